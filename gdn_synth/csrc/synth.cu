// synth.cu -- on-device twin of the seeded synthetic-input generator in gdn_synth/__init__.py.
//
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC 2011) keyed by (seed) with counter (element index lo, hi, step, stream = tag | layer << 16),
// and the same Irwin-Hall normal: four 22-bit uniforms summed, centred at 2^23, converted to fp32
// exactly and multiplied once by the caller's fp32 scale constant. Integer arithmetic and one
// correctly rounded multiply, so the values are bit-identical to the host generator's. This
// library holds no arithmetic of the decode method; it only fills buffers.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace {

struct Philox {
    uint32_t c0, c1, c2, c3;
};

__device__ __forceinline__ Philox philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1)
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += W0;
            k1 += W1;
        }
        const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
        const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return {c0, c1, c2, c3};
}

__device__ __forceinline__ float normal_at(uint64_t idx, uint64_t seed, uint32_t step,
                                           uint32_t stream, float c)
{
    const Philox r = philox4x32_10((uint32_t)idx, (uint32_t)(idx >> 32), step, stream,
                                   (uint32_t)seed, (uint32_t)(seed >> 32));
    const int32_t s = (int32_t)((r.c0 >> 10) + (r.c1 >> 10) + (r.c2 >> 10) + (r.c3 >> 10)) - (1 << 23);
    return __fmul_rn((float)s, c);
}

template <bool BF16>
__global__ void fill_kernel(void *out, int64_t n, uint64_t seed, uint32_t stream_id,
                            uint32_t step, const int32_t *step_ptr, int64_t start, float c)
{
    const uint32_t st = step_ptr ? (uint32_t)(step + *step_ptr) : step;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float x = normal_at((uint64_t)(start + i), seed, st, stream_id, c);
        if (BF16)
            static_cast<__nv_bfloat16 *>(out)[i] = __float2bfloat16_rn(x);
        else
            static_cast<float *>(out)[i] = x;
    }
}

__global__ void add_kernel(int32_t *p, int32_t d) { *p += d; }

}  // namespace

extern "C" {

// Fill out[0..n) with the normals of tensor elements start .. start+n-1 of stream
// (tag | layer << 16), at `step` (plus *step_ptr when step_ptr is not NULL: lets a captured CUDA
// graph draw fresh values on every replay). c is the fp32 scale constant std*sqrt(3)/2^22.
// bf16 != 0 stores bf16 (round to nearest even), else fp32. Returns 0 or a cudaError_t value.
int synth_fill_normal(void *out, int64_t n, uint64_t seed, uint32_t tag, uint32_t layer,
                      uint32_t step, const int32_t *step_ptr, int64_t start, float c, int bf16,
                      cudaStream_t stream)
{
    if (n <= 0) return 0;
    const uint32_t stream_id = (tag & 0xFFFFu) | ((layer & 0xFFFFu) << 16);
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 152 * 64) blocks = 152 * 64;
    if (bf16)
        fill_kernel<true><<<(unsigned)blocks, threads, 0, stream>>>(out, n, seed, stream_id, step, step_ptr, start, c);
    else
        fill_kernel<false><<<(unsigned)blocks, threads, 0, stream>>>(out, n, seed, stream_id, step, step_ptr, start, c);
    return (int)cudaGetLastError();
}

// *p += d on the device (advances a graph's step counter).
int synth_add_i32(int32_t *p, int32_t d, cudaStream_t stream)
{
    add_kernel<<<1, 1, 0, stream>>>(p, d);
    return (int)cudaGetLastError();
}

}  // extern "C"
