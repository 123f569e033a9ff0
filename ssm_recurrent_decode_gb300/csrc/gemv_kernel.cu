// gemv_kernel.cu -- the decode projection y = x W^T (gdn_gemv_bf16).
//
// A weight-streaming, HBM-bound matrix-vector product for a handful of token rows: each warp owns
// kRows = 4 output rows and walks its K range 256 inputs at a time, every lane loading 16 bytes
// (8 bf16) of each row and of each token row of x, so one x load feeds 4 rows of W (x comes from
// L1/L2: it is small and shared by every warp). Up to 8 token rows are handled per pass; their
// 4 x 8 partial sums are reduced with a butterfly reduce-scatter (31 shuffles, one result per
// lane). Split-K: blockIdx.y selects a K range whose partial sums go to the workspace, and a
// second small kernel adds the ranges in order (deterministic). No tensor cores: at decode batch
// sizes the weights' bytes, not the flops, set the time.
//
// Source: "Optimization Log: Qwen3.5-27B Dense on B200", Kernel 3 (BF16 GEMV with split-K).
#include <cstdint>

#include "gdn_common.cuh"
#include "gdn_gemv.h"

namespace gdn {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kRows = 4;          // output rows per warp
constexpr int kTok = 8;           // token rows per pass

__device__ __forceinline__ void unpack8(uint4 raw, float (&f)[8])
{
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Sum over the 32 lanes of each of the 32 values; lane l ends with the sum of value l.
__device__ __forceinline__ float reduce_scatter32(float (&x)[32], int lane)
{
#pragma unroll
    for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
            const float send = upper ? x[j] : x[j + n / 2];
            const float keep = upper ? x[j + n / 2] : x[j];
            x[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
    }
    return x[0];
}

// One pass over up to kTok token rows (t0 .. t0 + nt - 1) and one K range.
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const __grid_constant__ gdn_gemv_args P, int t0,
                                                            int nt, int k_per_split)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n0 = (blockIdx.x * kGemvWarps + warp) * kRows;
    if (n0 >= P.N) return;   // whole warps only: no shuffle below is left half-joined
    const int split = blockIdx.y;
    const int k_begin = split * k_per_split;
    const int k_end = min(P.Kd, k_begin + k_per_split);
    const bf16 *W = static_cast<const bf16 *>(P.W);
    const bf16 *X = static_cast<const bf16 *>(P.x);

    float acc[kRows][kTok];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < kTok; ++t) acc[r][t] = 0.f;

    for (int k = k_begin + lane * 8; k < k_end; k += 256) {
        float wf[kRows][8];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int n = n0 + r;
            if (n < P.N) {
                unpack8(__ldcs(reinterpret_cast<const uint4 *>(W + (size_t)n * P.Kd + k)), wf[r]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) wf[r][i] = 0.f;
            }
        }
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
            if (t < nt) {
                float xf[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(X + (size_t)(t0 + t) * P.x_stride + k)), xf);
#pragma unroll
                for (int r = 0; r < kRows; ++r)
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[r][t] = fmaf(wf[r][i], xf[i], acc[r][t]);
            }
        }
    }
    float v[32];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < kTok; ++t) v[r * kTok + t] = acc[r][t];
    const float sum = reduce_scatter32(v, lane);
    const int r = lane / kTok, t = lane - r * kTok, n = n0 + r;
    if (t >= nt || n >= P.N) return;
    if (gridDim.y > 1) {
        P.workspace[((size_t)split * P.T + t0 + t) * P.N + n] = sum;
    } else if (P.out_dtype == GDN_BF16) {
        static_cast<bf16 *>(P.y)[(size_t)(t0 + t) * P.y_stride + n] = __float2bfloat16_rn(sum);
    } else {
        static_cast<float *>(P.y)[(size_t)(t0 + t) * P.y_stride + n] = sum;
    }
}

// y[t, n] = sum over the splits, in order
__global__ void gemv_reduce_kernel(const __grid_constant__ gdn_gemv_args P, int splits)
{
    const long long total = (long long)P.T * P.N;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int j = 0; j < splits; ++j) s += P.workspace[(size_t)j * total + i];
        const int t = (int)(i / P.N), n = (int)(i - (long long)t * P.N);
        if (P.out_dtype == GDN_BF16)
            static_cast<bf16 *>(P.y)[(size_t)t * P.y_stride + n] = __float2bfloat16_rn(s);
        else
            static_cast<float *>(P.y)[(size_t)t * P.y_stride + n] = s;
    }
}

static int sm_count_gemv()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 152;
    return sms;
}

int gemv_launch(const gdn_gemv_args &p, int splits, cudaStream_t stream)
{
    const int ctas_n = (p.N + kGemvWarps * kRows - 1) / (kGemvWarps * kRows);
    // K ranges in whole 256-input steps
    const int steps = (p.Kd + 255) / 256;
    const int k_per_split = ((steps + splits - 1) / splits) * 256;
    const dim3 grid((unsigned)ctas_n, (unsigned)splits);
    for (int t0 = 0; t0 < p.T; t0 += kTok) {
        const int nt = p.T - t0 < kTok ? p.T - t0 : kTok;
        gemv_kernel<<<grid, kGemvThreads, 0, stream>>>(p, t0, nt, k_per_split);
    }
    if (splits > 1) {
        const long long total = (long long)p.T * p.N;
        long long blocks = (total + 255) / 256;
        if (blocks > 4 * 152) blocks = 4 * 152;
        gemv_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, splits);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

int gemv_default_splits(int N, int Kd)
{
    const int ctas_n = (N + kGemvWarps * kRows - 1) / (kGemvWarps * kRows);
    const int target = 4 * sm_count_gemv();
    int s = 1;
    while (s < 16 && ctas_n * s < target && Kd / (s * 2) >= 256) s *= 2;
    return s;
}

}  // namespace gdn

namespace {
bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}

extern "C" {

int32_t gdn_gemv_default_splits(int32_t T, int32_t N, int32_t Kd)
{
    (void)T;
    if (N < 1 || Kd < 1) return 1;
    return gdn::gemv_default_splits(N, Kd);
}

size_t gdn_gemv_workspace_bytes(int32_t T, int32_t N, int32_t splits)
{
    if (splits <= 1 || T < 0 || N < 0) return 0;
    return sizeof(float) * (size_t)splits * (size_t)T * (size_t)N;
}

int gdn_gemv_bf16(const gdn_gemv_args *a, gdn_stream_t stream)
{
    if (!a) return GDN_ERR_NULL;
    if (a->T < 0 || a->N < 0 || a->Kd < 0 || a->Kd % 8 != 0 || a->splits < 0 || a->splits > 64) return GDN_ERR_SHAPE;
    if (a->out_dtype != GDN_F32 && a->out_dtype != GDN_BF16) return GDN_ERR_DTYPE;
    if (a->T == 0 || a->N == 0) return GDN_OK;
    if (!a->x || !a->W || !a->y) return GDN_ERR_NULL;
    if (a->x_stride < a->Kd || a->x_stride % 8 != 0 || a->y_stride < a->N) return GDN_ERR_SHAPE;
    if (!al16(a->x) || !al16(a->W) || (reinterpret_cast<uintptr_t>(a->y) % (a->out_dtype == GDN_BF16 ? 2 : 4)) != 0)
        return GDN_ERR_ALIGN;
    const int splits = a->splits > 0 ? a->splits : (a->Kd == 0 ? 1 : gdn::gemv_default_splits(a->N, a->Kd));
    if (splits > 1) {
        if (!a->workspace) return GDN_ERR_NULL;
        if (a->workspace_bytes < gdn_gemv_workspace_bytes(a->T, a->N, splits)) return GDN_ERR_SHAPE;
        if ((reinterpret_cast<uintptr_t>(a->workspace) & 3u) != 0) return GDN_ERR_ALIGN;
    }
    return gdn::gemv_launch(*a, splits, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
