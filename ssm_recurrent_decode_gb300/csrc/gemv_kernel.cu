// gemv_kernel.cu -- the decode projection y = x W^T (gdn_gemv_bf16).
//
// A weight-streaming, HBM-bound product of a handful of token rows with a bf16 weight matrix, in
// two forms:
//  - one token row: CUDA cores. Each warp owns 4 output rows and walks its K range 512 inputs at a
//    time, every lane loading 16 bytes (8 bf16) of each row for two 256-input steps before using
//    them; one x value feeds 4 rows.
//  - two or more token rows: tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate), weight
//    rows as the M operand and groups of 8 token rows as N, loaded straight from global memory into
//    the operand registers; the tensor core sums 128-input groups and the groups are added in fp32
//    registers. At 8 token rows a CUDA-core form needs about 4 FMAs per weight byte, close to the
//    SM's FMA rate at HBM speed; the tensor core takes that work off the FMA pipe.
// In both, the token rows' slice of x is staged in shared memory (cp.async) when it fits.
// Split-K: blockIdx.y selects a K range whose partial sums go to the workspace, and a second small
// kernel adds the ranges in order (deterministic).
//
// Source: "Optimization Log: Qwen3.5-27B Dense on B200", Kernel 3 (BF16 GEMV with split-K).
#include <cstdint>
#include <mutex>

#include "gdn_common.cuh"
#include "gdn_gemv.h"

namespace gdn {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kRows = 4;          // output rows per warp (CUDA-core form)
// Largest staged x slice per CTA. Larger slices were slower than reading x through L1 on GB300:
// with 35 KB or more per CTA the shared-memory carve-out leaves too little L1 for the weight loads
// in flight.
constexpr size_t kStageMaxBytes = 24 * 1024;

__device__ __forceinline__ void unpack8(uint4 raw, float (&f)[8])
{
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// 16-byte asynchronous copy global -> shared (no register round trip; all of a thread's copies are
// in flight together until cp_async_wait_all)
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

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

// CUDA-core form: up to TOK token rows (t0 .. t0 + nt - 1; TOK = 1 is the instance in use) and one
// K range. The rows' slice of x is staged in shared memory when it fits (xs_elems > 0), otherwise
// read through L1. Each lane issues the weight loads of two 256-input steps before using them
// (8 x 16 bytes in flight per lane, 4 KB per warp); the 4 x TOK sums are reduced with a butterfly
// reduce-scatter. On GB300 this form (64 registers, four CTAs per SM) measured faster at one token
// row than a leaner single-row variant (44 registers, five CTAs per SM): 27.3 against 31.1 us for
// W [17408, 5120].
template <int TOK>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const __grid_constant__ gdn_gemv_args P, int t0,
                                                            int nt, int k_per_split, int xs_elems)
{
    extern __shared__ __align__(16) unsigned char gemv_sm[];
    bf16 *xs = reinterpret_cast<bf16 *>(gemv_sm);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int split = blockIdx.y;
    const int k_begin = split * k_per_split;
    const int k_end = min(P.Kd, k_begin + k_per_split);
    const int krange = max(0, k_end - k_begin);
    const bf16 *W = static_cast<const bf16 *>(P.W);
    const bf16 *X = static_cast<const bf16 *>(P.x);
    const bool staged = xs_elems > 0;
    if (staged) {
        const int per_row = krange / 8;
        for (int e = threadIdx.x; e < nt * per_row; e += kGemvThreads) {
            const int t = e / per_row, c = e - t * per_row;
            cp_async16(reinterpret_cast<uint4 *>(xs) + (size_t)t * per_row + c, X + (size_t)(t0 + t) * P.x_stride + k_begin + 8 * c);
        }
        cp_async_wait_all();
        __syncthreads();
    }
    const int n0 = (blockIdx.x * kGemvWarps + warp) * kRows;
    if (n0 >= P.N) return;
    float acc[kRows][TOK];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < TOK; ++t) acc[r][t] = 0.f;
    auto x_at = [&](int t, int k) -> uint4 {
        return staged ? reinterpret_cast<const uint4 *>(xs)[((size_t)t * krange + (k - k_begin)) / 8]
                      : __ldg(reinterpret_cast<const uint4 *>(X + (size_t)(t0 + t) * P.x_stride + k));
    };
    auto fma_step = [&](const uint4 (&wr)[kRows], int k) {
        float wf[kRows][8];
#pragma unroll
        for (int r = 0; r < kRows; ++r) unpack8(wr[r], wf[r]);
#pragma unroll
        for (int t = 0; t < TOK; ++t) {
            if (t < nt) {
                float xf[8];
                unpack8(x_at(t, k), xf);
#pragma unroll
                for (int r = 0; r < kRows; ++r)
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[r][t] = fmaf(wf[r][i], xf[i], acc[r][t]);
            }
        }
    };
    auto load_rows = [&](int k, uint4 (&wr)[kRows]) {
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            wr[r] = (n0 + r < P.N && k < k_end) ? __ldcs(reinterpret_cast<const uint4 *>(W + (size_t)(n0 + r) * P.Kd + k))
                                                : make_uint4(0u, 0u, 0u, 0u);
    };
    for (int k = k_begin + lane * 8; k < k_end; k += 512) {
        uint4 wa[kRows], wb[kRows];
        load_rows(k, wa);
        load_rows(k + 256, wb);
        fma_step(wa, k);
        if (k + 256 < k_end) fma_step(wb, k + 256);
    }
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < TOK; ++t) v[r * TOK + t] = acc[r][t];
    const float sum = reduce_scatter32(v, lane);
    if (lane >= kRows * TOK) return;
    const int r = lane / TOK, t = lane - r * TOK, n = n0 + r;
    if (t >= nt || n >= P.N) return;
    if (gridDim.y > 1) {
        P.workspace[((size_t)split * P.T + t0 + t) * P.N + n] = sum;
    } else if (P.out_dtype == GDN_BF16) {
        static_cast<bf16 *>(P.y)[(size_t)(t0 + t) * P.y_stride + n] = __float2bfloat16_rn(sum);
    } else {
        static_cast<float *>(P.y)[(size_t)(t0 + t) * P.y_stride + n] = sum;
    }
}

// Tensor-core form for passes of 2 or more token rows: one warp owns kMmaRows = 16 output rows and
// runs mma.sync m16n8k16 (bf16 in, fp32 accumulate) with the weight rows as the M operand and up
// to 8 token rows per group as the N operand. The k order inside a 32-input block is permuted the
// same way for both operands (a sum over k does not depend on its order), so that every lane's
// operands are one 16-byte load: lane (g, q) loads inputs 8q .. 8q + 7 of rows g and g + 8 and of
// token row g; its first mma takes the low 8 bytes of each load, its second the high 8 bytes. The
// weights go from global memory to registers with no shared-memory round trip; kMmaUnroll blocks
// of loads are in flight per lane.
constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kMmaRows = 16;
constexpr int kMmaUnroll = 4;
constexpr int kMmaKStep = 32 * kMmaUnroll;
constexpr int kMmaMaxGroups = 2;  // groups of 8 token rows per pass
// Token rows from which the tensor-core form runs. At one token row the CUDA-core form was as fast
// or faster on GB300 (28.2 vs 32.2 us for W [17408, 5120], 30.0 vs 30.3 us for W [5120, 17408]).
constexpr int kMmaMinTokens = 2;

__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One pass over up to 8G token rows (t0 .. t0 + nt - 1) and one K range. xs_stride > 0: the x slice
// is staged in shared memory, xs_stride uint4 per token row (padded so that the two token rows a
// quarter-warp reads fall in different banks).
template <int G>
__global__ void __launch_bounds__(kMmaThreads) gemv_mma_kernel(const __grid_constant__ gdn_gemv_args P, int t0,
                                                               int nt, int k_per_split, int xs_stride)
{
    extern __shared__ __align__(16) unsigned char gemv_sm[];
    uint4 *xs = reinterpret_cast<uint4 *>(gemv_sm);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int split = blockIdx.y;
    const int k_begin = split * k_per_split;
    const int k_end = min(P.Kd, k_begin + k_per_split);
    const int krange = max(0, k_end - k_begin);
    const bf16 *X = static_cast<const bf16 *>(P.x);
    const bool staged = xs_stride > 0;
    if (staged) {
        const int per_row = krange / 8;
        for (int e = threadIdx.x; e < nt * per_row; e += kMmaThreads) {
            const int t = e / per_row, c = e - t * per_row;
            cp_async16(xs + t * xs_stride + c, X + (size_t)(t0 + t) * P.x_stride + k_begin + 8 * c);
        }
    }
    const int n0 = (blockIdx.x * kMmaWarps + warp) * kMmaRows;
    const int ra = n0 + g, rb = n0 + g + 8;
    const bool va = ra < P.N, vb = rb < P.N;
    const uint4 *Wa = reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(P.W) + (size_t)(va ? ra : 0) * P.Kd);
    const uint4 *Wb = reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(P.W) + (size_t)(vb ? rb : 0) * P.Kd);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint4 wa[kMmaUnroll], wb[kMmaUnroll];
    auto load_w = [&](int kb) {
#pragma unroll
        for (int u = 0; u < kMmaUnroll; ++u) {
            const int k = kb + 32 * u + 8 * q;
            const bool in = k < k_end;
            wa[u] = (va && in) ? __ldcs(Wa + k / 8) : zero;
            wb[u] = (vb && in) ? __ldcs(Wb + k / 8) : zero;
        }
    };
    load_w(k_begin);   // the first group's weights are in flight while x lands in shared memory
    if (staged) {
        cp_async_wait_all();
        __syncthreads();
    }
    if (n0 >= P.N) return;   // whole warps only, after the CTA-wide barrier

    float acc[G][4];
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;

    for (int kb = k_begin; kb < k_end; kb += kMmaKStep) {
        if (kb != k_begin) load_w(kb);
        // the tensor core sums one 128-input group; the groups are added in fp32 registers with
        // round-to-nearest, so a long K range accumulates as a plain fp32 sum does
        float part[G][4];
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[j][e] = 0.f;
#pragma unroll
        for (int u = 0; u < kMmaUnroll; ++u) {
            const int k = kb + 32 * u + 8 * q;
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const int t = 8 * j + g;
                uint4 xv = zero;
                if (t < nt && k < k_end)
                    xv = staged ? xs[t * xs_stride + (k - k_begin) / 8]
                                : __ldg(reinterpret_cast<const uint4 *>(X + (size_t)(t0 + t) * P.x_stride + k));
                mma_16816_bf16(part[j], wa[u].x, wb[u].x, wa[u].y, wb[u].y, xv.x, xv.y);
                mma_16816_bf16(part[j], wa[u].z, wb[u].z, wa[u].w, wb[u].w, xv.z, xv.w);
            }
        }
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] += part[j][e];
    }
    // accumulator fragment: acc[j][0..1] row g, tokens 8j + 2q + {0, 1}; acc[j][2..3] row g + 8
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = e < 2 ? ra : rb;
            const int t = 8 * j + 2 * q + (e & 1);
            if (t >= nt || n >= P.N) continue;
            if (gridDim.y > 1) {
                P.workspace[((size_t)split * P.T + t0 + t) * P.N + n] = acc[j][e];
            } else if (P.out_dtype == GDN_BF16) {
                static_cast<bf16 *>(P.y)[(size_t)(t0 + t) * P.y_stride + n] = __float2bfloat16_rn(acc[j][e]);
            } else {
                static_cast<float *>(P.y)[(size_t)(t0 + t) * P.y_stride + n] = acc[j][e];
            }
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

// The layout of one call: which form runs, its grid, its K ranges and its staged x slice.
struct GemvPlan {
    bool mma;            // tensor-core form (T >= kMmaMinTokens) or CUDA-core form (one token row)
    int per_pass;        // token rows per pass over W
    int ctas_n;          // CTAs along N
    int k_per_split;     // inputs per K range (a whole number of the form's steps)
    int krange;          // inputs in the widest range
};

static GemvPlan make_plan(int T, int N, int Kd, int splits)
{
    GemvPlan pl;
    pl.mma = T >= kMmaMinTokens;
    pl.per_pass = pl.mma ? 8 * kMmaMaxGroups : 1;
    const int rows = pl.mma ? kMmaWarps * kMmaRows : kGemvWarps * kRows;
    pl.ctas_n = (N + rows - 1) / rows;
    const int gran = pl.mma ? kMmaKStep : 256;
    const int chunks = (Kd + gran - 1) / gran;
    pl.k_per_split = ((chunks + splits - 1) / splits) * gran;
    pl.krange = pl.k_per_split < Kd ? pl.k_per_split : Kd;
    return pl;
}

// Shared-memory bytes of a pass's staged x slice (0: it is too large and x is read through L1)
// and the kernel's staging argument (tensor-core form: row stride in uint4, padded to 64 bytes past
// a 128-byte boundary; CUDA-core form: elements).
static size_t stage_bytes(const GemvPlan &pl, int nt, int *arg)
{
    size_t bytes;
    int a;
    if (pl.mma) {
        a = ((pl.krange / 8 + 7) / 8) * 8 + 4;
        bytes = (size_t)nt * a * 16;
    } else {
        a = nt * pl.krange;
        bytes = (size_t)a * 2;
    }
    if (bytes > kStageMaxBytes) bytes = 0, a = 0;
    if (arg) *arg = a;
    return bytes;
}

int gemv_launch(const gdn_gemv_args &p, int splits, cudaStream_t stream)
{
    const GemvPlan pl = make_plan(p.T, p.N, p.Kd, splits);
    const dim3 grid((unsigned)pl.ctas_n, (unsigned)splits);
    for (int t0 = 0; t0 < p.T; t0 += pl.per_pass) {
        const int nt = p.T - t0 < pl.per_pass ? p.T - t0 : pl.per_pass;
        int xs = 0;
        const size_t smem = stage_bytes(pl, nt, &xs);
        if (!pl.mma)
            gemv_kernel<1><<<grid, kGemvThreads, smem, stream>>>(p, t0, 1, pl.k_per_split, xs);
        else if (nt <= 8)
            gemv_mma_kernel<1><<<grid, kMmaThreads, smem, stream>>>(p, t0, nt, pl.k_per_split, xs);
        else
            gemv_mma_kernel<2><<<grid, kMmaThreads, smem, stream>>>(p, t0, nt, pl.k_per_split, xs);
    }
    if (splits > 1) {
        const long long total = (long long)p.T * p.N;
        long long blocks = (total + 255) / 256;
        if (blocks > 4 * 152) blocks = 4 * 152;
        gemv_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, splits);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

// CTAs of the form that runs T token rows that fit on one SM with `smem` bytes of dynamic shared
// memory each (registers, threads and shared memory; the occupancy query is made once per device
// and form; without a device, the counts of the sm_103a build: 4 CUDA-core, 4 and 3 tensor-core
// CTAs for one and two token groups).
static int resident_ctas(bool mma, int groups, size_t smem)
{
    constexpr int kMaxDevices = 64;
    static std::mutex lock;
    static int occ[kMaxDevices][3];        // [device][CUDA-core, mma G=1, mma G=2], 0 = not asked
    static int smem_sm[kMaxDevices];
    int dev = 0, n = 0;
    const int which = mma ? groups : 0;
    static const int fallback[3] = {4, 4, 3};
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        n = fallback[which];
        if (smem > 0 && (int)(228 * 1024 / (smem + 1024)) < n) n = (int)(228 * 1024 / (smem + 1024));
        return n < 1 ? 1 : n;
    }
    {
        std::lock_guard<std::mutex> g(lock);
        if (!occ[dev][which]) {
            cudaError_t rc;
            if (which == 0) rc = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<1>, kGemvThreads, 0);
            else if (which == 1) rc = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_mma_kernel<1>, kMmaThreads, 0);
            else rc = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_mma_kernel<2>, kMmaThreads, 0);
            if (rc != cudaSuccess || n < 1) { cudaGetLastError(); n = fallback[which]; }
            occ[dev][which] = n;
            int sm = 0;
            if (cudaDeviceGetAttribute(&sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || sm <= 0) {
                cudaGetLastError();
                sm = 228 * 1024;
            }
            smem_sm[dev] = sm;
        }
        n = occ[dev][which];
        if (smem > 0) {
            const int by_smem = (int)(smem_sm[dev] / (smem + 1024));   // 1 KB reserved per CTA
            if (by_smem < n) n = by_smem;
        }
    }
    return n < 1 ? 1 : n;
}

// The split count for splits == 0, from measurements on GB300 at the decode shapes. Candidates are
// powers of two up to 64 with at least 512 inputs per range whose x slice fits the staging budget;
// the largest whose grid fits in one wave of resident CTAs wins (more CTAs per SM keep more weight
// loads in flight); failing that, the smallest that fills at least two waves (a grid of about 1.2
// waves leaves a tail of a few CTAs per SM and was the slowest choice).
int gemv_default_splits(int T, int N, int Kd)
{
    const long long sms = sm_count_gemv();
    int one_wave = 0, two_waves = 0, last_staged = 0, last = 1;
    for (int s = 1; s <= 64; s *= 2) {
        if (s > 1 && Kd / s < 512) break;
        last = s;
        const GemvPlan pl = make_plan(T, N, Kd, s);
        const int nt = T < pl.per_pass ? T : pl.per_pass;
        const size_t smem = stage_bytes(pl, nt, nullptr);
        if (smem == 0) continue;
        last_staged = s;
        const long long slots = resident_ctas(pl.mma, (nt + 7) / 8, smem) * sms;
        const long long ctas = (long long)pl.ctas_n * s;
        if (ctas <= slots) one_wave = s;
        else if (ctas >= 2 * slots && !two_waves) two_waves = s;
    }
    if (one_wave) return one_wave;
    if (two_waves) return two_waves;
    return last_staged ? last_staged : last;
}

}  // namespace gdn

namespace {
bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}

extern "C" {

int32_t gdn_gemv_default_splits(int32_t T, int32_t N, int32_t Kd)
{
    if (N < 1 || Kd < 1) return 1;
    return gdn::gemv_default_splits(T < 1 ? 1 : T, N, Kd);
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
    const int splits = a->splits > 0 ? a->splits : (a->Kd == 0 ? 1 : gdn::gemv_default_splits(a->T, a->N, a->Kd));
    if (splits > 1) {
        if (!a->workspace) return GDN_ERR_NULL;
        if (a->workspace_bytes < gdn_gemv_workspace_bytes(a->T, a->N, splits)) return GDN_ERR_SHAPE;
        if ((reinterpret_cast<uintptr_t>(a->workspace) & 3u) != 0) return GDN_ERR_ALIGN;
    }
    return gdn::gemv_launch(*a, splits, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
