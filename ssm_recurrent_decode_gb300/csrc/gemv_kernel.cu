// gemv_kernel.cu -- the decode projection y = x W^T (gdn_gemv_bf16).
//
// A weight-streaming, HBM-bound product of a handful of token rows with a bf16 weight matrix, in
// two forms:
//  - one token row: CUDA cores (this file). Each warp owns 4 output rows and walks its K range 512
//    inputs at a time, every lane loading 16 bytes (8 bf16) of each row for two 256-input steps
//    before using them; one x value feeds 4 rows. The row's slice of x is staged in shared memory
//    (cp.async) when it fits.
//  - two or more token rows: tcgen05 tensor cores with TMA-staged tiles (gemv_tc.cu). At 8 token
//    rows a CUDA-core form needs about 4 FMAs per weight byte, close to the SM's FMA rate at HBM
//    speed; the tensor core takes that work off the FMA pipe.
// Split-K: blockIdx.y selects a K range. Up to 8 ranges of a row block are one thread-block cluster
// and add their sums, in range order, through distributed shared memory; more ranges leave partial
// sums in the workspace and a second small kernel adds them in order (deterministic either way).
//
// Source: "Optimization Log: Qwen3.5-27B Dense on B200", Kernel 3 (BF16 GEMV with split-K).
#include <cstdint>
#include <mutex>

#include "gdn_chain.cuh"
#include "gdn_cluster.cuh"
#include "gdn_common.cuh"
#include "gdn_pipe.cuh"
#include "gdn_gemv.h"
#include "gemv_internal.h"

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
// reduce-scatter. On GB300 this form (56 registers, four CTAs per SM) measured faster at one token
// row than a leaner single-row variant (44 registers, five CTAs per SM): 27.3 against 31.1 us for
// W [17408, 5120].
template <int TOK>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const __grid_constant__ gdn_gemv_args P, int t0,
                                                            int nt, int k_per_split, int xs_elems, int mode,
                                                            int prefetch_w)
{
    extern __shared__ __align__(16) unsigned char gemv_sm[];
    __shared__ float red[kGemvWarps * kRows * TOK];   // this K range's sums, cluster mode
    bf16 *xs = reinterpret_cast<bf16 *>(gemv_sm);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int split = blockIdx.y;
    const int k_begin = split * k_per_split;
    const int k_end = min(P.Kd, k_begin + k_per_split);
    const int krange = max(0, k_end - k_begin);
    const bf16 *W = static_cast<const bf16 *>(P.W);
    const bf16 *X = static_cast<const bf16 *>(P.x);
    const bool staged = xs_elems > 0;
    const int n0 = (blockIdx.x * kGemvWarps + warp) * kRows;
    grid_launch_dependents();
    if (prefetch_w) {
        // A chained launch may start while the previous kernel still runs: bring this warp's
        // weight rows into L2 in the meantime, one 128-byte line per lane and prefetch.
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            if (n0 + r < P.N)
                for (int k = k_begin + lane * 64; k < k_end; k += 32 * 64)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(W + (size_t)(n0 + r) * P.Kd + k));
    }
    grid_dependency_wait();   // in a chained layer call x is the previous kernel's output
    if (staged) {
        const int per_row = krange / 8;
        for (int e = threadIdx.x; e < nt * per_row; e += kGemvThreads) {
            const int t = e / per_row, c = e - t * per_row;
            cp_async16(reinterpret_cast<uint4 *>(xs) + (size_t)t * per_row + c, X + (size_t)(t0 + t) * P.x_stride + k_begin + 8 * c);
        }
        cp_async_wait_all();
        __syncthreads();
    }
    float sum = 0.f;
    if (n0 < P.N) {   // whole warps
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
        sum = reduce_scatter32(v, lane);
    }
    // lane r * TOK + t holds (row n0 + r, token t0 + t)
    if (mode == kGemvReduceCluster) {
        // The K ranges of this row block are the CTAs of one cluster (rank = range). CTA r adds the
        // ranges' sums of its share of the block's outputs in range order, reading the other
        // CTAs' shared memory, and writes y.
        constexpr int kEntries = kGemvWarps * kRows * TOK;
        if (lane < kRows * TOK) red[warp * kRows * TOK + lane] = sum;
        __syncwarp();
        cluster_sync_all();
        const int rank = (int)cluster_ctarank(), nr = (int)gridDim.y;
        const int chunk = (kEntries + nr - 1) / nr;
        const int e = rank * chunk + threadIdx.x;
        if (threadIdx.x < chunk && e < kEntries) {
            float total = 0.f;
            for (int q = 0; q < nr; ++q) total += cluster_ld_f32(cluster_map(smem_u32(&red[e]), (uint32_t)q));
            const int t = e % TOK, n = blockIdx.x * kGemvWarps * kRows + e / TOK;
            if (t < nt && n < P.N) gemv_store(P, t0 + t, n, total);
        }
        cluster_sync_all();   // no CTA leaves while another still reads its shared memory
        return;
    }
    if (lane >= kRows * TOK || n0 >= P.N) return;
    const int r = lane / TOK, t = lane - r * TOK, n = n0 + r;
    if (t >= nt || n >= P.N) return;
    if (mode == kGemvReduceWorkspace) {
        const size_t wi = ((size_t)split * P.T + t0 + t) * P.N + n;
        if (gemv_ws_in_range(P, (long long)wi)) P.workspace[wi] = sum;   // (range: debug build)
    } else {
        gemv_store(P, t0 + t, n, sum);
    }
}

// y[t, n] = sum over the splits, in order
__global__ void gemv_reduce_kernel(const __grid_constant__ gdn_gemv_args P, int splits)
{
    const long long total = (long long)P.T * P.N;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int j = 0; j < splits; ++j)
            if (gemv_ws_in_range(P, (long long)j * total + i)) s += P.workspace[(size_t)j * total + i];
        const int t = (int)(i / P.N), n = (int)(i - (long long)t * P.N);
        gemv_store(P, t, n, s);
    }
}

static int sm_count_gemv()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 152;
    return sms;
}

// The form that runs T token rows: CUDA cores for one, tcgen05 (gemv_tc.cu) from two. At one token
// row the CUDA-core form was as fast or faster on GB300 (a tensor-core form measured 32.2 against
// 28.2 us for W [17408, 5120]).
constexpr int kTcMinTokens = 2;
enum class Form { kCore, kTc };
constexpr int kTcStages = 2;   // shared-memory stages of the tcgen05 form (36 KB each)

static Form form_for(int T) { return T < kTcMinTokens ? Form::kCore : Form::kTc; }

// The layout of one call: which form runs, its grid, its K ranges and its staged x slice.
struct GemvPlan {
    Form form;
    int per_pass;        // token rows per pass over W
    int ctas_n;          // CTAs along N
    int k_per_split;     // inputs per K range (a whole number of the form's steps)
    int krange;          // inputs in the widest range
};

static GemvPlan make_plan(int T, int N, int Kd, int splits)
{
    GemvPlan pl;
    pl.form = form_for(T);
    int rows, gran;
    if (pl.form == Form::kCore) pl.per_pass = 1, rows = kGemvWarps * kRows, gran = 256;
    else pl.per_pass = kTcTok, rows = kTcRows, gran = kTcStageK;
    pl.ctas_n = (N + rows - 1) / rows;
    const int chunks = (Kd + gran - 1) / gran;
    pl.k_per_split = ((chunks + splits - 1) / splits) * gran;
    pl.krange = pl.k_per_split < Kd ? pl.k_per_split : Kd;
    return pl;
}

// Dynamic shared memory of a pass. CUDA-core form: its staged x slice (0 when the slice is too
// large and x is read through L1), with the kernel's staging argument (elements). The tcgen05 form
// stages x with its weight tiles.
static size_t stage_bytes(const GemvPlan &pl, int nt, int *arg)
{
    if (arg) *arg = 0;
    if (pl.form == Form::kTc) return gemv_tc_smem_bytes(kTcStages);
    const int a = nt * pl.krange;
    const size_t bytes = (size_t)a * 2;
    if (bytes > kStageMaxBytes) return 0;
    if (arg) *arg = a;
    return bytes;
}

int gemv_launch(const gdn_gemv_args &p, int splits, cudaStream_t stream, bool chained)
{
    const GemvPlan pl = make_plan(p.T, p.N, p.Kd, splits);
    const int mode = gemv_reduce_mode(splits);
    if (pl.form == Form::kTc) {
        const int rc = gemv_tc_launch(p, splits, pl.k_per_split, kTcStages, stream, chained);
        if (rc != GDN_OK) return rc;
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        cfg.gridDim = dim3((unsigned)pl.ctas_n, (unsigned)splits);
        cfg.blockDim = dim3(kGemvThreads);
        cfg.stream = stream;
        cfg.attrs = attr;
        if (mode == kGemvReduceCluster) {
            attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;   // the K ranges of a row block
            attr[cfg.numAttrs].val.clusterDim.x = 1;
            attr[cfg.numAttrs].val.clusterDim.y = (unsigned)splits;
            attr[cfg.numAttrs].val.clusterDim.z = 1;
            ++cfg.numAttrs;
        }
        if (chained) set_programmatic(attr[cfg.numAttrs++]);
        const int prefetch_w = chained && gemv_prefetch_fits(p) ? 1 : 0;
        for (int t0 = 0; t0 < p.T; ++t0) {
            int xs = 0;
            cfg.dynamicSmemBytes = stage_bytes(pl, 1, &xs);
            if (cudaLaunchKernelEx(&cfg, gemv_kernel<1>, p, t0, 1, pl.k_per_split, xs, mode, prefetch_w) != cudaSuccess)
                return GDN_ERR_LAUNCH;
        }
    }
    if (mode == kGemvReduceWorkspace) {
        const long long total = (long long)p.T * p.N;
        long long blocks = (total + 255) / 256;
        if (blocks > 4 * 152) blocks = 4 * 152;
        gemv_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, splits);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

// CTAs of the form that runs T token rows that fit on one SM with `smem` bytes of dynamic shared
// memory each. CUDA-core form: the occupancy query (registers, threads, shared memory), made once
// per device; without a device, the count of the sm_103a build (4). tcgen05 form: its
// shared-memory bound (gemv_tc.cu).
static int resident_ctas(Form form, size_t smem)
{
    if (form == Form::kTc) return gemv_tc_resident_ctas(kTcStages);
    constexpr int kMaxDevices = 64;
    constexpr int kFallback = 4;
    static std::mutex lock;
    static int occ[kMaxDevices];        // 0 = not asked yet
    static int smem_sm[kMaxDevices];
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        n = kFallback;
        if (smem > 0 && (int)(228 * 1024 / (smem + 1024)) < n) n = (int)(228 * 1024 / (smem + 1024));
        return n < 1 ? 1 : n;
    }
    std::lock_guard<std::mutex> g(lock);
    if (!occ[dev]) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<1>, kGemvThreads, 0) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = kFallback;
        }
        occ[dev] = n;
        int sm = 0;
        if (cudaDeviceGetAttribute(&sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || sm <= 0) {
            cudaGetLastError();
            sm = 228 * 1024;
        }
        smem_sm[dev] = sm;
    }
    n = occ[dev];
    if (smem > 0) {
        const int by_smem = (int)(smem_sm[dev] / (smem + 1024));   // 1 KB reserved per CTA
        if (by_smem < n) n = by_smem;
    }
    return n < 1 ? 1 : n;
}

// The split count for splits == 0, from measurements on GB300 at the decode shapes. Candidates are
// powers of two up to the cluster size (so that no workspace is needed) with at least 512 inputs per range whose x slice fits the staging budget;
// the largest whose grid fits in one wave of resident CTAs wins (more CTAs per SM keep more weight
// loads in flight); failing that, the smallest that fills at least two waves (a grid of about 1.2
// waves leaves a tail of a few CTAs per SM and was the slowest choice).
int gemv_default_splits(int T, int N, int Kd)
{
    const long long sms = sm_count_gemv();
    int one_wave = 0, two_waves = 0, last_staged = 0, last = 1;
    for (int s = 1; s <= kGemvMaxCluster; s *= 2) {
        if (s > 1 && Kd / s < 512) break;
        last = s;
        const GemvPlan pl = make_plan(T, N, Kd, s);
        const int nt = T < pl.per_pass ? T : pl.per_pass;
        const size_t smem = stage_bytes(pl, nt, nullptr);
        if (smem == 0) continue;
        last_staged = s;
        const long long slots = resident_ctas(pl.form, smem) * sms;
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

namespace gdn {

// The host checks of gdn_gemv_bf16 (its status codes) and the split count it uses; *splits = 0
// when there is nothing to launch. No CUDA launch.
int gemv_check(const gdn_gemv_args *a, int *splits)
{
    *splits = 0;
    if (!a) return GDN_ERR_NULL;
    if (a->T < 0 || a->N < 0 || a->Kd < 0 || a->Kd % 8 != 0 || a->splits < 0 || a->splits > 64) return GDN_ERR_SHAPE;
    if (a->out_dtype != GDN_F32 && a->out_dtype != GDN_BF16) return GDN_ERR_DTYPE;
    if (a->T == 0 || a->N == 0) return GDN_OK;
    if (!a->x || !a->W || !a->y) return GDN_ERR_NULL;
    if (a->x_stride < a->Kd || a->x_stride % 8 != 0 || a->y_stride < a->N) return GDN_ERR_SHAPE;
    if (!al16(a->x) || !al16(a->W) || (reinterpret_cast<uintptr_t>(a->y) % (a->out_dtype == GDN_BF16 ? 2 : 4)) != 0)
        return GDN_ERR_ALIGN;
    const int s = a->splits > 0 ? a->splits : (a->Kd == 0 ? 1 : gemv_default_splits(a->T, a->N, a->Kd));
    if (gemv_reduce_mode(s) == kGemvReduceWorkspace) {
        if (!a->workspace) return GDN_ERR_NULL;
        if (a->workspace_bytes < gdn_gemv_workspace_bytes(a->T, a->N, s)) return GDN_ERR_SHAPE;
        if ((reinterpret_cast<uintptr_t>(a->workspace) & 3u) != 0) return GDN_ERR_ALIGN;
    }
    *splits = s;
    return GDN_OK;
}

}  // namespace gdn

extern "C" {

int32_t gdn_gemv_default_splits(int32_t T, int32_t N, int32_t Kd)
{
    if (N < 1 || Kd < 1) return 1;
    return gdn::gemv_default_splits(T < 1 ? 1 : T, N, Kd);
}

size_t gdn_gemv_workspace_bytes(int32_t T, int32_t N, int32_t splits)
{
    if (gdn::gemv_reduce_mode(splits) != gdn::kGemvReduceWorkspace || T < 0 || N < 0) return 0;
    return sizeof(float) * (size_t)splits * (size_t)T * (size_t)N;
}

int gdn_gemv_bf16(const gdn_gemv_args *a, gdn_stream_t stream)
{
    int splits = 0;
    const int rc = gdn::gemv_check(a, &splits);
    if (rc != GDN_OK || splits == 0) return rc;
    return gdn::gemv_launch(*a, splits, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
