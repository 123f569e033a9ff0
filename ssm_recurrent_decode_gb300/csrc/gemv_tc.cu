// gemv_tc.cu -- tcgen05 form of the decode projection y = x W^T (gdn_gemv_bf16) for passes of up
// to 16 token rows.
//
// One CTA owns 128 output rows (the MMA's M) and one K range. The range streams through a ring of
// shared-memory stages (kTcStages x kTcChunks tiles, see gemv_internal.h), each tile filled by two
// TMA copies (cp.async.bulk.tensor, 128-byte swizzle): 128 weight rows x 64 inputs (16 KB) and 16
// token rows x 64 inputs of x (2 KB; rows past T and inputs past Kd are zero-filled by the copy).
// The tiles of a stage are adjacent in K, so a stage reads 256 contiguous bytes of every weight
// row. One thread issues tcgen05.mma (kind::f16: bf16 operands, fp32 accumulation; M = 128,
// N = 16, K = 16, four per tile) into one of two 128-lane x 16-column fp32 accumulators in tensor
// memory, one buffer per 128 inputs; tcgen05.commit returns a stage to the producer once the MMAs
// reading it are done and hands a finished group to the epilogue. Four epilogue warps read each
// group's sum (tcgen05.ld, one output row per thread, 16 token columns), add it to fp32 registers
// while the next group accumulates in the other buffer, and finally write y or the partial sums.
// Adding the groups with round-to-nearest fp32 adds keeps a long K range as accurate as a plain
// fp32 sum; a single tensor-memory accumulation over 2560 inputs measured 2.1e-5 relative error.
//
// Roles: warp 0 allocates the tensor memory and runs the TMA producer on one lane, warp 1 issues
// the MMAs on one lane, warps 2 .. 5 (one per quarter of the tensor-memory lanes) are the epilogue.
// Every mbarrier wait is bounded. A wait that gives up raises GDN_DEVERR_TIMEOUT and a CTA-wide
// abort flag; the producer then waits (bounded) for its copies in flight, the MMA thread waits
// (bounded) for the MMAs it issued, the CTA frees its tensor memory and writes no output (with a
// workspace, it writes NaN into its partial-sum slots, so that the sums added later are NaN).
//
// Source: "Optimization Log: Qwen3.5-27B Dense on B200", Kernel 3 (BF16 GEMV with split-K).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "gdn_chain.cuh"
#include "gdn_cluster.cuh"
#include "gdn_common.cuh"
#include "gdn_gemv.h"
#include "gdn_pipe.cuh"
#include "gemv_internal.h"

namespace gdn {

constexpr int kTcEpiThreads = 128;                         // warps 2 .. 5
constexpr int kTcThreads = 64 + kTcEpiThreads;              // producer warp, MMA warp, epilogue
constexpr int kTcGroupStages = kTcChunks >= 2 ? 1 : 2;      // stages summed per accumulator buffer
constexpr uint32_t kTcABytes = kTcRows * kTcK * 2;          // weight tile, 16 KB
constexpr uint32_t kTcBBytes = kTcTok * kTcK * 2;           // token tile, 2 KB
constexpr uint32_t kTcStageBytes = kTcChunks * (kTcABytes + kTcBBytes);   // a multiple of 1024
constexpr uint32_t kTcTmemCols = 32;                        // two 16-column accumulators
constexpr long long kTcWaitLimit = 1LL << 31;               // SM clock cycles, about one second
// The limit of the waits that can give up (0: kTcWaitLimit); set only by the test hook below. The
// waits for copies and MMAs still in flight after a give-up always use kTcWaitLimit.
std::atomic<long long> g_wait_limit{0};

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9
// and 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTcTok >> 3) << 17) |
                              ((uint32_t)(kTcRows >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile as TMA writes it with the 128-byte swizzle:
// 128-byte rows, 8-row groups 1024 bytes apart (stride byte offset), start address in 16-byte
// units (bits 0-13), leading byte offset 16 (unused by swizzled K-major tiles), descriptor version
// 1 (bits 46-47), swizzle mode 128-byte (2, bits 61-63). The tile base is 1024-byte aligned, so
// stepping K by 16 elements is a 32-byte step of the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_tile_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// asks L2 to fetch a tile (no shared-memory destination, no completion to wait for)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int c0, int c1)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void tma_tile_2d_hint(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tensor memory) += A (shared, via descriptor) * B^T (shared, via descriptor); D is overwritten
// when accumulate == 0
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kTcIdesc), "r"(accumulate)
        : "memory");
}

// arrive once on `bar` when every tcgen05.mma this thread issued before has completed
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 16 columns of 32 bits: thread i of the warp gets lane (taddr.lane + i), columns
// taddr.col .. taddr.col + 15
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kTcThreads) gemv_tc_kernel(const __grid_constant__ gdn_gemv_args P,
                                                             const __grid_constant__ CUtensorMap wmap,
                                                             const __grid_constant__ CUtensorMap xmap, int t0, int nt,
                                                             int k_per_split, int stages, int mode,
                                                             int prefetch_w, long long wait_limit)
{
    extern __shared__ unsigned char tc_sm[];
    __shared__ __align__(8) uint64_t full[kTcMaxStages];    // stage filled (TMA bytes landed)
    __shared__ __align__(8) uint64_t empty[kTcMaxStages];   // stage read by its MMAs
    __shared__ __align__(8) uint64_t acc_full[2];           // accumulator buffer holds a group's sum
    __shared__ __align__(8) uint64_t acc_empty[2];          // accumulator buffer drained to registers
    __shared__ __align__(8) uint64_t done;                  // every MMA of the CTA completed
    __shared__ uint32_t tmem_holder;
    __shared__ int abort_flag, zero_flag;

    const uint32_t sbase = (smem_u32(tc_sm) + 1023u) & ~1023u;   // swizzled tiles need 1024-byte alignment
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.y;
    const int n0 = blockIdx.x * kTcRows;
    const int k_begin = split * k_per_split;
    const int k_end = min(P.Kd, k_begin + k_per_split);
    const int nk = k_end > k_begin ? (k_end - k_begin + kTcStageK - 1) / kTcStageK : 0;
    const int ngroups = (nk + kTcGroupStages - 1) / kTcGroupStages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kTcEpiThreads);
        }
        mbar_init(&done, 1);
        abort_flag = 0;
        zero_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        // 32 columns of tensor memory (128 lanes x 32 bit each): two 128 x 16 accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_holder)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    grid_launch_dependents();
    if (prefetch_w && threadIdx.x == 0) {
        // A chained launch may start while the previous kernel still runs: bring this CTA's weight
        // tiles (the same tiles the producer copies below) into L2 in the meantime.
        for (int it = 0; it < nk; ++it)
#pragma unroll
            for (int c = 0; c < kTcChunks; ++c) tma_prefetch_2d(&wmap, k_begin + it * kTcStageK + c * kTcK, n0);
    }
    grid_dependency_wait();   // in a chained layer call x is the previous kernel's output
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            const uint64_t pol = policy_evict_first();
            int it = 0;
            for (; it < nk; ++it) {
                const int s = it % stages;
                const uint32_t ph = (uint32_t)(it / stages) & 1u;
                if (it >= stages && !mbar_wait(&empty[s], ph ^ 1u, &abort_flag, wait_limit)) {
                    *(volatile int *)&abort_flag = 1;
                    raise_flag(P.err_flags, GDN_DEVERR_TIMEOUT);
                    break;
                }
                const uint32_t a = sbase + (uint32_t)s * kTcStageBytes;
                mbar_arrive_expect_tx(&full[s], kTcStageBytes);
#pragma unroll
                for (int c = 0; c < kTcChunks; ++c) {   // adjacent 64-input tiles of the same rows
                    const int k = k_begin + it * kTcStageK + c * kTcK;
                    tma_tile_2d_hint(a + c * kTcABytes, &wmap, k, n0, &full[s], pol);
                    tma_tile_2d(a + kTcChunks * kTcABytes + c * kTcBBytes, &xmap, k, t0, &full[s]);
                }
            }
            if (*(volatile int *)&abort_flag) {
                // let the copies of the stages still in flight land before the CTA exits
                for (int back = 1; back <= stages && it - back >= 0; ++back) {
                    const int m = it - back;
                    mbar_wait(&full[m % stages], (uint32_t)(m / stages) & 1u, &zero_flag, kTcWaitLimit);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            // Group g (kTcGroupStages stages, 128 inputs) accumulates in buffer g & 1, starting
            // from zero; its second use waits until the epilogue has drained the first.
            bool ok = true;
            for (int g = 0; g < ngroups && ok; ++g) {
                const int buf = g & 1;
                if (g >= 2 && !mbar_wait(&acc_empty[buf], (uint32_t)((g >> 1) - 1) & 1u, &abort_flag, wait_limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * kTcTok);
                const int it_end = min(nk, (g + 1) * kTcGroupStages);
                for (int it = g * kTcGroupStages; it < it_end; ++it) {
                    const int s = it % stages;
                    const uint32_t ph = (uint32_t)(it / stages) & 1u;
                    if (!mbar_wait(&full[s], ph, &abort_flag, wait_limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sbase + (uint32_t)s * kTcStageBytes, b0 = a0 + kTcChunks * kTcABytes;
                    const bool first = it == g * kTcGroupStages;
#pragma unroll
                    for (int c = 0; c < kTcChunks; ++c) {
                        const uint32_t a = a0 + c * kTcABytes, b = b0 + c * kTcBBytes;
#pragma unroll
                        for (int j = 0; j < kTcK / 16; ++j)
                            tc_mma(d, sw128_desc(a + 32u * j), sw128_desc(b + 32u * j),
                                   (first && c == 0 && j == 0) ? 0u : 1u);
                    }
                    tc_commit(&empty[s]);
                }
                if (ok) tc_commit(&acc_full[buf]);
            }
            if (!ok) {
                *(volatile int *)&abort_flag = 1;
                raise_flag(P.err_flags, GDN_DEVERR_TIMEOUT);
            }
            // every MMA issued above completes before the tensor memory is freed
            tc_commit(&done);
            mbar_wait(&done, 0u, &zero_flag, kTcWaitLimit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps 2 .. 5
        // Warp w reads tensor-memory lanes 32 (w % 4) .. 32 (w % 4) + 31: one output row per
        // thread, the 16 token columns of a group's sum, added to fp32 registers (round to
        // nearest), so a long K range accumulates as a plain fp32 sum does.
        const int quad = warp & 3;
        float acc[kTcTok];
#pragma unroll
        for (int i = 0; i < kTcTok; ++i) acc[i] = 0.f;
        bool ok = true;
        for (int g = 0; g < ngroups; ++g) {
            const int buf = g & 1;
            if (!mbar_wait(&acc_full[buf], (uint32_t)(g >> 1) & 1u, &abort_flag, wait_limit)) ok = false;
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[kTcTok];
            tc_ld16(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(buf * kTcTok), v);
#pragma unroll
            for (int i = 0; i < kTcTok; ++i) acc[i] += v[i];
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
        }
        if (!ok && lane == 0) {
            *(volatile int *)&abort_flag = 1;
            raise_flag(P.err_flags, GDN_DEVERR_TIMEOUT);
        }
        const int n = n0 + 32 * quad + lane;
        if (ok && mode == kGemvReduceCluster) {
            // this range's sums go to shared memory (the drained stage ring), token-major, for the
            // cluster reduction below
            float *red = reinterpret_cast<float *>(tc_sm + (sbase - smem_u32(tc_sm)));
#pragma unroll
            for (int t = 0; t < kTcTok; ++t) red[t * kTcRows + 32 * quad + lane] = acc[t];
        } else if (ok && n < P.N) {
#pragma unroll
            for (int t = 0; t < kTcTok; ++t) {
                if (t >= nt) break;
                if (mode == kGemvReduceWorkspace) {
                    const size_t wi = ((size_t)split * P.T + t0 + t) * P.N + n;
                    if (gemv_ws_in_range(P, (long long)wi)) P.workspace[wi] = acc[t];   // (range: debug build)
                } else {
                    gemv_store(P, t0 + t, n, acc[t]);
                }
            }
        } else if (!ok && mode == kGemvReduceWorkspace && n < P.N) {
            // The reduction kernel adds every range's slot; a range that gave up leaves NaN there
            // (not the buffer's previous contents), so the affected outputs of y come out NaN.
            for (int t = 0; t < nt; ++t) {
                const size_t wi = ((size_t)split * P.T + t0 + t) * P.N + n;
                if (gemv_ws_in_range(P, (long long)wi)) P.workspace[wi] = __int_as_float(0x7fc00000);
            }
        }
    }
    if (mode == kGemvReduceCluster) {
        // The K ranges of this row tile are the CTAs of one cluster (rank = range). CTA r adds the
        // ranges' sums of its share of the 16 x 128 outputs in range order, reading the other
        // CTAs' shared memory, and writes y; a CTA that gave up a wait makes the cluster skip.
        __syncwarp();
        cluster_sync_all();
        const uint32_t rank = cluster_ctarank();
        const int nr = (int)gridDim.y;
        int bad = 0;
        for (int q = 0; q < nr; ++q) bad |= cluster_ld_s32(cluster_map(smem_u32(&abort_flag), (uint32_t)q));
        if (!bad) {
            const int total = nt * kTcRows, chunk = (total + nr - 1) / nr;
            const int e_end = min(total, ((int)rank + 1) * chunk);
            for (int e = (int)rank * chunk + threadIdx.x; e < e_end; e += kTcThreads) {
                float sum = 0.f;
                for (int q = 0; q < nr; ++q) sum += cluster_ld_f32(cluster_map(sbase + 4u * (uint32_t)e, (uint32_t)q));
                const int t = e / kTcRows, n = n0 + (e - t * kTcRows);
                if (n < P.N) gemv_store(P, t0 + t, n, sum);
            }
        }
        cluster_sync_all();   // no CTA leaves while another still reads its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols) : "memory");
    }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::mutex lock;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::lock_guard<std::mutex> g(lock);
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// bf16 matrix [rows, cols] with a row pitch of `pitch` elements, tiles of box_rows x 64 columns
bool encode_bf16_tiles(CUtensorMap *map, const void *base, int rows, int cols, int64_t pitch, int box_rows)
{
    const auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;

// the dynamic shared-memory limit is raised once per device (a function attribute)
bool prepare_device(size_t smem)
{
    static std::mutex lock;
    static size_t raised[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> g(lock);
    if (raised[dev] < smem) {
        if (cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return false;
        raised[dev] = smem;
    }
    return true;
}

}  // namespace

size_t gemv_tc_smem_bytes(int stages) { return (size_t)stages * kTcStageBytes + 1024; }

// Resident CTAs per SM, from the shared-memory bound (each CTA holds its stages plus 1 KB of
// alignment slack, 1 KB is reserved per CTA; registers and threads allow more). The occupancy
// query reported one CTA per SM for this kernel on GB300, while timings over split counts follow
// the shared-memory bound (three CTAs at two stages of two tiles).
int gemv_tc_resident_ctas(int stages)
{
    static std::mutex lock;
    static int smem_sm[kMaxDevices];   // 0 = not asked yet
    const size_t smem = gemv_tc_smem_bytes(stages) + 256 + 1024;   // + static shared, + reserved
    int dev = 0, per_sm = 228 * 1024;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> g(lock);
        if (!smem_sm[dev]) {
            int v = 0;
            if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || v <= 0) {
                cudaGetLastError();
                v = 228 * 1024;
            }
            smem_sm[dev] = v;
        }
        per_sm = smem_sm[dev];
    } else {
        cudaGetLastError();
    }
    const int n = (int)(per_sm / smem);
    return n < 1 ? 1 : n;
}

int gemv_tc_launch(const gdn_gemv_args &p, int splits, int k_per_split, int stages, cudaStream_t stream,
                   bool chained)
{
    if (stages < 2 || stages > kTcMaxStages || k_per_split % kTcStageK != 0) return GDN_ERR_ARG;
    CUtensorMap wmap, xmap;
    if (!encode_bf16_tiles(&wmap, p.W, p.N, p.Kd, p.Kd, kTcRows) ||
        !encode_bf16_tiles(&xmap, p.x, p.T, p.Kd, p.x_stride, kTcTok))
        return GDN_ERR_LAUNCH;
    const size_t smem = gemv_tc_smem_bytes(stages);
    if (!prepare_device(smem)) return GDN_ERR_LAUNCH;
    const int mode = gemv_reduce_mode(splits);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3((unsigned)((p.N + kTcRows - 1) / kTcRows), (unsigned)splits);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    if (mode == kGemvReduceCluster) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;   // the K ranges of a row tile
        attr[cfg.numAttrs].val.clusterDim.x = 1;
        attr[cfg.numAttrs].val.clusterDim.y = (unsigned)splits;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (chained) set_programmatic(attr[cfg.numAttrs++]);
    const int prefetch_w = chained && gemv_prefetch_fits(p) ? 1 : 0;
    const long long limit_set = g_wait_limit.load(std::memory_order_relaxed);
    const long long wait_limit = limit_set > 0 ? limit_set : kTcWaitLimit;
    for (int t0 = 0; t0 < p.T; t0 += kTcTok) {
        const int nt = p.T - t0 < kTcTok ? p.T - t0 : kTcTok;
        if (cudaLaunchKernelEx(&cfg, gemv_tc_kernel, p, wmap, xmap, t0, nt, k_per_split, stages, mode,
                               prefetch_w, wait_limit) != cudaSuccess)
            return GDN_ERR_LAUNCH;
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

}  // namespace gdn

extern "C" int64_t gdn_gemv_set_wait_limit(int64_t cycles)
{
    return gdn::g_wait_limit.exchange(cycles > 0 ? cycles : 0);
}
