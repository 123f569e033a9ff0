// mamba_kernel.cu -- the Mamba-1 selective-scan decode step (mamba_selective_scan_decode).
//
// A diagonal recurrence: every (row, channel) owns an N-entry fp32 state row, updated
// element-wise and contracted with C into one output. LPR = NP / 8 lanes share a row (NP / 4 when
// N < 8), each holding eight (four) consecutive state entries as 16-byte accesses when N is a
// power of two, so a warp moves 32 / LPR consecutive rows, 1 KB of contiguous state; the output
// is a group sum over the LPR lanes. B and C rows are shared by every channel of a row (L1 hits), A rows by every row of
// a channel (L2 hits). Memory-bound: about 8 flops and an exp per 8 bytes of state.
//
// Source: "Triton decode kernel + MBU analysis", "Kernel design" (the math, fp32 accumulation and
// state); that page's kernel runs one program per (row, channel) with BLOCK_N = next_pow2(N).
#include <cmath>
#include <cstdint>

#include "gdn_chain.cuh"
#include "gdn_common.cuh"
#include "gdn_pipe.cuh"
#include "mamba_decode.h"

namespace gdn {

constexpr int kMambaThreads = 256;
constexpr int kMambaGsCtasPerSmBound = 5;   // resident CTAs of the grid-stride form (48 registers)

template <typename T> __device__ __forceinline__ float ld1(const void *p, size_t i)
{
    return to_f32(static_cast<const T *>(p)[i]);
}

// EPL state entries per lane (4, or 8 when N >= 8): fewer lanes per row means fewer repeated
// loads of the row's scalars and a shorter group sum. The state loads are issued first and the
// A, B, C rows read four entries at a time, so that the kernel fits 32 registers: eight CTAs
// (64 warps) per SM keep more state loads in flight. On GB300 this took B = 1024, D = 1536, N = 16
// from 38.4 to 36.0 us (48 registers, five CTAs per SM, with all rows loaded up front). The kernel
// waits for the previous kernel before it touches memory and is launched with the programmatic
// attribute, so consecutive small calls hide each other's launch (B = 4 / 16, N = 16: 2.14 / 2.51
// against 2.55 / 2.91 us).
template <int NP, typename Tin, bool VEC>
__global__ void __launch_bounds__(kMambaThreads, 7) mamba_decode_kernel(const __grid_constant__ mamba_decode_args P)
{
    constexpr int EPL = NP >= 8 ? 8 : 4;
    constexpr int LPR = NP / EPL;
    const int N = P.N, D = P.D;
    const long long rows = (long long)P.B * D;
    const long long tid = (long long)blockIdx.x * kMambaThreads + threadIdx.x;
    const long long r = tid / LPR;
    const int sub = (int)(tid % LPR);
    const bool live = r < rows;
    const int b = live ? (int)(r / D) : 0, d = live ? (int)(r - (long long)b * D) : 0;
    const int n0 = sub * EPL;
    ordinary_launch_start();
    // 16-byte accesses: entries 4 sub + VS q .. + 3 of the row (q < EPL / 4), so that each access
    // of a row's lanes covers 16 LPR contiguous bytes
    constexpr int VS = 4 * LPR;
    const int vc = 4 * sub;

    float hv[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) hv[j] = 0.f;
    const float *hp = P.h + (size_t)r * N + n0;
    const float x = live ? ld1<Tin>(P.x, (size_t)r) : 0.f;
    const float dt = live ? ld1<Tin>(P.dt, (size_t)r) : 0.f;
    float y = 0.f;
    if (live) {
        if (VEC) {
#pragma unroll
            for (int q = 0; q < EPL / 4; ++q) {
                const float4 h4 = ld_stream(P.h + (size_t)r * N + vc + VS * q);
                hv[4 * q] = h4.x; hv[4 * q + 1] = h4.y; hv[4 * q + 2] = h4.z; hv[4 * q + 3] = h4.w;
            }
            const float dtx = dt * x;
#pragma unroll
            for (int q = 0; q < EPL / 4; ++q) {
                const float4 a4 = *reinterpret_cast<const float4 *>(P.A + (size_t)d * N + vc + VS * q);
                const float4 b4 = load4(static_cast<const Tin *>(P.Bm) + (size_t)b * N + vc + VS * q);
                const float4 c4 = load4(static_cast<const Tin *>(P.Cm) + (size_t)b * N + vc + VS * q);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w},
                            cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float &h = hv[4 * q + j];
                    h = fmaf(__expf(dt * av[j]), h, dtx * bv[j]);
                    y = fmaf(cv[j], h, y);
                }
            }
        } else {
            const float dtx = dt * x;
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                if (n0 + j < N) {
                    const float a = P.A[(size_t)d * N + n0 + j];
                    hv[j] = fmaf(__expf(dt * a), hp[j], dtx * ld1<Tin>(P.Bm, (size_t)b * N + n0 + j));
                    y = fmaf(ld1<Tin>(P.Cm, (size_t)b * N + n0 + j), hv[j], y);
                }
            }
        }
    }
    y = group_sum<LPR>(y);   // every lane of the group takes part, live or not
    if (!live) return;
    float *op = (P.h_out ? P.h_out : P.h) + (size_t)r * N + n0;
    if (VEC) {
        float *ov = (P.h_out ? P.h_out : P.h) + (size_t)r * N + vc;
#pragma unroll
        for (int q = 0; q < EPL / 4; ++q)
            st_stream(ov + VS * q, make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]));
    } else {
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (n0 + j < N) op[j] = hv[j];
    }
    if (sub == 0) {
        if (P.Dskip) y = fmaf(P.Dskip[d], x, y);
        if (P.z) {
            const float z = ld1<Tin>(P.z, (size_t)r);
            y *= z * sigmoid_f(z);
        }
        if (P.out_dtype == GDN_BF16)
            static_cast<bf16 *>(P.y)[r] = __float2bfloat16_rn(y);
        else
            static_cast<float *>(P.y)[r] = y;
    }
}

// Grid-stride form for large batches at N = 32 .. 128 (powers of two): a grid of five CTAs per SM
// walks the rows, each thread issuing the next row's state loads before it computes the current
// row, so a lane keeps its state loads in flight across rows instead of ending its CTA after one
// row. At N = 64, B = 1024 the one-row-per-thread kernel kept every warp slot busy with HBM 60%
// busy (22 long-scoreboard stalls per issue); this form took 144.1 against 151.1 us (38.4 against
// 40.0 at B = 256). With only a few rows per thread it was slower (B = 16: 5.32 against 4.45 us),
// so it runs only when the rows fill the grid at least twice.
template <int NP, typename Tin>
__global__ void __launch_bounds__(kMambaThreads, kMambaGsCtasPerSmBound) mamba_gs_kernel(const __grid_constant__ mamba_decode_args P)
{
    constexpr int EPL = 8;
    constexpr int LPR = NP / EPL;
    const int N = P.N, D = P.D;
    const long long rows = (long long)P.B * D;
    const long long tid = (long long)blockIdx.x * kMambaThreads + threadIdx.x;
    const long long rstep = (long long)gridDim.x * kMambaThreads / LPR;
    const int sub = (int)(tid % LPR);
    // entries 4 sub .. 4 sub + 3 and HALF + 4 sub .. + 3 of a row: each access of a row's lanes
    // covers 16 LPR contiguous bytes
    constexpr int HALF = 4 * LPR;
    const int n0 = 4 * sub;
    long long r = tid / LPR;
    // the row's state and its per-row scalars (x, dt and, for the lane that writes y, z) are
    // loaded one row ahead, so that no load from HBM waits in the computing row's path
    float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
    float cx = 0.f, cdt = 0.f, cz = 0.f;
    if (r < rows) {
        c0 = ld_stream(P.h + (size_t)r * N + n0);
        c1 = ld_stream(P.h + (size_t)r * N + n0 + HALF);
        cx = ld1<Tin>(P.x, (size_t)r);
        cdt = ld1<Tin>(P.dt, (size_t)r);
        if (P.z && sub == 0) cz = ld1<Tin>(P.z, (size_t)r);
    }
    // every lane of the warp stays in the loop until none of its rows is left (the group sums
    // take all 32 lanes); lanes past the end compute on zeros and store nothing
    for (;; r += rstep) {
        const bool live = r < rows;
        if (!__any_sync(0xFFFFFFFFu, live)) break;
        const long long rn = r + rstep;
        float4 n0v = make_float4(0.f, 0.f, 0.f, 0.f), n1v = n0v;
        float nx = 0.f, ndt = 0.f, nz = 0.f;
        if (rn < rows) {
            n0v = ld_stream(P.h + (size_t)rn * N + n0);
            n1v = ld_stream(P.h + (size_t)rn * N + n0 + HALF);
            nx = ld1<Tin>(P.x, (size_t)rn);
            ndt = ld1<Tin>(P.dt, (size_t)rn);
            if (P.z && sub == 0) nz = ld1<Tin>(P.z, (size_t)rn);
        }
        const long long rr = live ? r : 0;
        const int b = (int)(rr / D), d = (int)(rr - (long long)b * D);
        const float x = cx, dt = cdt;
        const float dtx = dt * x;
        float hv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        float y = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 a4 = *reinterpret_cast<const float4 *>(P.A + (size_t)d * N + n0 + HALF * q);
            const float4 b4 = load4(static_cast<const Tin *>(P.Bm) + (size_t)b * N + n0 + HALF * q);
            const float4 c4 = load4(static_cast<const Tin *>(P.Cm) + (size_t)b * N + n0 + HALF * q);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w}, cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float &h = hv[4 * q + j];
                h = fmaf(__expf(dt * av[j]), h, dtx * bv[j]);
                y = fmaf(cv[j], h, y);
            }
        }
        y = group_sum<LPR>(y);
        if (live) {
            float *op = (P.h_out ? P.h_out : P.h) + (size_t)r * N + n0;
            st_stream(op, make_float4(hv[0], hv[1], hv[2], hv[3]));
            st_stream(op + HALF, make_float4(hv[4], hv[5], hv[6], hv[7]));
        }
        if (live && sub == 0) {
            if (P.Dskip) y = fmaf(P.Dskip[d], x, y);
            if (P.z) y *= cz * sigmoid_f(cz);
            if (P.out_dtype == GDN_BF16)
                static_cast<bf16 *>(P.y)[r] = __float2bfloat16_rn(y);
            else
                static_cast<float *>(P.y)[r] = y;
        }
        c0 = n0v;
        c1 = n1v;
        cx = nx;
        cdt = ndt;
        cz = nz;
    }
}

// Staged form for N = 16 .. 128 (powers of two) and large batches: one CTA per block of NB = 4 (or
// 2) batch rows b0 .. by RPP consecutive channels d0 .. (32 KB, or 16 KB, of state: NB contiguous
// runs of RPP state rows). Thread 0 bulk-copies the runs and the NB B and C rows (cp.async.bulk,
// completion on one mbarrier) into shared memory as the CTA starts; meanwhile every thread loads
// the eight A entries of its channel, which all NB batch rows share, and the x, dt and z scalars
// of its NB rows. The update then reads only shared memory and registers, one batch row per
// pass, and stores with streaming stores, so a CTA's shared memory is busy for the copy and a short
// arithmetic phase, not for round trips to L2 (NB = 4: 58 registers, four CTAs per SM, 128 KB of
// copies in flight per SM; NB = 2: 48 registers, five CTAs per SM). An earlier form, one block of consecutive rows per CTA with the A, B and C rows
// read from L2 during the update, was slower than the grid-stride form (158.7 against 142.0 us at
// B = 1024, N = 64), and bounding this one to five CTAs per SM (48 registers, a few spilled) lost
// 2-8%. The wait is bounded: on a timeout the CTA raises
// GDN_DEVERR_TIMEOUT in err_flags, thread 0 waits (bounded) for its copies, and the block's rows are
// left as they were.
constexpr long long kMambaWaitLimit = 1LL << 31;   // SM clock cycles, about one second

// NB batch rows per block (one per pass): 4 (32 KB of state) or 2 (16 KB)
template <int NP, int NB, typename Tin>
__global__ void __launch_bounds__(kMambaThreads) mamba_stage_kernel(const __grid_constant__ mamba_decode_args P)
{
    constexpr int EPL = 8;
    constexpr int LPR = NP / EPL;                    // lanes per state row
    constexpr int RPP = kMambaThreads / LPR;         // channels of a block
    static_assert(RPP * NP * 4 == 8192, "a batch row of a block is 8 KB of state");
    __shared__ __align__(128) float hs[NB * RPP * NP];
    __shared__ __align__(16) Tin bs[NB * NP];
    __shared__ __align__(16) Tin cs[NB * NP];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag, zero_flag;
    const int D = P.D;
    const int dblocks = (D + RPP - 1) / RPP;
    const int bblk = blockIdx.x / dblocks, dblk = blockIdx.x - bblk * dblocks;
    const int b0 = bblk * NB, d0 = dblk * RPP;
    const int nb = P.B - b0 < NB ? P.B - b0 : NB, nd = D - d0 < RPP ? D - d0 : RPP;
    // lane `sub` of a row holds the entries 4 sub .. 4 sub + 3 and 4 LPR + 4 sub .. + 3, so that
    // the LPR lanes of a row read and write 16 LPR contiguous bytes per access (no bank conflicts
    // in shared memory, whole sectors in global memory)
    const int sub = threadIdx.x % LPR, lrow = threadIdx.x / LPR;
    constexpr int HALF = 4 * LPR;
    const int n0 = 4 * sub;
    const bool dlive = lrow < nd;
    const int d = d0 + (dlive ? lrow : 0);

    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        zero_flag = 0;
        fence_barrier_init();
        const uint32_t run = (uint32_t)nd * NP * 4u, brow = (uint32_t)nb * NP * (uint32_t)sizeof(Tin);
        mbar_arrive_expect_tx(&bar, (uint32_t)nb * run + 2u * brow);
        const uint64_t pol = policy_evict_first();
        for (int p = 0; p < nb; ++p)
            bulk_g2s_hint(hs + p * RPP * NP, P.h + ((size_t)(b0 + p) * D + d0) * NP, run, &bar, pol);
        bulk_g2s(bs, static_cast<const Tin *>(P.Bm) + (size_t)b0 * NP, brow, &bar);
        bulk_g2s(cs, static_cast<const Tin *>(P.Cm) + (size_t)b0 * NP, brow, &bar);
    }
    // this channel's A entries and the scalars of its four rows, while the copies are in flight
    const float4 a_lo = *reinterpret_cast<const float4 *>(P.A + (size_t)d * NP + n0);
    const float4 a_hi = *reinterpret_cast<const float4 *>(P.A + (size_t)d * NP + n0 + HALF);
    const float av[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
    float xs[NB], dts[NB], zs[NB];
#pragma unroll
    for (int p = 0; p < NB; ++p) {
        const bool live = dlive && p < nb;
        const size_t r = (size_t)(b0 + p) * D + d;
        xs[p] = live ? ld1<Tin>(P.x, r) : 0.f;
        dts[p] = live ? ld1<Tin>(P.dt, r) : 0.f;
        zs[p] = live && P.z && sub == 0 ? ld1<Tin>(P.z, r) : 0.f;
    }
    __syncthreads();   // the barrier is initialised before anyone waits on it
    if (!mbar_wait_warp(&bar, 0u, &abort_flag, kMambaWaitLimit)) {
        if ((threadIdx.x & 31) == 0) raise_flag(P.err_flags, GDN_DEVERR_TIMEOUT);
        if (threadIdx.x == 0) mbar_wait(&bar, 0u, &zero_flag, kMambaWaitLimit);   // the copies land first
        return;
    }
    float *out = P.h_out ? P.h_out : P.h;
#pragma unroll
    for (int p = 0; p < NB; ++p) {
        const bool live = dlive && p < nb;   // rows past the edges: computed on zeros, never stored
        const int hrow = p * RPP + lrow;
        const float x = xs[p], dt = dts[p], dtx = dt * x;
        float hv[8];
        float y = 0.f;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            // rows past the edges of a ragged block were not copied: they compute on zeros
            const float4 h4 = live ? *reinterpret_cast<const float4 *>(hs + hrow * NP + n0 + HALF * q) : z4;
            const float4 b4 = live ? load4(bs + p * NP + n0 + HALF * q) : z4;
            const float4 c4 = live ? load4(cs + p * NP + n0 + HALF * q) : z4;
            const float hq[4] = {h4.x, h4.y, h4.z, h4.w}, bq[4] = {b4.x, b4.y, b4.z, b4.w}, cq[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                hv[4 * q + j] = fmaf(__expf(dt * av[4 * q + j]), hq[j], dtx * bq[j]);
                y = fmaf(cq[j], hv[4 * q + j], y);
            }
        }
        y = group_sum<LPR>(y);
        if (!live) continue;
        const size_t r = (size_t)(b0 + p) * D + d;
        float *op = out + r * NP + n0;
        st_stream(op, make_float4(hv[0], hv[1], hv[2], hv[3]));
        st_stream(op + HALF, make_float4(hv[4], hv[5], hv[6], hv[7]));
        if (sub == 0) {
            if (P.Dskip) y = fmaf(P.Dskip[d], x, y);
            if (P.z) y *= zs[p] * sigmoid_f(zs[p]);
            if (P.out_dtype == GDN_BF16)
                static_cast<bf16 *>(P.y)[r] = __float2bfloat16_rn(y);
            else
                static_cast<float *>(P.y)[r] = y;
        }
    }
}

template <int NP, typename Tin>
static int launch_mamba_np(const mamba_decode_args &p, cudaStream_t s)
{
    const long long threads = (long long)p.B * p.D * (NP / (NP >= 8 ? 8 : 4));
    const unsigned blocks = (unsigned)((threads + kMambaThreads - 1) / kMambaThreads);
    if constexpr (NP >= 16) {
        if (p.N == NP) {
            int dev = 0, sms = 0;
            if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return GDN_ERR_LAUNCH;
            // The staged form (B and C rows 16-byte aligned for their bulk copies): 32 KB blocks
            // from six waves of them, 16 KB blocks from two waves. On GB300 at D = 1536: B = 1024,
            // N = 64 118.6 us with 32 KB blocks against 120.9 with 16 KB and 142.1 for the
            // grid-stride form; N = 128 233.2 against 241.3 and 288.9; B = 256, N = 16 10.40 with
            // 16 KB blocks against 10.69 for the per-row kernel; B = 512, N = 16 17.95 against
            // 18.40 with 32 KB blocks; B = 256, N = 64 32.59 against 32.82.
            constexpr int rpp = kMambaThreads / (NP / 8);
            const long long dblocks = (p.D + rpp - 1) / rpp;
            const long long sb4 = dblocks * ((p.B + 3) / 4), sb2 = dblocks * ((p.B + 1) / 2);
            const bool al16 = (reinterpret_cast<uintptr_t>(p.Bm) & 15u) == 0 && (reinterpret_cast<uintptr_t>(p.Cm) & 15u) == 0;
            if (al16 && sb4 >= 24LL * sms) {
                mamba_stage_kernel<NP, 4, Tin><<<(unsigned)sb4, kMambaThreads, 0, s>>>(p);
                return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
            }
            if (al16 && sb2 >= 8LL * sms) {
                mamba_stage_kernel<NP, 2, Tin><<<(unsigned)sb2, kMambaThreads, 0, s>>>(p);
                return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
            }
            const unsigned cap = (unsigned)sms * kMambaGsCtasPerSmBound;
            if (NP >= 32 && blocks >= 2u * cap) {
                mamba_gs_kernel<NP, Tin><<<cap, kMambaThreads, 0, s>>>(p);
                return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
            }
        }
    }
    if (p.N == NP)
        launch_ordinary(mamba_decode_kernel<NP, Tin, true>, dim3(blocks), dim3(kMambaThreads), 0, s, p);
    else
        launch_ordinary(mamba_decode_kernel<NP, Tin, false>, dim3(blocks), dim3(kMambaThreads), 0, s, p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

template <typename Tin>
static int launch_mamba_t(const mamba_decode_args &p, cudaStream_t s)
{
    if (p.N <= 4) return launch_mamba_np<4, Tin>(p, s);
    if (p.N <= 8) return launch_mamba_np<8, Tin>(p, s);
    if (p.N <= 16) return launch_mamba_np<16, Tin>(p, s);
    if (p.N <= 32) return launch_mamba_np<32, Tin>(p, s);
    if (p.N <= 64) return launch_mamba_np<64, Tin>(p, s);
    return launch_mamba_np<128, Tin>(p, s);
}

}  // namespace gdn

namespace {
bool al(const void *p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }
}

extern "C" int mamba_selective_scan_decode(const mamba_decode_args *a, gdn_stream_t stream)
{
    if (!a) return GDN_ERR_NULL;
    if (a->B < 0 || a->D < 0 || a->N < 1 || a->N > 128) return GDN_ERR_SHAPE;
    if ((long long)a->B * a->D * 32 > 0x7FFFFFFFLL * 256) return GDN_ERR_SHAPE;
    if ((a->in_dtype != GDN_F32 && a->in_dtype != GDN_BF16) || (a->out_dtype != GDN_F32 && a->out_dtype != GDN_BF16))
        return GDN_ERR_DTYPE;
    if (a->B == 0 || a->D == 0) return GDN_OK;
    if (!a->x || !a->dt || !a->A || !a->Bm || !a->Cm || !a->h || !a->y) return GDN_ERR_NULL;
    const size_t es = a->in_dtype == GDN_BF16 ? 2 : 4;
    if (!al(a->x, es) || !al(a->dt, es) || !al(a->Bm, es) || !al(a->Cm, es) || (a->z && !al(a->z, es)) ||
        !al(a->h, 4) || !al(a->A, 4) || (a->h_out && !al(a->h_out, 4)) || (a->Dskip && !al(a->Dskip, 4)) ||
        !al(a->y, a->out_dtype == GDN_BF16 ? 2 : 4))
        return GDN_ERR_ALIGN;
    const bool pow2 = a->N == 4 || a->N == 8 || a->N == 16 || a->N == 32 || a->N == 64 || a->N == 128;
    if (pow2 && (!al(a->h, 16) || !al(a->A, 16) || (a->h_out && !al(a->h_out, 16)) || !al(a->Bm, 4 * es) ||
                 !al(a->Cm, 4 * es)))
        return GDN_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return a->in_dtype == GDN_BF16 ? gdn::launch_mamba_t<gdn::bf16>(*a, s) : gdn::launch_mamba_t<float>(*a, s);
}
