// buffered_pipe.cu -- the buffered, output-only decode as a persistent, warp-specialised kernel
// for K = V = 128 (the shapes of every workload on the source pages).
//
// Same arithmetic as buffered_kernel.cu (low-rank replay of the ring records; the flush step at
// write_pos == L-1 folds them into the checkpoint and writes it back), organised so that HBM
// streams continuously:
//   - one CTA per SM: two groups of 8 consumer warps that take alternate tiles, and 1 producer warp;
//   - the producer walks the CTA's tiles ahead of the consumers and, for each, moves the 64 KB
//     checkpoint tile, the q/k/v rows and the tile's ring records (p delta rows, p key rows) into
//     a shared-memory stage with 1-D bulk copies (cp.async.bulk) that complete on the stage's
//     "full" mbarrier, and writes the tile's scalars (slot, cursor, gate inputs, the records'
//     log-decays) beside them;
//   - NST stages (2 or 3, as many as fit) keep up to NST tiles in flight per SM while the
//     consumers compute, so the tile loads of the next tiles overlap the current tile's
//     arithmetic and write-back;
//   - consumers take both dot products straight from the staged tile (16 rows x 4 columns per
//     lane); a flush step re-reads it eight rows at a time, folds the records in and writes the
//     new checkpoint with streaming stores; then the stage is released on its "empty" mbarrier.
// Every wait is bounded: a wait that runs past its limit sets GDN_DEVERR_TIMEOUT, raises a
// CTA-wide abort flag and ends the CTA's loop; the producer then waits (bounded) for the copies
// it issued, so no copy is in flight when the CTA exits.
//
// Source: "Microbenchmark: buffered output-only GDN decode (ReplaySSM Part A)" (module docstring,
// _bench_cfg / run_replay); the step of "Optimization Log: Qwen3.5-27B Dense on B200", Kernel 4.
#include "gdn_launch.h"
#include "gdn_pipe.cuh"
#include "gdn_tile.cuh"

namespace gdn {

constexpr int kPipeGW = 8;                            // warps of one consumer group
constexpr int kPipeGroups = 2;                        // consumer groups, alternating tiles
constexpr int kPipeCW = kPipeGW * kPipeGroups;        // consumer warps
constexpr int kPipeThreads = (kPipeCW + 1) * 32;      // plus one producer warp
constexpr int kPipeLMax = 64;
constexpr long long kWaitLimit = 1LL << 31;           // SM clock cycles, about one second

// Per-stage scalars. gr is filled by a bulk copy of the tile's log-decay records (first, so that
// it is 16-byte aligned); status .. beta by the producer; c, alpha, gamma are consumer scratch.
struct PipeMeta {
    float gr[kPipeLMax];        // log-decays of records j < p
    int status;                 // 0 run, 1 pad row, 2 bad slot index, 3 bad cursor, 4 out of range (debug)
    int slot, p;
    float g, beta;              // this step's log-decay and beta
    float c[kPipeLMax];         // c_j = exp(g_{j+1} + ... + g_p)
    float alpha[kPipeLMax];     // c_j (k_j . k)
    float gamma[kPipeLMax];     // c_j (k_j . q)
};

__host__ __device__ inline uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

// Byte offsets inside one stage: S tile, q, k, v rows, delta records, key records, scalars.
struct PipeLayout {
    uint32_t q, k, v, d, kr, meta, stage;
    __host__ __device__ PipeLayout(int L, uint32_t es, uint32_t rs)
    {
        q = 128u * 128u * 4u;
        k = q + round16(128u * es);
        v = k + round16(128u * es);
        d = v + round16(128u * es);
        kr = d + round16((uint32_t)(L - 1) * 128u * rs);
        meta = kr + round16((uint32_t)(L - 1) * 128u * rs);
        stage = (meta + (uint32_t)sizeof(PipeMeta) + 127u) & ~127u;
    }
};

template <typename Tring> __device__ __forceinline__ Tring ring_out(float x);
template <> __device__ __forceinline__ float ring_out<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 ring_out<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float ring_in(float x) { return x; }
__device__ __forceinline__ float ring_in(bf16 x) { return __bfloat162float(x); }

// eight consecutive ring values (rows of one warp) from shared memory
__device__ __forceinline__ void load8(const float *p, float (&o)[8])
{
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16 *p, float (&o)[8])
{
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <typename Tin, typename Tring>
__global__ void __launch_bounds__(kPipeThreads, 1) buffered_pipe_kernel(const __grid_constant__ StepLaunch P)
{
    constexpr int K = 128, V = 128;
    using TL = Tile<128, 16, kPipeGW>;
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ int abort_flag;
    __shared__ int zero_flag;

    const gdn_step_args &a = P.a;
    const int HV = a.HV, L = P.L, NST = P.nst, G = P.G;
    const int ntiles = a.B * HV;
    const PipeLayout lay(L, sizeof(Tin), sizeof(Tring));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + (size_t)NST * lay.stage);
    uint64_t *empty = full + NST;
    uint64_t *scr = empty + NST;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 32);
            mbar_init(&empty[s], kPipeGW);
            mbar_init(&scr[s], kPipeGW);
        }
        abort_flag = 0;
        zero_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kPipeCW) {
        // ---------------------------------------------------------------- producer warp
        // Tile scalars are fetched 32 tiles at a time (lane i for the i-th next tile), so the
        // producer pays one global round trip per 32 tiles; per tile it only waits for a free
        // stage, writes the scalars and issues the bulk copies.
        const uint64_t pol = policy_evict_first();
        const uint32_t es = sizeof(Tin), rs = sizeof(Tring);
        int n = 0;
        bool stop = false;
        for (int base = blockIdx.x; base < ntiles && !stop; base += 32 * gridDim.x) {
            const int my_tile = base + lane * gridDim.x;
            int my_slot = 0, my_status = 1, my_p = 0;
            float my_g = 0.f, my_beta = 0.f;
            if (my_tile < ntiles) {
                const int b = my_tile / HV, hv = my_tile - b * HV;
                my_slot = b;
                my_status = 0;
                if (P.idx) {
                    my_slot = P.idx[b];
                    if (my_slot == P.pad) my_status = 1;
                    else if (my_slot < 0 || my_slot >= a.num_slots) my_status = 2;
                }
                my_p = P.write_pos[b];
                if (my_status == 0 && (my_p < 0 || my_p >= L)) my_status = 3;
                if (my_status == 0 && (!step_tile_in_range(a, b, hv, hv / G, my_slot) ||
                                       !ring_in_range(a, L, my_slot, hv, hv / G, my_p)))
                    my_status = 4;   // an index out of range (debug build): skipped, nothing written
                if (my_status != 0) my_p = 0;
                step_gates<Tin>(a, b, hv, my_g, my_beta);
            }
            for (int i = 0; i < 32; ++i) {
                const int tile = base + i * gridDim.x;
                if (tile >= ntiles) break;
                const int st = n % NST;
                const uint32_t ph = (uint32_t)(n / NST) & 1u;
                if (n >= NST && !mbar_wait_warp(&empty[st], ph ^ 1u, &abort_flag, kWaitLimit)) {
                    if (lane == 0) {
                        *(volatile int *)&abort_flag = 1;
                        raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
                    }
                    stop = true;
                    break;
                }
                const int slot = __shfl_sync(kFull, my_slot, i);
                const int status = __shfl_sync(kFull, my_status, i);
                const int p = __shfl_sync(kFull, my_p, i);
                const float g = __shfl_sync(kFull, my_g, i);
                const float beta = __shfl_sync(kFull, my_beta, i);
                ++n;
                if (lane != 0) {
                    mbar_arrive(&full[st]);
                    continue;
                }
                unsigned char *stage = sm + (size_t)st * lay.stage;
                PipeMeta *meta = reinterpret_cast<PipeMeta *>(stage + lay.meta);
                meta->status = status;
                meta->slot = slot;
                meta->p = p;
                meta->g = g;
                meta->beta = beta;
                const uint32_t gbytes = p > 0 ? round16((uint32_t)p * 4u) : 0u;
                const uint32_t bytes = status == 0 ? 128u * 128u * 4u + 3u * 128u * es + 2u * (uint32_t)p * 128u * rs + gbytes : 0u;
                fence_proxy_async();
                mbar_arrive_expect_tx(&full[st], bytes);
                if (status == 0) {
                    const int b = tile / HV, hv = tile - b * HV, h = hv / G;
                    const float *S = static_cast<const float *>(a.state) + ((size_t)slot * HV + hv) * (size_t)(V * K);
                    bulk_g2s_hint(stage, S, 128u * 128u * 4u, &full[st], pol);
                    bulk_g2s(stage + lay.q, static_cast<const Tin *>(a.q) + (size_t)b * a.q_stride + (size_t)h * K, 128u * es, &full[st]);
                    bulk_g2s(stage + lay.k, static_cast<const Tin *>(a.k) + (size_t)b * a.k_stride + (size_t)h * K, 128u * es, &full[st]);
                    bulk_g2s(stage + lay.v, static_cast<const Tin *>(a.v) + (size_t)b * a.v_stride + (size_t)hv * V, 128u * es, &full[st]);
                    if (p > 0) {
                        const Tring *dr = static_cast<const Tring *>(P.d_cache) + ((size_t)slot * HV + hv) * L * V;
                        const Tring *kr = static_cast<const Tring *>(P.k_cache) + ((size_t)slot * a.H + h) * L * K;
                        bulk_g2s(stage + lay.d, dr, (uint32_t)p * 128u * rs, &full[st]);
                        bulk_g2s(stage + lay.kr, kr, (uint32_t)p * 128u * rs, &full[st]);
                        bulk_g2s(meta->gr, P.g_cache + ((size_t)slot * HV + hv) * L, gbytes, &full[st]);
                    }
                }
            }
        }
        if (*(volatile int *)&abort_flag) {
            // let every copy issued for the stages still in flight land before the CTA exits
            for (int back = 1; back <= NST && n - back >= 0; ++back) {
                const int m = n - back;
                mbar_wait(&full[m % NST], (uint32_t)(m / NST) & 1u, &zero_flag, kWaitLimit);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumer warps
    // Two groups of eight warps take alternate tiles, so two tiles are in their arithmetic at once.
    const int group = warp / kPipeGW, gwarp = warp - group * kPipeGW;
    TL t;
    t.init(gwarp);
    const int tid = threadIdx.x - group * kPipeGW * 32;   // 0 .. 255 within the group
    int n = group;
    for (int tile = blockIdx.x + group * gridDim.x; tile < ntiles; tile += kPipeGroups * gridDim.x, n += kPipeGroups) {
        const int st = n % NST;
        const uint32_t ph = (uint32_t)(n / NST) & 1u;
        // A stage's uses alternate between the groups, so this group may reach tile n while the
        // other group still holds tile n - NST on the same stage. A parity wait can only tell
        // apart a phase from the one before it, so first wait for that earlier use to be released
        // (after which the stage's barriers are at most one phase away from tile n's).
        if ((n >= NST && !mbar_wait_warp(&empty[st], ph ^ 1u, &abort_flag, kWaitLimit)) ||
            !mbar_wait_warp(&full[st], ph, &abort_flag, kWaitLimit)) {
            if (lane == 0) {
                *(volatile int *)&abort_flag = 1;
                raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
            }
            break;
        }
        const unsigned char *stage = sm + (size_t)st * lay.stage;
        PipeMeta *meta = reinterpret_cast<PipeMeta *>(sm + (size_t)st * lay.stage + lay.meta);
        const int status = meta->status, slot = meta->slot, p = meta->p;
        const int b = tile / HV, hv = tile - b * HV;
        const size_t out_base = ((size_t)b * HV + hv) * V;
        if (status != 0) {
            if ((status == 2 || status == 3) && tid == 0)
                raise_flag(a.err_flags, status == 2 ? GDN_DEVERR_BAD_INDEX : GDN_DEVERR_BAD_WRITE_POS);
            if (status != 4 && tid < V) store_out(a.out, a.out_dtype, out_base + tid, 0.f);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&scr[st]);
                mbar_arrive(&empty[st]);
            }
            continue;
        }
        const bool flush = p == L - 1;
        const Tin *qs = reinterpret_cast<const Tin *>(stage + lay.q);
        const Tin *ks = reinterpret_cast<const Tin *>(stage + lay.k);
        const Tin *vs = reinterpret_cast<const Tin *>(stage + lay.v);
        const Tring *ds = reinterpret_cast<const Tring *>(stage + lay.d);
        const Tring *krs = reinterpret_cast<const Tring *>(stage + lay.kr);
        const float *Ss = reinterpret_cast<const float *>(stage);

        const float4 kh = l2_normalise4<32>(load4(ks + t.col), a.use_qk_l2norm != 0, 1.f);
        const float4 qh = l2_normalise4<32>(load4(qs + t.col), a.use_qk_l2norm != 0, P.scale);
        const float kq = group_sum<32>(dot4(kh, qh));
        const float g = meta->g, beta = meta->beta;
        // record scalars, one warp per record
        for (int j = gwarp; j < p; j += kPipeGW) {
            const float4 kj = load4(krs + (size_t)j * K + t.col);
            const float dk = group_sum<32>(dot4(kj, kh));
            const float dq = group_sum<32>(dot4(kj, qh));
            if (lane == 0) {
                float acc = g;
                for (int i = j + 1; i < p; ++i) acc += meta->gr[i];
                const float c = expf(acc);
                meta->c[j] = c;
                meta->alpha[j] = c * dk;
                meta->gamma[j] = c * dq;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&scr[st]);

        float gsum = g;
        for (int i = 0; i < p; ++i) gsum += meta->gr[i];
        const float Gam = expf(gsum);

        // the two dots, straight from the staged tile (16 rows x 4 columns per lane)
        const int row0 = t.row(0, 0);   // this warp's TL::R consecutive rows
        const int r_own = t.row(0, t.owned_chunk(0));
        const float vv = t.holds_k_dot() ? to_f32(vs[r_own]) : 0.f;
        float x[TL::N];
        {
            const float4 gk = scale4(kh, Gam), gq = scale4(qh, Gam);
#pragma unroll
            for (int i = 0; i < TL::R; ++i) {
                const float4 srow = *reinterpret_cast<const float4 *>(Ss + (size_t)(row0 + i) * K + t.col);
                x[i] = dot4(srow, gk);
                x[TL::R + i] = dot4(srow, gq);
            }
        }
        t.reduce_scatter(x);

        if (!mbar_wait_warp(&scr[st], ph, &abort_flag, kWaitLimit)) {
            if (lane == 0) {
                *(volatile int *)&abort_flag = 1;
                raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
            }
            break;
        }
        // ring corrections: lower lanes on u, upper lanes on o
        {
            const float *coef = t.holds_k_dot() ? meta->alpha : meta->gamma;
            float acc = x[0];
            for (int j = 0; j < p; ++j) acc = fmaf(ring_in(ds[(size_t)j * V + r_own]), coef[j], acc);
            x[0] = acc;
        }
        float dv[TL::M];
        dv[0] = beta * (vv - x[0]);
        const float dq = t.delta_for_q(dv[0]);
        Tring *dring = static_cast<Tring *>(P.d_cache) + ((size_t)slot * HV + hv) * L * V;
        if (t.writer()) {
            if (t.holds_k_dot())
                dring[(size_t)p * V + r_own] = ring_out<Tring>(dv[0]);
            else
                store_out(a.out, a.out_dtype, out_base + r_own, fmaf(dq, kq, x[0]));
        }
        if (flush) {
            // S = Gamma S_c + delta k^T + sum_j d_j (c_j k_j)^T, eight rows at a time
            float *S = static_cast<float *>(a.state) + ((size_t)slot * HV + hv) * (size_t)(V * K);
#pragma unroll
            for (int i8 = 0; i8 < TL::R; i8 += 8) {
                // the fold's FMAs on fp32 pairs (fma.rn.f32x2: each element rounded as by fmaf, so
                // the result is the scalar loop's bit for bit, in half the instructions; the L = 16
                // flush took 205.0 against 211.4 us at B = 256)
                float2 alo[8], ahi[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 srow = *reinterpret_cast<const float4 *>(Ss + (size_t)(row0 + i8 + i) * K + t.col);
                    const float4 a0 = axpby4(Gam, srow, t.delta_of(dv, i8 + i), kh);
                    alo[i] = make_float2(a0.x, a0.y);
                    ahi[i] = make_float2(a0.z, a0.w);
                }
                for (int j = 0; j < p; ++j) {
                    const float4 kj = scale4(load4(krs + (size_t)j * K + t.col), meta->c[j]);
                    const float2 klo = make_float2(kj.x, kj.y), khi = make_float2(kj.z, kj.w);
                    float dj[8];
                    load8(ds + (size_t)j * V + row0 + i8, dj);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float2 d2 = make_float2(dj[i], dj[i]);
                        alo[i] = __ffma2_rn(d2, klo, alo[i]);
                        ahi[i] = __ffma2_rn(d2, khi, ahi[i]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    st_stream(S + (size_t)(row0 + i8 + i) * K + t.col, make_float4(alo[i].x, alo[i].y, ahi[i].x, ahi[i].y));
            }
        }
        // everything of this stage has been read
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);

        // this step's key record (first value head of the group) and log-decay record
        if (hv % G == 0 && gwarp == 0) {
            Tring *dst = static_cast<Tring *>(P.k_cache) + (((size_t)slot * a.H + hv / G) * L + p) * K + t.col;
            dst[0] = ring_out<Tring>(kh.x);
            dst[1] = ring_out<Tring>(kh.y);
            dst[2] = ring_out<Tring>(kh.z);
            dst[3] = ring_out<Tring>(kh.w);
        }
        if (tid == 0) P.g_cache[((size_t)slot * HV + hv) * L + p] = g;
    }
}

// dynamic shared memory of the pipelined kernel for NST stages
static size_t pipe_smem(const PipeLayout &lay, int nst) { return (size_t)nst * lay.stage + 3 * nst * sizeof(uint64_t); }

template <typename Tin, typename Tring>
static int launch_pipe_t(const StepLaunch &p0, cudaStream_t stream)
{
    StepLaunch p = p0;
    const PipeLayout lay(p.L, sizeof(Tin), sizeof(Tring));
    int dev = 0, sms = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const size_t budget = (size_t)max_smem - 1024;   // room for the kernel's static shared memory
    int nst = 3;
    while (nst >= 2 && pipe_smem(lay, nst) > budget) --nst;
    if (nst < 2) return GDN_ERR_SHAPE;
    p.nst = nst;
    const size_t smem = pipe_smem(lay, nst);
    auto kern = buffered_pipe_kernel<Tin, Tring>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int tiles = p.a.B * p.a.HV;
    const int grid = tiles < sms ? tiles : sms;
    kern<<<grid, kPipeThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

bool buffered_pipe_fits(int L, int in_dtype, int ring_dtype, int max_smem)
{
    const PipeLayout lay(L, in_dtype == GDN_BF16 ? 2 : 4, ring_dtype == GDN_BF16 ? 2 : 4);
    return pipe_smem(lay, 2) + 1024 <= (size_t)max_smem;
}

int launch_buffered_pipe(const StepLaunch &p, int ring_dtype, cudaStream_t stream)
{
    if (p.a.in_dtype == GDN_BF16)
        return ring_dtype == GDN_BF16 ? launch_pipe_t<bf16, bf16>(p, stream) : launch_pipe_t<bf16, float>(p, stream);
    return ring_dtype == GDN_BF16 ? launch_pipe_t<float, bf16>(p, stream) : launch_pipe_t<float, float>(p, stream);
}


// ------------------------------------------------------------------------------------------------
// One tile per CTA of 256 threads with the same staging: thread 0 reads the row's slot and cursor
// and bulk-copies the 64 KB checkpoint tile, the q/k/v rows and the tile's p ring records (delta
// rows, key rows, log-decays) into the CTA's shared memory on one mbarrier; the arithmetic is the
// consumer group's above with block barriers in place of the group's mbarrier. 73 KB of shared
// memory at L = 16 with a bf16 ring: three CTAs per SM, each with its copies in flight, and
// consecutive launches overlap like any per-tile kernel.
// ------------------------------------------------------------------------------------------------
template <typename Tin, typename Tring>
__global__ void __launch_bounds__(kThreads, 3) buffered_stage_kernel(const __grid_constant__ StepLaunch P)
{
    constexpr int K = 128, V = 128;
    using TL = Tile<128, 16, kWarps>;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag, zero_flag, s_status, s_slot, s_p;

    const gdn_step_args &a = P.a;
    const int HV = a.HV, L = P.L, G = P.G;
    const int tile = blockIdx.x, b = tile / HV, hv = tile - b * HV, h = hv / G;
    const int lane = threadIdx.x & 31, tid = threadIdx.x;
    const PipeLayout lay(L, sizeof(Tin), sizeof(Tring));
    PipeMeta *meta = reinterpret_cast<PipeMeta *>(stage + lay.meta);
    const size_t out_base = ((size_t)b * HV + hv) * V;
    const uint32_t es = sizeof(Tin), rs = sizeof(Tring);

    if (tid == 0) {
        int slot = b, status = 0;
        if (P.idx) {
            slot = P.idx[b];
            if (slot == P.pad) status = 1;
            else if (slot < 0 || slot >= a.num_slots) status = 2;
        }
        int p = P.write_pos[b];
        if (status == 0 && (p < 0 || p >= L)) status = 3;
        if (status == 0 && (!step_tile_in_range(a, b, hv, h, slot) || !ring_in_range(a, L, slot, hv, h, p)))
            status = 4;   // an index out of range (debug build): skipped, nothing written
        if (status != 0) p = 0;
        s_status = status;
        s_slot = slot;
        s_p = p;
        abort_flag = 0;
        zero_flag = 0;
        if (status == 0) {
            mbar_init(&bar, 1);
            fence_barrier_init();
            const uint32_t gbytes = p > 0 ? round16((uint32_t)p * 4u) : 0u;
            mbar_arrive_expect_tx(&bar, 128u * 128u * 4u + 3u * 128u * es + 2u * (uint32_t)p * 128u * rs + gbytes);
            const float *S = static_cast<const float *>(a.state) + ((size_t)slot * HV + hv) * (size_t)(V * K);
            bulk_g2s_hint(stage, S, 128u * 128u * 4u, &bar, policy_evict_first());
            bulk_g2s(stage + lay.q, static_cast<const Tin *>(a.q) + (size_t)b * a.q_stride + (size_t)h * K, 128u * es, &bar);
            bulk_g2s(stage + lay.k, static_cast<const Tin *>(a.k) + (size_t)b * a.k_stride + (size_t)h * K, 128u * es, &bar);
            bulk_g2s(stage + lay.v, static_cast<const Tin *>(a.v) + (size_t)b * a.v_stride + (size_t)hv * V, 128u * es, &bar);
            if (p > 0) {
                const Tring *dr = static_cast<const Tring *>(P.d_cache) + ((size_t)slot * HV + hv) * L * V;
                const Tring *kr = static_cast<const Tring *>(P.k_cache) + ((size_t)slot * a.H + h) * L * K;
                bulk_g2s(stage + lay.d, dr, (uint32_t)p * 128u * rs, &bar);
                bulk_g2s(stage + lay.kr, kr, (uint32_t)p * 128u * rs, &bar);
                bulk_g2s(meta->gr, P.g_cache + ((size_t)slot * HV + hv) * L, gbytes, &bar);
            }
        }
    }
    float g, beta;
    step_gates<Tin>(a, b, hv, g, beta);
    TL t;
    t.init();
    __syncthreads();
    const int status = s_status, slot = s_slot, p = s_p;
    if (status != 0) {   // uniform over the CTA
        if ((status == 2 || status == 3) && tid == 0)
            raise_flag(a.err_flags, status == 2 ? GDN_DEVERR_BAD_INDEX : GDN_DEVERR_BAD_WRITE_POS);
        if (status != 4 && tid < V) store_out(a.out, a.out_dtype, out_base + tid, 0.f);
        return;
    }
    if (!mbar_wait_warp(&bar, 0u, &abort_flag, kWaitLimit)) {
        if (lane == 0) raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
        if (tid == 0) mbar_wait(&bar, 0u, &zero_flag, kWaitLimit);   // copies still in flight land first
        return;
    }
    const bool flush = p == L - 1;
    const Tin *qs = reinterpret_cast<const Tin *>(stage + lay.q);
    const Tin *ks = reinterpret_cast<const Tin *>(stage + lay.k);
    const Tin *vs = reinterpret_cast<const Tin *>(stage + lay.v);
    const Tring *ds = reinterpret_cast<const Tring *>(stage + lay.d);
    const Tring *krs = reinterpret_cast<const Tring *>(stage + lay.kr);
    const float *Ss = reinterpret_cast<const float *>(stage);

    const float4 kh = l2_normalise4<32>(load4(ks + t.col), a.use_qk_l2norm != 0, 1.f);
    const float4 qh = l2_normalise4<32>(load4(qs + t.col), a.use_qk_l2norm != 0, P.scale);
    const float kq = group_sum<32>(dot4(kh, qh));
    // record scalars, one warp per record
    for (int j = t.warp; j < p; j += kWarps) {
        const float4 kj = load4(krs + (size_t)j * K + t.col);
        const float dk = group_sum<32>(dot4(kj, kh));
        const float dq = group_sum<32>(dot4(kj, qh));
        if (lane == 0) {
            float acc = g;
            for (int i = j + 1; i < p; ++i) acc += meta->gr[i];
            const float c = expf(acc);
            meta->c[j] = c;
            meta->alpha[j] = c * dk;
            meta->gamma[j] = c * dq;
        }
    }
    float gsum = g;
    for (int i = 0; i < p; ++i) gsum += meta->gr[i];
    const float Gam = expf(gsum);

    // the two dots, straight from the staged tile (16 rows x 4 columns per lane)
    const int row0 = t.row(0, 0);
    const int r_own = t.row(0, t.owned_chunk(0));
    const float vv = t.holds_k_dot() ? to_f32(vs[r_own]) : 0.f;
    float x[TL::N];
    {
        const float4 gk = scale4(kh, Gam), gq = scale4(qh, Gam);
#pragma unroll
        for (int i = 0; i < TL::R; ++i) {
            const float4 srow = *reinterpret_cast<const float4 *>(Ss + (size_t)(row0 + i) * K + t.col);
            x[i] = dot4(srow, gk);
            x[TL::R + i] = dot4(srow, gq);
        }
    }
    t.reduce_scatter(x);
    __syncthreads();   // the record scalars are complete
    {
        const float *coef = t.holds_k_dot() ? meta->alpha : meta->gamma;
        float acc = x[0];
        for (int j = 0; j < p; ++j) acc = fmaf(ring_in(ds[(size_t)j * V + r_own]), coef[j], acc);
        x[0] = acc;
    }
    float dv[TL::M];
    dv[0] = beta * (vv - x[0]);
    const float dq = t.delta_for_q(dv[0]);
    Tring *dring = static_cast<Tring *>(P.d_cache) + ((size_t)slot * HV + hv) * L * V;
    if (t.writer()) {
        if (t.holds_k_dot())
            dring[(size_t)p * V + r_own] = ring_out<Tring>(dv[0]);
        else
            store_out(a.out, a.out_dtype, out_base + r_own, fmaf(dq, kq, x[0]));
    }
    if (flush) {
        // S = Gamma S_c + delta k^T + sum_j d_j (c_j k_j)^T, eight rows at a time
        float *S = static_cast<float *>(a.state) + ((size_t)slot * HV + hv) * (size_t)(V * K);
#pragma unroll
        for (int i8 = 0; i8 < TL::R; i8 += 8) {
            float4 acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 srow = *reinterpret_cast<const float4 *>(Ss + (size_t)(row0 + i8 + i) * K + t.col);
                acc[i] = axpby4(Gam, srow, t.delta_of(dv, i8 + i), kh);
            }
            for (int j = 0; j < p; ++j) {
                const float4 kj = scale4(load4(krs + (size_t)j * K + t.col), meta->c[j]);
                float dj[8];
                load8(ds + (size_t)j * V + row0 + i8, dj);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[i].x = fmaf(dj[i], kj.x, acc[i].x);
                    acc[i].y = fmaf(dj[i], kj.y, acc[i].y);
                    acc[i].z = fmaf(dj[i], kj.z, acc[i].z);
                    acc[i].w = fmaf(dj[i], kj.w, acc[i].w);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) st_stream(S + (size_t)(row0 + i8 + i) * K + t.col, acc[i]);
        }
    }
    // this step's key record (first value head of the group) and log-decay record
    if (hv % G == 0 && t.warp == 0) {
        Tring *dst = static_cast<Tring *>(P.k_cache) + (((size_t)slot * a.H + h) * L + p) * K + t.col;
        dst[0] = ring_out<Tring>(kh.x);
        dst[1] = ring_out<Tring>(kh.y);
        dst[2] = ring_out<Tring>(kh.z);
        dst[3] = ring_out<Tring>(kh.w);
    }
    if (tid == 0) P.g_cache[((size_t)slot * HV + hv) * L + p] = g;
}

template <typename Tin, typename Tring>
static int launch_stage_t(const StepLaunch &p, cudaStream_t stream)
{
    const PipeLayout lay(p.L, sizeof(Tin), sizeof(Tring));
    const size_t smem = lay.stage;
    auto kern = buffered_stage_kernel<Tin, Tring>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    kern<<<(unsigned)(p.a.B * p.a.HV), kThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

int launch_buffered_stage(const StepLaunch &p, int ring_dtype, cudaStream_t stream)
{
    if (p.a.in_dtype == GDN_BF16)
        return ring_dtype == GDN_BF16 ? launch_stage_t<bf16, bf16>(p, stream) : launch_stage_t<bf16, float>(p, stream);
    return ring_dtype == GDN_BF16 ? launch_stage_t<float, bf16>(p, stream) : launch_stage_t<float, float>(p, stream);
}

}  // namespace gdn
