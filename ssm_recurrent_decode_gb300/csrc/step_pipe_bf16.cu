// step_pipe_bf16.cu -- the packed / indexed decode step with a bf16 state, K = V = 128, as a
// persistent, warp-specialised kernel (gdn_decode_step and gdn_decode_step_indexed).
//
// A bf16 state tile is 32 KB, and the step does about as much arithmetic per tile as with an fp32
// state, in half the bytes: the per-tile kernel (step_kernel_bf16) spent so long on each tile's
// arithmetic that HBM sat idle for much of the launch. Here the state tiles stream into shared
// memory ahead of the arithmetic:
//   - one CTA per SM: a producer warp and NG groups of 8 consumer warps taking tiles in turn;
//   - the producer walks the CTA's tiles and, for each, moves the 32 KB state tile and the q, k, v
//     rows into a shared-memory stage with 1-D bulk copies (cp.async.bulk) that complete on the
//     stage's "full" mbarrier, and writes the tile's slot, status and gates beside them (fetched
//     32 tiles at a time, one lane per tile);
//   - NST stages (up to six, about 200 KB) keep that many tiles in flight per SM;
//   - a consumer group reads a staged row as 16-byte vectors of eight bf16 values (16 lanes per
//     row, two rows per warp instruction, eight rows per lane in two halves of four), takes S.k
//     and S.q with a reduce-scatter over the 16 lanes of a row, then reads the rows again, applies
//     the update in
//     fp32 and stores the rounded rows to HBM with 16-byte streaming stores; then the stage is
//     released on its "empty" mbarrier.
// Arithmetic as in step_kernel_bf16: u = e (S k_hat), o = e (S q_hat) + delta (k_hat . q_hat),
// S' = e S + delta k_hat^T in fp32, rounded to nearest even as it is stored.
// Every wait is bounded: a wait that runs past its limit sets GDN_DEVERR_TIMEOUT, raises a
// CTA-wide abort flag and ends the CTA's loop; the producer then waits (bounded) for the copies
// it issued, so no copy is in flight when the CTA exits.
//
// Sources: "Optimization Log: Qwen3.5-27B Dense on B200", "Kernel 4: Fused DeltaNet Recurrent
// (FLAGSHIP)" (the Math block; 32 KB bf16 state per head); "Microbenchmark: buffered output-only
// GDN decode (ReplaySSM Part A)", _bench_cfg / run_packed (packed mixed_qkv, gates, slot pool).
#include "gdn_launch.h"
#include "gdn_pipe.cuh"
#include "gdn_tile.cuh"

namespace gdn {

constexpr int kBpGW = 8;                               // warps of one consumer group
constexpr int kBpMaxStages = 6;
constexpr long long kBpWaitLimit = 1LL << 31;          // SM clock cycles, about one second
constexpr uint32_t kBpTileBytes = 128u * 128u * 2u;    // one bf16 state tile

template <int NG> constexpr int bp_threads() { return (NG * kBpGW + 1) * 32; }

struct BpMeta {
    int status;   // 0 run, 1 pad row, 2 bad slot index, 3 an index out of range (debug build)
    int slot;
    float g, beta;
};

// Byte offsets inside one stage: S tile, q, k, v rows, scalars.
struct BpLayout {
    uint32_t q, k, v, meta, stage;
    __host__ __device__ explicit BpLayout(uint32_t es)
    {
        q = kBpTileBytes;
        k = q + 128u * es;
        v = k + 128u * es;
        meta = v + 128u * es;
        stage = (meta + (uint32_t)sizeof(BpMeta) + 127u) & ~127u;
    }
};

// Arithmetic on pairs of fp32 values (fma.rn.f32x2 and mul.rn.f32x2 of sm_100 and later): the
// same rounding per element as the scalar operations, in half the instructions.
// eight bf16 values of a 16-byte vector as four fp32 pairs (element 2 j in .x, 2 j + 1 in .y)
__device__ __forceinline__ void unpack8(uint4 r, float2 (&o)[4])
{
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
}
// eight consecutive q/k/v values of a staged row
__device__ __forceinline__ void lds8(const bf16 *p, float2 (&o)[4]) { unpack8(*reinterpret_cast<const uint4 *>(p), o); }
__device__ __forceinline__ void lds8(const float *p, float2 (&o)[4])
{
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    o[0] = make_float2(a.x, a.y); o[1] = make_float2(a.z, a.w); o[2] = make_float2(b.x, b.y); o[3] = make_float2(b.z, b.w);
}

// sum of the eight products a . b, accumulated as two interleaved partial sums
__device__ __forceinline__ float dot8(const float2 (&a)[4], const float2 (&b)[4])
{
    float2 acc = __fmul2_rn(a[0], b[0]);
#pragma unroll
    for (int i = 1; i < 4; ++i) acc = __ffma2_rn(a[i], b[i], acc);
    return acc.x + acc.y;
}

// round two fp32 values to nearest even bf16 and pack them (low half first)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// Butterfly reduce-scatter over the 16 lanes of a row group: at offset O a lane keeps one half of
// its NN values and adds the partner's copy of that half; once one value is left, the remaining
// offsets are plain butterflies. For 8 values (4 rows x 2 dots) lanes 2j and 2j + 1 of a row group
// end with the complete sum of index j in x[0]: 8 shuffles instead of 8 x 4 for separate sums.
template <int O, int NN>
__device__ __forceinline__ void bp_reduce(float (&x)[8], int lane)
{
    if constexpr (O >= 1) {
        if constexpr (NN > 1) {
            const bool upper = (lane & O) != 0;
#pragma unroll
            for (int j = 0; j < NN / 2; ++j) {
                const float send = upper ? x[j] : x[j + NN / 2];
                const float keep = upper ? x[j + NN / 2] : x[j];
                x[j] = keep + __shfl_xor_sync(kFull, send, O);
            }
            bp_reduce<O / 2, NN / 2>(x, lane);
        } else {
            x[0] += __shfl_xor_sync(kFull, x[0], O);
            bp_reduce<O / 2, 1>(x, lane);
        }
    }
}

template <typename Tin, int NG>
__global__ void __launch_bounds__(bp_threads<NG>(), 1) step_pipe_bf16_kernel(const __grid_constant__ StepLaunch P)
{
    constexpr int K = 128, V = 128;
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ int abort_flag;
    __shared__ int zero_flag;

    const gdn_step_args &a = P.a;
    const int HV = a.HV, NST = P.nst, G = P.G;
    const int ntiles = a.B * HV;
    const BpLayout lay(sizeof(Tin));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + (size_t)NST * lay.stage);
    uint64_t *empty = full + NST;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBpGW);
        }
        abort_flag = 0;
        zero_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NG * kBpGW) {
        // ---------------------------------------------------------------- producer warp
        const uint64_t pol = policy_evict_first();
        const uint32_t es = sizeof(Tin);
        int n = 0;
        bool stop = false;
        for (int base = blockIdx.x; base < ntiles && !stop; base += 32 * gridDim.x) {
            const int my_tile = base + lane * gridDim.x;
            int my_slot = 0, my_status = 1;
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
                if (my_status == 0 && !step_tile_in_range(a, b, hv, hv / G, my_slot)) my_status = 3;   // debug build
                if (my_status != 3) step_gates<Tin>(a, b, hv, my_g, my_beta);
            }
            for (int i = 0; i < 32; ++i) {
                const int tile = base + i * gridDim.x;
                if (tile >= ntiles) break;
                const int st = n % NST;
                const uint32_t ph = (uint32_t)(n / NST) & 1u;
                if (n >= NST && !mbar_wait_warp(&empty[st], ph ^ 1u, &abort_flag, kBpWaitLimit)) {
                    if (lane == 0) {
                        *(volatile int *)&abort_flag = 1;
                        raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
                    }
                    stop = true;
                    break;
                }
                const int slot = __shfl_sync(kFull, my_slot, i);
                const int status = __shfl_sync(kFull, my_status, i);
                const float g = __shfl_sync(kFull, my_g, i);
                const float beta = __shfl_sync(kFull, my_beta, i);
                ++n;
                if (lane != 0) continue;
                unsigned char *stage = sm + (size_t)st * lay.stage;
                BpMeta *meta = reinterpret_cast<BpMeta *>(stage + lay.meta);
                meta->status = status;
                meta->slot = slot;
                meta->g = g;
                meta->beta = beta;
                const uint32_t bytes = status == 0 ? kBpTileBytes + 3u * 128u * es : 0u;
                fence_proxy_async();
                mbar_arrive_expect_tx(&full[st], bytes);
                if (status == 0) {
                    const int b = tile / HV, hv = tile - b * HV, h = hv / G;
                    const bf16 *S = static_cast<const bf16 *>(a.state) + ((size_t)slot * HV + hv) * (size_t)(V * K);
                    bulk_g2s_hint(stage, S, kBpTileBytes, &full[st], pol);
                    bulk_g2s(stage + lay.q, static_cast<const Tin *>(a.q) + (size_t)b * a.q_stride + (size_t)h * K, 128u * es, &full[st]);
                    bulk_g2s(stage + lay.k, static_cast<const Tin *>(a.k) + (size_t)b * a.k_stride + (size_t)h * K, 128u * es, &full[st]);
                    bulk_g2s(stage + lay.v, static_cast<const Tin *>(a.v) + (size_t)b * a.v_stride + (size_t)hv * V, 128u * es, &full[st]);
                }
            }
        }
        if (lane == 0 && *(volatile int *)&abort_flag) {
            // let every copy issued for the stages still in flight land before the CTA exits
            for (int back = 1; back <= NST && n - back >= 0; ++back) {
                const int m = n - back;
                mbar_wait(&full[m % NST], (uint32_t)(m / NST) & 1u, &zero_flag, kBpWaitLimit);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumer warps
    const int group = warp / kBpGW, gwarp = warp - group * kBpGW;
    const int grp = lane >> 4, sub = lane & 15, col = sub * 8;
    const int tid = threadIdx.x - group * kBpGW * 32;   // 0 .. 255 within the group
    const int rbase = gwarp * 16 + grp;                 // row of vector i: rbase + 2 i
    int n = group;
    for (int tile = blockIdx.x + group * gridDim.x; tile < ntiles; tile += NG * gridDim.x, n += NG) {
        const int st = n % NST;
        const uint32_t ph = (uint32_t)(n / NST) & 1u;
        // the stage's previous use (another group's tile) is released first, then this tile's
        // copies have landed
        if ((n >= NST && !mbar_wait_warp(&empty[st], ph ^ 1u, &abort_flag, kBpWaitLimit)) ||
            !mbar_wait_warp(&full[st], ph, &abort_flag, kBpWaitLimit)) {
            if (lane == 0) {
                *(volatile int *)&abort_flag = 1;
                raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
            }
            break;
        }
        const unsigned char *stage = sm + (size_t)st * lay.stage;
        const BpMeta *meta = reinterpret_cast<const BpMeta *>(stage + lay.meta);
        const int status = meta->status, slot = meta->slot;
        const int b = tile / HV, hv = tile - b * HV;
        const size_t out_base = ((size_t)b * HV + hv) * V;
        if (status != 0) {
            if (status == 2 && tid == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_INDEX);
            if (status != 3 && tid < V) store_out(a.out, a.out_dtype, out_base + tid, 0.f);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            continue;
        }
        const float g = meta->g, beta = meta->beta;
        const Tin *qs = reinterpret_cast<const Tin *>(stage + lay.q);
        const Tin *ks = reinterpret_cast<const Tin *>(stage + lay.k);
        const Tin *vs = reinterpret_cast<const Tin *>(stage + lay.v);
        const bf16 *Ss = reinterpret_cast<const bf16 *>(stage);

        // normalised q and k on this lane's eight columns (sums over the 16 lanes of a row)
        float2 kh[4], qh[4];
        lds8(ks + col, kh);
        lds8(qs + col, qh);
        {
            const bool l2 = a.use_qk_l2norm != 0;
            const float sk = group_sum<16>(dot8(kh, kh));
            const float sq = group_sum<16>(dot8(qh, qh));
            const float rk = l2 ? 1.0f / sqrtf(sk + 1e-6f) : 1.0f;
            const float rq = (l2 ? 1.0f / sqrtf(sq + 1e-6f) : 1.0f) * P.scale;
            const float2 rk2 = make_float2(rk, rk), rq2 = make_float2(rq, rq);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                kh[c] = __fmul2_rn(kh[c], rk2);
                qh[c] = __fmul2_rn(qh[c], rq2);
            }
        }
        const float kq = group_sum<16>(dot8(kh, qh));
        const float e = expf(g);
        const float2 e2 = make_float2(e, e);

        // The lane's eight rows in two halves of four (8 partial dots live at a time). Per half:
        // partial dots over the lane's eight columns and a reduce-scatter over the 16 lanes of the
        // row, after which lane sub holds index sub / 2 (S.k of row 4 h + sub / 2 for sub < 8, S.q
        // of row 4 h + sub / 2 - 4 for sub >= 8), so delta of row 4 h + j sits on lane 2 j. Then the
        // rows are read again, updated (S' = e S + delta k^T, rounded to bf16) and stored with
        // 16-byte streaming stores, one half at a time.
        float dh0 = 0.f, dh1 = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float x[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float2 sv[4];
                lds8(Ss + (size_t)(rbase + 2 * (4 * h + i)) * K + col, sv);
                x[i] = dot8(sv, kh);
                x[4 + i] = dot8(sv, qh);
            }
            bp_reduce<8, 8>(x, lane);
            const int r_own = rbase + 2 * (4 * h + ((sub >> 1) & 3));
            float d = 0.f;
            if (sub < 8) d = beta * (to_f32(vs[r_own]) - e * x[0]);
            const float d_lo = __shfl_xor_sync(kFull, d, 8);
            if (sub >= 8 && (sub & 1) == 0) store_out(a.out, a.out_dtype, out_base + r_own, fmaf(d_lo, kq, e * x[0]));
            if (h == 0) dh0 = d; else dh1 = d;
        }
        bf16 *S = static_cast<bf16 *>(a.state) + ((size_t)slot * HV + hv) * (size_t)(V * K);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            const float d = h == 0 ? dh0 : dh1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float di = __shfl_sync(kFull, d, (lane & 16) + 2 * i);
                const float2 d2 = make_float2(di, di);
                const int r = rbase + 2 * (4 * h + i);
                float2 sv[4];
                lds8(Ss + (size_t)r * K + col, sv);
                uint32_t w[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float2 nv = __ffma2_rn(d2, kh[c], __fmul2_rn(e2, sv[c]));   // fmaf(d, k, e s) per element
                    w[c] = pack_bf16x2(nv.x, nv.y);
                }
                __stcs(reinterpret_cast<uint4 *>(S + (size_t)r * K + col), make_uint4(w[0], w[1], w[2], w[3]));
            }
        }
        // everything of this stage has been read
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
}

// dynamic shared memory for NST stages
static size_t bp_smem(const BpLayout &lay, int nst) { return (size_t)nst * lay.stage + 2 * nst * sizeof(uint64_t); }

template <typename Tin, int NG>
static int launch_bp_t(const StepLaunch &p0, cudaStream_t stream)
{
    StepLaunch p = p0;
    const BpLayout lay(sizeof(Tin));
    int dev = 0, sms = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const size_t budget = (size_t)max_smem - 1024;   // room for the kernel's static shared memory
    int nst = kBpMaxStages;
    while (nst > NG && bp_smem(lay, nst) > budget) --nst;
    if (bp_smem(lay, nst) > budget) return GDN_ERR_SHAPE;
    p.nst = nst;
    const size_t smem = bp_smem(lay, nst);
    auto kern = step_pipe_bf16_kernel<Tin, NG>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int tiles = p.a.B * p.a.HV;
    const int grid = tiles < sms ? tiles : sms;
    kern<<<grid, bp_threads<NG>(), smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

constexpr int kBpGroups = 3;

bool step_pipe_bf16_ok(const gdn_step_args &a)
{
    auto al16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    const int64_t es = a.in_dtype == GDN_BF16 ? 2 : 4;
    return a.state_dtype == GDN_BF16 && a.K == 128 && a.V == 128 && al16(a.state) && al16(a.q) &&
           al16(a.k) && al16(a.v) && (a.q_stride * es) % 16 == 0 && (a.k_stride * es) % 16 == 0 &&
           (a.v_stride * es) % 16 == 0;
}

int launch_step_pipe_bf16(const StepLaunch &p, cudaStream_t stream)
{
    return p.a.in_dtype == GDN_BF16 ? launch_bp_t<bf16, kBpGroups>(p, stream) : launch_bp_t<float, kBpGroups>(p, stream);
}

}  // namespace gdn
