// step_stage_bf16.cu -- the packed / indexed decode step with a bf16 state at K = V = 128
// (gdn_decode_step and gdn_decode_step_indexed, from 128 tiles per call).
//
// One CTA of 256 threads per (row, value head) tile. Thread 0 bulk-copies the 32 KB state tile and
// the q, k, v rows into the CTA's shared memory (cp.async.bulk, completion counted on one
// mbarrier) as soon as the CTA starts; every thread computes the gates while the copies are in
// flight. The arithmetic then reads the staged rows as 16-byte vectors of eight bf16 values (16
// lanes per row, two rows per warp instruction, eight rows per lane in two halves of four):
// partial dots S.k and S.q over the lane's eight columns in fp32 pairs, a reduce-scatter over the
// 16 lanes of a row, delta and the output, then the rows are read again, updated
// (S' = e S + delta k^T in fp32, rounded to nearest even) and stored with 16-byte streaming
// stores. No thread holds the tile in registers, so a CTA needs 40 registers per thread and
// 33.5 KB of shared memory: six CTAs per SM keep 192 KB of copies in flight per SM, and
// consecutive launches overlap like any per-tile kernel. The wait for the copies is bounded;
// on a timeout the CTA raises GDN_DEVERR_TIMEOUT, thread 0 waits (bounded) for the copies still in
// flight, and the tile is left as it was.
//
// Measured on GB300 at B = 256, HV = 32: 80.5 us per step against 93.7 for the per-tile kernel
// that held its rows in registers as 8-byte vectors (step_kernel_bf16), and 90.4 for a persistent
// warp-specialised form (a producer warp and six shared-memory stages), whose tiles waited for
// their consumer groups.
//
// Sources: "Optimization Log: Qwen3.5-27B Dense on B200", "Kernel 4: Fused DeltaNet Recurrent
// (FLAGSHIP)" (the Math block; 32 KB bf16 state per head); "Microbenchmark: buffered output-only
// GDN decode (ReplaySSM Part A)", _bench_cfg / run_packed (packed mixed_qkv, gates, slot pool).
#include "gdn_launch.h"
#include "gdn_pipe.cuh"
#include "gdn_tile.cuh"

namespace gdn {

constexpr long long kBsWaitLimit = 1LL << 31;          // SM clock cycles, about one second
constexpr uint32_t kBsTileBytes = 128u * 128u * 2u;    // one bf16 state tile

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

template <typename Tin>
__global__ void __launch_bounds__(256, 6) step_stage_bf16_kernel(const __grid_constant__ StepLaunch P)
{
    constexpr int K = 128;
    __shared__ __align__(128) unsigned char st[kBsTileBytes + 3u * 128u * sizeof(Tin)];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag, zero_flag;
    const gdn_step_args &a = P.a;
    const int HV = a.HV, V = a.V;
    const int tile = blockIdx.x, b = tile / HV, hv = tile - b * HV, h = hv / P.G;
    const int lane = threadIdx.x & 31;
    const int grp = lane >> 4, sub = lane & 15, col = sub * 8;
    const int rbase = (int)(threadIdx.x >> 5) * 16 + grp;   // row of vector i: rbase + 2 i
    const size_t out_base = ((size_t)b * HV + hv) * V;

    int slot = b;
    if (P.idx) {
        slot = P.idx[b];
        const bool pad = slot == P.pad;
        if (pad || slot < 0 || slot >= a.num_slots) {   // uniform over the CTA
            if (!pad && threadIdx.x == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_INDEX);
            if ((int)threadIdx.x < V) store_out(a.out, a.out_dtype, out_base + threadIdx.x, 0.f);
            return;
        }
    }
    if (!step_tile_in_range(a, b, hv, h, slot)) return;   // debug build only
    bf16 *S = static_cast<bf16 *>(a.state) + ((size_t)slot * HV + hv) * (size_t)V * K;
    const uint32_t es = sizeof(Tin);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        zero_flag = 0;
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar, kBsTileBytes + 3u * 128u * es);
        bulk_g2s_hint(st, S, kBsTileBytes, &bar, policy_evict_first());
        bulk_g2s(st + kBsTileBytes, static_cast<const Tin *>(a.q) + (size_t)b * a.q_stride + (size_t)h * K, 128u * es, &bar);
        bulk_g2s(st + kBsTileBytes + 128u * es, static_cast<const Tin *>(a.k) + (size_t)b * a.k_stride + (size_t)h * K,
                 128u * es, &bar);
        bulk_g2s(st + kBsTileBytes + 256u * es, static_cast<const Tin *>(a.v) + (size_t)b * a.v_stride + (size_t)hv * V,
                 128u * es, &bar);
    }
    float g, beta;
    step_gates<Tin>(a, b, hv, g, beta);
    const float e = expf(g);
    __syncthreads();   // the barrier is initialised before anyone waits on it
    if (!mbar_wait_warp(&bar, 0u, &abort_flag, kBsWaitLimit)) {
        if (lane == 0) raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
        // the copies may still be in flight: thread 0 waits (bounded) for them before the CTA exits
        if (threadIdx.x == 0) mbar_wait(&bar, 0u, &zero_flag, kBsWaitLimit);
        return;
    }
    const bf16 *Ss = reinterpret_cast<const bf16 *>(st);
    const Tin *qs = reinterpret_cast<const Tin *>(st + kBsTileBytes);
    const Tin *ks = reinterpret_cast<const Tin *>(st + kBsTileBytes + 128u * es);
    const Tin *vs = reinterpret_cast<const Tin *>(st + kBsTileBytes + 256u * es);
    float2 kh[4], qh[4];
    lds8(ks + col, kh);
    lds8(qs + col, qh);
    {
        const bool l2 = a.use_qk_l2norm != 0;
        const float sk = group_sum<16>(dot8(kh, kh));
        const float sq = group_sum<16>(dot8(qh, qh));
        const float rk = l2 ? rsqrtf(sk + 1e-6f) : 1.0f;
        const float rq = (l2 ? rsqrtf(sq + 1e-6f) : 1.0f) * P.scale;
        const float2 rk2 = make_float2(rk, rk), rq2 = make_float2(rq, rq);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            kh[c] = __fmul2_rn(kh[c], rk2);
            qh[c] = __fmul2_rn(qh[c], rq2);
        }
    }
    const float kq = group_sum<16>(dot8(kh, qh));
    const float2 e2 = make_float2(e, e);
    float dh0 = 0.f, dh1 = 0.f;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float x[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 sv[4];
            lds8(Ss + (size_t)(rbase + 2 * (4 * hh + i)) * K + col, sv);
            x[i] = dot8(sv, kh);
            x[4 + i] = dot8(sv, qh);
        }
        bp_reduce<8, 8>(x, lane);
        const int r_own = rbase + 2 * (4 * hh + ((sub >> 1) & 3));
        const float d = sub < 8 && r_own < V ? beta * (to_f32(vs[r_own]) - e * x[0]) : 0.f;
        const float d_lo = __shfl_xor_sync(kFull, d, 8);
        if (sub >= 8 && (sub & 1) == 0 && r_own < V) store_out(a.out, a.out_dtype, out_base + r_own, fmaf(d_lo, kq, e * x[0]));
        if (hh == 0) dh0 = d; else dh1 = d;
    }
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        const float d = hh == 0 ? dh0 : dh1;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float di = __shfl_sync(kFull, d, (lane & 16) + 2 * i);
            const float2 d2 = make_float2(di, di);
            const int r = rbase + 2 * (4 * hh + i);
            float2 sv[4];
            lds8(Ss + (size_t)r * K + col, sv);
            uint32_t w[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 nv = __ffma2_rn(d2, kh[c], __fmul2_rn(e2, sv[c]));   // fmaf(d, k, e s) per element
                w[c] = pack_bf16x2(nv.x, nv.y);
            }
            if (r < V) __stcs(reinterpret_cast<uint4 *>(S + (size_t)r * K + col), make_uint4(w[0], w[1], w[2], w[3]));
        }
    }
}

int launch_step_stage_bf16(const StepLaunch &p, cudaStream_t stream)
{
    const unsigned tiles = (unsigned)p.a.B * (unsigned)p.a.HV;
    if (p.a.in_dtype == GDN_BF16)
        step_stage_bf16_kernel<bf16><<<tiles, 256, 0, stream>>>(p);
    else
        step_stage_bf16_kernel<float><<<tiles, 256, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

bool step_stage_bf16_ok(const gdn_step_args &a)
{
    auto al16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    const int64_t es = a.in_dtype == GDN_BF16 ? 2 : 4;
    return a.state_dtype == GDN_BF16 && a.K == 128 && a.V == 128 && al16(a.state) && al16(a.q) &&
           al16(a.k) && al16(a.v) && (a.q_stride * es) % 16 == 0 && (a.k_stride * es) % 16 == 0 &&
           (a.v_stride * es) % 16 == 0;
}

}  // namespace gdn
