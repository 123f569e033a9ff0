// gdn_tile.cuh -- the per-tile machinery of the decode kernels (internal to libgdn_decode.so).
//
// One CTA of 8 warps owns one state tile S[V, K] (fp32, key index contiguous). A state row of K
// floats is read by LPR = K/4 lanes, one 16-byte vector each, so a warp instruction moves 512
// contiguous bytes. Every thread keeps R = 16 such vectors in registers: the tile is read from
// HBM once, both row dots (S.k and S.q) are taken from the registers, and the updated tile is
// written back from the same registers. Nothing of the tile is re-read.
//
// Step arithmetic (single pass over S). With the decay D = diag(exp(g_k)) (all equal for the
// per-head gate), S_bar = S D and the update S' = S_bar + delta k^T give
//     u     = S_bar k  = S (D k)
//     delta = beta (v - u)
//     o     = S' q     = S (D q) + delta (k . q)
//     S'    = S D + delta k^T
// so one read of S feeds both dots. This is the step of "Optimization Log: Qwen3.5-27B Dense on
// B200", section "Kernel 4: Fused DeltaNet Recurrent (FLAGSHIP)" (Math block: decay, S^T k,
// delta, rank-1 update, S^T q), regrouped; that page's two-pass design reads S twice.
#pragma once

#include "gdn_common.cuh"
#include "gdn_decode.h"

namespace gdn {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xFFFFFFFFu;

template <int K, int R_ = 16, int NW = kWarps>
struct Tile {
    static_assert(K == 16 || K == 32 || K == 64 || K == 128, "K must be 16, 32, 64 or 128");
    static constexpr int LPR = K / 4;               // lanes per state row
    static constexpr int RPI = 32 / LPR;            // rows per warp instruction
    static constexpr int R = R_;                    // 16-byte vectors per thread per pass
    static constexpr int N = 2 * R;                 // partial dots per thread (R for S.k, R for S.q)
    static constexpr int DUP = N >= LPR ? 1 : LPR / N;  // lanes left holding the same reduced dot
    static constexpr int M = N >= LPR ? N / LPR : 1;    // fully reduced dots per lane
    static constexpr int HALF = LPR / 2;            // lanes [0, HALF) of a row group end with S.k
    static constexpr int ROWS_WARP = R * RPI;
    static constexpr int ROWS_PASS = NW * ROWS_WARP;

    int lane, warp, sub, grp, col;
    float4 s[R];

    __device__ __forceinline__ void init(int warp_index = threadIdx.x >> 5)
    {
        lane = threadIdx.x & 31;
        warp = warp_index;
        sub = lane % LPR;
        grp = lane / LPR;
        col = sub * 4;
    }

    // state row held in vector i of the pass that starts at row0
    __device__ __forceinline__ int row(int row0, int i) const
    {
        return row0 + warp * ROWS_WARP + i * RPI + grp;
    }

    // chunk index whose reduced dot this lane holds in slot m (see reduce_scatter)
    __device__ __forceinline__ int owned_chunk(int m) const { return ((sub % HALF) / DUP) * M + m; }
    __device__ __forceinline__ bool holds_k_dot() const { return sub < HALF; }
    // one lane of each group of DUP identical lanes writes the row's results
    __device__ __forceinline__ bool writer() const { return (sub % DUP) == 0; }

    template <typename TS>
    __device__ __forceinline__ void load(const TS *tile, int V, int row0)
    {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = row(row0, i);
            s[i] = r < V ? ld_stream(tile + (size_t)r * K + col) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    // x[i] = S_i . kd, x[R + i] = S_i . qd over this lane's four columns
    __device__ __forceinline__ void partial_dots(float4 kd, float4 qd, float (&x)[N]) const
    {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            x[i] = dot4(s[i], kd);
            x[R + i] = dot4(s[i], qd);
        }
    }

    // Butterfly reduce-scatter over the LPR lanes of a row group: at offset o a lane keeps one
    // half of its values and adds the partner's copy of that half. After the halving steps lane
    // `sub` holds the complete sums of indices (sub/DUP)*M .. (sub/DUP)*M + M-1 in x[0 .. M);
    // when there are fewer values than lanes (DUP > 1) the last steps are plain butterflies and
    // DUP neighbouring lanes end with the same sums. That is about N shuffles per lane instead of
    // N * log2(LPR) for N separate reductions.
    __device__ __forceinline__ void reduce_scatter(float (&x)[N]) const { rs_step<LPR / 2, N>(x); }

    // one butterfly step at lane offset O with NN live values (compile-time, fully unrolled)
    template <int O, int NN>
    __device__ __forceinline__ void rs_step(float (&x)[N]) const
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
                rs_step<O / 2, NN / 2>(x);
            } else {
                x[0] += __shfl_xor_sync(kFull, x[0], O);
                rs_step<O / 2, 1>(x);
            }
        }
    }

    // delta of chunk i (the value sits on lane grp*LPR + (i/M)*DUP, slot i%M)
    __device__ __forceinline__ float delta_of(const float (&dv)[M], int i) const
    {
        return __shfl_sync(kFull, dv[i % M], (lane & ~(LPR - 1)) + (i / M) * DUP);
    }

    // upper lanes receive the delta of the lower lane that owns the same chunk
    __device__ __forceinline__ float delta_for_q(float dm) const
    {
        return __shfl_up_sync(kFull, dm, HALF);
    }

    // S' = S * dec + delta k^T, written back with streaming stores (rounded for a bf16 state)
    template <typename TS>
    __device__ __forceinline__ void update_store(TS *tile, int V, int row0, float4 dec,
                                                 float4 kh, const float (&dv)[M])
    {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float d = delta_of(dv, i);
            const int r = row(row0, i);
            if (r < V) st_stream(tile + (size_t)r * K + col, decay_update4(dec, s[i], d, kh));
        }
    }
};

// L2 normalisation of the q/k head held in four-element chunks by every row group of a warp:
// returns x / sqrt(|x|^2 + eps) * s (or x * s when disabled).
template <int LPR>
__device__ __forceinline__ float4 l2_normalise4(float4 x, bool enabled, float s)
{
    const float ss = group_sum<LPR>(dot4(x, x));
    const float r = enabled ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    return scale4(x, r * s);
}

__device__ __forceinline__ void store_out(void *out, int dtype, size_t i, float x)
{
    if (dtype == GDN_BF16)
        static_cast<bf16 *>(out)[i] = __float2bfloat16_rn(x);
    else
        static_cast<float *>(out)[i] = x;
}

// Debug build: the buffers one step tile (request row b, value head hv, q/k head h, state slot)
// reads and writes lie inside the extents its arguments describe: the state tile, the q, k and v
// rows, the gate inputs and the output row. A failed check has raised GDN_DEVERR_RANGE and the
// caller skips the tile. The release build compiles this to the constant true.
__device__ __forceinline__ bool step_tile_in_range(const gdn_step_args &a, int b, int hv, int h, int slot)
{
#ifdef GDN_DEBUG
    const long long VK = (long long)a.V * a.K, B1 = (long long)a.B - 1;
    bool ok = GDN_IN(a.err_flags, ((long long)slot * a.HV + hv) * VK + VK - 1, (long long)a.num_slots * a.HV * VK);
    ok = ok && GDN_IN(a.err_flags, (long long)b * a.q_stride + (long long)(h + 1) * a.K - 1, B1 * a.q_stride + (long long)a.H * a.K);
    ok = ok && GDN_IN(a.err_flags, (long long)b * a.k_stride + (long long)(h + 1) * a.K - 1, B1 * a.k_stride + (long long)a.H * a.K);
    ok = ok && GDN_IN(a.err_flags, (long long)b * a.v_stride + (long long)(hv + 1) * a.V - 1, B1 * a.v_stride + (long long)a.HV * a.V);
    ok = ok && GDN_IN(a.err_flags, (long long)b * a.HV + hv, (long long)a.B * a.HV);
    ok = ok && GDN_IN(a.err_flags, ((long long)b * a.HV + hv + 1) * a.V - 1, (long long)a.B * a.HV * a.V);
    return ok;
#else
    (void)a;
    return true;
#endif
}

// Debug build: the ring records of a tile at cursor p lie inside the rings (d_cache [slots, HV,
// L, V], k_cache [slots, H, L, K], g_cache [slots, HV, L]).
__device__ __forceinline__ bool ring_in_range(const gdn_step_args &a, int L, int slot, int hv, int h, int p)
{
#ifdef GDN_DEBUG
    bool ok = GDN_IN(a.err_flags, p, L);
    ok = ok && GDN_IN(a.err_flags, (((long long)slot * a.HV + hv) * L + p + 1) * a.V - 1, (long long)a.num_slots * a.HV * L * a.V);
    ok = ok && GDN_IN(a.err_flags, (((long long)slot * a.H + h) * L + p + 1) * a.K - 1, (long long)a.num_slots * a.H * L * a.K);
    ok = ok && GDN_IN(a.err_flags, ((long long)slot * a.HV + hv) * L + p, (long long)a.num_slots * a.HV * L);
    return ok;
#else
    (void)a;
    return true;
#endif
}

// Debug build: the buffers one fused tile (token t, head h, slot) reads and writes lie inside the
// extents its arguments describe: the state tile, the conv state of the head's q, k and v channels
// (all three taps), the x row, the output gate, raw_g, raw_beta, dt_bias and the output row.
__device__ __forceinline__ bool fused_tile_in_range(const gdn_fused_args &a, int t, int h, int slot)
{
#ifdef GDN_DEBUG
    const long long D = a.head_dim, dim = (long long)a.heads * D, T1 = (long long)a.T - 1;
    bool ok = GDN_IN(a.err_flags, (((long long)slot * a.heads + h + 1) * D) * D - 1, (long long)a.num_slots * a.heads * D * D);
    const long long cs_end = (long long)(a.num_slots - 1) * a.cs_stride_slot + (3 * dim - 1) * a.cs_stride_chan +
                             2 * a.cs_stride_tap + 1;
    for (int part = 0; part < 3; ++part) {
        const long long c0 = part * dim + (long long)h * D;
        ok = ok && GDN_IN(a.err_flags, slot * a.cs_stride_slot + c0 * a.cs_stride_chan, cs_end);
        ok = ok && GDN_IN(a.err_flags, slot * a.cs_stride_slot + (c0 + D - 1) * a.cs_stride_chan + 2 * a.cs_stride_tap, cs_end);
    }
    ok = ok && GDN_IN(a.err_flags, t * a.x_stride + 2 * dim + (h + 1) * D - 1, T1 * a.x_stride + 3 * dim);
    ok = ok && GDN_IN(a.err_flags, t * a.out_gate_stride + (h + 1) * D - 1, T1 * a.out_gate_stride + dim);
    ok = ok && GDN_IN(a.err_flags, t * a.raw_beta_stride + h, T1 * a.raw_beta_stride + a.heads);
    if (a.gate_kind == GDN_FUSED_GATE_KDA) {
        ok = ok && GDN_IN(a.err_flags, t * a.raw_g_stride + (h + 1) * D - 1, T1 * a.raw_g_stride + dim);
        ok = ok && GDN_IN(a.err_flags, (h + 1) * D - 1, dim);
    } else {
        ok = ok && GDN_IN(a.err_flags, t * a.raw_g_stride + h, T1 * a.raw_g_stride + a.heads);
    }
    ok = ok && GDN_IN(a.err_flags, ((long long)t * a.heads + h + 1) * D - 1, (long long)a.T * dim);
    return ok;
#else
    (void)a;
    return true;
#endif
}

// g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b) (raw mode) or the given values
template <typename Tin>
__device__ __forceinline__ void step_gates(const gdn_step_args &a, int b, int hv, float &g,
                                           float &beta)
{
    const size_t gi = (size_t)b * a.HV + hv;
    if (a.gate_mode == GDN_GATE_RAW) {
        const float av = to_f32(static_cast<const Tin *>(a.a)[gi]);
        const float bv = to_f32(static_cast<const Tin *>(a.b)[gi]);
        g = -expf(a.A_log[hv]) * softplus_f(av + a.dt_bias[hv]);
        beta = sigmoid_f(bv);
    } else {
        g = a.g[gi];
        beta = a.beta[gi];
    }
}

}  // namespace gdn
