// fused_kernel.cu -- one launch for the fused decode (gdn_decode_fused):
//   (1) width-4 causal conv1d update with SiLU on the head's q, k and v channels; the conv
//       state is shifted in place (tap 0 oldest, tap 3 = the current input);
//   (2) the delta-rule step with one log-decay per key channel (KDA) or per head (GDN gate),
//       beta = sigmoid(raw_beta), in-kernel q/k L2 norm and q scale;
//   (3) the gated RMSNorm out = o / sqrt(mean(o^2) + eps) * w * act(gate), stored as bf16.
// One CTA per (token t, head h): the conv channels of a head belong to that CTA alone, so the
// in-place conv-state shift needs no synchronisation across CTAs, and the conv output, the
// step's output and the norm's statistics stay in shared memory. HBM traffic is the state tile
// in and out (64 KB each at head_dim 128) plus a few KB of inputs, conv state and output.
//
// Sources: "Microbenchmark for the fused Kimi-K3 KDA decode kernel on ROCm" (module docstring:
// conv update -> delta-rule step -> gated RMSNorm in one launch; class Inputs: shapes, the NULL
// slot 0, lower_bound -5; triton_chain: causal_conv1d_update with SiLU, the KDA packed decode with
// raw_g/raw_beta/A_log/dt_bias; _gated_rmsnorm); "Optimization Log: Qwen3.5-27B Dense on B200",
// "Kernel 2" (rmsnorm times silu(gate)) and "Kernel 5" (shift + insert + dot product + SiLU).
// The KDA decay formula is not printed on those pages; kda_gate_form selects one of two readings.
#include "gdn_chain.cuh"
#include "gdn_launch.h"
#include "gdn_tile.cuh"

namespace gdn {

__device__ __forceinline__ float bf(const void *p, size_t i)
{
    return __bfloat162float(static_cast<const bf16 *>(p)[i]);
}

// CHAIN: the instance for chained launches (gdn_decode_front), which waits for the kernel before it
// after its state loads. Ordinary launches run the other instance, which is launched with the same
// attribute but waits before it touches memory and only then lets the next kernel start
// (ordinary_launch_start), so consecutive calls hide each other's launch: on GB300 6.44 against
// 6.63 us at T = 1 and 8.59 against 8.74 at T = 2 (a wait after the state loads had made
// ordinary launches about 1% slower).
template <int D, bool CHAIN>
__global__ void __launch_bounds__(kThreads, 2) fused_kernel(const __grid_constant__ FusedLaunch P)
{
    using TL = Tile<D>;
    static_assert(TL::ROWS_PASS >= D, "one pass covers the tile");
    const gdn_fused_args &a = P.a;
    const int heads = a.heads;
    const int t_ = blockIdx.x / heads, h = blockIdx.x - t_ * heads;
    const size_t dim = (size_t)heads * D;
    bf16 *out = static_cast<bf16 *>(a.out) + ((size_t)t_ * heads + h) * D;

    __shared__ float qkv[3 * D];
    __shared__ float o_s[D];
    __shared__ float red[kWarps];

    if constexpr (CHAIN) grid_launch_dependents();
    else ordinary_launch_start();
    const int slot = a.state_indices[t_];
    const bool skip = slot == a.pad_slot_id || slot < 0 || slot >= a.num_slots;   // uniform over the CTA
    const bool out_of_range = !skip && !fused_tile_in_range(a, t_, h, slot);      // debug build only
    float *S = a.state + ((size_t)(skip ? 0 : slot) * heads + h) * (size_t)D * D;
    TL t;
    t.init();
    if (!skip && !out_of_range) t.load(S, D, 0);
    // In a chained layer call the previous kernel (the input projection) writes x and the gate
    // rows, never the state or the slot indices: the state tile is already in flight here.
    if constexpr (CHAIN) grid_dependency_wait();
    if (out_of_range) return;
    if (skip) {
        if (slot != a.pad_slot_id && threadIdx.x == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_INDEX);
        for (int r = threadIdx.x; r < D; r += kThreads) out[r] = __float2bfloat16_rn(0.f);
        return;
    }

    // (1) conv update of the 3*D channels of this head
    bf16 *cs = static_cast<bf16 *>(a.conv_state);
    for (int c = threadIdx.x; c < 3 * D; c += kThreads) {
        const int part = c / D, j = c - part * D;
        const size_t ch = part * dim + (size_t)h * D + j;
        const float xin = bf(a.x, (size_t)t_ * a.x_stride + ch);
        bf16 *cp = cs + (size_t)slot * a.cs_stride_slot + ch * a.cs_stride_chan;
        const bf16 x0 = cp[0], x1 = cp[a.cs_stride_tap], x2 = cp[2 * a.cs_stride_tap];
        const float4 w = *reinterpret_cast<const float4 *>(a.conv_w + ch * 4);
        float acc = w.x * __bfloat162float(x0);
        acc = fmaf(w.y, __bfloat162float(x1), acc);
        acc = fmaf(w.z, __bfloat162float(x2), acc);
        acc = fmaf(w.w, xin, acc);
        if (a.conv_b) acc += a.conv_b[ch];
        qkv[c] = acc * sigmoid_f(acc);
        cp[0] = x1;
        cp[a.cs_stride_tap] = x2;
        cp[2 * a.cs_stride_tap] = __float2bfloat16_rn(xin);
    }

    // (2) gates for this lane's four key columns
    float4 gk;
    const float A = expf(a.A_log[h]);
    if (a.gate_kind == GDN_FUSED_GATE_KDA) {
        const size_t gi = (size_t)t_ * a.raw_g_stride + (size_t)h * D + t.col;
        const float *db = a.dt_bias + (size_t)h * D + t.col;
        float gv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float xg = bf(a.raw_g, gi + c) + db[c];
            gv[c] = a.kda_gate_form == 0 ? fmaxf(a.lower_bound, -A * softplus_f(xg))
                                         : a.lower_bound * sigmoid_f(A * xg);
        }
        gk = make_float4(gv[0], gv[1], gv[2], gv[3]);
    } else {
        const float gv = -A * softplus_f(bf(a.raw_g, (size_t)t_ * a.raw_g_stride + h) + a.dt_bias[h]);
        gk = make_float4(gv, gv, gv, gv);
    }
    const float4 dec = make_float4(expf(gk.x), expf(gk.y), expf(gk.z), expf(gk.w));
    const float beta = sigmoid_f(bf(a.raw_beta, (size_t)t_ * a.raw_beta_stride + h));
    __syncthreads();

    const float4 q4 = *reinterpret_cast<const float4 *>(qkv + t.col);
    const float4 k4 = *reinterpret_cast<const float4 *>(qkv + D + t.col);
    const float4 kh = l2_normalise4<TL::LPR>(k4, a.use_qk_l2norm != 0, 1.f);
    const float4 qh = l2_normalise4<TL::LPR>(q4, a.use_qk_l2norm != 0, P.scale);
    const float kq = group_sum<TL::LPR>(dot4(kh, qh));
    const float4 kd = mul4(kh, dec), qd = mul4(qh, dec);

    float vv[TL::M];
#pragma unroll
    for (int m = 0; m < TL::M; ++m) {
        const int r = t.row(0, t.owned_chunk(m));
        vv[m] = (t.holds_k_dot() && r < D) ? qkv[2 * D + r] : 0.f;
    }
    float x[TL::N];
    t.partial_dots(kd, qd, x);
    t.reduce_scatter(x);
    float dv[TL::M];
#pragma unroll
    for (int m = 0; m < TL::M; ++m) dv[m] = beta * (vv[m] - x[m]);
#pragma unroll
    for (int m = 0; m < TL::M; ++m) {
        const float dq = t.delta_for_q(dv[m]);
        const int r = t.row(0, t.owned_chunk(m));
        if (!t.holds_k_dot() && r < D) o_s[r] = fmaf(dq, kq, x[m]);
    }
    t.update_store(S, D, 0, dec, kh, dv);
    __syncthreads();

    // (3) gated RMSNorm over the head's D outputs
    float sq = 0.f;
    for (int r = threadIdx.x; r < D; r += kThreads) sq = fmaf(o_s[r], o_s[r], sq);
    sq = group_sum<32>(sq);
    if (t.lane == 0) red[t.warp] = sq;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += red[w];
    const float rs = 1.0f / sqrtf(tot / D + a.norm_eps);
    const size_t gbase = (size_t)t_ * a.out_gate_stride + (size_t)h * D;
    for (int r = threadIdx.x; r < D; r += kThreads) {
        const float gt = bf(a.out_gate, gbase + r);
        const float act = a.gate_act == GDN_ACT_SILU ? gt * sigmoid_f(gt) : sigmoid_f(gt);
        out[r] = __float2bfloat16_rn(o_s[r] * rs * a.norm_w[r] * act);
    }
}

template <int D>
static int launch_fused_t(const FusedLaunch &p, cudaStream_t stream, bool chained)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)p.a.T * (unsigned)p.a.heads);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    set_programmatic(attr[cfg.numAttrs++]);   // the ordinary instance waits before it touches memory
    if (cudaLaunchKernelEx(&cfg, chained ? fused_kernel<D, true> : fused_kernel<D, false>, p) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

int launch_fused(const FusedLaunch &p, cudaStream_t stream, bool chained)
{
    switch (p.a.head_dim) {
    case 16: return launch_fused_t<16>(p, stream, chained);
    case 32: return launch_fused_t<32>(p, stream, chained);
    case 64: return launch_fused_t<64>(p, stream, chained);
    case 128: return launch_fused_t<128>(p, stream, chained);
    default: return GDN_ERR_SHAPE;
    }
}

}  // namespace gdn
