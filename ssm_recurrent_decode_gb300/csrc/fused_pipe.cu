// fused_pipe.cu -- the fused decode (conv update -> delta step -> gated RMSNorm) as a persistent,
// warp-specialised kernel for head_dim 128.
//
// Same arithmetic as fused_kernel.cu, organised like buffered_pipe.cu so that HBM streams
// continuously: one CTA per SM with a producer warp and two groups of 8 consumer warps that take
// alternate (token, head) tiles. For each tile the producer moves, with 1-D bulk copies into a
// shared-memory stage: the 64 KB state tile, the head's q/k/v input channels of x (3 x 256 B), its
// conv state (the "DS" layout as 3 runs of 768 B, the "SD" layout as 9 runs of 256 B), the KDA
// gate inputs (raw_g row, dt_bias row) and the output-gate row; slot, beta and the per-head decay
// come from a batched scalar prefetch (32 tiles per global round trip). The conv weights of a
// tile are requested (read-only path, L2-resident) before its stage is waited for. Within a group, two mbarriers order
// conv outputs -> step and step -> RMSNorm. Every wait is bounded; a timeout sets
// GDN_DEVERR_TIMEOUT and stops the CTA (the producer then waits, bounded, for its copies).
//
// Sources: "Microbenchmark for the fused Kimi-K3 KDA decode kernel on ROCm" (module docstring,
// Inputs, triton_chain, _gated_rmsnorm, fused); "Optimization Log: Qwen3.5-27B Dense on B200",
// Kernel 2, Kernel 4 and Kernel 5.
#include "gdn_chain.cuh"
#include "gdn_launch.h"
#include "gdn_pipe.cuh"
#include "gdn_tile.cuh"

namespace gdn {

constexpr int kFGW = 8;                       // warps of one consumer group
constexpr int kFGroups = 2;
constexpr int kFCW = kFGW * kFGroups;
constexpr int kFThreads = (kFCW + 1) * 32;
constexpr long long kFWaitLimit = 1LL << 31;  // SM clock cycles, about one second

struct FusedMeta {
    int status;       // 0 run, 1 pad row, 2 bad slot, 3 an index out of range (debug build)
    int slot;
    float beta;
    float g_head;     // GDN gate: the head's log-decay
    float A;          // exp(A_log[h]) for the KDA gate
};

// byte offsets in one stage
struct FusedLayout {
    static constexpr uint32_t x = 128u * 128u * 4u;   // after the state tile
    static constexpr uint32_t cs = x + 3u * 256u;      // conv state, 3 x 128 channels x 3 taps bf16
    static constexpr uint32_t rg = cs + 2304u;         // raw_g row (bf16 x 128)
    static constexpr uint32_t db = rg + 256u;          // dt_bias row (fp32 x 128)
    static constexpr uint32_t og = db + 512u;          // output gate row (bf16 x 128)
    static constexpr uint32_t meta = og + 256u;
    static constexpr uint32_t stage = (meta + (uint32_t)sizeof(FusedMeta) + 127u) & ~127u;
};

// a . b over four elements as two fp32 pairs (fma.rn.f32x2: the same rounding per element as the
// scalar operations, half the instructions)
__device__ __forceinline__ float dot4_pairs(float4 a, float4 b)
{
    float2 p = __fmul2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y));
    p = __ffma2_rn(make_float2(a.z, a.w), make_float2(b.z, b.w), p);
    return p.x + p.y;
}

// dec * s + d * k elementwise, as two fp32 pairs
__device__ __forceinline__ float4 decay_update_pairs(float4 dec, float4 s, float d, float4 k)
{
    const float2 d2 = make_float2(d, d);
    const float2 lo = __ffma2_rn(d2, make_float2(k.x, k.y), __fmul2_rn(make_float2(dec.x, dec.y), make_float2(s.x, s.y)));
    const float2 hi = __ffma2_rn(d2, make_float2(k.z, k.w), __fmul2_rn(make_float2(dec.z, dec.w), make_float2(s.z, s.w)));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ float bfs(const unsigned char *base, uint32_t off, int i)
{
    return __bfloat162float(reinterpret_cast<const bf16 *>(base + off)[i]);
}

template <bool SD>
__global__ void __launch_bounds__(kFThreads, 1) fused_pipe_kernel(const __grid_constant__ FusedLaunch P)
{
    constexpr int D = 128;
    using TR = Tile<128, 8, kFGW>;   // one 8-row chunk: 16 dots over 32 lanes, 2 lanes per result
    using FL = FusedLayout;
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ float ysm[kFGroups][3 * D];      // conv outputs q | k | v of the group's tile
    __shared__ __align__(16) float decsm[kFGroups][D];   // per-key decays exp(g_k) of the group's tile (KDA)
    __shared__ float red[kFGroups][2][kFGW];    // per-warp sums of o^2 (double-buffered)
    __shared__ __align__(8) uint64_t gbar[kFGroups][2];   // group syncs: conv -> step, o^2 -> norm
    __shared__ int abort_flag;
    __shared__ int zero_flag;

    const gdn_fused_args &a = P.a;
    const int heads = a.heads, T = a.T, NST = 3;
    const int ntiles = T * heads;
    const size_t dim = (size_t)heads * D;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + (size_t)NST * FL::stage);
    uint64_t *empty = full + NST;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    bf16 *const cstate = static_cast<bf16 *>(a.conv_state);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 32);
            mbar_init(&empty[s], kFGW);
        }
        for (int g = 0; g < kFGroups; ++g) {
            mbar_init(&gbar[g][0], kFGW);
            mbar_init(&gbar[g][1], kFGW);
        }
        abort_flag = 0;
        zero_flag = 0;
        fence_barrier_init();
    }
    grid_launch_dependents();
    grid_dependency_wait();   // in a chained layer call x and the gate rows are the previous kernel's output
    __syncthreads();

    if (warp == kFCW) {
        // ---------------------------------------------------------------- producer warp
        const uint64_t pol = policy_evict_first();
        int n = 0;
        bool stop = false;
        for (int base = blockIdx.x; base < ntiles && !stop; base += 32 * gridDim.x) {
            const int my_tile = base + lane * gridDim.x;
            int my_slot = 0, my_status = 1;
            float my_beta = 0.f, my_g = 0.f, my_A = 0.f;
            if (my_tile < ntiles) {
                const int t = my_tile / heads, h = my_tile - t * heads;
                my_slot = a.state_indices[t];
                my_status = my_slot == a.pad_slot_id ? 1 : (my_slot < 0 || my_slot >= a.num_slots) ? 2 : 0;
                if (my_status == 0 && !fused_tile_in_range(a, t, h, my_slot)) my_status = 3;   // debug build
                my_beta = sigmoid_f(__bfloat162float(static_cast<const bf16 *>(a.raw_beta)[(size_t)t * a.raw_beta_stride + h]));
                my_A = expf(a.A_log[h]);
                if (a.gate_kind == GDN_FUSED_GATE_GDN)
                    my_g = -my_A * softplus_f(__bfloat162float(static_cast<const bf16 *>(a.raw_g)[(size_t)t * a.raw_g_stride + h]) + a.dt_bias[h]);
            }
            for (int i = 0; i < 32; ++i) {
                const int tile = base + i * gridDim.x;
                if (tile >= ntiles) break;
                const int st = n % NST;
                const uint32_t ph = (uint32_t)(n / NST) & 1u;
                if (n >= NST && !mbar_wait_warp(&empty[st], ph ^ 1u, &abort_flag, kFWaitLimit)) {
                    if (lane == 0) {
                        *(volatile int *)&abort_flag = 1;
                        raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
                    }
                    stop = true;
                    break;
                }
                const int slot = __shfl_sync(kFull, my_slot, i);
                const int status = __shfl_sync(kFull, my_status, i);
                const float beta = __shfl_sync(kFull, my_beta, i);
                const float gh = __shfl_sync(kFull, my_g, i);
                const float A = __shfl_sync(kFull, my_A, i);
                ++n;
                if (lane != 0) {
                    mbar_arrive(&full[st]);
                    continue;
                }
                unsigned char *stage = sm + (size_t)st * FL::stage;
                FusedMeta *meta = reinterpret_cast<FusedMeta *>(stage + FL::meta);
                meta->status = status;
                meta->slot = slot;
                meta->beta = beta;
                meta->g_head = gh;
                meta->A = A;
                const bool kda = a.gate_kind == GDN_FUSED_GATE_KDA;
                const uint32_t bytes = status == 0 ? 65536u + 768u + 2304u + 256u + (kda ? 256u + 512u : 0u) : 0u;
                fence_proxy_async();
                mbar_arrive_expect_tx(&full[st], bytes);
                if (status == 0) {
                    const int t = tile / heads, h = tile - t * heads;
                    const float *S = a.state + ((size_t)slot * heads + h) * (size_t)(D * D);
                    bulk_g2s_hint(stage, S, 65536u, &full[st], pol);
                    const bf16 *xr = static_cast<const bf16 *>(a.x) + (size_t)t * a.x_stride + (size_t)h * D;
                    const bf16 *csr = cstate + (size_t)slot * a.cs_stride_slot;
                    for (int part = 0; part < 3; ++part) {
                        bulk_g2s(stage + FL::x + part * 256u, xr + part * dim, 256u, &full[st]);
                        const size_t ch0 = part * dim + (size_t)h * D;
                        if (SD) {
                            for (int tap = 0; tap < 3; ++tap)
                                bulk_g2s(stage + FL::cs + (part * 3 + tap) * 256u, csr + ch0 + tap * a.cs_stride_tap, 256u, &full[st]);
                        } else {
                            bulk_g2s(stage + FL::cs + part * 768u, csr + ch0 * 3, 768u, &full[st]);
                        }
                    }
                    bulk_g2s(stage + FL::og, static_cast<const bf16 *>(a.out_gate) + (size_t)t * a.out_gate_stride + (size_t)h * D, 256u, &full[st]);
                    if (kda) {
                        bulk_g2s(stage + FL::rg, static_cast<const bf16 *>(a.raw_g) + (size_t)t * a.raw_g_stride + (size_t)h * D, 256u, &full[st]);
                        bulk_g2s(stage + FL::db, a.dt_bias + (size_t)h * D, 512u, &full[st]);
                    }
                }
            }
        }
        if (*(volatile int *)&abort_flag) {
            for (int back = 1; back <= NST && n - back >= 0; ++back) {
                const int m = n - back;
                mbar_wait(&full[m % NST], (uint32_t)(m / NST) & 1u, &zero_flag, kFWaitLimit);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumer groups
    const int group = warp / kFGW, gwarp = warp - group * kFGW;
    const int tid = threadIdx.x - group * kFGW * 32;   // 0 .. 255
    TR t;
    t.init(gwarp);
    const int row0 = gwarp * 16;                       // this warp's 16 consecutive rows
    // after a chunk's reduce-scatter, lanes 2i and 2i+1 (and 16+2i, 17+2i) hold row 8c+i
    const int rsub = (t.sub % 16) / 2;
    float w_norm[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) w_norm[c] = a.norm_w[row0 + 8 * c + rsub];
    float *ys = ysm[group];
    const bool kda = a.gate_kind == GDN_FUSED_GATE_KDA;

    // conv weights of a tile's channels (this thread's channels tid and tid + 256)
    auto load_w = [&](int tile, float4 (&w)[2]) {
        const int h = tile % heads;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c = tid + u * 256;
            if (c < 3 * D && tile < ntiles) {
                const int part = c / D, j = c - part * D;
                w[u] = __ldg(reinterpret_cast<const float4 *>(a.conv_w + (part * dim + (size_t)h * D + j) * 4));
            }
        }
    };
    const int first = blockIdx.x + group * gridDim.x;

    int n = group, lt = 0;
    for (int tile = first; tile < ntiles; tile += kFGroups * gridDim.x, n += kFGroups) {
        // the tile's conv weights are requested before waiting for its stage
        float4 w_cur[2];
        load_w(tile, w_cur);
        const int st = n % NST;
        const uint32_t ph = (uint32_t)(n / NST) & 1u;
        // wait for the previous use of the stage to be released first (the groups alternate)
        if ((n >= NST && !mbar_wait_warp(&empty[st], ph ^ 1u, &abort_flag, kFWaitLimit)) ||
            !mbar_wait_warp(&full[st], ph, &abort_flag, kFWaitLimit)) {
            if (lane == 0) {
                *(volatile int *)&abort_flag = 1;
                raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
            }
            break;
        }
        const unsigned char *stage = sm + (size_t)st * FL::stage;
        const FusedMeta *meta = reinterpret_cast<const FusedMeta *>(stage + FL::meta);
        const int status = meta->status, slot = meta->slot;
        const int tt = tile / heads, h = tile - tt * heads;
        bf16 *out = static_cast<bf16 *>(a.out) + ((size_t)tt * heads + h) * D;
        if (status != 0) {
            if (status == 2 && tid == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_INDEX);
            if (status != 3 && tid < D) out[tid] = __float2bfloat16_rn(0.f);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            continue;
        }
        const uint32_t gp = (uint32_t)lt & 1u;
        ++lt;

        // (1) conv update of the head's 3 x 128 channels
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c = tid + u * 256;
            if (c < 3 * D) {
                const int part = c / D, j = c - part * D;
                float x0, x1, x2;
                if (SD) {
                    x0 = bfs(stage, FL::cs, (part * 3 + 0) * D + j);
                    x1 = bfs(stage, FL::cs, (part * 3 + 1) * D + j);
                    x2 = bfs(stage, FL::cs, (part * 3 + 2) * D + j);
                } else {
                    x0 = bfs(stage, FL::cs, part * 3 * D + j * 3 + 0);
                    x1 = bfs(stage, FL::cs, part * 3 * D + j * 3 + 1);
                    x2 = bfs(stage, FL::cs, part * 3 * D + j * 3 + 2);
                }
                const float xin = bfs(stage, FL::x, part * D + j);
                const float4 w = w_cur[u];
                float acc = w.x * x0;
                acc = fmaf(w.y, x1, acc);
                acc = fmaf(w.z, x2, acc);
                acc = fmaf(w.w, xin, acc);
                const size_t ch = part * dim + (size_t)h * D + j;
                if (a.conv_b) acc += a.conv_b[ch];
                ys[c] = acc * sigmoid_f(acc);
                bf16 *cp = cstate + (size_t)slot * a.cs_stride_slot + ch * a.cs_stride_chan;
                cp[0] = __float2bfloat16_rn(x1);
                cp[a.cs_stride_tap] = __float2bfloat16_rn(x2);
                cp[2 * a.cs_stride_tap] = __float2bfloat16_rn(xin);
            }
        }
        // (2) the KDA per-key decays, once per tile: threads 128..255 (one conv channel each above)
        // take one key column each; the other warps read them after the group barrier. (Each warp
        // computing all 128 itself cost 1.5-1.9k of a tile's 9k cycles per group at T = 8; with
        // fp32-pair dots and updates the call took 20.37 against 20.61 us, T = 4: 13.47 against
        // 13.86, as the other phases, which share the SM with the second group, took up the rest.)
        if (kda && tid >= 128) {
            const int col = tid - 128;
            const float xg = bfs(stage, FL::rg, col) + reinterpret_cast<const float *>(stage + FL::db)[col];
            const float gv = a.kda_gate_form == 0 ? fmaxf(a.lower_bound, -meta->A * softplus_f(xg))
                                                  : a.lower_bound * sigmoid_f(meta->A * xg);
            decsm[group][col] = expf(gv);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&gbar[group][0]);

        const float beta = meta->beta;
        float gate[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) gate[c] = bfs(stage, FL::og, row0 + 8 * c + rsub);
        if (!mbar_wait_warp(&gbar[group][0], gp, &abort_flag, kFWaitLimit)) {
            if (lane == 0) {
                *(volatile int *)&abort_flag = 1;
                raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
            }
            break;
        }
        float4 dec;
        if (kda) {
            dec = *reinterpret_cast<const float4 *>(&decsm[group][t.col]);
        } else {
            const float e = expf(meta->g_head);
            dec = make_float4(e, e, e, e);
        }

        // (3) the step, both dots straight from the staged tile, eight rows at a time
        const float4 kh = l2_normalise4<32>(*reinterpret_cast<const float4 *>(ys + D + t.col), a.use_qk_l2norm != 0, 1.f);
        const float4 qh = l2_normalise4<32>(*reinterpret_cast<const float4 *>(ys + t.col), a.use_qk_l2norm != 0, P.scale);
        const float kq = group_sum<32>(dot4(kh, qh));
        const float *Ss = reinterpret_cast<const float *>(stage);
        float dvc0 = 0.f, dvc1 = 0.f, oc0 = 0.f, oc1 = 0.f;
        {
            const float4 kd = mul4(kh, dec), qd = mul4(qh, dec);
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                float x[TR::N];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 srow = *reinterpret_cast<const float4 *>(Ss + (size_t)(row0 + 8 * c + i) * D + t.col);
                    x[i] = dot4_pairs(srow, kd);
                    x[8 + i] = dot4_pairs(srow, qd);
                }
                t.reduce_scatter(x);
                const float vv = t.holds_k_dot() ? ys[2 * D + row0 + 8 * c + rsub] : 0.f;
                const float d = beta * (vv - x[0]);   // lanes [0, 16)
                const float dq = __shfl_up_sync(kFull, d, 16);
                const float o = fmaf(dq, kq, x[0]);  // lanes [16, 32)
                if (c == 0) {
                    dvc0 = d;
                    oc0 = o;
                } else {
                    dvc1 = d;
                    oc1 = o;
                }
            }
        }
        {
            float *S = a.state + ((size_t)slot * heads + h) * (size_t)(D * D);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float d = __shfl_sync(kFull, c == 0 ? dvc0 : dvc1, 2 * i);
                    const float4 srow = *reinterpret_cast<const float4 *>(Ss + (size_t)(row0 + 8 * c + i) * D + t.col);
                    st_stream(S + (size_t)(row0 + 8 * c + i) * D + t.col, decay_update_pairs(dec, srow, d, kh));
                }
            }
        }
        // the warp's share of sum(o^2) (one lane per row), then the stage is no longer needed
        const bool owner = !t.holds_k_dot() && (t.sub & 1) == 0;
        float sq = owner ? oc0 * oc0 + oc1 * oc1 : 0.f;
        sq = group_sum<32>(sq);
        if (lane == 0) red[group][gp][gwarp] = sq;
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[st]);
            mbar_arrive(&gbar[group][1]);
        }
        if (!mbar_wait_warp(&gbar[group][1], gp, &abort_flag, kFWaitLimit)) {
            if (lane == 0) {
                *(volatile int *)&abort_flag = 1;
                raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
            }
            break;
        }
        // (4) gated RMSNorm over the head's 128 outputs
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kFGW; ++w) tot += red[group][gp][w];
        const float rs = 1.0f / sqrtf(tot / D + a.norm_eps);
        if (owner) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float act = a.gate_act == GDN_ACT_SILU ? gate[c] * sigmoid_f(gate[c]) : sigmoid_f(gate[c]);
                out[row0 + 8 * c + rsub] = __float2bfloat16_rn((c == 0 ? oc0 : oc1) * rs * w_norm[c] * act);
            }
        }
    }
}

static size_t fused_pipe_smem() { return 3 * (size_t)FusedLayout::stage + 2 * 3 * sizeof(uint64_t); }

bool fused_pipe_fits(int max_smem) { return fused_pipe_smem() + 8192 <= (size_t)max_smem; }

int launch_fused_pipe(const FusedLaunch &p, bool sd, cudaStream_t stream, bool chained)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const size_t smem = fused_pipe_smem();
    auto kern = sd ? fused_pipe_kernel<true> : fused_pipe_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int tiles = p.a.T * p.a.heads;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms));
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    if (chained) set_programmatic(attr[cfg.numAttrs++]);
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return GDN_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}


// ------------------------------------------------------------------------------------------------
// One (token, head) tile per CTA of 256 threads with the same staging: thread 0 bulk-copies the
// state tile and the conv-state rows (neither is written by a chained launch's previous kernel),
// waits for that kernel, then copies x and the gate rows; all threads compute the tile's scalars
// meanwhile. The arithmetic is the consumer group's above, with block barriers in place of the
// group's mbarriers. 68 KB of shared memory per CTA: three CTAs per SM.
// ------------------------------------------------------------------------------------------------
template <bool SD>
__global__ void __launch_bounds__(256, 3) fused_stage_kernel(const __grid_constant__ FusedLaunch P)
{
    constexpr int D = 128;
    using TR = Tile<128, 8, kFGW>;
    using FL = FusedLayout;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ float ys[3 * D];
    __shared__ float red[kFGW];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag, zero_flag;

    const gdn_fused_args &a = P.a;
    const int heads = a.heads;
    const size_t dim = (size_t)heads * D;
    const int tile = blockIdx.x, tt = tile / heads, h = tile - tt * heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    bf16 *const cstate = static_cast<bf16 *>(a.conv_state);
    bf16 *out = static_cast<bf16 *>(a.out) + ((size_t)tt * heads + h) * D;
    const bool kda = a.gate_kind == GDN_FUSED_GATE_KDA;

    grid_launch_dependents();
    const int slot = a.state_indices[tt];
    const bool skip = slot == a.pad_slot_id || slot < 0 || slot >= a.num_slots;   // uniform over the CTA
    const bool out_of_range = !skip && !fused_tile_in_range(a, tt, h, slot);      // debug build only
    if (skip || out_of_range) {
        grid_dependency_wait();
        if (skip && slot != a.pad_slot_id && tid == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_INDEX);
        if (skip && tid < D) out[tid] = __float2bfloat16_rn(0.f);
        return;
    }
    const uint64_t pol = policy_evict_first();
    const bf16 *csr = cstate + (size_t)slot * a.cs_stride_slot;
    if (tid == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        zero_flag = 0;
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar, 65536u + 768u + 2304u + 256u + (kda ? 256u + 512u : 0u));
        bulk_g2s_hint(stage, a.state + ((size_t)slot * heads + h) * (size_t)(D * D), 65536u, &bar, pol);
        for (int part = 0; part < 3; ++part) {
            const size_t ch0 = part * dim + (size_t)h * D;
            if (SD) {
                for (int tap = 0; tap < 3; ++tap)
                    bulk_g2s(stage + FL::cs + (part * 3 + tap) * 256u, csr + ch0 + tap * a.cs_stride_tap, 256u, &bar);
            } else {
                bulk_g2s(stage + FL::cs + part * 768u, csr + ch0 * 3, 768u, &bar);
            }
        }
        if (kda) bulk_g2s(stage + FL::db, a.dt_bias + (size_t)h * D, 512u, &bar);
    }
    // a chained launch: x and the gate rows may be the previous kernel's output
    grid_dependency_wait();
    if (tid == 0) {
        const bf16 *xr = static_cast<const bf16 *>(a.x) + (size_t)tt * a.x_stride + (size_t)h * D;
        for (int part = 0; part < 3; ++part) bulk_g2s(stage + FL::x + part * 256u, xr + part * dim, 256u, &bar);
        bulk_g2s(stage + FL::og, static_cast<const bf16 *>(a.out_gate) + (size_t)tt * a.out_gate_stride + (size_t)h * D, 256u, &bar);
        if (kda) bulk_g2s(stage + FL::rg, static_cast<const bf16 *>(a.raw_g) + (size_t)tt * a.raw_g_stride + (size_t)h * D, 256u, &bar);
    }
    // the tile's scalars, the conv weights of this thread's channels and the norm weights
    const float beta = sigmoid_f(__bfloat162float(static_cast<const bf16 *>(a.raw_beta)[(size_t)tt * a.raw_beta_stride + h]));
    const float A = expf(a.A_log[h]);
    float g_head = 0.f;
    if (!kda) g_head = -A * softplus_f(__bfloat162float(static_cast<const bf16 *>(a.raw_g)[(size_t)tt * a.raw_g_stride + h]) + a.dt_bias[h]);
    float4 w_cur[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c = tid + u * 256;
        if (c < 3 * D) {
            const int part = c / D, j = c - part * D;
            w_cur[u] = __ldg(reinterpret_cast<const float4 *>(a.conv_w + (part * dim + (size_t)h * D + j) * 4));
        }
    }
    TR t;
    t.init(warp);
    const int row0 = warp * 16;
    const int rsub = (t.sub % 16) / 2;
    float w_norm[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) w_norm[c] = a.norm_w[row0 + 8 * c + rsub];
    __syncthreads();   // the barrier is initialised before anyone waits on it
    if (!mbar_wait_warp(&bar, 0u, &abort_flag, kFWaitLimit)) {
        if (lane == 0) raise_flag(a.err_flags, GDN_DEVERR_TIMEOUT);
        if (tid == 0) mbar_wait(&bar, 0u, &zero_flag, kFWaitLimit);   // copies still in flight land first
        return;
    }

    // (1) conv update of the head's 3 x 128 channels
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c = tid + u * 256;
        if (c < 3 * D) {
            const int part = c / D, j = c - part * D;
            float x0, x1, x2;
            if (SD) {
                x0 = bfs(stage, FL::cs, (part * 3 + 0) * D + j);
                x1 = bfs(stage, FL::cs, (part * 3 + 1) * D + j);
                x2 = bfs(stage, FL::cs, (part * 3 + 2) * D + j);
            } else {
                x0 = bfs(stage, FL::cs, part * 3 * D + j * 3 + 0);
                x1 = bfs(stage, FL::cs, part * 3 * D + j * 3 + 1);
                x2 = bfs(stage, FL::cs, part * 3 * D + j * 3 + 2);
            }
            const float xin = bfs(stage, FL::x, part * D + j);
            const float4 w = w_cur[u];
            float acc = w.x * x0;
            acc = fmaf(w.y, x1, acc);
            acc = fmaf(w.z, x2, acc);
            acc = fmaf(w.w, xin, acc);
            const size_t ch = part * dim + (size_t)h * D + j;
            if (a.conv_b) acc += a.conv_b[ch];
            ys[c] = acc * sigmoid_f(acc);
            bf16 *cp = cstate + (size_t)slot * a.cs_stride_slot + ch * a.cs_stride_chan;
            cp[0] = __float2bfloat16_rn(x1);
            cp[a.cs_stride_tap] = __float2bfloat16_rn(x2);
            cp[2 * a.cs_stride_tap] = __float2bfloat16_rn(xin);
        }
    }
    // (2) gates of this lane's four key columns, output gate of its rows
    float4 dec;
    if (kda) {
        float gv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float xg = bfs(stage, FL::rg, t.col + c) + reinterpret_cast<const float *>(stage + FL::db)[t.col + c];
            gv[c] = a.kda_gate_form == 0 ? fmaxf(a.lower_bound, -A * softplus_f(xg)) : a.lower_bound * sigmoid_f(A * xg);
        }
        dec = make_float4(expf(gv[0]), expf(gv[1]), expf(gv[2]), expf(gv[3]));
    } else {
        const float e = expf(g_head);
        dec = make_float4(e, e, e, e);
    }
    float gate[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) gate[c] = bfs(stage, FL::og, row0 + 8 * c + rsub);
    __syncthreads();   // conv outputs complete

    // (3) the step, both dots straight from the staged tile, eight rows at a time
    const float4 kh = l2_normalise4<32>(*reinterpret_cast<const float4 *>(ys + D + t.col), a.use_qk_l2norm != 0, 1.f);
    const float4 qh = l2_normalise4<32>(*reinterpret_cast<const float4 *>(ys + t.col), a.use_qk_l2norm != 0, P.scale);
    const float kq = group_sum<32>(dot4(kh, qh));
    const float *Ss = reinterpret_cast<const float *>(stage);
    float dvc0 = 0.f, dvc1 = 0.f, oc0 = 0.f, oc1 = 0.f;
    {
        const float4 kd = mul4(kh, dec), qd = mul4(qh, dec);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
            float x[TR::N];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 srow = *reinterpret_cast<const float4 *>(Ss + (size_t)(row0 + 8 * c + i) * D + t.col);
                x[i] = dot4(srow, kd);
                x[8 + i] = dot4(srow, qd);
            }
            t.reduce_scatter(x);
            const float vv = t.holds_k_dot() ? ys[2 * D + row0 + 8 * c + rsub] : 0.f;
            const float d = beta * (vv - x[0]);
            const float dq = __shfl_up_sync(kFull, d, 16);
            const float o = fmaf(dq, kq, x[0]);
            if (c == 0) {
                dvc0 = d;
                oc0 = o;
            } else {
                dvc1 = d;
                oc1 = o;
            }
        }
    }
    {
        float *S = a.state + ((size_t)slot * heads + h) * (size_t)(D * D);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float d = __shfl_sync(kFull, c == 0 ? dvc0 : dvc1, 2 * i);
                const float4 srow = *reinterpret_cast<const float4 *>(Ss + (size_t)(row0 + 8 * c + i) * D + t.col);
                st_stream(S + (size_t)(row0 + 8 * c + i) * D + t.col, decay_update4(dec, srow, d, kh));
            }
        }
    }
    // (4) gated RMSNorm over the head's 128 outputs
    const bool owner = !t.holds_k_dot() && (t.sub & 1) == 0;
    float sq = owner ? oc0 * oc0 + oc1 * oc1 : 0.f;
    sq = group_sum<32>(sq);
    if (lane == 0) red[warp] = sq;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kFGW; ++w) tot += red[w];
    const float rs = 1.0f / sqrtf(tot / D + a.norm_eps);
    if (owner) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const float act = a.gate_act == GDN_ACT_SILU ? gate[c] * sigmoid_f(gate[c]) : sigmoid_f(gate[c]);
            out[row0 + 8 * c + rsub] = __float2bfloat16_rn((c == 0 ? oc0 : oc1) * rs * w_norm[c] * act);
        }
    }
}

int launch_fused_stage(const FusedLaunch &p, bool sd, cudaStream_t stream, bool chained)
{
    const size_t smem = FusedLayout::meta;   // state tile, x, conv state, raw_g, dt_bias, out_gate
    auto kern = sd ? fused_stage_kernel<true> : fused_stage_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)(p.a.T * p.a.heads));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    if (chained) set_programmatic(attr[cfg.numAttrs++]);
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return GDN_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

}  // namespace gdn
