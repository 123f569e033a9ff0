// step_kernel.cu -- the packed / indexed single-token decode step (gdn_decode_step and
// gdn_decode_step_indexed).
//
// The state is fp32, or bf16 when it is stored in bf16 (8-byte accesses of four values, fp32
// arithmetic, the updated tile rounded to nearest even as it is stored).
//
// Grid: 1, 2, 4 or 8 CTAs per (row b, value head hv) tile, tiles ordered b * HV + hv, so the G
// value heads that share a q/k head sit next to each other and find its q/k in L2. At K = 128
// with an fp32 state a tile is two CTAs of 64 rows each (8 rows per thread, four CTAs per SM),
// the fastest split on GB300 at every batch size; small batches split further. Each CTA streams
// its rows in with 16-byte loads, takes S.(Dk) and S.(Dq) from registers, and writes S' back with
// 16-byte streaming stores: one HBM read and one HBM write of the state, which is the whole
// roofline of this memory-bound matrix-vector step.
//
// Sources: "Optimization Log: Qwen3.5-27B Dense on B200", "Kernel 4: Fused DeltaNet Recurrent
// (FLAGSHIP)" (the Math block); "Microbenchmark: buffered output-only GDN decode (ReplaySSM Part
// A)", _bench_cfg / run_packed (packed mixed_qkv, gates from a, b, A_log, dt_bias, in-kernel q/k
// L2 norm with scale K^-1/2, ssm_state_indices, state [num_slots, HV, V, K] updated in place,
// out [B, 1, HV, V]); _state_bytes_per_step (k [H, K] shared across HV // H value heads).
#include "gdn_chain.cuh"
#include "gdn_launch.h"
#include "gdn_tile.cuh"

namespace gdn {

// R rows per warp: R = 16 lets a CTA own a whole tile (looping over row passes when V is larger
// than 128); R = 8, 4 or 2 split a tile's rows over `splits` CTAs (R = 8 at K = 128 with an fp32
// state, and smaller R for batches with too few tiles to fill the GPU). Row dots are complete within a row, so the
// split needs no exchange between CTAs; each CTA normalises q and k itself.
//
// CHAIN: the instance behind gdn_decode_step_indexed_chained, launched as a programmatic dependent
// launch (a layer of a multi-layer graph). It lets the next kernel start its CTAs at once, reads
// the slot index and issues its state loads, and only then waits for the kernel before it on the
// stream to complete; every other input is read, and every output written, after that wait. The
// ordinary instance is launched with the same attribute but waits before it touches memory and
// only then lets the next kernel start (ordinary_launch_start), so the next call's CTAs can be
// resident when this one ends: on GB300 3.20 against 3.42 us per call at B = 1, 13.28 against
// 13.39 at B = 16, no change from B = 64 (a wait after outstanding loads, by contrast, slowed
// ordinary launches). The bf16-state kernels of their own (step_kernel_bf16, and the staged one
// from 128 tiles) keep plain launches: with tiles staged in shared memory the early CTAs made
// B = 16 slower (9.47 against 8.48 us).
template <int K, typename Tin, typename TS, int R, bool CHAIN>
__global__ void __launch_bounds__(kThreads, R >= 16 ? 2 : 4) step_kernel(const __grid_constant__ StepLaunch P, int splits)
{
    using TL = Tile<K, R>;
    const gdn_step_args &a = P.a;
    const int HV = a.HV, V = a.V;
    const int tile = blockIdx.x / splits, blk = blockIdx.x - tile * splits;
    const int b = tile / HV, hv = tile - b * HV, h = hv / P.G;
    const size_t out_base = ((size_t)b * HV + hv) * V;
    const int first_row = blk * TL::ROWS_PASS, row_step = splits * TL::ROWS_PASS;
    if constexpr (CHAIN) grid_launch_dependents();
    else ordinary_launch_start();

    int slot = b;
    if (P.idx) {
        slot = P.idx[b];
        const bool pad = slot == P.pad;
        if (pad || slot < 0 || slot >= a.num_slots) {   // uniform over the CTA
            if constexpr (CHAIN) grid_dependency_wait();
            if (!pad && blk == 0 && threadIdx.x == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_INDEX);
            for (int r = threadIdx.x; r < V; r += kThreads)
                if ((r / TL::ROWS_PASS) % splits == blk) store_out(a.out, a.out_dtype, out_base + r, 0.f);
            return;
        }
    }
    if (!step_tile_in_range(a, b, hv, h, slot)) return;   // debug build only
    TS *S = static_cast<TS *>(a.state) + ((size_t)slot * HV + hv) * (size_t)V * K;

    TL t;
    t.init();
    t.load(S, V, first_row);   // the tile's loads go out first; everything below overlaps them
    if constexpr (CHAIN) grid_dependency_wait();

    const Tin *qp = static_cast<const Tin *>(a.q) + (size_t)b * a.q_stride + (size_t)h * K;
    const Tin *kp = static_cast<const Tin *>(a.k) + (size_t)b * a.k_stride + (size_t)h * K;
    const Tin *vp = static_cast<const Tin *>(a.v) + (size_t)b * a.v_stride + (size_t)hv * V;
    const float4 q4 = load4(qp + t.col), k4 = load4(kp + t.col);
    float g, beta;
    step_gates<Tin>(a, b, hv, g, beta);

    const float4 kh = l2_normalise4<TL::LPR>(k4, a.use_qk_l2norm != 0, 1.f);
    const float4 qh = l2_normalise4<TL::LPR>(q4, a.use_qk_l2norm != 0, P.scale);
    const float kq = group_sum<TL::LPR>(dot4(kh, qh));
    const float e = expf(g);
    const float4 dec = make_float4(e, e, e, e);
    const float4 kd = scale4(kh, e), qd = scale4(qh, e);

    for (int row0 = first_row; row0 < V; row0 += row_step) {
        if (row0 != first_row) t.load(S, V, row0);
        float vv[TL::M];
#pragma unroll
        for (int m = 0; m < TL::M; ++m) {
            const int r = t.row(row0, t.owned_chunk(m));
            vv[m] = (t.holds_k_dot() && r < V) ? to_f32(vp[r]) : 0.f;
        }
        float x[TL::N];
        t.partial_dots(kd, qd, x);
        t.reduce_scatter(x);
        // lanes [0, HALF) of a row group: x[m] = u of their rows -> delta
        float dv[TL::M];
#pragma unroll
        for (int m = 0; m < TL::M; ++m) dv[m] = beta * (vv[m] - x[m]);
        // lanes [HALF, LPR): x[m] = S (D q) of the same rows -> o = x + delta (k . q)
#pragma unroll
        for (int m = 0; m < TL::M; ++m) {
            const float dq = t.delta_for_q(dv[m]);
            const int r = t.row(row0, t.owned_chunk(m));
            if (!t.holds_k_dot() && t.writer() && r < V) store_out(a.out, a.out_dtype, out_base + r, fmaf(dq, kq, x[m]));
        }
        t.update_store(S, V, row0, dec, kh, dv);
    }
}

__device__ __forceinline__ float4 widen_bf16x4(uint2 raw)
{
    return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                       __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
}

// bf16 state, one row pass (V <= rows per pass): NT tiles per CTA, whose loads are all issued
// before any is computed; rows stay in registers as packed bf16 (8 bytes per four values), are
// widened to fp32 where they are used, and the update is rounded to nearest even as it is stored.
// Each tile's rows are reduced in two 8-row chunks (16 partial dots live, not 32) and the decay is
// applied to the reduced dots, so one tile fits in 80 registers: launched with NT = 1 at three CTAs
// per SM (92.7 us per step at B = 256, HV = 32; two tiles per CTA at two CTAs per SM: 105.4 us;
// four CTAs per SM spill: 95.2 us).
template <int K, typename Tin, int NT>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 3 : 2) step_kernel_bf16(const __grid_constant__ StepLaunch P)
{
    using TL = Tile<K>;      // row geometry: 16 rows per warp
    using TR = Tile<K, 8>;   // reduction of one 8-row chunk (same lane layout)
    const gdn_step_args &a = P.a;
    const int HV = a.HV, V = a.V;
    const int ntiles = a.B * HV;
    TL t;
    t.init();
    TR t8;
    t8.init();
    uint2 raw[NT][TL::R];
    int slots[NT];
    bool run[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
        const int tile = blockIdx.x * NT + u;
        run[u] = false;
        slots[u] = 0;
        if (tile < ntiles) {
            const int b = tile / HV, hv = tile - b * HV;
            int slot = b;
            bool skip = false;
            if (P.idx) {
                slot = P.idx[b];
                const bool pad = slot == P.pad;
                if (pad || slot < 0 || slot >= a.num_slots) {
                    if (!pad && threadIdx.x == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_INDEX);
                    const size_t out_base = ((size_t)b * HV + hv) * V;
                    for (int r = threadIdx.x; r < V; r += kThreads) store_out(a.out, a.out_dtype, out_base + r, 0.f);
                    skip = true;
                }
            }
            if (!skip && step_tile_in_range(a, b, hv, hv / P.G, slot)) {   // (range: debug build)
                run[u] = true;
                slots[u] = slot;
                const bf16 *S = static_cast<const bf16 *>(a.state) + ((size_t)slot * HV + hv) * (size_t)V * K;
#pragma unroll
                for (int i = 0; i < TL::R; ++i) {
                    const int r = t.row(0, i);
                    raw[u][i] = r < V ? __ldcs(reinterpret_cast<const uint2 *>(S + (size_t)r * K + t.col))
                                      : make_uint2(0u, 0u);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NT; ++u) {
        if (!run[u]) continue;   // uniform over the CTA
        const int tile = blockIdx.x * NT + u;
        const int b = tile / HV, hv = tile - b * HV, h = hv / P.G;
        const size_t out_base = ((size_t)b * HV + hv) * V;
        const Tin *qp = static_cast<const Tin *>(a.q) + (size_t)b * a.q_stride + (size_t)h * K;
        const Tin *kp = static_cast<const Tin *>(a.k) + (size_t)b * a.k_stride + (size_t)h * K;
        const Tin *vp = static_cast<const Tin *>(a.v) + (size_t)b * a.v_stride + (size_t)hv * V;
        const float4 q4 = load4(qp + t.col), k4 = load4(kp + t.col);
        float g, beta;
        step_gates<Tin>(a, b, hv, g, beta);
        const float4 kh = l2_normalise4<TL::LPR>(k4, a.use_qk_l2norm != 0, 1.f);
        const float4 qh = l2_normalise4<TL::LPR>(q4, a.use_qk_l2norm != 0, P.scale);
        const float kq = group_sum<TL::LPR>(dot4(kh, qh));
        const float e = expf(g);   // applied to the reduced dots: u = e (S k), and e (S q)
        // two chunks of 8 rows: 16 partial dots live at a time instead of 32
        float dch[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float x[TR::N];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 sv = widen_bf16x4(raw[u][8 * c + i]);
                x[i] = dot4(sv, kh);
                x[8 + i] = dot4(sv, qh);
            }
            t8.reduce_scatter(x);
            const int r = t.row(0, 8 * c + t8.owned_chunk(0));
            const float vv = (t8.holds_k_dot() && r < V) ? to_f32(vp[r]) : 0.f;
            const float d = beta * (vv - e * x[0]);
            const float dq = t8.delta_for_q(d);
            if (!t8.holds_k_dot() && t8.writer() && r < V)
                store_out(a.out, a.out_dtype, out_base + r, fmaf(dq, kq, e * x[0]));
            dch[c] = d;
        }
        bf16 *S = static_cast<bf16 *>(a.state) + ((size_t)slots[u] * HV + hv) * (size_t)V * K;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const float dc[1] = {dch[c]};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float d = t8.delta_of(dc, i);
                const int r = t.row(0, 8 * c + i);
                if (r < V) st_stream(S + (size_t)r * K + t.col, axpby4(e, widen_bf16x4(raw[u][8 * c + i]), d, kh));
            }
        }
    }
}

static int sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

template <int K, typename Tin, typename TS, int R>
static void launch_rows(const StepLaunch &p, unsigned tiles, cudaStream_t stream, bool chained)
{
    const int splits = R >= 16 ? 1 : (p.a.V + Tile<K, R>::ROWS_PASS - 1) / Tile<K, R>::ROWS_PASS;
    // A chained launch gains the previous layer's tail, which matters when a layer is a few waves
    // of CTAs: on GB300 the 48-layer graph took 18.68 against 19.50 us per layer at B = 16 (2.5
    // waves) but 244.3 against 242.5 at B = 256 (40 waves). From eight waves on it launches as usual.
    const unsigned per_sm = R >= 16 ? 2u : 4u;
    const unsigned waves_x8 = 8u * per_sm * (unsigned)(sm_count() > 0 ? sm_count() : 152);
    if (chained && tiles * (unsigned)splits >= waves_x8) chained = false;
    if (!chained) {
        launch_ordinary(step_kernel<K, Tin, TS, R, false>, dim3(tiles * (unsigned)splits), dim3(kThreads), 0, stream, p, splits);
        return;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_programmatic(attr[0]);
    cfg.gridDim = dim3(tiles * (unsigned)splits);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, step_kernel<K, Tin, TS, R, true>, p, splits);
}

template <int K, typename Tin, typename TS>
static int launch_step_t(const StepLaunch &p, cudaStream_t stream, bool chained)
{
    const unsigned tiles = (unsigned)p.a.B * (unsigned)p.a.HV;
    // Enough CTAs to cover every SM about four times over: whole tiles when the batch allows it,
    // otherwise the fewest row splits that get there (at most 8 per tile at V = 128).
    const unsigned target = 4u * (unsigned)(sm_count() > 0 ? sm_count() : 152);
    auto ctas = [&](int rows_pass) { return tiles * (unsigned)((p.a.V + rows_pass - 1) / rows_pass); };
    // fp32 state at K = 128: 8 rows per thread (two CTAs per tile, 64 registers, four CTAs per SM)
    // measured faster than whole-tile CTAs at every batch size on GB300 (156.1 against 157.4 us at
    // B = 256, 22.6 against 24.0 at B = 32)
    if (sizeof(TS) == 4 && K == 128 && ctas(Tile<K, 8>::ROWS_PASS) >= target) {
        launch_rows<K, Tin, TS, 8>(p, tiles, stream, chained);
        return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
    }
    if constexpr (sizeof(TS) == 2 && K == 128) {
        // bf16 state at K = V = 128: each tile staged in shared memory by a bulk copy
        // (step_stage_bf16.cu) from 128 tiles on; on GB300 it beat the row split at B = 8 and 16
        // (HV = 32: 5.92 against 7.47 us, 8.52 against 10.37) and lost at B = 1 (3.52 against 3.29)
        if (tiles >= 128u && step_stage_bf16_ok(p.a)) return launch_step_stage_bf16(p, stream);
    }
    if (tiles >= target) {
        bool paired = false;
        if constexpr (sizeof(TS) == 2 && K >= 64) {
            if (p.a.V <= Tile<K>::ROWS_PASS) {
                step_kernel_bf16<K, Tin, 1><<<tiles, kThreads, 0, stream>>>(p);
                paired = true;
            }
        }
        if (!paired) launch_rows<K, Tin, TS, 16>(p, tiles, stream, chained);
    } else if (ctas(Tile<K, 8>::ROWS_PASS) >= target) {
        launch_rows<K, Tin, TS, 8>(p, tiles, stream, chained);
    } else if (ctas(Tile<K, 4>::ROWS_PASS) >= target) {
        launch_rows<K, Tin, TS, 4>(p, tiles, stream, chained);
    } else {
        launch_rows<K, Tin, TS, 2>(p, tiles, stream, chained);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

template <typename Tin, typename TS>
static int launch_step_k(const StepLaunch &p, cudaStream_t stream, bool chained)
{
    switch (p.a.K) {
    case 16: return launch_step_t<16, Tin, TS>(p, stream, chained);
    case 32: return launch_step_t<32, Tin, TS>(p, stream, chained);
    case 64: return launch_step_t<64, Tin, TS>(p, stream, chained);
    case 128: return launch_step_t<128, Tin, TS>(p, stream, chained);
    default: return GDN_ERR_SHAPE;
    }
}

int launch_step(const StepLaunch &p, cudaStream_t stream, bool chained)
{
    if (p.a.state_dtype == GDN_BF16)
        return p.a.in_dtype == GDN_BF16 ? launch_step_k<bf16, bf16>(p, stream, chained)
                                        : launch_step_k<float, bf16>(p, stream, chained);
    return p.a.in_dtype == GDN_BF16 ? launch_step_k<bf16, float>(p, stream, chained)
                                    : launch_step_k<float, float>(p, stream, chained);
}

}  // namespace gdn
