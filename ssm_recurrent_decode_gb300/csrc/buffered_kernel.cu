// buffered_kernel.cu -- the buffered, output-only decode (gdn_decode_buffered).
//
// The pool holds checkpoints S_c. Row b at ring cursor p = write_pos[b] acts on the state that
// p replayed records (d_j, k_j, g_j), j < p, would give, but it never builds that state unless
// p == L-1. With G_i the log-decays of the records and of this step (g_p = g),
//     Gamma = exp(sum_{i<=p} g_i),   c_j = exp(sum_{j<i<=p} g_i),
//     S_bar = Gamma S_c + sum_{j<p} c_j d_j k_j^T          (decayed state before this update)
//     u     = Gamma (S_c k) + sum_j c_j d_j (k_j . k)
//     delta = beta (v - u)
//     o     = Gamma (S_c q) + sum_j c_j d_j (k_j . q) + delta (k . q)
// so a non-flush step reads S_c once, reads the small ring, and writes only its own records and
// the output. The flush step (p == L-1) forms S_bar + delta k^T from registers with p FMAs per
// element and writes it back to S_c. Over a cycle of L steps the state traffic is L reads and one
// write per tile instead of L reads and L writes.
//
// Source: "Microbenchmark: buffered output-only GDN decode (ReplaySSM Part A)": module docstring
// (read S every step, append d/k/g ring records, fold the ring into the checkpoint only when
// write_pos == L-1), _bench_cfg (d_cache [slots, HV, L, V], k_cache [slots, H, L, K], g_cache
// [slots, HV, L] fp32, write_pos [B]), _amortize (each phase replays one more record than the
// last); the step itself as in step_kernel.cu. The page replays the records element by element
// (walking nk key chunks); the low-rank form above is this library's own regrouping.
#include "gdn_launch.h"
#include "gdn_tile.cuh"

namespace gdn {

// Shared memory of one CTA: cd[L][V] = c_j d_j, kr[L][K] = k_j (flush only), kk[L] = k_j . k,
// kqr[L] = k_j . q, c[L] = c_j.
size_t buffered_smem_bytes(int L, int V, int K)
{
    return sizeof(float) * ((size_t)L * V + (size_t)L * K + 3 * (size_t)L);
}

template <typename T> __device__ __forceinline__ T ring_cast(float x);
template <> __device__ __forceinline__ float ring_cast<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 ring_cast<bf16>(float x) { return __float2bfloat16_rn(x); }

template <int K, typename Tin, typename Tring>
__global__ void __launch_bounds__(kThreads, 2) buffered_kernel(const __grid_constant__ StepLaunch P)
{
    using TL = Tile<K>;
    extern __shared__ float sm[];
    const gdn_step_args &a = P.a;
    const int H = a.H, HV = a.HV, V = a.V, L = P.L;
    const int b = blockIdx.x / HV, hv = blockIdx.x - b * HV, h = hv / P.G;
    const size_t out_base = ((size_t)b * HV + hv) * V;

    int slot = b;
    bool skip = false;
    if (P.idx) {
        slot = P.idx[b];
        const bool pad = slot == P.pad;
        if (pad || slot < 0 || slot >= a.num_slots) {
            if (!pad && threadIdx.x == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_INDEX);
            skip = true;
        }
    }
    const int p = P.write_pos[b];
    if (!skip && (p < 0 || p >= L)) {
        if (threadIdx.x == 0) raise_flag(a.err_flags, GDN_DEVERR_BAD_WRITE_POS);
        skip = true;
    }
    if (skip) {   // uniform over the CTA
        for (int r = threadIdx.x; r < V; r += kThreads) store_out(a.out, a.out_dtype, out_base + r, 0.f);
        return;
    }
    if (!step_tile_in_range(a, b, hv, h, slot) || !ring_in_range(a, L, slot, hv, h, p)) return;   // debug build
    const bool flush = p == L - 1;
    float *S = static_cast<float *>(a.state) + ((size_t)slot * HV + hv) * (size_t)V * K;

    TL t;
    t.init();
    t.load(S, V, 0);

    float *cd = sm;                         // [L][V]
    float *kr = cd + (size_t)L * V;         // [L][K]
    float *kk = kr + (size_t)L * K;         // [L]
    float *kqr = kk + L;                    // [L]
    float *cj = kqr + L;                    // [L]

    const Tin *qp = static_cast<const Tin *>(a.q) + (size_t)b * a.q_stride + (size_t)h * K;
    const Tin *kp = static_cast<const Tin *>(a.k) + (size_t)b * a.k_stride + (size_t)h * K;
    const Tin *vp = static_cast<const Tin *>(a.v) + (size_t)b * a.v_stride + (size_t)hv * V;
    const float4 q4 = load4(qp + t.col), k4 = load4(kp + t.col);
    float g, beta;
    step_gates<Tin>(a, b, hv, g, beta);
    const float4 kh = l2_normalise4<TL::LPR>(k4, a.use_qk_l2norm != 0, 1.f);
    const float4 qh = l2_normalise4<TL::LPR>(q4, a.use_qk_l2norm != 0, P.scale);
    const float kq = group_sum<TL::LPR>(dot4(kh, qh));

    Tring *dring = static_cast<Tring *>(P.d_cache) + ((size_t)slot * HV + hv) * L * V;
    Tring *kring = static_cast<Tring *>(P.k_cache) + ((size_t)slot * H + h) * L * K;
    float *gring = P.g_cache + ((size_t)slot * HV + hv) * L;

    // decay factors: cj[j] = exp(g_{j+1} + ... + g_p), Gamma = exp(g_0 + ... + g_p)
    if ((int)threadIdx.x < p) kk[threadIdx.x] = gring[threadIdx.x];   // staged log-decays
    __syncthreads();
    float gsum = g;
    for (int i = 0; i < p; ++i) gsum += kk[i];
    const float Gam = expf(gsum);
    if ((int)threadIdx.x < p) {
        float acc = g;
        for (int i = threadIdx.x + 1; i < p; ++i) acc += kk[i];
        cj[threadIdx.x] = expf(acc);
    }
    __syncthreads();
    // record dots k_j . k and k_j . q (one warp per record), staged k_j for the flush
    for (int j = t.warp; j < p; j += kWarps) {
        const float4 kj = load4(kring + (size_t)j * K + t.col);
        const float dk = group_sum<TL::LPR>(dot4(kj, kh));
        const float dq = group_sum<TL::LPR>(dot4(kj, qh));
        if (flush && t.grp == 0) *reinterpret_cast<float4 *>(kr + (size_t)j * K + t.col) = kj;
        __syncwarp();
        if (t.lane == 0) {
            kk[j] = dk;   // overwrites the staged g_j; every thread has read it before the sync
            kqr[j] = dq;
        }
    }
    // c_j d_j for every record and row
    for (int e = threadIdx.x; e < p * V; e += kThreads) {
        const int j = e / V;
        cd[e] = cj[j] * to_f32(dring[e]);
    }
    __syncthreads();

    const float4 gk = scale4(kh, Gam), gq = scale4(qh, Gam);
    for (int row0 = 0; row0 < V; row0 += TL::ROWS_PASS) {
        if (row0) t.load(S, V, row0);
        float vv[TL::M];
#pragma unroll
        for (int m = 0; m < TL::M; ++m) {
            const int r = t.row(row0, t.owned_chunk(m));
            vv[m] = (t.holds_k_dot() && r < V) ? to_f32(vp[r]) : 0.f;
        }
        float x[TL::N];
        t.partial_dots(gk, gq, x);
        t.reduce_scatter(x);
        // ring corrections: lower lanes add sum_j c_j d_j (k_j . k), upper lanes sum_j c_j d_j (k_j . q)
        const float *coef = t.holds_k_dot() ? kk : kqr;
#pragma unroll
        for (int m = 0; m < TL::M; ++m) {
            const int r = min(t.row(row0, t.owned_chunk(m)), V - 1);
            float acc = x[m];
            for (int j = 0; j < p; ++j) acc = fmaf(cd[(size_t)j * V + r], coef[j], acc);
            x[m] = acc;
        }
        float dv[TL::M];
#pragma unroll
        for (int m = 0; m < TL::M; ++m) dv[m] = beta * (vv[m] - x[m]);
#pragma unroll
        for (int m = 0; m < TL::M; ++m) {
            const float dq = t.delta_for_q(dv[m]);
            const int r = t.row(row0, t.owned_chunk(m));
            if (r < V) {
                if (t.holds_k_dot())
                    dring[(size_t)p * V + r] = ring_cast<Tring>(dv[m]);
                else
                    store_out(a.out, a.out_dtype, out_base + r, fmaf(dq, kq, x[m]));
            }
        }
        if (flush) {
            // S = Gamma S_c + sum_j c_j d_j k_j^T + delta k^T
#pragma unroll
            for (int i = 0; i < TL::R; ++i) {
                const float d = t.delta_of(dv, i);
                t.s[i] = axpby4(Gam, t.s[i], d, kh);
            }
            for (int j = 0; j < p; ++j) {
                const float4 kj = *reinterpret_cast<const float4 *>(kr + (size_t)j * K + t.col);
#pragma unroll
                for (int i = 0; i < TL::R; ++i) {
                    const int r = min(t.row(row0, i), V - 1);
                    const float c = cd[(size_t)j * V + r];
                    t.s[i] = make_float4(fmaf(c, kj.x, t.s[i].x), fmaf(c, kj.y, t.s[i].y),
                                         fmaf(c, kj.z, t.s[i].z), fmaf(c, kj.w, t.s[i].w));
                }
            }
#pragma unroll
            for (int i = 0; i < TL::R; ++i) {
                const int r = t.row(row0, i);
                if (r < V) st_stream(S + (size_t)r * K + t.col, t.s[i]);
            }
        }
    }
    // this step's records: k_hat by the first value head of the group, g by every value head
    if (hv % P.G == 0 && t.warp == 0 && t.grp == 0) {
        Tring *dst = kring + (size_t)p * K + t.col;
        dst[0] = ring_cast<Tring>(kh.x);
        dst[1] = ring_cast<Tring>(kh.y);
        dst[2] = ring_cast<Tring>(kh.z);
        dst[3] = ring_cast<Tring>(kh.w);
    }
    if (threadIdx.x == 0) gring[p] = g;
}

template <int K, typename Tin, typename Tring>
static int launch_buf_t(const StepLaunch &p, cudaStream_t stream)
{
    const size_t smem = buffered_smem_bytes(p.L, p.a.V, K);
    auto kern = buffered_kernel<K, Tin, Tring>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const unsigned tiles = (unsigned)p.a.B * (unsigned)p.a.HV;
    kern<<<tiles, kThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

template <typename Tin, typename Tring>
static int launch_buf_k(const StepLaunch &p, cudaStream_t stream)
{
    switch (p.a.K) {
    case 16: return launch_buf_t<16, Tin, Tring>(p, stream);
    case 32: return launch_buf_t<32, Tin, Tring>(p, stream);
    case 64: return launch_buf_t<64, Tin, Tring>(p, stream);
    case 128: return launch_buf_t<128, Tin, Tring>(p, stream);
    default: return GDN_ERR_SHAPE;
    }
}

int launch_buffered(const StepLaunch &p, int ring_dtype, cudaStream_t stream)
{
    if (p.a.in_dtype == GDN_BF16)
        return ring_dtype == GDN_BF16 ? launch_buf_k<bf16, bf16>(p, stream) : launch_buf_k<bf16, float>(p, stream);
    return ring_dtype == GDN_BF16 ? launch_buf_k<float, bf16>(p, stream) : launch_buf_k<float, float>(p, stream);
}

}  // namespace gdn
