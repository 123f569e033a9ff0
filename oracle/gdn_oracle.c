/*
 * gdn_oracle.c -- plain, slow fp64 CPU oracle for the single-token gated delta-rule decode step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this library. It shares no code with the CUDA library (no headers, helpers or tables) and the
 * CUDA library never calls it.
 *
 * Every routine is the plain definition, written in the order the sources state it:
 *   - the delta-rule step: "Optimization Log: Qwen3.5-27B Dense on B200", section "Kernel 4: Fused
 *     DeltaNet Recurrent (FLAGSHIP)", Math block: decay S by exp(g), residual against S k, scale by
 *     beta, rank-1 update, output from the updated state.
 *   - in-kernel q/k L2 normalisation, the K^-1/2 q scale, GQA sharing and the slot indirection:
 *     "Microbenchmark: buffered output-only GDN decode (ReplaySSM Part A)", functions _bench_cfg
 *     (run_packed: scale, use_qk_l2norm_in_kernel, ssm_state_indices) and _state_bytes_per_step
 *     (k: [H,K] shared across HV//H).
 *   - the buffered (output-only) variant: same page, module docstring and _bench_cfg (run_replay):
 *     read S every step, append d/k/g ring records, fold the ring into the checkpoint at
 *     write_pos == L-1.
 *   - conv update, KDA gate, beta and gated RMSNorm: "Microbenchmark for the fused Kimi-K3 KDA decode
 *     kernel on ROCm", functions Inputs, triton_chain and _gated_rmsnorm; "Optimization Log", section
 *     "Kernel 5: Fused Causal Conv1d Update" (shift + insert + dot product + SiLU).
 *   - the Mamba-1 selective-scan decode step: "Triton decode kernel + MBU analysis", section
 *     "Kernel design" (the per-element math block).
 *   - the decode projection y = x W^T: "Optimization Log", section "Kernel 3: BF16 GEMV with
 *     Split-K" (one sum over all inputs per output here; the split-K order is the kernels' choice).
 * No single-pass or low-rank rewrite of the step appears here: those identities are what the
 * tests check this code against.
 *
 * All arrays are dense row-major fp64 (int32 for indices). Build with -ffp-contract=off so that no
 * multiply-add is fused and the result is the same on every host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double softplus(double x) { return log1p(exp(x)); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Round to the nearest bf16 value, ties to even (8 significant bits). Finite inputs. */
double oracle_round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    double m = frexp(x, &e);                 /* x = m * 2^e, 0.5 <= |m| < 1 */
    return ldexp(nearbyint(ldexp(m, 8)), e - 8);
}

/* GDN gates: g = -exp(A_log[hv]) * softplus(a + dt_bias[hv]), beta = sigmoid(b).
 * a, b, g, beta: [B, HV]; A_log, dt_bias: [HV]. */
void oracle_gdn_gates(int B, int HV, const double *a, const double *b, const double *A_log,
                      const double *dt_bias, double *g, double *beta)
{
    for (int i = 0; i < B; ++i)
        for (int hv = 0; hv < HV; ++hv) {
            size_t o = (size_t)i * HV + hv;
            g[o] = -exp(A_log[hv]) * softplus(a[o] + dt_bias[hv]);
            beta[o] = sigmoid(b[o]);
        }
}

/* KDA per-key-channel gate, bounded below by lower_bound.
 * raw_g, g: [T, heads, D]; A_log: [heads]; dt_bias: [heads * D].
 * form 0: g = max(lower_bound, -exp(A_log[h]) * softplus(raw_g + dt_bias))
 * form 1: g = lower_bound * sigmoid(exp(A_log[h]) * (raw_g + dt_bias)) */
void oracle_kda_gate(int T, int heads, int D, const double *raw_g, const double *A_log,
                     const double *dt_bias, double lower_bound, int form, double *g)
{
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < heads; ++h)
            for (int d = 0; d < D; ++d) {
                size_t o = ((size_t)t * heads + h) * D + d;
                double x = raw_g[o] + dt_bias[(size_t)h * D + d];
                double val;
                if (form == 0) {
                    val = -exp(A_log[h]) * softplus(x);
                    if (val < lower_bound) val = lower_bound;
                } else {
                    val = lower_bound * sigmoid(exp(A_log[h]) * x);
                }
                g[o] = val;
            }
}

/* beta = sigmoid(raw) elementwise, n values. */
void oracle_sigmoid(size_t n, const double *raw, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = sigmoid(raw[i]);
}

/* x / sqrt(sum x^2 + eps) over n values, times s. */
static void l2_normalise(int n, const double *x, double eps, double s, int enabled, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = enabled ? 1.0 / sqrt(ss + eps) : 1.0;
    for (int i = 0; i < n; ++i) y[i] = x[i] * r * s;
}

/* One step of the recurrence on one state tile S[V, K] (row v, column k).
 * decay: one value (per_key == 0) or K values, one per key column. */
static void delta_rule_tile(int K, int V, double *S, const double *khat, const double *qhat,
                            const double *vin, const double *decay_log, int per_key, double beta,
                            double *u, double *d, double *o)
{
    /* S <- exp(g) * S */
    for (int vv = 0; vv < V; ++vv)
        for (int kk = 0; kk < K; ++kk)
            S[(size_t)vv * K + kk] *= exp(per_key ? decay_log[kk] : decay_log[0]);
    /* u = S k */
    for (int vv = 0; vv < V; ++vv) {
        double acc = 0.0;
        for (int kk = 0; kk < K; ++kk) acc += S[(size_t)vv * K + kk] * khat[kk];
        u[vv] = acc;
    }
    /* delta = beta * (v - u) */
    for (int vv = 0; vv < V; ++vv) d[vv] = beta * (vin[vv] - u[vv]);
    /* S <- S + delta k^T */
    for (int vv = 0; vv < V; ++vv)
        for (int kk = 0; kk < K; ++kk) S[(size_t)vv * K + kk] += d[vv] * khat[kk];
    /* o = S q */
    for (int vv = 0; vv < V; ++vv) {
        double acc = 0.0;
        for (int kk = 0; kk < K; ++kk) acc += S[(size_t)vv * K + kk] * qhat[kk];
        o[vv] = acc;
    }
}

/* Slot of row b: idx[b], or b when idx is NULL. Returns -1 for a pad row, -2 for a bad slot. */
static long slot_of(int b, const int32_t *idx, int32_t pad_slot, int num_slots)
{
    long s = idx ? (long)idx[b] : (long)b;
    if (idx && s == pad_slot) return -1;
    if (s < 0 || s >= num_slots) return -2;
    return s;
}

/* Decode step for every (row b, value head hv).
 *   q, k: [B, H, K]; v: [B, HV, V]; g: [B, HV] (g_per_key = 0) or [B, HV, K] (g_per_key = 1);
 *   beta: [B, HV]; state: [num_slots, HV, V, K], updated in place; out: [B, HV, V].
 *   q/k head of value head hv is hv / (HV / H). With use_qk_l2norm, k_hat = k / sqrt(|k|^2 + l2_eps)
 *   and q_hat = scale * q / sqrt(|q|^2 + l2_eps); otherwise q_hat = scale * q.
 *   A pad row (idx[b] == pad_slot) and a row with an out-of-range slot leave the state as it is and
 *   get out = 0. Returns the number of out-of-range rows.
 *   state_bf16 != 0: the state is stored in bf16 ("Optimization Log", Kernel 4: a 32 KB bf16 state
 *   per head). The step runs on the stored values as above, out comes from the updated state before
 *   storage, and the updated state is then rounded to bf16 (nearest, ties to even). */
int oracle_delta_step(int B, int H, int HV, int K, int V, int num_slots,
                      const double *q, const double *k, const double *v,
                      const double *g, int g_per_key, const double *beta,
                      double scale, int use_qk_l2norm, double l2_eps,
                      const int32_t *idx, int32_t pad_slot, int state_bf16, double *state, double *out)
{
    int G = HV / H, bad = 0;
    double *kh = malloc(sizeof(double) * K), *qh = malloc(sizeof(double) * K);
    double *u = malloc(sizeof(double) * V), *d = malloc(sizeof(double) * V);
    for (int b = 0; b < B; ++b) {
        long s = slot_of(b, idx, pad_slot, num_slots);
        if (s < 0) {
            if (s == -2) ++bad;
            memset(out + (size_t)b * HV * V, 0, sizeof(double) * HV * V);
            continue;
        }
        for (int hv = 0; hv < HV; ++hv) {
            int h = hv / G;
            l2_normalise(K, k + ((size_t)b * H + h) * K, l2_eps, 1.0, use_qk_l2norm, kh);
            l2_normalise(K, q + ((size_t)b * H + h) * K, l2_eps, scale, use_qk_l2norm, qh);
            const double *gl = g_per_key ? g + ((size_t)b * HV + hv) * K : g + (size_t)b * HV + hv;
            double *S = state + ((size_t)s * HV + hv) * V * K;
            delta_rule_tile(K, V, S, kh, qh, v + ((size_t)b * HV + hv) * V, gl, g_per_key,
                            beta[(size_t)b * HV + hv], u, d, out + ((size_t)b * HV + hv) * V);
            if (state_bf16)
                for (size_t e = 0; e < (size_t)V * K; ++e) S[e] = oracle_round_bf16(S[e]);
        }
    }
    free(kh); free(qh); free(u); free(d);
    return bad;
}

/* Buffered (output-only) decode step. Per row b with cursor p = write_pos[b] (0 <= p < L):
 *   the checkpoint S_c = state[slot, hv] is replayed through the ring records j = 0 .. p-1,
 *     S <- exp(g_j) * S + d_j k_j^T
 *   (d_cache [num_slots, HV, L, V], k_cache [num_slots, H, L, K], g_cache [num_slots, HV, L]),
 *   then this step runs on S exactly as oracle_delta_step does; its records (d, k_hat, g) are
 *   written at ring position p, rounded to bf16 when ring_bf16 != 0; and if p == L-1 the result is
 *   written back to the checkpoint. write_pos is not advanced. Rows with a pad slot, a bad slot or
 *   a bad cursor are skipped with out = 0. Returns the number of bad rows. */
int oracle_gdn_buffered(int B, int H, int HV, int K, int V, int num_slots,
                        const double *q, const double *k, const double *v,
                        const double *g, const double *beta,
                        double scale, int use_qk_l2norm, double l2_eps,
                        const int32_t *idx, int32_t pad_slot,
                        int L, int ring_bf16, double *d_cache, double *k_cache, double *g_cache,
                        const int32_t *write_pos, double *state, double *out)
{
    int G = HV / H, bad = 0;
    double *kh = malloc(sizeof(double) * K), *qh = malloc(sizeof(double) * K);
    double *u = malloc(sizeof(double) * V), *d = malloc(sizeof(double) * V);
    double *S = malloc(sizeof(double) * (size_t)V * K);
    for (int b = 0; b < B; ++b) {
        long s = slot_of(b, idx, pad_slot, num_slots);
        int p = write_pos[b];
        if (s < 0 || p < 0 || p >= L) {
            if (s == -2 || (s >= 0 && (p < 0 || p >= L))) ++bad;
            memset(out + (size_t)b * HV * V, 0, sizeof(double) * HV * V);
            continue;
        }
        for (int hv = 0; hv < HV; ++hv) {
            int h = hv / G;
            double *Sc = state + ((size_t)s * HV + hv) * V * K;
            double *dring = d_cache + ((size_t)s * HV + hv) * L * V;
            double *kring = k_cache + ((size_t)s * H + h) * L * K;
            double *gring = g_cache + ((size_t)s * HV + hv) * L;
            memcpy(S, Sc, sizeof(double) * (size_t)V * K);
            for (int j = 0; j < p; ++j)
                for (int vv = 0; vv < V; ++vv)
                    for (int kk = 0; kk < K; ++kk)
                        S[(size_t)vv * K + kk] = exp(gring[j]) * S[(size_t)vv * K + kk]
                                                 + dring[(size_t)j * V + vv] * kring[(size_t)j * K + kk];
            l2_normalise(K, k + ((size_t)b * H + h) * K, l2_eps, 1.0, use_qk_l2norm, kh);
            l2_normalise(K, q + ((size_t)b * H + h) * K, l2_eps, scale, use_qk_l2norm, qh);
            double gv = g[(size_t)b * HV + hv];
            delta_rule_tile(K, V, S, kh, qh, v + ((size_t)b * HV + hv) * V, &gv, 0,
                            beta[(size_t)b * HV + hv], u, d, out + ((size_t)b * HV + hv) * V);
            for (int vv = 0; vv < V; ++vv)
                dring[(size_t)p * V + vv] = ring_bf16 ? oracle_round_bf16(d[vv]) : d[vv];
            for (int kk = 0; kk < K; ++kk)
                kring[(size_t)p * K + kk] = ring_bf16 ? oracle_round_bf16(kh[kk]) : kh[kk];
            gring[p] = gv;
            if (p == L - 1) memcpy(Sc, S, sizeof(double) * (size_t)V * K);
        }
    }
    free(kh); free(qh); free(u); free(d); free(S);
    return bad;
}

/* Causal conv1d update of width 4 with SiLU, for T rows of C channels.
 *   x: [T, C]; w: [C, 4]; bias: [C] or NULL; conv_state: [num_slots, C, 3] with tap 0 the oldest
 *   input; y: [T, C].
 *   y[c] = silu(w[c,0]*cs[c,0] + w[c,1]*cs[c,1] + w[c,2]*cs[c,2] + w[c,3]*x[c] + bias[c]),
 *   then cs[c] <- (cs[c,1], cs[c,2], x[c]).
 *   Rows with a pad slot or a bad slot leave the conv state as it is and get y = 0.
 *   Returns the number of bad rows. */
int oracle_conv_update(int T, int C, const double *x, const double *w, const double *bias,
                       double *conv_state, int num_slots, const int32_t *idx, int32_t pad_slot,
                       double *y)
{
    int bad = 0;
    for (int t = 0; t < T; ++t) {
        long s = slot_of(t, idx, pad_slot, num_slots);
        if (s < 0) {
            if (s == -2) ++bad;
            memset(y + (size_t)t * C, 0, sizeof(double) * C);
            continue;
        }
        for (int c = 0; c < C; ++c) {
            double *cs = conv_state + ((size_t)s * C + c) * 3;
            double xin = x[(size_t)t * C + c];
            const double *wc = w + (size_t)c * 4;
            double acc = wc[0] * cs[0] + wc[1] * cs[1] + wc[2] * cs[2] + wc[3] * xin;
            if (bias) acc += bias[c];
            y[(size_t)t * C + c] = acc * sigmoid(acc);
            cs[0] = cs[1];
            cs[1] = cs[2];
            cs[2] = xin;
        }
    }
    return bad;
}

/* Gated RMSNorm over the last dimension: out = x / sqrt(mean(x^2) + eps) * w * act(gate),
 * act = silu (act == 0) or sigmoid (act == 1). x, gate, out: [rows, D]; w: [D]. */
void oracle_gated_rmsnorm(int rows, int D, const double *x, const double *gate, const double *w,
                          double eps, int act, double *out)
{
    for (int r = 0; r < rows; ++r) {
        const double *xr = x + (size_t)r * D;
        double ss = 0.0;
        for (int i = 0; i < D; ++i) ss += xr[i] * xr[i];
        double rs = 1.0 / sqrt(ss / D + eps);
        for (int i = 0; i < D; ++i) {
            double gt = gate[(size_t)r * D + i];
            double a = act == 0 ? gt * sigmoid(gt) : sigmoid(gt);
            out[(size_t)r * D + i] = xr[i] * rs * w[i] * a;
        }
    }
}

/* Mamba-1 selective-scan decode step ("Triton decode kernel + MBU analysis", section "Kernel
 * design"), per (row b, channel d) with state h[b, d, 0..N):
 *   dA = exp(dt * A[d, :]);  dB = dt * B[b, :];  h <- dA * h + dB * x;  y = sum_n C[b, n] h[n];
 *   y += Dskip[d] * x (when Dskip is given);  y *= silu(z) (when z is given).
 * x, dt, z, y: [B, D]; A: [D, N]; Bm, Cm: [B, N]; Dskip: [D] or NULL; z: [B, D] or NULL;
 * h: [B, D, N], updated in place. */
void oracle_mamba_decode(int B, int D, int N, const double *x, const double *dt, const double *A,
                         const double *Bm, const double *Cm, const double *Dskip, const double *z,
                         double *h, double *y)
{
    for (int b = 0; b < B; ++b)
        for (int d = 0; d < D; ++d) {
            size_t r = (size_t)b * D + d;
            double *hr = h + r * N;
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                double dA = exp(dt[r] * A[(size_t)d * N + n]);
                double dB = dt[r] * Bm[(size_t)b * N + n];
                hr[n] = dA * hr[n] + dB * x[r];
                acc += Cm[(size_t)b * N + n] * hr[n];
            }
            if (Dskip) acc += Dskip[d] * x[r];
            if (z) acc *= z[r] * sigmoid(z[r]);
            y[r] = acc;
        }
}

/* Projection for decode ("Optimization Log: Qwen3.5-27B Dense on B200", Kernel 3: BF16 GEMV):
 * y[t, n] = sum_k x[t, k] W[n, k] for T rows, N outputs, Kd inputs; W stored one output row per
 * line ([N, Kd]). */
void oracle_gemv(int T, int N, int Kd, const double *x, const double *W, double *y)
{
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < Kd; ++k) acc += x[(size_t)t * Kd + k] * W[(size_t)n * Kd + k];
            y[(size_t)t * N + n] = acc;
        }
}
