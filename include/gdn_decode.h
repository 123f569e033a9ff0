/*
 * gdn_decode.h -- C ABI of the GB300 (sm_103a) single-token gated delta-rule decode library
 * (libgdn_decode.so).
 *
 * The operation. For each request row b and value head hv, with state tile S = state[slot, hv]
 * (V rows, K columns, fp32, key index contiguous) and q/k head h = hv / (HV / H):
 *     k_hat = k[b,h] / sqrt(|k[b,h]|^2 + 1e-6),   q_hat = scale * q[b,h] / sqrt(|q[b,h]|^2 + 1e-6)
 *     S     <- exp(g) * S                       (g one value, or one value per key column)
 *     u      = S k_hat
 *     delta  = beta * (v[b,hv] - u)
 *     S     <- S + delta k_hat^T                (written back in place)
 *     out[b,hv] = S q_hat
 * This is the Math block of "Optimization Log: Qwen3.5-27B Dense on B200", section "Kernel 4:
 * Fused DeltaNet Recurrent (FLAGSHIP)", with the state stored [V, K] so that S^T k there is S k
 * here. The in-kernel L2 norm, the K^-1/2 scale, the slot pool and GQA sharing follow
 * "Microbenchmark: buffered output-only GDN decode (ReplaySSM Part A)" (_bench_cfg, run_packed;
 * _state_bytes_per_step: k [H,K] shared across HV//H value heads).
 *
 * Conventions shared by every entry point:
 *   - Every pointer in an args struct is a DEVICE pointer. The caller allocates and owns every
 *     buffer; the library allocates nothing, never synchronises, and launches only on `stream`.
 *     Calls are asynchronous; a call may be captured in a CUDA graph.
 *   - Sizes are element counts; strides are in elements.
 *   - The return value is GDN_OK or a negative gdn_status. A non-zero return means nothing was
 *     launched (except GDN_ERR_LAUNCH, which reports a failed launch). Arguments are checked on
 *     the host before any CUDA call: NULL pointers, unsupported sizes, dtypes and alignment.
 *   - Device-resident data (slot indices, ring cursors) is checked in the kernel. A row whose slot
 *     index or cursor is out of range is skipped: its state is not touched, its output is zeroed,
 *     and the matching GDN_DEVERR_* bit is OR-ed into *err_flags when err_flags is not NULL. The
 *     kernels never trap.
 *   - Two non-pad rows of one call must not name the same slot (the result is then undefined).
 *   - Supported sizes: K (key/head dim) in {16, 32, 64, 128}; V (value dim) in [1, 1024];
 *     HV a multiple of H. q and k must be 4-element aligned (8 bytes for bf16, 16 for fp32) and
 *     their row strides multiples of 4; state must be 16-byte aligned.
 */
#ifndef GDN_DECODE_H
#define GDN_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                         /* cudaStream_t is a pointer to this */
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_dtype { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef enum gdn_gate_mode {
    GDN_GATE_RAW = 0,    /* g = -exp(A_log[hv]) * softplus(a[b,hv] + dt_bias[hv]); beta = sigmoid(b[b,hv]) */
    GDN_GATE_DIRECT = 1  /* g[b,hv] and beta[b,hv] are given (fp32) */
} gdn_gate_mode;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL = -1,     /* a required pointer is NULL */
    GDN_ERR_SHAPE = -2,    /* unsupported or inconsistent size */
    GDN_ERR_DTYPE = -3,    /* unsupported dtype or dtype combination */
    GDN_ERR_ALIGN = -4,    /* a pointer or stride breaks the alignment rule */
    GDN_ERR_LAUNCH = -5,   /* the CUDA launch failed (cudaGetLastError) */
    GDN_ERR_ARG = -6,      /* another invalid argument (e.g. L < 1, unknown enum value) */
    GDN_ERR_SCRATCH = -7   /* the call needs more scratch than a no-allocation entry point's fixed
                              buffer holds */
} gdn_status;

/* Bits OR-ed into *err_flags by the kernels. */
#define GDN_DEVERR_BAD_INDEX 0x1      /* a slot index outside [0, num_slots) that is not the pad id */
#define GDN_DEVERR_BAD_WRITE_POS 0x2  /* a ring cursor outside [0, L) */
#define GDN_DEVERR_TIMEOUT 0x4        /* a bounded wait inside a pipelined kernel gave up; the CTA
                                         stopped early and its remaining rows were not computed */
#define GDN_DEVERR_RANGE 0x8          /* debug build only (libgdn_decode_debug.so, compiled with
                                         -DGDN_DEBUG): a kernel computed a global-memory index outside
                                         the buffer its arguments describe; that access was skipped */

/* Arguments of one decode step (all entry points but gdn_decode_fused). */
typedef struct gdn_step_args {
    int32_t B;            /* request rows */
    int32_t H;            /* q/k heads */
    int32_t HV;           /* value heads; HV % H == 0, q/k head of hv is hv / (HV / H) */
    int32_t K;            /* key dim (q, k head dim, state columns) */
    int32_t V;            /* value dim (v head dim, state rows, output dim) */
    int32_t num_slots;    /* state pool size */
    int32_t in_dtype;     /* gdn_dtype of q, k, v, a, b */
    int32_t out_dtype;    /* gdn_dtype of out */
    const void *q;        /* q[b,h,:] at q + b*q_stride + h*K */
    const void *k;        /* k[b,h,:] at k + b*k_stride + h*K */
    const void *v;        /* v[b,hv,:] at v + b*v_stride + hv*V */
    int64_t q_stride, k_stride, v_stride;
                          /* a packed mixed_qkv [B, 2*H*K + HV*V] row = [q | k | v] is passed as
                             q = x, k = x + H*K, v = x + 2*H*K, all strides 2*H*K + HV*V */
    int32_t gate_mode;    /* gdn_gate_mode */
    const void *a;        /* RAW: [B, HV] in_dtype */
    const void *b;        /* RAW: [B, HV] in_dtype */
    const float *A_log;   /* RAW: [HV] */
    const float *dt_bias; /* RAW: [HV] */
    const float *g;       /* DIRECT: [B, HV] log-decay */
    const float *beta;    /* DIRECT: [B, HV] */
    float scale;          /* multiplies q after normalisation; 0 selects K^-1/2 */
    int32_t use_qk_l2norm;/* 1: normalise q and k in the kernel (as above); 0: use them as given */
    void *state;          /* [num_slots, HV, V, K] in state_dtype, read and written in place */
    void *out;            /* [B, HV, V] out_dtype (the [B, 1, HV, V] decode output) */
    int32_t *err_flags;   /* optional, may be NULL: GDN_DEVERR_* bits are OR-ed in */
    int32_t state_dtype;  /* GDN_F32 (default), or GDN_BF16: the state is stored in bf16 and the
                             step computes in fp32; out comes from the updated state before it is
                             rounded (nearest even) for storage. bf16 storage is supported by
                             gdn_decode_step and gdn_decode_step_indexed; gdn_decode_buffered
                             returns GDN_ERR_DTYPE for it. */
} gdn_step_args;

/* Ring of the buffered (output-only) decode; see gdn_decode_buffered. */
typedef struct gdn_ring_args {
    int32_t L;                /* ring length, 1 <= L <= 64 */
    int32_t ring_dtype;       /* gdn_dtype of d_cache and k_cache */
    void *d_cache;            /* [num_slots, HV, L, V] delta records */
    void *k_cache;            /* [num_slots, H, L, K] normalised-key records */
    float *g_cache;           /* [num_slots, HV, L] log-decay records */
    const int32_t *write_pos; /* [B] cursor of each row, 0 <= write_pos[b] < L; read only */
    int32_t kernel;           /* GDN_KERNEL_AUTO (0): the persistent pipelined kernel when it applies and
                                 L > 1, else the per-tile kernel; GDN_KERNEL_TILE (1) / GDN_KERNEL_PIPE
                                 (2) / GDN_KERNEL_STAGE (3, one CTA per tile staged in shared memory)
                                 force one
                                 (PIPE and STAGE need K == V == 128, L == 1 or a multiple of 4, and
                                 16-byte aligned rows and rings: GDN_ERR_SHAPE or GDN_ERR_ALIGN
                                 otherwise) */
} gdn_ring_args;

typedef enum gdn_kernel { GDN_KERNEL_AUTO = 0, GDN_KERNEL_TILE = 1, GDN_KERNEL_PIPE = 2, GDN_KERNEL_STAGE = 3 } gdn_kernel;

typedef enum gdn_fused_gate {
    GDN_FUSED_GATE_KDA = 0,   /* one log-decay per key channel, bounded below by lower_bound */
    GDN_FUSED_GATE_GDN = 1    /* one log-decay per head: -exp(A_log[h]) * softplus(raw_g[t,h] + dt_bias[h]) */
} gdn_fused_gate;

typedef enum gdn_act { GDN_ACT_SILU = 0, GDN_ACT_SIGMOID = 1 } gdn_act;

/* Arguments of the fused decode (conv update -> delta step -> gated RMSNorm). H == HV == heads,
 * K == V == head_dim, dim = heads * head_dim. All bf16 tensors are bf16; all others fp32. */
typedef struct gdn_fused_args {
    int32_t T;                /* tokens (rows) */
    int32_t heads;
    int32_t head_dim;         /* 16, 32, 64 or 128 */
    int32_t num_slots;        /* pool size of both state and conv_state */
    const void *x;            /* bf16 [T, 3*dim], row = [q | k | v] channels before the conv */
    int64_t x_stride;         /* row stride of x */
    const float *conv_w;      /* [3*dim, 4]; tap 3 multiplies the current input */
    const float *conv_b;      /* [3*dim] or NULL */
    void *conv_state;         /* bf16, logical [num_slots, 3*dim, 3] (tap 0 = oldest input), in place */
    int64_t cs_stride_slot, cs_stride_chan, cs_stride_tap;
                              /* "DS" physical [slots, 3*dim, 3]: (9*dim, 3, 1);
                                 "SD" physical [slots, 3, 3*dim] seen transposed: (9*dim, 1, 3*dim) */
    int32_t gate_kind;        /* gdn_fused_gate */
    int32_t kda_gate_form;    /* KDA only. 0: g = max(lower_bound, -exp(A_log[h]) * softplus(raw + dt_bias));
                                 1: g = lower_bound * sigmoid(exp(A_log[h]) * (raw + dt_bias)) */
    const void *raw_g;        /* bf16: KDA [T, heads, head_dim]; GDN [T, heads] */
    const void *raw_beta;     /* bf16 [T, heads]; beta = sigmoid(raw_beta) */
    const float *A_log;       /* [heads] */
    const float *dt_bias;     /* KDA [heads*head_dim]; GDN [heads] */
    float lower_bound;        /* KDA bound, e.g. -5 */
    float scale;              /* q scale after normalisation; 0 selects head_dim^-1/2 */
    int32_t use_qk_l2norm;
    float *state;             /* [num_slots, heads, head_dim, head_dim] fp32, in place */
    const int32_t *state_indices; /* [T] slot of each token (for state and conv_state) */
    int32_t pad_slot_id;      /* rows with this index are skipped, out = 0 */
    const void *out_gate;     /* bf16 [T, heads, head_dim] */
    const float *norm_w;      /* [head_dim] */
    float norm_eps;           /* e.g. 1e-5 */
    int32_t gate_act;         /* gdn_act applied to out_gate */
    void *out;                /* bf16 [T, heads, head_dim] */
    int32_t *err_flags;       /* optional */
    int32_t kernel;           /* GDN_KERNEL_AUTO: when head_dim == 128, the conv state is in the DS or
                                 SD layout, rows are 16-byte aligned and there are more than two
                                 (token, head) tiles per SM, one CTA per tile staged in shared memory
                                 by bulk copies from twelve tiles per SM and the persistent pipelined
                                 kernel below that; else the per-tile kernel. GDN_KERNEL_TILE /
                                 GDN_KERNEL_PIPE / GDN_KERNEL_STAGE force one */
    int64_t raw_g_stride;     /* row (token) strides in elements of raw_g, raw_beta and out_gate, at
                                 least the dense row width; 0 selects the dense width. The pipelined */
    int64_t raw_beta_stride;  /* kernel needs out_gate's (and a KDA raw_g's) to be a multiple of 8, */
    int64_t out_gate_stride;  /* like x_stride. Lets the op read views of one projection output. */
} gdn_fused_args;

/*
 * gdn_decode_step -- one decode step, row b on slot b (num_slots >= B).
 * Source: "Optimization Log: Qwen3.5-27B Dense on B200", Kernel 4 Math block; q/k treatment as
 * in "Microbenchmark: buffered output-only GDN decode", _bench_cfg (run_packed).
 * HBM traffic: the state tile is read once and written once (2*B*HV*V*K*4 bytes per call, or
 * 2*B*HV*V*K*2 with a bf16 state).
 */
int gdn_decode_step(const gdn_step_args *args, gdn_stream_t stream);

/*
 * gdn_decode_step_indexed -- the packed decode over a slot pool: row b uses state slot
 * cache_indices[b] (device int32 [B]); a row whose index equals pad_slot_id is skipped (state
 * untouched, out zeroed). Source: "Microbenchmark: buffered output-only GDN decode", _bench_cfg
 * (run_packed: ssm_state_indices); the pad convention follows "Microbenchmark for the fused
 * Kimi-K3 KDA decode kernel on ROCm", class Inputs (slot 0 is the NULL block, skipped).
 */
int gdn_decode_step_indexed(const gdn_step_args *args, const int32_t *cache_indices,
                            int32_t pad_slot_id, gdn_stream_t stream);

/*
 * gdn_decode_step_indexed_chained -- gdn_decode_step_indexed for the layers of a multi-layer
 * decode (one call per layer, each with its own state pool, e.g. under one CUDA graph). The
 * kernel is a programmatic dependent launch: it may start while the kernel before it on `stream`
 * is still running, reads cache_indices and loads its state tiles, and waits for that kernel to
 * complete before it reads q, k, v, the gate inputs or the gates and before it writes anything.
 * Every other buffer may be that kernel's output. Because each chained kernel lets the next one
 * start at once, a chained call may overlap any kernel of the run of consecutive chained calls
 * before it and the library call just before that run (an ordinary step call lets the next kernel
 * start once the work before it is complete): no kernel in that run, nor that call, may write this
 * call's state tiles or cache_indices. Give every chained layer its own state pool, and make the
 * first call of each step an ordinary call on a pool of its own, so that two calls on the same
 * pool are never in one run. The overlap takes one launch gap and the
 * previous layer's tail off each layer. A bf16 state at K = V = 128 from 128 tiles on, and grids
 * of eight or more waves of CTAs, run the ordinary kernel (no overlap). Arguments, results and
 * status codes as for gdn_decode_step_indexed. Source: as gdn_decode_step_indexed; the layer loop is the model of
 * "Optimization Log: Qwen3.5-27B Dense on B200" (decode is launch-bound at small batch, "Triton
 * decode kernel + MBU analysis", Kernel design).
 */
int gdn_decode_step_indexed_chained(const gdn_step_args *args, const int32_t *cache_indices,
                                    int32_t pad_slot_id, gdn_stream_t stream);

/*
 * gdn_decode_buffered -- the buffered, output-only decode. The state pool holds checkpoints S_c.
 * For row b with cursor p = write_pos[b]: the step acts on the state reached by replaying ring
 * records j < p on S_c (S <- exp(g_j) S + d_j k_j^T), appends its own records (delta, k_hat, g)
 * at ring position p (rounded to ring_dtype), and only when p == L-1 writes the resulting state
 * back to S_c. The kernel reads write_pos and never advances it: the caller moves each cursor to
 * (p + 1) % L between calls. L = 1 is the packed step. The k record of q/k head h is written by
 * one value head of its group. Source: "Microbenchmark: buffered output-only GDN decode", module
 * docstring and _bench_cfg (run_replay, time_at); traffic per call is a read of every tile plus,
 * on the flush call, a write: (1 + 1/L) x state bytes per step over a cycle.
 */
int gdn_decode_buffered(const gdn_step_args *args, const int32_t *cache_indices,
                        int32_t pad_slot_id, const gdn_ring_args *ring, gdn_stream_t stream);

/*
 * gdn_decode_fused -- one launch for: width-4 causal conv1d update with SiLU on the 3*dim q/k/v
 * channels (conv state shifted in place), the delta step with per-key-channel (KDA) or per-head
 * (GDN) decay and beta = sigmoid(raw_beta), and the gated RMSNorm
 *     out = o / sqrt(mean(o^2) + norm_eps) * norm_w * act(out_gate)
 * over each head's head_dim outputs, stored as bf16. The conv output is not rounded between
 * the conv and the step. Source: "Microbenchmark for the fused Kimi-K3 KDA decode kernel on
 * ROCm": module docstring, class Inputs, triton_chain, _gated_rmsnorm and fused;
 * "Optimization Log", Kernel 2 (rmsnorm * silu(gate)) and Kernel 5 (shift + insert + dot + SiLU).
 */
int gdn_decode_fused(const gdn_fused_args *args, gdn_stream_t stream);

/*
 * gdn_selftest_bounded_wait -- a check of the bounded waits inside the pipelined kernels (the
 * pages have no counterpart; it is a library self-test). One CTA of 128 threads waits on an
 * mbarrier; with arrive != 0 one thread arrives and the wait completes; with arrive == 0 nothing
 * arrives, the waits give up after limit_cycles SM clock cycles, GDN_DEVERR_TIMEOUT is OR-ed into
 * *err_flags (a device int32) and the kernel returns normally. Returns GDN_OK, GDN_ERR_NULL,
 * GDN_ERR_ARG (limit_cycles < 1) or GDN_ERR_LAUNCH.
 */
int gdn_selftest_bounded_wait(int32_t *err_flags, int64_t limit_cycles, int32_t arrive, gdn_stream_t stream);

/* Static text for a gdn_status code. */
const char *gdn_strerror(int status);

/* ABI checks for bindings: sizeof of the args structs (which: 0 step, 1 ring, 2 fused, 3 the
 * decode projection's gdn_gemv_args of gdn_gemv.h, 4 gdn_front_args of gdn_front.h, 5
 * mamba_decode_args of mamba_decode.h). */
size_t gdn_abi_struct_size(int which);

/* Library ABI version (incremented on any change of the args structs; currently 7). */
int gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DECODE_H */
