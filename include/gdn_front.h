/*
 * gdn_front.h -- C ABI of the decode layer front in libgdn_decode.so: one DeltaNet layer's decode
 * forward for T token rows, from the hidden state in to the hidden state out. Conventions as in
 * gdn_decode.h (device pointers owned by the caller, nothing allocated or synchronised, launches
 * only on `stream`, host-side checks before any CUDA call, negative gdn_status on error).
 *
 * The operation ("Optimization Log: Qwen3.5-27B Dense on B200", Integration: the DeltaNet forward
 * of the model patcher is "fused proj + conv1d + recurrent + norm_gated + output"), with
 * dim = heads * head_dim and G = dim (KDA gate) or heads (GDN gate):
 *     z = x W_in^T          z [T, P] bf16, P = 4*dim + G + heads, columns
 *                           [ q | k | v (3*dim) | out_gate (dim) | raw_g (G) | raw_beta (heads) ]
 *     o = fused(z)          width-4 conv update of q|k|v -> delta step -> gated RMSNorm
 *                           (gdn_decode_fused on views of z), o [T, dim] bf16
 *     y = o W_out^T         y [T, hidden]
 * The projections are gdn_gemv_bf16 (bf16 weights, fp32 accumulation, K ranges added inside a
 * thread-block cluster), the middle step gdn_decode_fused: three launches on `stream`, all
 * checked on the host before the first one. The layout of z (which columns feed which input) is
 * this library's; a model's own projection is mapped to it by ordering the rows of W_in.
 */
#ifndef GDN_FRONT_H
#define GDN_FRONT_H

#include <stddef.h>
#include <stdint.h>

#include "gdn_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gdn_front_args {
    int32_t T;              /* token rows, >= 0 */
    int32_t hidden;         /* model width, a multiple of 8 */
    const void *x;          /* bf16 [T, hidden], row stride x_stride (a multiple of 8), 16-byte aligned */
    int64_t x_stride;
    const void *W_in;       /* bf16 [P, hidden] dense, 16-byte aligned (P from gdn_front_proj_width) */
    const void *W_out;      /* bf16 [hidden, dim] dense, 16-byte aligned */
    void *z;                /* bf16 [T, P] dense, 16-byte aligned: caller-owned scratch */
    void *o;                /* bf16 [T, dim] dense, 16-byte aligned: caller-owned scratch */
    void *y;                /* [T, hidden] y_dtype, row stride y_stride */
    int32_t y_dtype;        /* gdn_dtype of y */
    int64_t y_stride;
    int32_t in_splits;      /* K ranges of the projections, 0 .. 8 (0: the library's choice); */
    int32_t out_splits;     /* up to 8 ranges need no workspace */
    gdn_fused_args core;    /* the middle step's arguments: heads, head_dim, num_slots, conv
                               weights and state, gate kind and parameters, state, state_indices,
                               pad_slot_id, norm_w, norm_eps, gate_act, err_flags, kernel. Its T,
                               x, raw_g, raw_beta, out_gate, out and their strides are ignored and
                               set from z and o. */
} gdn_front_args;

/* P, the width of z for these head sizes and gate kind (0 for an unknown gate kind). */
int64_t gdn_front_proj_width(int32_t heads, int32_t head_dim, int32_t gate_kind);

/*
 * gdn_decode_front -- the layer's decode forward as above. Returns GDN_OK or the codes of
 * gdn_gemv_bf16 and gdn_decode_fused for the stage whose arguments fail (GDN_ERR_ARG for splits
 * outside 0 .. 8); then nothing was launched. Device-side errors go to core.err_flags as in
 * gdn_decode_fused (and GDN_DEVERR_TIMEOUT from a projection).
 * Three launches on `stream`, ordered as ordinary stream work towards the caller: the first is an
 * ordinary launch; the second and third are programmatic dependent launches that may start while
 * the launch before them finishes and wait for it before reading its output.
 */
int gdn_decode_front(const gdn_front_args *args, gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_FRONT_H */
