/*
 * gdn_gemv.h -- C ABI of the decode projection (GEMV) in libgdn_decode.so; conventions as in
 * gdn_decode.h (device pointers owned by the caller, nothing allocated or synchronised, launches
 * only on `stream`, host-side checks before any CUDA call, negative gdn_status on error).
 *
 * The operation ("Optimization Log: Qwen3.5-27B Dense on B200", Kernel 3: BF16 GEMV with
 * split-K, the projections that dominate decode time): for T token rows (decode batch, T >= 1),
 *     y[t, n] = sum_k x[t, k] * W[n, k]        (bf16 x and W, fp32 accumulation)
 * with W stored one output row per line ([N, Kd], the nn.Linear weight layout). Split-K divides
 * the Kd inputs into `splits` ranges whose fp32 partial sums go to a caller workspace and are then
 * added in a fixed order (deterministic), so that narrow projections still spread over every SM.
 * HBM traffic: the weights once per 8 token rows, 2 * N * Kd bytes for T <= 8.
 */
#ifndef GDN_GEMV_H
#define GDN_GEMV_H

#include <stddef.h>
#include <stdint.h>

#include "gdn_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gdn_gemv_args {
    int32_t T;              /* token rows, >= 0 */
    int32_t N;              /* outputs */
    int32_t Kd;             /* inputs, a multiple of 8 */
    int32_t out_dtype;      /* gdn_dtype of y */
    const void *x;          /* bf16 [T, Kd], row stride x_stride (a multiple of 8), 16-byte aligned */
    int64_t x_stride;
    const void *W;          /* bf16 [N, Kd] dense, 16-byte aligned */
    void *y;                /* [T, N] out_dtype, row stride y_stride */
    int64_t y_stride;
    int32_t splits;         /* K ranges: 0 lets the library choose (gdn_gemv_default_splits) */
    float *workspace;       /* fp32, at least gdn_gemv_workspace_bytes(T, N, splits) bytes when the
                               split count is above 1; unused (may be NULL) otherwise */
    size_t workspace_bytes;
} gdn_gemv_args;

/* The split count gdn_gemv_bf16 uses when args->splits == 0 (enough CTAs to cover every SM about
 * four times; at most 16, and at least 256 inputs per range). */
int32_t gdn_gemv_default_splits(int32_t T, int32_t N, int32_t Kd);

/* Workspace bytes a call with this split count needs (0 when splits <= 1). */
size_t gdn_gemv_workspace_bytes(int32_t T, int32_t N, int32_t splits);

/*
 * gdn_gemv_bf16 -- y = x W^T for decode. Source: "Optimization Log: Qwen3.5-27B Dense on B200",
 * Kernel 3 (BF16 GEMV with split-K; M = 1 decode; key shapes [5120, 17408] and [17408, 5120]).
 * Returns GDN_OK, GDN_ERR_NULL (a missing pointer, or no workspace when one is needed),
 * GDN_ERR_SHAPE (negative sizes, Kd not a multiple of 8, workspace too small, splits > 64),
 * GDN_ERR_DTYPE, GDN_ERR_ALIGN or GDN_ERR_LAUNCH.
 */
int gdn_gemv_bf16(const gdn_gemv_args *args, gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GEMV_H */
