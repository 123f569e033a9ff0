/*
 * gdn_gemv.h -- C ABI of the decode projection (GEMV) in libgdn_decode.so; conventions as in
 * gdn_decode.h (device pointers owned by the caller, nothing allocated or synchronised, launches
 * only on `stream`, host-side checks before any CUDA call, negative gdn_status on error).
 *
 * The operation ("Optimization Log: Qwen3.5-27B Dense on B200", Kernel 3: BF16 GEMV with
 * split-K, the projections that dominate decode time): for T token rows (decode batch, T >= 1),
 *     y[t, n] = sum_k x[t, k] * W[n, k]        (bf16 x and W, fp32 accumulation)
 * with W stored one output row per line ([N, Kd], the nn.Linear weight layout). Split-K divides
 * the Kd inputs into `splits` ranges so that narrow projections still spread over every SM; the
 * ranges' fp32 partial sums are added in range order (deterministic): with up to 8 ranges inside
 * the launch (the ranges of a row tile form a thread-block cluster and add through distributed
 * shared memory), with more in a caller workspace and a second launch.
 * HBM traffic: the weights once per pass of up to 16 token rows, 2 * N * Kd bytes for T <= 16.
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
                               split count is above 8; unused (may be NULL) otherwise */
    size_t workspace_bytes;
    int32_t *err_flags;     /* optional device word; a kernel that gives up a bounded wait ORs
                               GDN_DEVERR_TIMEOUT into it and leaves its outputs unwritten (with
                               more than 8 K ranges: sets them to NaN) */
} gdn_gemv_args;

/* The split count gdn_gemv_bf16 uses when args->splits == 0: a power of two up to 8 (so no
 * workspace is needed) with at least 512 inputs per range, chosen so that the grid fills one wave
 * of resident CTAs (or at least two) and each CTA's slice of x fits its shared-memory staging
 * budget. Queries the current device's SM count and kernel occupancy once (no allocation, no
 * launch). */
int32_t gdn_gemv_default_splits(int32_t T, int32_t N, int32_t Kd);

/* Workspace bytes a call with this split count needs (0 when splits <= 8). */
size_t gdn_gemv_workspace_bytes(int32_t T, int32_t N, int32_t splits);

/*
 * gdn_gemv_bf16 -- y = x W^T for decode. Source: "Optimization Log: Qwen3.5-27B Dense on B200",
 * Kernel 3 (BF16 GEMV with split-K; M = 1 decode; key shapes [5120, 17408] and [17408, 5120]).
 * Returns GDN_OK, GDN_ERR_NULL (a missing pointer, or no workspace when one is needed),
 * GDN_ERR_SHAPE (negative sizes, Kd not a multiple of 8, workspace too small, splits > 64),
 * GDN_ERR_DTYPE, GDN_ERR_ALIGN or GDN_ERR_LAUNCH. From 2 token rows on the library's tensor-core
 * kernel waits on mbarriers with a bound; a wait that gives up ORs GDN_DEVERR_TIMEOUT into
 * args->err_flags (when given) and leaves that CTA's outputs of y unwritten, or, with more than 8
 * K ranges (a workspace), writes NaN into its partial sums so that those outputs of y come out
 * NaN rather than sums of stale workspace values.
 */
int gdn_gemv_bf16(const gdn_gemv_args *args, gdn_stream_t stream);

/*
 * gdn_gemv_set_wait_limit -- test hook, not for production use: sets, for the whole process, the
 * number of SM clock cycles after which a wait of the tensor-core projection (T >= 2) gives up;
 * 0 restores the default (2^31 cycles, about one second). With a limit far below a copy's latency
 * a test can make the waits run out and check that the call returns normally, reports
 * GDN_DEVERR_TIMEOUT and leaves y unwritten or NaN; the waits that let copies and MMAs in flight
 * finish after a give-up keep the default limit. Returns the previous setting. Launches nothing.
 * No counterpart on the source pages.
 */
int64_t gdn_gemv_set_wait_limit(int64_t cycles);

/* Size of the fixed buffer behind gdn_gemv_bf16_noalloc, in fp32 values (4 MiB). */
#define GDN_GEMV_NOALLOC_MAX_FLOATS (1 << 20)

/*
 * gdn_gemv_bf16_noalloc -- the same projection for callers that cannot allocate device memory:
 * code handed only raw device pointers by a host framework that owns every allocation, serving
 * loops that must never call cudaMalloc (it can synchronise the device and stall other work),
 * and runtimes with a fixed, pre-planned memory budget. The source pages have no counterpart; it
 * is a library convenience.
 *
 * Arguments as for gdn_gemv_bf16, except that workspace and workspace_bytes are ignored: when the
 * call needs a workspace (more than 8 K ranges), its fp32 partial sums go to a buffer of
 * GDN_GEMV_NOALLOC_MAX_FLOATS values that the library keeps on every GPU that loads it, until the
 * process exits. A call whose splits * T * N exceeds that size is rejected with GDN_ERR_SCRATCH
 * before anything is launched, after the argument checks of gdn_gemv_bf16 (pass 8 or fewer
 * ranges, which need no buffer, or use gdn_gemv_bf16 with your own workspace). Nothing here
 * allocates: the first call in a CUDA context that uses the buffer looks up that context's buffer
 * address (cudaGetSymbolAddress) with the device current, so make that first call before any
 * stream capture. With lazy module loading (CUDA's default) that first lookup may also be what
 * makes the driver load this library's device code, and with it the 4 MiB array, on that device;
 * later calls change no device memory reservation. The address is remembered per context: after
 * cudaDeviceReset (a new primary context) the next call looks it up again. Every call in a context
 * shares the one buffer, which keeps the last call's partial sums (each call writes all the sums
 * it reads, so no clearing is needed); calls that can run at the same time on the GPU, e.g. on two
 * streams, race on it and must be ordered.
 * Returns the codes of gdn_gemv_bf16, and GDN_ERR_SCRATCH.
 */
int gdn_gemv_bf16_noalloc(const gdn_gemv_args *args, gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GEMV_H */
