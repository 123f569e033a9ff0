/*
 * mamba_decode.h -- C ABI of the Mamba-1 selective-scan decode step in libgdn_decode.so (the
 * GB300 / sm_103a decode library; see gdn_decode.h for the conventions both headers share:
 * device pointers owned by the caller, nothing allocated or synchronised, launches only on
 * `stream`, host-side argument checks before any CUDA call, negative gdn_status on error).
 *
 * The operation ("Triton decode kernel + MBU analysis", section "Kernel design"), for each row b
 * and channel d with state h[b, d, 0..N) (fp32):
 *     dA = exp(dt[b,d] * A[d, :])          dB = dt[b,d] * Bm[b, :]
 *     h  <- dA * h + dB * x[b,d]           (element-wise over the N state entries)
 *     y[b,d] = sum_n Cm[b,n] h[n]  (+ Dskip[d] x[b,d])  (* silu(z[b,d]))
 * dt is used as given (the softplus of the projection, if any, is the caller's). Arithmetic is
 * fp32 whatever the input dtype; the state is fp32 end to end.
 * HBM traffic (the page's bytes model): B * D * (20 N + 24) bytes per call; the state alone is
 * 8 * B * D * N bytes.
 */
#ifndef MAMBA_DECODE_H
#define MAMBA_DECODE_H

#include <stdint.h>

#include "gdn_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mamba_decode_args {
    int32_t B;              /* rows */
    int32_t D;              /* channels (d_inner) */
    int32_t N;              /* state size per channel, 1 .. 128 */
    int32_t in_dtype;       /* gdn_dtype of x, dt, Bm, Cm, z */
    int32_t out_dtype;      /* gdn_dtype of y */
    const void *x;          /* [B, D] dense */
    const void *dt;         /* [B, D] dense */
    const float *A;         /* [D, N] dense (negative for a decaying state) */
    const void *Bm;         /* [B, N] dense: the SSM's input matrix row of each b */
    const void *Cm;         /* [B, N] dense: the SSM's output matrix row of each b */
    const float *Dskip;     /* [D] or NULL: skip term */
    const void *z;          /* [B, D] or NULL: output gate */
    float *h;               /* [B, D, N] fp32 state: read; updated in place when h_out is NULL */
    float *h_out;           /* [B, D, N] or NULL: where the new state goes (may not overlap h) */
    void *y;                /* [B, D] out_dtype */
    int32_t *err_flags;     /* optional device word: GDN_DEVERR_TIMEOUT is ORed in when a bounded
                               wait of the staged kernel gives up (its rows are then left as they
                               were); NULL: not reported */
} mamba_decode_args;

/*
 * mamba_selective_scan_decode -- one decode step of the Mamba-1 selective scan, one launch.
 * Source: "Triton decode kernel + MBU analysis", sections "Kernel design" (the per-element math,
 * fp32 accumulation, fp32 state) and "Microbench" (the bytes-moved model). Returns GDN_OK,
 * GDN_ERR_NULL, GDN_ERR_SHAPE (N outside 1..128, negative sizes), GDN_ERR_DTYPE, GDN_ERR_ALIGN
 * (h, h_out and A must be 16-byte aligned when N is a multiple of 4) or GDN_ERR_LAUNCH. For
 * N = 16, 32, 64 or 128 and batches of at least two waves of its 16 KB blocks (two batch rows of a
 * channel range; 32 KB, four rows, from six waves), the call runs a kernel that bulk-copies
 * blocks of state, B and C into shared memory (B and C must then be 16-byte aligned, else another
 * kernel runs); a bounded wait there reports GDN_DEVERR_TIMEOUT through err_flags. Launches only;
 * no allocation, no synchronisation.
 */
int mamba_selective_scan_decode(const mamba_decode_args *args, gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_DECODE_H */
