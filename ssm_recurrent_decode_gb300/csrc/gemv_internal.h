// gemv_internal.h -- declarations shared by the decode projection's translation units (internal to
// libgdn_decode.so).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>

#include "gdn_common.cuh"
#include "gdn_gemv.h"

namespace gdn {

// How a launch's K ranges are combined: one range writes y itself; up to kGemvMaxCluster ranges
// of a row tile form one thread-block cluster and add their sums through distributed shared
// memory, in range order; more ranges write partial sums to the caller's workspace, added in range
// order by a second kernel.
constexpr int kGemvReduceNone = 0;
constexpr int kGemvReduceWorkspace = 1;
constexpr int kGemvReduceCluster = 2;
constexpr int kGemvMaxCluster = 8;   // the portable cluster size

inline int gemv_reduce_mode(int splits)
{
    return splits <= 1 ? kGemvReduceNone : (splits <= kGemvMaxCluster ? kGemvReduceCluster : kGemvReduceWorkspace);
}

// Debug build: y[t, n] and the workspace slot (split, t, n) lie inside y [T, y_stride] and the
// workspace the arguments describe (GDN_IN of gdn_common.cuh; the constant true in release).
__device__ __forceinline__ bool gemv_y_in_range(const gdn_gemv_args &P, int t, int n)
{
    return GDN_IN(P.err_flags, (long long)t * P.y_stride + n, (long long)(P.T - 1) * P.y_stride + P.N) &&
           GDN_IN(P.err_flags, n, P.N);
}
__device__ __forceinline__ bool gemv_ws_in_range(const gdn_gemv_args &P, long long i)
{
    return GDN_IN(P.err_flags, i, (long long)(P.workspace_bytes / 4));
}

// y[t, n] = v, rounded to y's dtype
__device__ __forceinline__ void gemv_store(const gdn_gemv_args &P, int t, int n, float v)
{
    if (!gemv_y_in_range(P, t, n)) return;   // debug build only
    if (P.out_dtype == GDN_BF16)
        static_cast<__nv_bfloat16 *>(P.y)[(size_t)t * P.y_stride + n] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(P.y)[(size_t)t * P.y_stride + n] = v;
}

// A chained launch (below) prefetches its weights into L2 while it waits for the kernel before it
// when W takes at most half of L2; larger weights would evict one another before use.
constexpr size_t kPrefetchMaxBytes = 64u << 20;
inline bool gemv_prefetch_fits(const gdn_gemv_args &p) { return (size_t)p.N * (size_t)p.Kd * 2 <= kPrefetchMaxBytes; }

// The host checks of gdn_gemv_bf16 and its split count (*splits = 0: nothing to launch), without
// any CUDA launch; gemv_launch then launches a checked call. chained: the launch may start while
// the previous kernel on the stream finishes (programmatic dependent launch; the kernel waits for
// that kernel before it reads x).
int gemv_check(const gdn_gemv_args *a, int *splits);
int gemv_launch(const gdn_gemv_args &p, int splits, cudaStream_t stream, bool chained = false);

// tcgen05 form: output rows per CTA (the MMA's M), inputs per stage, token rows per pass (N)
constexpr int kTcRows = 128;
constexpr int kTcK = 64;              // inputs per TMA tile (one 128-byte swizzle span)
// Adjacent 64-input tiles per shared-memory stage, loaded back to back: each stage reads 256
// contiguous bytes of every weight row. On GB300 two tiles per stage in a 2-stage ring (3 CTAs
// per SM) streamed faster than one tile in a 4-stage ring (0.84 against 0.81 of the copy
// bandwidth for W [17408, 5120], 0.87 against 0.83 for [5120, 17408]); four or six tiles per
// stage fit only one CTA per SM.
constexpr int kTcChunks = 2;
constexpr int kTcStageK = kTcK * kTcChunks;
constexpr int kTcTok = 16;
constexpr int kTcMaxStages = 8;

// dynamic shared memory of a tcgen05-form CTA with `stages` stages
size_t gemv_tc_smem_bytes(int stages);

// CTAs of the tcgen05 form resident on one SM of the current device
int gemv_tc_resident_ctas(int stages);

// launches the tcgen05 form over every pass of 16 token rows (as a cluster launch when the ranges
// are combined in a cluster; a workspace sum is left to the caller); k_per_split is a multiple of
// kTcStageK
int gemv_tc_launch(const gdn_gemv_args &p, int splits, int k_per_split, int stages, cudaStream_t stream,
                   bool chained = false);

}  // namespace gdn
