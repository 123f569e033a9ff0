// gdn_launch.h -- launch parameters shared by the host layer (api.cu) and the kernels
// (internal to libgdn_decode.so; the public interface is include/gdn_decode.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gdn_decode.h"

namespace gdn {

// Everything one launch of the step or buffered kernel needs, resolved and validated on the host.
struct StepLaunch {
    gdn_step_args a;          // the caller's arguments (device pointers, sizes, strides)
    const int32_t *idx;       // slot of each row, or nullptr for row b -> slot b
    int32_t pad;              // rows whose index equals this are skipped
    int32_t G;                // value heads per q/k head
    float scale;              // resolved q scale
    // buffered decode only
    int32_t L;
    void *d_cache;
    void *k_cache;
    float *g_cache;
    const int32_t *write_pos;
    int32_t nst;              // pipelined kernel: shared-memory stages
};

struct FusedLaunch {
    gdn_fused_args a;
    float scale;
};

// A checked gdn_decode_fused call: its launch arguments and kernel choice.
struct FusedPlan {
    FusedLaunch p;
    bool empty;      // T == 0: nothing to launch
    bool use_pipe;   // the persistent pipelined kernel (or, with use_stage, the staged one)
    bool use_stage;  // one CTA per tile staged in shared memory
    bool sd;         // its conv state is in the SD layout
};

// The host checks of gdn_decode_fused (the same status codes) and its kernel choice; no CUDA launch.
// chained (launch_fused_plan and the launchers below): the launch may start while the previous
// kernel on the stream finishes (programmatic dependent launch); the kernel waits for that kernel
// before it reads its inputs, and reads before the wait only the state tile and the slot indices.
int prepare_fused(const gdn_fused_args *a, FusedPlan *plan);
int launch_fused_plan(const FusedPlan &plan, cudaStream_t stream, bool chained = false);

// Host launchers, one per kernel family; each dispatches on K and the dtypes. They return
// GDN_OK or GDN_ERR_LAUNCH / GDN_ERR_SHAPE and never synchronise.
// launch_step with chained: the row kernels run their chained instance as a programmatic
// dependent launch (gdn_decode_step_indexed_chained); the bf16-state kernels launch as usual.
int launch_step(const StepLaunch &p, cudaStream_t stream, bool chained = false);
int launch_buffered(const StepLaunch &p, int ring_dtype, cudaStream_t stream);
int launch_fused(const FusedLaunch &p, cudaStream_t stream, bool chained = false);

// The step for a bf16 state at K = V = 128 with each tile staged in shared memory by a bulk copy
// (step_stage_bf16.cu), and whether a call qualifies for it (bf16 state, K = V = 128, 16-byte
// aligned state and q/k/v rows).
bool step_stage_bf16_ok(const gdn_step_args &a);
int launch_step_stage_bf16(const StepLaunch &p, cudaStream_t stream);

// Dynamic shared memory the buffered kernel needs for ring length L, value dim V and key dim K.
size_t buffered_smem_bytes(int L, int V, int K);

// The persistent, warp-specialised buffered kernel (K = V = 128, 16-byte aligned rows).
int launch_buffered_pipe(const StepLaunch &p, int ring_dtype, cudaStream_t stream);
// Whether its two-stage shared-memory footprint fits in max_smem bytes per CTA.
bool buffered_pipe_fits(int L, int in_dtype, int ring_dtype, int max_smem);
// The same step with one tile per CTA staged in shared memory (the pipelined kernel's
// requirements; one stage of shared memory per CTA).
int launch_buffered_stage(const StepLaunch &p, int ring_dtype, cudaStream_t stream);

// The persistent, warp-specialised fused kernel (head_dim 128; conv state in the DS layout, or in
// the SD layout when sd is true).
int launch_fused_pipe(const FusedLaunch &p, bool sd, cudaStream_t stream, bool chained = false);
bool fused_pipe_fits(int max_smem);
// The same op with one (token, head) tile per CTA staged in shared memory (the pipelined kernel's
// requirements).
int launch_fused_stage(const FusedLaunch &p, bool sd, cudaStream_t stream, bool chained = false);

}  // namespace gdn
