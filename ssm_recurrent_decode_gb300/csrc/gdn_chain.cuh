// gdn_chain.cuh -- programmatic dependent launch for the chained launches of one layer call
// (internal to libgdn_decode.so).
#pragma once

#include <cuda_runtime.h>

namespace gdn {

// A kernel launched with the programmatic-serialization attribute may start while the kernel
// before it on the stream is still running. It must call grid_dependency_wait, in every CTA and
// on every path, before it touches memory that kernel writes; the wait returns once that kernel
// has completed and its writes are visible, and at once when the attribute was not given.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allows the next kernel on the stream, if launched with the attribute, to start its CTAs.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Host side: marks a launch as programmatically dependent on the previous kernel of its stream.
inline void set_programmatic(cudaLaunchAttribute &attr)
{
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
}

// The start of an ordinary (not chained) launch: wait for the kernel before it on the stream, then
// let the next kernel start its CTAs. The kernel touches no memory before the wait, so the stream
// order is the usual one; the next call's CTAs may become resident while this one drains (they
// block in their own wait, or, for a chained call, load only their own state). The trigger comes
// after the wait, so a chained call that follows can overlap this kernel and no earlier one.
__device__ __forceinline__ void ordinary_launch_start()
{
    grid_dependency_wait();
    grid_launch_dependents();
}

// An ordinary launch with the programmatic attribute (for kernels that begin with
// ordinary_launch_start): consecutive library calls on a stream hide each other's launch.
template <typename Kern, typename... Args>
inline cudaError_t launch_ordinary(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_programmatic(attr[0]);
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace gdn
