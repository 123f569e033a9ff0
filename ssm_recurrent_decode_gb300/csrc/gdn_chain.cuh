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

}  // namespace gdn
