// gdn_cluster.cuh -- thread-block cluster primitives (internal to libgdn_decode.so): the cluster-wide
// barrier and loads from another CTA's shared memory (distributed shared memory). No multicast.
#pragma once

#include <cstdint>

namespace gdn {

// every thread of every CTA of the cluster arrives (release) and waits (acquire); all threads of a
// warp execute it together
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// the shared::cluster address of this CTA's shared-memory address `saddr` in CTA `rank`
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ float cluster_ld_f32(uint32_t caddr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(caddr) : "memory");
    return v;
}

__device__ __forceinline__ int cluster_ld_s32(uint32_t caddr)
{
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(caddr) : "memory");
    return v;
}

}  // namespace gdn
