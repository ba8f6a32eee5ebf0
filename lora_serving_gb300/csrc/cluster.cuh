// cluster.cuh -- thread-block cluster helpers shared by the kernels that
// split work over a cluster: rank, barrier, and distributed shared memory
// (a peer CTA's shared memory addressed through mapa).
#pragma once

#include <stdint.h>

namespace lora {

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }

// The address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(uint32_t local_addr, uint32_t rank)
{
    uint32_t remote;
    asm("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}
// Plain (non-volatile) DSMEM loads: ordering against the peers' writes is
// given by the cluster barrier, so independent loads may be issued together.
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t remote)
{
    float2 v;
    asm("ld.shared::cluster.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(remote));
    return v;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t remote)
{
    float4 v;
    asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote));
    return v;
}

}  // namespace lora
