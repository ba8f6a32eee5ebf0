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
// A 32-bit store into a peer CTA's shared memory (published to it by the
// next cluster barrier).
__device__ __forceinline__ void st_dsmem_u32(uint32_t remote, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(remote), "r"(v) : "memory");
}

// Four fp32 values into a peer CTA's shared memory, completing 16 bytes of
// the transaction count of the peer's mbarrier at remote_bar.
__device__ __forceinline__ void st_async_f4(uint32_t remote, float a, float b, float c, float d, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];\n" ::"r"(
                     remote),
                 "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t remote)
{
    float4 v;
    asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote));
    return v;
}

}  // namespace lora
