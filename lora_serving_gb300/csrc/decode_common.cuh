// decode_common.cuh -- device helpers shared by the decode-row kernels
// (the one-launch grouped kernel and the two-launch grouped shrink/expand):
// mbarriers with bounded waits, bulk and 16-byte asynchronous copies,
// programmatic-dependent-launch controls, cluster/DSMEM access, the
// mma.sync m16n8k16 building blocks, and the unit lookup over gather groups.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "cluster.cuh"
#include "common.cuh"

namespace lora {
namespace dec {

constexpr int kRB = 16;                                   // decode rows per unit (the mma M)
constexpr unsigned long long kTimeoutNs = 200000000ull;   // bounded waits: 0.2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long gtime()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same test, letting the hardware suspend the thread for up to
// kSuspendNs while the phase is incomplete (it resumes when the phase
// completes): a waiting warp does not spin through issue slots.
constexpr uint32_t kSuspendNs = 1000000u;
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity to complete; false after
// kTimeoutNs (the caller flags the timeout and winds down).
static __device__ __noinline__ bool mbar_wait(uint64_t* bar, unsigned parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = gtime();
    while (!mbar_try_wait_suspend(bar, parity))
        if (gtime() - t0 > kTimeoutNs) return false;
    return true;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid)
{
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Requests the 128-byte line holding p into L2 (no completion, no registers).
__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// v (two fp32 values) -> packed bf16 hi pair and bf16 lo pair (v ~= hi + lo).
__device__ __forceinline__ void split_hi_lo(float a, float b, uint32_t& hi, uint32_t& lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // .x = a (low half)
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Units of a group: ceil(len / 16), or 0 (and bad) when its bounds fall
// outside [0, n_pos) -- so perm is never read out of range.
__device__ __forceinline__ int group_units(int s, int e, int n_pos, bool& bad)
{
    const bool sane = s >= 0 && e <= n_pos && s <= e;
    bad |= !sane;
    return sane ? (e - s + kRB - 1) / kRB : 0;
}

struct UnitInfo {
    int g, pos0, nrows, slot, found, bad;
};

// Unit u -> (group, first position, rows, slot).  Every thread of the CTA
// takes part and the answer is uniform across the CTA (and across a
// cluster, whose CTAs all map to the same unit).  The group table is read
// NT groups per round trip (one group per thread, block-wide prefix sum),
// together with the permutation when it fits in s_perm.  `bad` is set for
// a malformed table (a group outside [0, n_pos), or a table that does not
// start at 0 and end at n_pos), and when the table holds more units than the grid's
// grid_units (the host's bound on the longest group was understated, so
// some rows have no CTA): every CTA sees the same total and reports it.
template <int NT, class Params>
__device__ __forceinline__ UnitInfo find_unit(const Params& p, int u, int* s_perm, bool stage_perm, int grid_units)
{
    __shared__ int s_warp[NT / 32];
    __shared__ UnitInfo s_info;
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_info.found = 0;
        // the table must cover [0, n_pos): its first entry 0, its last n_pos
        s_bad = p.n_groups > 0 && (__ldg(p.gstarts) != 0 || __ldg(p.gstarts + p.n_groups) != p.n_pos);
    }
    if (stage_perm)
        for (int i = tid; i < p.n_pos; i += NT) s_perm[i] = __ldg(p.perm + i);
    int base = 0;   // units in the groups of earlier rounds
    for (int g0 = 0; g0 < p.n_groups; g0 += NT) {
        const int gi = g0 + tid;
        int s = 0, e = 0, sl = -1;
        bool bad = false;
        int n = 0;
        if (gi < p.n_groups) {
            s = __ldg(p.gstarts + gi);
            e = __ldg(p.gstarts + gi + 1);
            sl = __ldg(p.gslot + gi);
            n = group_units(s, e, p.n_pos, bad);
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) {
            const int c = s_warp[w];
            if (w < warp) before += c;
            total += c;
        }
        incl += base + before;
        const int excl = incl - n;
        if (bad) atomicOr(&s_bad, 1);
        if (gi < p.n_groups && u >= excl && u < incl) {
            UnitInfo info;
            info.g = gi;
            info.pos0 = s + (u - excl) * kRB;
            info.nrows = min(kRB, e - info.pos0);
            info.slot = sl;
            info.found = 1;
            info.bad = 0;
            s_info = info;
        }
        base += total;
        __syncthreads();   // s_warp is rewritten by the next round
    }
    if (p.n_groups <= 0) __syncthreads();
    UnitInfo r = s_info;
    r.bad = s_bad || base > grid_units;
    return r;
}

}  // namespace dec
}  // namespace lora
