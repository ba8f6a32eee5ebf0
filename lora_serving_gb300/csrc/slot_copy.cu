// slot_copy.cu -- one launch that gathers a batch's adapter loads from the
// slot manager's pinned host cache into the device slots.
//
// vLLM offline multi-LoRA page, step 2: adapters wait in host memory
// (max_cpu_loras) and are copied into one of max_loras GPU slots when a
// batch needs them.  A prepared adapter is one piece per projection for A
// and for B (80 KB each for a rank-16 Llama-3.2-3B projection); issued as
// separate copies, per-copy overhead bounds the load rate.  Here the GPU
// reads the mapped host buffers itself: the pieces of every adapter the
// batch loads are laid end to end in 16-byte units, each CTA moves a
// contiguous 32 KB of that range (8 units in flight per thread before the
// stores), and one launch covers the batch.

#include "launch.h"
#include "slot_copy.h"

namespace lora {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;
constexpr uint64_t kUnitsPerCta = static_cast<uint64_t>(kCopyThreads) * kCopyUnroll;   // 2048 x 16 B

struct CopyParams {
    CopySeg seg[kMaxCopySegs];
    uint64_t start[kMaxCopySegs + 1];   // first unit of each piece; start[n] = total units
    int n;
};

__global__ void __launch_bounds__(kCopyThreads) slot_copy_kernel(const __grid_constant__ CopyParams p)
{
    const uint64_t u0 = static_cast<uint64_t>(blockIdx.x) * kUnitsPerCta;
    // the piece holding this CTA's first unit
    int s = 0;
    while (s + 1 < p.n && p.start[s + 1] <= u0) ++s;
    uint4 v[kCopyUnroll];
    uint64_t u[kCopyUnroll];
    int sg[kCopyUnroll];
#pragma unroll
    for (int i = 0; i < kCopyUnroll; ++i) {
        u[i] = u0 + static_cast<uint64_t>(i) * kCopyThreads + threadIdx.x;
        int k = s;
        while (k + 1 < p.n && p.start[k + 1] <= u[i]) ++k;
        sg[i] = k;
        if (u[i] < p.start[p.n])
            v[i] = reinterpret_cast<const uint4*>(p.seg[k].src)[u[i] - p.start[k]];
    }
#pragma unroll
    for (int i = 0; i < kCopyUnroll; ++i)
        if (u[i] < p.start[p.n]) reinterpret_cast<uint4*>(p.seg[sg[i]].dst)[u[i] - p.start[sg[i]]] = v[i];
}

}  // namespace

cudaError_t launch_slot_copy(const CopySeg* segs, int n, cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    if (n > kMaxCopySegs) return cudaErrorInvalidValue;
    CopyParams p{};
    p.n = n;
    uint64_t total = 0;
    for (int i = 0; i < n; ++i) {
        if ((segs[i].bytes & 15u) || (reinterpret_cast<uintptr_t>(segs[i].src) & 15u) ||
            (reinterpret_cast<uintptr_t>(segs[i].dst) & 15u))
            return cudaErrorInvalidValue;
        p.seg[i] = segs[i];
        p.start[i] = total;
        total += segs[i].bytes / 16;
    }
    p.start[n] = total;
    if (total == 0) return cudaSuccess;
    const uint64_t grid = (total + kUnitsPerCta - 1) / kUnitsPerCta;
    if (grid > 0x7FFFFFFFull) return cudaErrorInvalidConfiguration;
    slot_copy_kernel<<<static_cast<unsigned>(grid), kCopyThreads, 0, stream>>>(p);
    note_launch();
    return cudaGetLastError();
}

}  // namespace lora
