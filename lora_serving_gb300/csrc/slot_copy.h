// slot_copy.h -- the adapter slot manager's load copy (host-side declaration;
// plain C++ so that host-only translation units can include it).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lora {

// One contiguous piece to move: `bytes` (a multiple of 16) from src to dst,
// both 16-byte aligned.  src may be pinned, mapped host memory (its device
// address), dst device memory.
struct CopySeg {
    const void* src;
    void* dst;
    uint64_t bytes;
};

constexpr int kMaxCopySegs = 64;   // pieces per launch

// Moves n (<= kMaxCopySegs) pieces in one kernel launch on `stream`.
cudaError_t launch_slot_copy(const CopySeg* segs, int n, cudaStream_t stream);

}  // namespace lora
