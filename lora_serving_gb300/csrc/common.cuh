// common.cuh -- device helpers shared by the LoRA kernels: bf16 vector
// unpacking, the position -> (row, slot) map used by BGMV (per-token ids)
// and SGMV (segments, optionally through a row permutation), and the
// non-trapping device status flags.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lora.h"

namespace lora {

typedef uint16_t bf16_t;

// Upper/lower bf16 of a 32-bit word, as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Dot product of 8 bf16 pairs packed in two uint4, accumulated in fp32.
__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc)
{
    acc = fmaf(bf16_lo(a.x), bf16_lo(b.x), acc);
    acc = fmaf(bf16_hi(a.x), bf16_hi(b.x), acc);
    acc = fmaf(bf16_lo(a.y), bf16_lo(b.y), acc);
    acc = fmaf(bf16_hi(a.y), bf16_hi(b.y), acc);
    acc = fmaf(bf16_lo(a.z), bf16_lo(b.z), acc);
    acc = fmaf(bf16_hi(a.z), bf16_hi(b.z), acc);
    acc = fmaf(bf16_lo(a.w), bf16_lo(b.w), acc);
    acc = fmaf(bf16_hi(a.w), bf16_hi(b.w), acc);
    return acc;
}

// Dot product of 8 bf16 (one uint4) with 8 fp32 values.
__device__ __forceinline__ float dot8f(const uint4& a, const float* f, float acc)
{
    acc = fmaf(bf16_lo(a.x), f[0], acc);
    acc = fmaf(bf16_hi(a.x), f[1], acc);
    acc = fmaf(bf16_lo(a.y), f[2], acc);
    acc = fmaf(bf16_hi(a.y), f[3], acc);
    acc = fmaf(bf16_lo(a.z), f[4], acc);
    acc = fmaf(bf16_hi(a.z), f[5], acc);
    acc = fmaf(bf16_lo(a.w), f[6], acc);
    acc = fmaf(bf16_hi(a.w), f[7], acc);
    return acc;
}

// Two fp32 values -> packed bf16 pair (lo in the low half), each rounded to
// nearest-even: one conversion instruction for the pair.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);   // .x = lo (low half), .y = hi
    return *reinterpret_cast<const uint32_t*>(&h2);
}

// y8 <- bf16_rne(y8 + acc) for 8 packed bf16 values.
__device__ __forceinline__ uint4 add_round8(const uint4& y, const float* acc)
{
    uint4 o;
    o.x = pack_bf16x2(bf16_lo(y.x) + acc[0], bf16_hi(y.x) + acc[1]);
    o.y = pack_bf16x2(bf16_lo(y.y) + acc[2], bf16_hi(y.y) + acc[3]);
    o.z = pack_bf16x2(bf16_lo(y.z) + acc[4], bf16_hi(y.z) + acc[5]);
    o.w = pack_bf16x2(bf16_lo(y.w) + acc[6], bf16_hi(y.w) + acc[7]);
    return o;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ void flag(int32_t* status, int32_t bits)
{
    if (status) atomicOr(status, bits);
}

// Maps a position p in [0, n_pos) to the row it updates and the adapter slot
// it uses.  Two forms:
//   per-token ids (BGMV): row = row_base + p, slot = ids[row];
//   segments (SGMV): the segment s with seg_starts[s] <= p < seg_starts[s+1]
//     gives slot = seg_slot[s]; row = perm ? perm[p] : p.
struct RowMap {
    const int32_t* ids;
    int row_base;
    const int32_t* seg_starts;
    const int32_t* seg_slot;
    int n_segs;
    const int32_t* perm;
    int n_pos;
    int n_rows;
    int n_slots;
};

// Largest s in [0, n_segs) with seg_starts[s] <= p (binary search).
__device__ __forceinline__ int find_segment(const int32_t* seg_starts, int n_segs, int p)
{
    int lo = 0, hi = n_segs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(seg_starts + mid) <= p) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Returns true when position p has an adapter to apply; sets row and slot.
// Malformed entries are flagged and skipped, never trapped.
__device__ __forceinline__ bool resolve(const RowMap& m, int p, int& row, int& slot, int32_t* status)
{
    if (m.seg_starts == nullptr) {
        row = m.row_base + p;
        slot = __ldg(m.ids + row);
    } else {
        const int s = find_segment(m.seg_starts, m.n_segs, p);
        if (!(__ldg(m.seg_starts + s) <= p && p < __ldg(m.seg_starts + s + 1))) {
            flag(status, LORA_DEV_BAD_SEGMENT);
            return false;
        }
        slot = __ldg(m.seg_slot + s);
        row = m.perm ? __ldg(m.perm + p) : p;
        if (row < 0 || row >= m.n_rows) {
            flag(status, LORA_DEV_BAD_SEGMENT);
            return false;
        }
    }
    if (slot == -1) return false;
    if (slot < -1 || slot >= m.n_slots) {
        flag(status, LORA_DEV_SLOT_OUT_OF_RANGE);
        return false;
    }
    return true;
}

// A set of up to LORA_MAX_PROJ projections sharing one input.
struct ProjSet {
    const bf16_t* A[LORA_MAX_PROJ];
    const bf16_t* B[LORA_MAX_PROJ];
    int out_off[LORA_MAX_PROJ];
    int width[LORA_MAX_PROJ];
    int n_proj;
    int r_slot;
};

}  // namespace lora
