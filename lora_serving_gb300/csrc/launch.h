// launch.h -- internal kernel launchers (C++; not part of the C ABI).
#pragma once

#include <cstdlib>

#include <cuda_runtime.h>

#include "common.cuh"

namespace lora {

// Counts every kernel launch the library issues (see lora_kernel_launch_count).
void note_launch();

// Test hook for the bounded waits: LORA_TEST_STALL names one kernel
// (kStallShrinkTc, kStallExpandTc or kStallFusedDecode) whose first copy
// barrier is armed for 16 bytes more than its copies deliver, so that wait
// runs out and the kernel takes its timeout path (LORA_DEV_TIMEOUT).  The
// copies themselves complete as usual.  Unset outside the tests.
constexpr int kStallShrinkTc = 1, kStallExpandTc = 2, kStallFusedDecode = 3;
unsigned test_stall_bytes(int kernel);

// Integer tuning override from the environment (dflt when unset or empty).
inline int env_int(const char* name, int dflt)
{
    const char* e = std::getenv(name);
    return (e && *e) ? std::atoi(e) : dflt;
}

// LORA_MAX_SHARED_CARVEOUT=1 makes every kernel of the library prefer the
// largest shared-memory carveout, so an SM runs all of them under one
// L1/shared split and CTAs of consecutive kernels can share an SM without
// the SM first draining to change its carveout.  Measured: calls with no
// dependency between them overlap better (3B decode, independent ordering,
// 0.139 -> 0.119 ms per step), the dependent chain and the mixed batch do
// not gain (0.1577 -> 0.1598 ms; 3.734 -> 3.738 ms), so the driver's
// per-kernel choice stays the default.
inline cudaError_t prefer_max_shared(const void* fn)
{
    if (env_int("LORA_MAX_SHARED_CARVEOUT", 0) == 0) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

// One position per CTA, CUDA cores: v[row][p*r_slot + j] = A_p[slot][j] . x[row].
cudaError_t launch_shrink_rowwise(float* v, int ld_v, const bf16_t* x, int ld_x, int h_in,
                                  const ProjSet& ps, const RowMap& map, int32_t* status,
                                  cudaStream_t stream);

// One position per CTA, CUDA cores:
// y[row][out_off_p + c] = bf16(y + B_p[slot][c] . v[row][p*r_slot ...]).
cudaError_t launch_expand_rowwise(bf16_t* y, int ld_y, const float* v, int ld_v,
                                  const ProjSet& ps, const RowMap& map, int32_t* status,
                                  cudaStream_t stream);

// Tensor-core SGMV (long contiguous segments).  Shrink writes fp32 v when
// v != nullptr, else the bf16 hi/lo planes vh/vl ([n_rows][n_proj*r_pad64]);
// the expand reads the planes.
bool sgmv_tc_supported(int n_proj, int r_slot, int h_in);
size_t sgmv_tc_plane_bytes(int n_rows, int n_proj, int r_slot);
// Both take lora_apply's ordering flags (programmatic dependent launch unless
// LORA_APPLY_NO_PDL; the shrink reads x before the wait with X_READY).
// tickets (device, or null): a work-item counter the shrink zeroes and the
// expand that follows it in the same call draws its items from (null: the
// expand's static item order).  Calls that may overlap need their own.
cudaError_t launch_sgmv_shrink_tc(float* v, int ld_v, bf16_t* vh, bf16_t* vl, const bf16_t* x, int ld_x, int h_in,
                                  const ProjSet& ps, const int32_t* seg_starts, const int32_t* seg_slot, int n_segs,
                                  int n_pos, int n_rows, int n_slots, unsigned flags, int32_t* status,
                                  cudaStream_t stream, unsigned* tickets = nullptr);
cudaError_t launch_sgmv_expand_tc(bf16_t* y, int ld_y, const bf16_t* vh, const bf16_t* vl, const ProjSet& ps,
                                  const int32_t* seg_starts, const int32_t* seg_slot, int n_segs, int n_pos,
                                  int n_rows, int n_slots, unsigned flags, int32_t* status, cudaStream_t stream,
                                  unsigned* tickets = nullptr);

// Whether the fused decode kernel handles this projection set.
bool fused_decode_supported(int n_proj, int r_slot);

// Decode rows in gather form (perm / gstarts / gslot over n_pos positions):
// shrink + cluster reduction + expand in one launch, no workspace.
cudaError_t launch_bgmv_fused(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                              const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                              int n_pos, int max_group_len, int n_rows, int n_slots, unsigned flags,
                              int32_t* status, cudaStream_t stream);

// Whether a decode call takes the two-launch form (wide outputs, or many
// weight bytes streamed per call) rather than the one-launch kernel.
bool decode_two_launch(const ProjSet& ps, int h_in, int n_groups);

// The same rows in two launches: a grouped shrink that stores v as bf16
// hi/lo planes vh, vl ([n_rows][n_proj * r_pad64], the layout of the
// tensor-core SGMV route), then a grouped expand that streams B'.
cudaError_t launch_bgmv_grouped(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                                const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                                int n_pos, int max_group_len, int n_rows, int n_slots, unsigned flags,
                                bf16_t* vh, bf16_t* vl, int32_t* status, cudaStream_t stream);

// The grouped shrink alone (the planes, no expand); perm == nullptr takes
// positions as rows (contiguous prefill segments as groups).
cudaError_t launch_bgmv_grouped_shrink(const bf16_t* x, int ld_x, int h_in, const ProjSet& ps, const int32_t* perm,
                                       const int32_t* gstarts, const int32_t* gslot, int n_groups, int n_pos,
                                       int max_group_len, int n_rows, int n_slots, unsigned flags, bf16_t* vh,
                                       bf16_t* vl, int32_t* status, cudaStream_t stream);

// The grouped pair with an fp32 intermediate (the standalone SGMV calls):
// v[row][j] (ld_v) instead of the planes; r_slot <= 64.  Programmatic
// dependent launch, as lora_apply's default ordering.
cudaError_t launch_group_shrink_f32(float* v, int ld_v, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                                    const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                                    int n_pos, int max_group_len, int n_rows, int n_slots, int32_t* status,
                                    cudaStream_t stream);
cudaError_t launch_group_expand_f32(bf16_t* y, int ld_y, const float* v, int ld_v, const ProjSet& ps,
                                    const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                                    int n_pos, int max_group_len, int n_rows, int n_slots, int32_t* status,
                                    cudaStream_t stream);

// The grouped pair driven by per-row adapter ids (the standalone BGMV calls,
// no gather metadata): unit = (slot, run of 16 rows with that id, in row
// order), found by each CTA with a block-wide scan of the ids.  fp32 v;
// r_slot <= 64 and at most 65536 units (bgmv_ids_supported).  Programmatic
// dependent launch, as lora_apply's default ordering.
bool bgmv_ids_supported(int r_slot, int n_rows, int n_slots);
cudaError_t launch_bgmv_ids_shrink_f32(float* v, int ld_v, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                                       const int32_t* ids, int n_rows, int n_slots, int32_t* status,
                                       cudaStream_t stream);
cudaError_t launch_bgmv_ids_expand_f32(bf16_t* y, int ld_y, const float* v, int ld_v, const ProjSet& ps,
                                       const int32_t* ids, int n_rows, int n_slots, int32_t* status,
                                       cudaStream_t stream);

// The LoRA linear layer: y[:, off_p + c] = bf16(x W^T + B'_p v_p) for every
// row (ids per row, -1 = base only), W [n_out][ld_w] stacking the
// projections' base weights, v from the bf16 hi/lo planes.
cudaError_t launch_linear_tc(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const bf16_t* W, int ld_w,
                             int n_out, const ProjSet& ps, const bf16_t* vh, const bf16_t* vl,
                             const int32_t* ids, int n_rows, int n_slots, int32_t* status, cudaStream_t stream,
                             unsigned* tickets = nullptr);

// The same layer for decode-sized batches (n_rows <= 64, r_slot <= 64): the
// tile turned around (128 output columns as the MMA's M, the rows as its N),
// K split over a cluster, the delta a K extension per adapter slot present.
// Internal launch flag (beside the public LORA_APPLY_* bits) for the grouped
// shrink: its dependents may launch only once its grid dependency has
// resolved, i.e. once everything enqueued before it has completed.  A
// following kernel that reads x (or anything else written earlier) at
// once may then start early behind a shrink that itself starts early.
constexpr unsigned kShrinkTriggerLate = 0x100u;

bool linear_swap_supported(int n_rows, int r_slot);
cudaError_t launch_linear_swap(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const bf16_t* W, int ld_w,
                               int n_out, const ProjSet& ps, const bf16_t* vh, const bf16_t* vl, const int32_t* ids,
                               int n_rows, int n_slots, int32_t* status, cudaStream_t stream);

// W += sign * B A over one adapter slot (merge / unmerge), one rounding.
cudaError_t launch_merge(bf16_t* W, int ld_w, int out, int h_in, const bf16_t* A, const bf16_t* B, int r_slot,
                         int sign, cudaStream_t stream);
// The same over n weights (host arrays of device pointers), one launch per 32.
cudaError_t launch_merge_batch(int n, bf16_t* const* W, const int* ld_w, const int* out, const int* h_in,
                               const bf16_t* const* A, const bf16_t* const* B, int r_slot, int sign,
                               cudaStream_t stream);
// The tensor-memory form of both (slot ranks up to 64).
bool merge_tc_supported(int r_slot);
cudaError_t launch_merge_tc(int n, bf16_t* const* W, const int* ld_w, const int* out, const int* h_in,
                            const bf16_t* const* A, const bf16_t* const* B, int r_slot, int sign, cudaStream_t stream);

}  // namespace lora
