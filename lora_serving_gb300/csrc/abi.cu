// abi.cu -- C ABI entry points: host-side validation and dispatch.
//
// Every entry point checks its arguments before enqueueing anything and
// returns a status code (vLLM offline LoRA page, "limits": invalid requests
// are rejected at submission, not silently ignored).  The route rule of
// lora_apply follows the TGI page, "4. SGMV and BGMV at inference": SGMV for
// prefill rows or when the rank exceeds the BGMV cap, BGMV otherwise.

#include <atomic>
#include <cstdint>

#include "launch.h"

namespace lora {
namespace {
std::atomic<uint64_t> g_launches{0};
}
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
unsigned test_stall_bytes(int kernel) { return env_int("LORA_TEST_STALL", 0) == kernel ? 16u : 0u; }
}  // namespace lora

using lora::bf16_t;
using lora::ProjSet;
using lora::RowMap;

namespace {

constexpr int kMaxHin = 65536;
// Segments at least this long send a prefill batch to the tensor-core SGMV
// kernels (128-row tiles); shorter ones stay on the CUDA-core kernels.
constexpr int kTcMinSegment = 64;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lora_status_t check_common(int n_rows, int r_slot, int n_slots)
{
    if (n_rows < 0 || n_slots <= 0 || r_slot <= 0) return LORA_ERR_INVALID_ARG;
    if (r_slot > LORA_MAX_RANK) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (r_slot % 8 != 0) return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

lora_status_t check_x(const bf16_t* x, int ld_x, int h_in)
{
    if (!x || h_in <= 0) return LORA_ERR_INVALID_ARG;
    if (h_in > kMaxHin || ld_x < h_in) return LORA_ERR_SHAPE;
    if (!aligned16(x) || h_in % 8 != 0 || ld_x % 8 != 0) return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

lora_status_t check_y(const bf16_t* y, int ld_y, int y_off, int width)
{
    if (!y || width <= 0 || y_off < 0) return LORA_ERR_INVALID_ARG;
    if (static_cast<long long>(y_off) + width > ld_y) return LORA_ERR_SHAPE;
    if (!aligned16(y) || ld_y % 8 != 0 || y_off % 8 != 0 || width % 8 != 0) return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

lora_status_t check_v(const float* v, int ld_v, int cols)
{
    if (!v) return LORA_ERR_INVALID_ARG;
    if (ld_v < cols) return LORA_ERR_SHAPE;
    if (!aligned16(v) || ld_v % 4 != 0) return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

lora_status_t check_store(const bf16_t* s)
{
    if (!s) return LORA_ERR_INVALID_ARG;
    if (!aligned16(s)) return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

lora_status_t check_segments(const int32_t* seg_starts, const int32_t* seg_slot, int n_segs,
                             int n_pos, int n_rows, const int32_t* perm)
{
    if (n_segs < 0 || n_pos < 0 || n_rows < 0) return LORA_ERR_INVALID_ARG;
    if (n_pos == 0) return LORA_OK;
    if (n_segs == 0 || !seg_starts || !seg_slot) return LORA_ERR_METADATA;
    if (!perm && n_pos > n_rows) return LORA_ERR_METADATA;
    return LORA_OK;
}

// Projections of one call update disjoint column ranges of y: two kernels'
// read-modify-writes of one element would race.
lora_status_t check_disjoint(const lora_proj_t* projs, int n_proj)
{
    for (int p = 0; p < n_proj; ++p)
        for (int q = 0; q < p; ++q) {
            const long long a0 = projs[p].out_off, a1 = a0 + projs[p].width;
            const long long b0 = projs[q].out_off, b1 = b0 + projs[q].width;
            if (a0 < b1 && b0 < a1) return LORA_ERR_SHAPE;
        }
    return LORA_OK;
}

#define LORA_TRY(expr)                          \
    do {                                        \
        lora_status_t _st = (expr);             \
        if (_st != LORA_OK) return _st;         \
    } while (0)

inline lora_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

inline int env_int_abi(const char* name, int dflt) { return lora::env_int(name, dflt); }

RowMap ids_map(const int32_t* ids, int row_base, int n_pos, int n_rows, int n_slots)
{
    RowMap m{};
    m.ids = ids;
    m.row_base = row_base;
    m.n_pos = n_pos;
    m.n_rows = n_rows;
    m.n_slots = n_slots;
    return m;
}

RowMap seg_map(const int32_t* seg_starts, const int32_t* seg_slot, int n_segs,
               const int32_t* perm, int n_pos, int n_rows, int n_slots)
{
    RowMap m{};
    m.seg_starts = seg_starts;
    m.seg_slot = seg_slot;
    m.n_segs = n_segs;
    m.perm = perm;
    m.n_pos = n_pos;
    m.n_rows = n_rows;
    m.n_slots = n_slots;
    return m;
}

ProjSet single_proj(const bf16_t* A, const bf16_t* B, int y_off, int width, int r_slot)
{
    ProjSet ps{};
    ps.A[0] = A;
    ps.B[0] = B;
    ps.out_off[0] = y_off;
    ps.width[0] = width;
    ps.n_proj = 1;
    ps.r_slot = r_slot;
    return ps;
}

}  // namespace

extern "C" {

lora_status_t lora_bgmv_shrink(float* v, int ld_v, const lora_bf16_t* x, int ld_x,
                               const lora_bf16_t* A, const int32_t* lora_ids, int n_rows,
                               int h_in, int r_slot, int n_slots, int32_t* dev_status,
                               lora_stream_t stream)
{
    // The shrink accepts a rank-stacked A (n_proj * slot rank rows), so its
    // bound is the fused limit rather than one slot's LORA_MAX_RANK.
    if (n_rows < 0 || n_slots <= 0 || r_slot <= 0) return LORA_ERR_INVALID_ARG;
    if (r_slot > LORA_MAX_RANK * LORA_MAX_PROJ) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (r_slot % 8 != 0) return LORA_ERR_ALIGNMENT;
    if (n_rows == 0) return LORA_OK;
    if (!lora_ids) return LORA_ERR_INVALID_ARG;
    LORA_TRY(check_x(x, ld_x, h_in));
    LORA_TRY(check_store(A));
    LORA_TRY(check_v(v, ld_v, r_slot));
    ProjSet ps = single_proj(A, nullptr, 0, 0, r_slot);
    // Rows grouped by their ids on the device (each adapter's A streamed once
    // per 16 rows) where the grouped kernels take the rank; per row otherwise.
    if (lora::bgmv_ids_supported(r_slot, n_rows, n_slots))
        return cuda_status(lora::launch_bgmv_ids_shrink_f32(v, ld_v, x, ld_x, h_in, ps, lora_ids, n_rows, n_slots,
                                                            dev_status, reinterpret_cast<cudaStream_t>(stream)));
    RowMap m = ids_map(lora_ids, 0, n_rows, n_rows, n_slots);
    return cuda_status(lora::launch_shrink_rowwise(v, ld_v, x, ld_x, h_in, ps, m, dev_status,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_bgmv_expand(lora_bf16_t* y, int ld_y, int y_off, int width,
                               const float* v, int ld_v, const lora_bf16_t* B,
                               const int32_t* lora_ids, int n_rows, int r_slot, int n_slots,
                               int32_t* dev_status, lora_stream_t stream)
{
    LORA_TRY(check_common(n_rows, r_slot, n_slots));
    if (n_rows == 0) return LORA_OK;
    if (!lora_ids) return LORA_ERR_INVALID_ARG;
    LORA_TRY(check_y(y, ld_y, y_off, width));
    LORA_TRY(check_store(B));
    LORA_TRY(check_v(v, ld_v, r_slot));
    ProjSet ps = single_proj(nullptr, B, y_off, width, r_slot);
    if (lora::bgmv_ids_supported(r_slot, n_rows, n_slots))
        return cuda_status(lora::launch_bgmv_ids_expand_f32(y, ld_y, v, ld_v, ps, lora_ids, n_rows, n_slots,
                                                            dev_status, reinterpret_cast<cudaStream_t>(stream)));
    RowMap m = ids_map(lora_ids, 0, n_rows, n_rows, n_slots);
    return cuda_status(lora::launch_expand_rowwise(y, ld_y, v, ld_v, ps, m, dev_status,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_sgmv_shrink(float* v, int ld_v, const lora_bf16_t* x, int ld_x,
                               const lora_bf16_t* A, const int32_t* seg_starts,
                               const int32_t* seg_slot, int n_segs, const int32_t* row_perm,
                               int n_pos, int n_rows, int max_seg_len, int h_in, int r_slot,
                               int n_slots, int32_t* dev_status, lora_stream_t stream)
{
    if (n_rows < 0 || n_slots <= 0 || r_slot <= 0) return LORA_ERR_INVALID_ARG;
    if (r_slot > LORA_MAX_RANK * LORA_MAX_PROJ) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (r_slot % 8 != 0) return LORA_ERR_ALIGNMENT;
    LORA_TRY(check_segments(seg_starts, seg_slot, n_segs, n_pos, n_rows, row_perm));
    if (n_pos == 0) return LORA_OK;
    LORA_TRY(check_x(x, ld_x, h_in));
    LORA_TRY(check_store(A));
    LORA_TRY(check_v(v, ld_v, r_slot));
    ProjSet ps = single_proj(A, nullptr, 0, 0, r_slot);
    if (!row_perm && max_seg_len >= kTcMinSegment && lora::sgmv_tc_supported(1, r_slot, h_in))
        return cuda_status(lora::launch_sgmv_shrink_tc(v, ld_v, nullptr, nullptr, x, ld_x, h_in, ps, seg_starts,
                                                       seg_slot, n_segs, n_pos, n_rows, n_slots, 0u, dev_status,
                                                       reinterpret_cast<cudaStream_t>(stream)));
    // Short segments and gathered rows: the segments as groups of the
    // grouped shrink (units of 16 rows, each adapter's A streamed once per
    // unit), for ranks the grouped kernels take.
    if (r_slot <= 64)
        return cuda_status(lora::launch_group_shrink_f32(v, ld_v, x, ld_x, h_in, ps, row_perm, seg_starts, seg_slot,
                                                         n_segs, n_pos, max_seg_len, n_rows, n_slots, dev_status,
                                                         reinterpret_cast<cudaStream_t>(stream)));
    RowMap m = seg_map(seg_starts, seg_slot, n_segs, row_perm, n_pos, n_rows, n_slots);
    return cuda_status(lora::launch_shrink_rowwise(v, ld_v, x, ld_x, h_in, ps, m, dev_status,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_sgmv_expand(lora_bf16_t* y, int ld_y, int y_off, int width,
                               const float* v, int ld_v, const lora_bf16_t* B,
                               const int32_t* seg_starts, const int32_t* seg_slot, int n_segs,
                               const int32_t* row_perm, int n_pos, int n_rows, int max_seg_len,
                               int r_slot, int n_slots, int32_t* dev_status,
                               lora_stream_t stream)
{
    LORA_TRY(check_common(n_rows, r_slot, n_slots));
    LORA_TRY(check_segments(seg_starts, seg_slot, n_segs, n_pos, n_rows, row_perm));
    if (n_pos == 0) return LORA_OK;
    LORA_TRY(check_y(y, ld_y, y_off, width));
    LORA_TRY(check_store(B));
    LORA_TRY(check_v(v, ld_v, r_slot));
    ProjSet ps = single_proj(nullptr, B, y_off, width, r_slot);
    // The segments as groups of the grouped expand (each unit's B' columns
    // brought by bulk copies, the tensor cores on v split hi/lo).
    if (r_slot <= 64)
        return cuda_status(lora::launch_group_expand_f32(y, ld_y, v, ld_v, ps, row_perm, seg_starts, seg_slot, n_segs,
                                                         n_pos, max_seg_len, n_rows, n_slots, dev_status,
                                                         reinterpret_cast<cudaStream_t>(stream)));
    RowMap m = seg_map(seg_starts, seg_slot, n_segs, row_perm, n_pos, n_rows, n_slots);
    return cuda_status(lora::launch_expand_rowwise(y, ld_y, v, ld_v, ps, m, dev_status,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

// Workspace layout: [bf16 hi/lo planes of v for the tensor-core SGMV route]
// [fp32 v for the other routes][the tensor-core expand's work-item counter],
// each part 256-byte aligned.
static size_t plane_region_bytes(int n_rows, int n_proj, int r_slot)
{
    return (lora::sgmv_tc_plane_bytes(n_rows, n_proj, r_slot) + 255) / 256 * 256;
}
static size_t fp32_region_bytes(int n_rows, int n_proj, int r_slot)
{
    return (static_cast<size_t>(n_rows) * n_proj * r_slot * sizeof(float) + 255) / 256 * 256;
}
constexpr size_t kTicketRegionBytes = 256;

size_t lora_apply_workspace_bytes(int n_rows, int n_proj, int r_slot)
{
    if (n_rows <= 0 || n_proj <= 0 || r_slot <= 0) return 0;
    if (n_proj > LORA_MAX_PROJ || r_slot > LORA_MAX_RANK) return 0;   // lora_apply rejects these
    return plane_region_bytes(n_rows, n_proj, r_slot) + fp32_region_bytes(n_rows, n_proj, r_slot) + kTicketRegionBytes;
}

lora_status_t lora_apply(lora_bf16_t* y, int ld_y, const lora_bf16_t* x, int ld_x, int h_in,
                         const lora_proj_t* projs, int n_proj, int r_slot, int n_slots,
                         const lora_meta_t* meta, void* workspace, size_t ws_bytes,
                         uint32_t flags, int32_t* dev_status, lora_stream_t stream)
{
    if (!projs || !meta || n_proj <= 0 || n_proj > LORA_MAX_PROJ) return LORA_ERR_INVALID_ARG;
    const int T = meta->n_rows, P = meta->n_prefill;
    LORA_TRY(check_common(T, r_slot, n_slots));
    if (P < 0 || P > T) return LORA_ERR_METADATA;
    if (T == 0) return LORA_OK;
    LORA_TRY(check_x(x, ld_x, h_in));
    ProjSet ps{};
    ps.n_proj = n_proj;
    ps.r_slot = r_slot;
    for (int p = 0; p < n_proj; ++p) {
        LORA_TRY(check_y(y, ld_y, projs[p].out_off, projs[p].width));
        LORA_TRY(check_store(projs[p].A));
        LORA_TRY(check_store(projs[p].B));
        ps.A[p] = projs[p].A;
        ps.B[p] = projs[p].B;
        ps.out_off[p] = projs[p].out_off;
        ps.width[p] = projs[p].width;
    }
    LORA_TRY(check_disjoint(projs, n_proj));
    const int R = n_proj * r_slot;
    if (!workspace) return LORA_ERR_WORKSPACE;
    if (ws_bytes < lora_apply_workspace_bytes(T, n_proj, r_slot)) return LORA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LORA_ERR_ALIGNMENT;
    bf16_t* vh = static_cast<bf16_t*>(workspace);
    bf16_t* vl = vh + plane_region_bytes(T, n_proj, r_slot) / 2 / sizeof(bf16_t);
    float* v = reinterpret_cast<float*>(static_cast<char*>(workspace) + plane_region_bytes(T, n_proj, r_slot));
    unsigned* tickets = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + plane_region_bytes(T, n_proj, r_slot) +
                                                    fp32_region_bytes(T, n_proj, r_slot));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int D = T - P;
    if (P > 0) LORA_TRY(check_segments(meta->seg_starts, meta->seg_slot, meta->n_segs, P, T, nullptr));
    if (D > 0) {
        if (!meta->lora_ids) return LORA_ERR_INVALID_ARG;
        if (r_slot > LORA_BGMV_MAX_RANK) {
            if (!meta->perm) return LORA_ERR_METADATA;
            LORA_TRY(check_segments(meta->gseg_starts, meta->gseg_slot, meta->n_gsegs, D, T, meta->perm));
        }
    }

    // A mixed batch whose prefill rows take the tensor cores launches the
    // prefill shrink first (one CTA per SM), then the decode rows' kernel,
    // which fills the SMs' remaining room beside it (programmatic dependent
    // launch), then the prefill expand: the shrink and the decode kernel
    // touch disjoint rows of y and of the workspace.  Otherwise the decode
    // rows' kernel comes first and the prefill kernels follow.
    const bool tc_prefill = P > 0 && meta->max_seg_len >= kTcMinSegment && lora::sgmv_tc_supported(n_proj, r_slot, h_in);
    const bool shrink_first = tc_prefill && D > 0 && env_int_abi("LORA_APPLY_SHRINK_FIRST", 1) != 0;
    if (shrink_first)
        LORA_TRY(cuda_status(lora::launch_sgmv_shrink_tc(nullptr, 0, vh, vl, x, ld_x, h_in, ps, meta->seg_starts,
                                                         meta->seg_slot, meta->n_segs, P, T, n_slots, flags,
                                                         dev_status, s, tickets)));
    if (D > 0) {
        const bool gathered = meta->perm && meta->gseg_starts && meta->gseg_slot && meta->n_gsegs > 0;
        const bool fused_ok = gathered && lora::fused_decode_supported(n_proj, r_slot);
        const bool grouped_ok = gathered && r_slot <= 64;
        // Decode rows grouped by adapter: the BGMV route for r_slot <=
        // LORA_BGMV_MAX_RANK and the SGMV-over-gather-groups route above it
        // share one grouping.  One launch (cluster split-K) for small calls;
        // two (grouped shrink, grouped expand) for wide or weight-heavy ones.
        if (grouped_ok && (!fused_ok || lora::decode_two_launch(ps, h_in, meta->n_gsegs))) {
            LORA_TRY(cuda_status(lora::launch_bgmv_grouped(y, ld_y, x, ld_x, h_in, ps, meta->perm,
                                                           meta->gseg_starts, meta->gseg_slot, meta->n_gsegs, D,
                                                           meta->max_gseg_len, T, n_slots, flags, vh, vl,
                                                           dev_status, s)));
        } else if (fused_ok) {
            LORA_TRY(cuda_status(lora::launch_bgmv_fused(y, ld_y, x, ld_x, h_in, ps, meta->perm,
                                                         meta->gseg_starts, meta->gseg_slot, meta->n_gsegs,
                                                         D, meta->max_gseg_len, T, n_slots, flags,
                                                         dev_status, s)));
        } else {
            RowMap m = r_slot <= LORA_BGMV_MAX_RANK
                           ? ids_map(meta->lora_ids, P, D, T, n_slots)
                           : seg_map(meta->gseg_starts, meta->gseg_slot, meta->n_gsegs, meta->perm, D, T, n_slots);
            LORA_TRY(cuda_status(lora::launch_shrink_rowwise(v, R, x, ld_x, h_in, ps, m, dev_status, s)));
            LORA_TRY(cuda_status(lora::launch_expand_rowwise(y, ld_y, v, R, ps, m, dev_status, s)));
        }
    }
    if (P > 0) {
        if (tc_prefill) {
            // long segments: tensor-core shrink into the hi/lo planes, then expand
            if (!shrink_first)
                LORA_TRY(cuda_status(lora::launch_sgmv_shrink_tc(nullptr, 0, vh, vl, x, ld_x, h_in, ps,
                                                                 meta->seg_starts, meta->seg_slot, meta->n_segs, P,
                                                                 T, n_slots, flags, dev_status, s, tickets)));
            LORA_TRY(cuda_status(lora::launch_sgmv_expand_tc(y, ld_y, vh, vl, ps, meta->seg_starts,
                                                             meta->seg_slot, meta->n_segs, P, T, n_slots, flags,
                                                             dev_status, s, tickets)));
        } else if (r_slot <= 64) {
            // short segments: the segments as groups of the grouped pair (no
            // permutation: a segment's positions are its rows)
            LORA_TRY(cuda_status(lora::launch_bgmv_grouped(y, ld_y, x, ld_x, h_in, ps, nullptr, meta->seg_starts,
                                                           meta->seg_slot, meta->n_segs, P, meta->max_seg_len, T,
                                                           n_slots, flags, vh, vl, dev_status, s)));
        } else {
            RowMap m = seg_map(meta->seg_starts, meta->seg_slot, meta->n_segs, nullptr, P, T, n_slots);
            LORA_TRY(cuda_status(lora::launch_shrink_rowwise(v, R, x, ld_x, h_in, ps, m, dev_status, s)));
            LORA_TRY(cuda_status(lora::launch_expand_rowwise(y, ld_y, v, R, ps, m, dev_status, s)));
        }
    }
    return LORA_OK;
}

lora_status_t lora_linear(lora_bf16_t* y, int ld_y, const lora_bf16_t* x, int ld_x, int h_in,
                          const lora_bf16_t* W, int ld_w, const lora_proj_t* projs, int n_proj, int r_slot,
                          int n_slots, const lora_meta_t* meta, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, lora_stream_t stream)
{
    if (!projs || !meta || !W || n_proj <= 0 || n_proj > LORA_MAX_PROJ) return LORA_ERR_INVALID_ARG;
    const int T = meta->n_rows, P = meta->n_prefill, D = T - P;
    LORA_TRY(check_common(T, r_slot, n_slots));
    if (P < 0 || P > T) return LORA_ERR_METADATA;
    if (T == 0) return LORA_OK;
    LORA_TRY(check_x(x, ld_x, h_in));
    if (ld_w < h_in) return LORA_ERR_SHAPE;
    if (!aligned16(W) || ld_w % 8 != 0) return LORA_ERR_ALIGNMENT;
    ProjSet ps{};
    ps.n_proj = n_proj;
    ps.r_slot = r_slot;
    int n_out = 0;
    for (int p = 0; p < n_proj; ++p) {
        LORA_TRY(check_y(y, ld_y, projs[p].out_off, projs[p].width));
        LORA_TRY(check_store(projs[p].A));
        LORA_TRY(check_store(projs[p].B));
        if (projs[p].out_off != n_out) return LORA_ERR_SHAPE;   // the projections tile [0, n_out)
        n_out += projs[p].width;
        ps.A[p] = projs[p].A;
        ps.B[p] = projs[p].B;
        ps.out_off[p] = projs[p].out_off;
        ps.width[p] = projs[p].width;
    }
    const bool tc_shrink = lora::sgmv_tc_supported(n_proj, r_slot, h_in);
    if (r_slot > 64 && (D > 0 || !tc_shrink)) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (!meta->lora_ids) return LORA_ERR_INVALID_ARG;
    if (!workspace) return LORA_ERR_WORKSPACE;
    if (ws_bytes < lora_apply_workspace_bytes(T, n_proj, r_slot)) return LORA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LORA_ERR_ALIGNMENT;
    if (P > 0) LORA_TRY(check_segments(meta->seg_starts, meta->seg_slot, meta->n_segs, P, T, nullptr));
    if (D > 0) {
        if (!meta->perm) return LORA_ERR_METADATA;
        LORA_TRY(check_segments(meta->gseg_starts, meta->gseg_slot, meta->n_gsegs, D, T, meta->perm));
    }
    bf16_t* vh = static_cast<bf16_t*>(workspace);
    bf16_t* vl = vh + plane_region_bytes(T, n_proj, r_slot) / 2 / sizeof(bf16_t);
    unsigned* tickets = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + plane_region_bytes(T, n_proj, r_slot) +
                                                    fp32_region_bytes(T, n_proj, r_slot));
    bool tickets_zeroed = false;   // the tensor-core shrink zeroes the linear kernel's tile counter
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // v = A x into the hi/lo planes: tensor-core shrink over the prefill
    // segments (grouped shrink over them where the tensor-core form does not
    // apply), grouped shrink over the decode groups
    if (P > 0 && meta->n_segs > 0) {
        if (tc_shrink) {
            LORA_TRY(cuda_status(lora::launch_sgmv_shrink_tc(nullptr, 0, vh, vl, x, ld_x, h_in, ps, meta->seg_starts,
                                                             meta->seg_slot, meta->n_segs, P, T, n_slots,
                                                             LORA_APPLY_NO_PDL, dev_status, s, tickets)));
            tickets_zeroed = true;
        }
        else
            LORA_TRY(cuda_status(lora::launch_bgmv_grouped_shrink(x, ld_x, h_in, ps, nullptr, meta->seg_starts,
                                                                  meta->seg_slot, meta->n_segs, P,
                                                                  meta->max_seg_len, T, n_slots, LORA_APPLY_NO_PDL,
                                                                  vh, vl, dev_status, s)));
    }
    // The decode rows' shrink, when it is the call's first kernel, starts
    // early (its adapter rows load while the kernel before it finishes) and
    // lets the linear kernel launch once everything before the call has
    // completed, since that kernel reads x at once.
    const bool first_kernel = !(P > 0 && meta->n_segs > 0);
    const unsigned dshrink_flags = first_kernel && env_int_abi("LORA_LINEAR_SHRINK_PDL", 1) != 0
                                       ? lora::kShrinkTriggerLate
                                       : LORA_APPLY_NO_PDL;
    if (D > 0 && meta->n_gsegs > 0)
        LORA_TRY(cuda_status(lora::launch_bgmv_grouped_shrink(x, ld_x, h_in, ps, meta->perm, meta->gseg_starts,
                                                              meta->gseg_slot, meta->n_gsegs, D, meta->max_gseg_len,
                                                              T, n_slots, dshrink_flags, vh, vl, dev_status,
                                                              s)));
    // base product with the delta in the same accumulator: decode-sized
    // batches turn the tile around (the weights are the bytes), larger ones
    // take the persistent tile kernel
    if (lora::linear_swap_supported(T, r_slot) && env_int_abi("LORA_LINEAR_SWAP", 1) != 0)
        return cuda_status(lora::launch_linear_swap(y, ld_y, x, ld_x, h_in, W, ld_w, n_out, ps, vh, vl,
                                                    meta->lora_ids, T, n_slots, dev_status, s));
    return cuda_status(lora::launch_linear_tc(y, ld_y, x, ld_x, h_in, W, ld_w, n_out, ps, vh, vl, meta->lora_ids, T,
                                              n_slots, dev_status, s, tickets_zeroed ? tickets : nullptr));
}

lora_status_t lora_merge(lora_bf16_t* W, int ld_w, int out, int h_in, const lora_bf16_t* A,
                         const lora_bf16_t* B, int r_slot, int sign, lora_stream_t stream)
{
    if (!W || out <= 0 || h_in <= 0 || r_slot <= 0 || (sign != 1 && sign != -1)) return LORA_ERR_INVALID_ARG;
    if (r_slot > LORA_MAX_RANK) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (ld_w < h_in || out > (1 << 22)) return LORA_ERR_SHAPE;
    if (!aligned16(W) || ld_w % 8 != 0 || h_in % 8 != 0 || r_slot % 8 != 0) return LORA_ERR_ALIGNMENT;
    LORA_TRY(check_store(A));
    LORA_TRY(check_store(B));
    return cuda_status(lora::launch_merge(W, ld_w, out, h_in, A, B, r_slot, sign,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_merge_batch(int n, lora_bf16_t* const* W, const int* ld_w, const int* out, const int* h_in,
                               const lora_bf16_t* const* A, const lora_bf16_t* const* B, int r_slot, int sign,
                               lora_stream_t stream)
{
    if (n < 0 || (n > 0 && (!W || !ld_w || !out || !h_in || !A || !B))) return LORA_ERR_INVALID_ARG;
    if (r_slot <= 0 || (sign != 1 && sign != -1)) return LORA_ERR_INVALID_ARG;
    if (r_slot > LORA_MAX_RANK) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (r_slot % 8 != 0) return LORA_ERR_ALIGNMENT;
    for (int i = 0; i < n; ++i) {
        if (!W[i] || out[i] <= 0 || h_in[i] <= 0) return LORA_ERR_INVALID_ARG;
        if (ld_w[i] < h_in[i] || out[i] > (1 << 22)) return LORA_ERR_SHAPE;
        if (!aligned16(W[i]) || ld_w[i] % 8 != 0 || h_in[i] % 8 != 0) return LORA_ERR_ALIGNMENT;
        LORA_TRY(check_store(A[i]));
        LORA_TRY(check_store(B[i]));
    }
    if (n == 0) return LORA_OK;
    return cuda_status(lora::launch_merge_batch(n, W, ld_w, out, h_in, A, B, r_slot, sign,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

uint64_t lora_kernel_launch_count(void) { return lora::g_launches.load(std::memory_order_relaxed); }

lora_status_t lora_read_device_status(const int32_t* dev_status, int32_t* out, lora_stream_t stream)
{
    if (!dev_status || !out) return LORA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // extern "C"
