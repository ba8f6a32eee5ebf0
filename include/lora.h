/*
 * lora.h -- C ABI of the GB300 multi-LoRA delta library (liblora.so).
 *
 * The library adds, for every row t of a batch, the low-rank delta of the
 * adapter that row names to a shared base-layer output:
 *
 *     y[t, off : off+w] += B'_id(t) ( A_id(t) x_t )        (id(t) >= 0)
 *
 * and leaves rows whose id is -1 (base model only) untouched.
 *
 * Sources (page title, section):
 *   [MLS]  "Multi-LoRA serving: one base, many adapters" -- "direct answer":
 *          Delta W = B A with B in R^{d x r}, A in R^{r x k}; the base GEMM
 *          runs once for the batch and each row's B(Ax) is added by a grouped
 *          kernel keyed by adapter id (SGMV/BGMV).
 *   [TGI]  "Text Generation Inference multi-LoRA adapter serving in
 *          practice" -- "implementation 3. weight preprocessing" (scale
 *          lora_alpha/r or rsLoRA lora_alpha/sqrt(r) folded into lora_B; rank
 *          padded to the kernel's vector width), "4. SGMV and BGMV at
 *          inference" (SGMV for prefill segments or ranks above the BGMV cap,
 *          BGMV token by token otherwise), "5. tensor parallelism" (slicing
 *          for uneven q/k/v widths, fused gate_up), and the backend note
 *          naming bgmv_shrink / bgmv_expand / sgmv_shrink / sgmv_expand.
 *   [VLLM] "How vLLM attaches a different LoRA adapter per request in
 *          offline inference" -- step 2 (max_loras slots, max_lora_rank =
 *          the largest rank in use), step 3 (None runs the base model) and
 *          "limits" (invalid requests are rejected before submission).
 *
 * Conventions for every entry point:
 *   - bf16 values are passed as their 16-bit patterns (lora_bf16_t).
 *   - Device pointers (marked [dev]) are owned by the caller; the kernel
 *     entry points allocate no memory and keep no state between calls
 *     except what the caller passes (the slot manager, below, owns a pinned
 *     host cache).  Host pointers are marked [host].
 *   - Kernel entry points validate their arguments on the host, enqueue on
 *     `stream` and return without synchronising.  A host-detectable error
 *     returns a non-OK status BEFORE anything is enqueued.
 *   - Device-detected faults (an adapter id >= n_slots, a segment table that
 *     does not cover its rows) never trap: the row is skipped and a bit is
 *     OR-ed into *dev_status (LORA_DEV_*), which may be NULL to ignore them.
 *     Kernels contain no device printf and no unbounded wait: a wait for an
 *     asynchronous copy gives up after 0.2 s and sets LORA_DEV_TIMEOUT.
 *   - Alignment: every bf16/fp32 matrix pointer is 16-byte aligned, and all
 *     leading dimensions, widths, column offsets and h_in are multiples of 8
 *     elements (one 128-bit vector of bf16); r_slot is a multiple of 8.
 *   - Row-major everywhere.  Adapter stores keep the peft orientation [MLS]:
 *       A store: [n_slots][r_slot][h_in]      (lora_A, K-major)
 *       B store: [n_slots][width][r_slot]     (scaled lora_B, K-major)
 *     The intermediate v is fp32 [n_rows][ld_v] and is never rounded to bf16.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lora_bf16_t;           /* bf16 bit pattern */
typedef struct CUstream_st* lora_stream_t; /* same handle as cudaStream_t */

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,       /* NULL pointer, negative size, n_proj out of range */
    LORA_ERR_SHAPE = 2,             /* leading dimension too small, slice outside the row */
    LORA_ERR_RANK_EXCEEDS_SLOT = 3, /* adapter rank > r_slot, or r_slot > LORA_MAX_RANK */
    LORA_ERR_SLOT_RANGE = 4,        /* adapter id outside [-1, n_slots); more adapters than slots */
    LORA_ERR_ALIGNMENT = 5,         /* pointer or size violates the 16-byte rule above */
    LORA_ERR_METADATA = 6,          /* segment table inconsistent with the row counts */
    LORA_ERR_WORKSPACE = 7,         /* workspace NULL or smaller than required */
    LORA_ERR_CUDA = 8               /* a CUDA call failed (launch, copy, attribute) */
} lora_status_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define LORA_DEV_SLOT_OUT_OF_RANGE 0x1 /* a row named an id >= n_slots or < -1; row skipped */
#define LORA_DEV_BAD_SEGMENT 0x2       /* a segment/perm entry fell outside its rows, or a
                                          group outgrew meta->max_gseg_len; rows skipped */
#define LORA_DEV_TIMEOUT 0x4           /* an asynchronous copy did not land within 0.2 s (never
                                          expected): the kernel that waited stops; rows of y it
                                          had not finished keep their previous values (a shrink
                                          stores a zero intermediate for its unfinished rows, so
                                          the expand adds nothing); the call returns and later
                                          calls are unaffected */

/* Largest r_slot (rank of one projection's slot) the kernels accept. */
#define LORA_MAX_RANK 128
/* BGMV cap: decode rows use BGMV when r_slot <= this, SGMV otherwise [TGI 4].
 * The page does not print the cap; 32 is this library's choice. */
#define LORA_BGMV_MAX_RANK 32
/* Most projections one fused lora_apply call handles (q/k/v: 3, gate/up: 2). */
#define LORA_MAX_PROJ 4

/* ------------------------------------------------------------------ *
 *  Kernel entry points (device pointers, asynchronous on `stream`)
 * ------------------------------------------------------------------ */

/*
 * Ordering of the four standalone calls below: as lora_apply with flags 0.
 * Their kernels use programmatic dependent launch and may start while the
 * kernel enqueued before them is still running.  They read the adapter store,
 * lora_ids and the segment tables at once, so these must not be written by
 * that kernel (copies made with cudaMemcpyAsync are ordered as usual).  They
 * read x and v, and write v, y and dev_status, only once that kernel has
 * completed.  None completes before the kernel before it.  The row-by-row
 * form (slot ranks above 64) runs in plain stream order.
 */

/*
 * BGMV shrink [TGI 4, decode, token by token]:
 *   v[t][j] = sum_i A[id_t][j][i] * x[t][i]      for j < r_slot, id_t >= 0
 * x        [dev] bf16 [n_rows][ld_x], ld_x >= h_in
 * A        [dev] bf16 [n_slots][r_slot][h_in] (for q/k/v stacked along rank,
 *                pass the stacked store and r_slot = n_proj * slot rank)
 * lora_ids [dev] int32 [n_rows], -1 = base (v row not written)
 * v        [dev] fp32 [n_rows][ld_v], ld_v >= r_slot; fp32 accumulation
 * n_rows == 0 is a no-op.  For r_slot <= 64 (and n_slots * ceil(n_rows/16)
 * <= 65536) the rows are grouped by id on the device, each adapter's A read
 * once per run of 16 of its rows; otherwise row by row.  The form does not
 * change the result.  An id outside [-1, n_slots) sets
 * LORA_DEV_SLOT_OUT_OF_RANGE and its row is skipped.
 */
lora_status_t lora_bgmv_shrink(float* v, int ld_v, const lora_bf16_t* x, int ld_x,
                               const lora_bf16_t* A, const int32_t* lora_ids, int n_rows,
                               int h_in, int r_slot, int n_slots, int32_t* dev_status,
                               lora_stream_t stream);

/*
 * BGMV expand [TGI 4; slicing per TGI 5]:
 *   y[t][y_off+c] = bf16_rne( y[t][y_off+c] + sum_j B[id_t][c][j] * v[t][j] )
 * for c < width, id_t >= 0; rows with id -1 are never written.
 * y        [dev] bf16 [n_rows][ld_y], y_off + width <= ld_y
 * v        [dev] fp32 [n_rows][ld_v] (pass v + p*r_slot for projection p of
 *                a stacked shrink), ld_v >= r_slot
 * B        [dev] bf16 [n_slots][width][r_slot], already scaled (B')
 * Kernel form and id checks as in lora_bgmv_shrink.
 */
lora_status_t lora_bgmv_expand(lora_bf16_t* y, int ld_y, int y_off, int width,
                               const float* v, int ld_v, const lora_bf16_t* B,
                               const int32_t* lora_ids, int n_rows, int r_slot, int n_slots,
                               int32_t* dev_status, lora_stream_t stream);

/*
 * SGMV shrink [TGI 4, prefill, "variable-length segments"]:
 * segment s covers positions [seg_starts[s], seg_starts[s+1]) and uses slot
 * seg_slot[s] (-1: skipped).  Position p maps to row row_perm[p], or to row p
 * when row_perm is NULL (contiguous segments).  For every covered row:
 *   v[row][j] = sum_i A[slot][j][i] * x[row][i]       j < r_slot
 * seg_starts [dev] int32 [n_segs+1], non-decreasing, seg_starts[0] == 0,
 *            seg_starts[n_segs] == n_pos
 * seg_slot   [dev] int32 [n_segs]
 * row_perm   [dev] int32 [n_pos] or NULL; every entry in [0, n_rows)
 * n_rows     rows of x / v (bounds for the row indices)
 * max_seg_len  [host] an upper bound on the longest segment (0 = unknown).
 *              It picks the kernel form (tensor cores for contiguous
 *              segments of 64 rows or more; otherwise, for r_slot <= 64, the
 *              grouped kernels, whose grid it sizes: a value below the true
 *              longest segment leaves rows without their result and sets
 *              LORA_DEV_BAD_SEGMENT).
 */
lora_status_t lora_sgmv_shrink(float* v, int ld_v, const lora_bf16_t* x, int ld_x,
                               const lora_bf16_t* A, const int32_t* seg_starts,
                               const int32_t* seg_slot, int n_segs, const int32_t* row_perm,
                               int n_pos, int n_rows, int max_seg_len, int h_in, int r_slot,
                               int n_slots, int32_t* dev_status, lora_stream_t stream);

/*
 * SGMV expand: for every row covered by a segment with slot >= 0,
 *   y[row][y_off+c] = bf16_rne( y[row][y_off+c] + sum_j B[slot][c][j] * v[row][j] )
 * Arguments as in lora_sgmv_shrink and lora_bgmv_expand (max_seg_len sizes
 * the grouped kernels' grid for r_slot <= 64, as in lora_sgmv_shrink).
 */
lora_status_t lora_sgmv_expand(lora_bf16_t* y, int ld_y, int y_off, int width,
                               const float* v, int ld_v, const lora_bf16_t* B,
                               const int32_t* seg_starts, const int32_t* seg_slot, int n_segs,
                               const int32_t* row_perm, int n_pos, int n_rows, int max_seg_len,
                               int r_slot, int n_slots, int32_t* dev_status,
                               lora_stream_t stream);

/* One projection of a fused call: its own A/B stores and its output slice. */
typedef struct {
    const lora_bf16_t* A; /* [dev] [n_slots][r_slot][h_in] */
    const lora_bf16_t* B; /* [dev] [n_slots][width][r_slot], scaled */
    int out_off;          /* first column of this projection in y */
    int width;            /* its number of output columns (uneven for GQA k/v) */
} lora_proj_t;

/*
 * Batch metadata as built by lora_build_metadata and copied to the device.
 * Rows [0, n_prefill) are prefill rows, rows [n_prefill, n_rows) decode rows.
 */
typedef struct {
    const int32_t* lora_ids;    /* [dev] [n_rows], -1 = base */
    int n_rows;
    int n_prefill;
    const int32_t* seg_starts;  /* [dev] [n_segs+1] prefill segments over [0, n_prefill) */
    const int32_t* seg_slot;    /* [dev] [n_segs] */
    int n_segs;
    int max_seg_len;            /* longest prefill segment (host value; an upper bound,
                                   0 = unknown).  It picks the kernel form; where
                                   lora_linear's grouped shrink takes the segments, it
                                   also sizes that grid, as max_gseg_len below. */
    const int32_t* perm;        /* [dev] [n_rows-n_prefill] decode rows sorted by slot */
    const int32_t* gseg_starts; /* [dev] [n_gsegs+1] groups over positions of perm */
    const int32_t* gseg_slot;   /* [dev] [n_gsegs] */
    int n_gsegs;
    int max_gseg_len;           /* largest decode group (host value; an upper bound,
                                   0 = unknown).  The decode kernels size their grids
                                   from it: a value below the true largest group leaves
                                   rows without their delta and sets
                                   LORA_DEV_BAD_SEGMENT. */
} lora_meta_t;

/* lora_apply flags.
 * Ordering against the kernel enqueued just before the call: lora_apply's
 * kernels (decode rows first, then prefill rows) use programmatic dependent
 * launch, so each may start while the kernel before it is still running.
 * They read the adapter store and the batch metadata at once (neither may
 * be written by that kernel; copies made with cudaMemcpyAsync are ordered
 * as usual), and touch y, the workspace and dev_status only after that
 * kernel has completed.  None completes before the kernel before it.
 *   LORA_APPLY_X_READY: x is not written by the kernel just before the call
 *     (in a model layer x comes from earlier than the base GEMM that writes
 *     y), so the shrinks may read x before that kernel completes.
 *   LORA_APPLY_Y_READY: y is neither read nor written by the kernel just
 *     before the call (e.g. the delta goes to a buffer of its own), so the
 *     decode kernel may update y before that kernel completes; with X_READY
 *     as well, calls that share no buffers overlap fully.
 *   LORA_APPLY_NO_PDL: plain stream ordering, nothing starts early. */
#define LORA_APPLY_X_READY 0x1u
#define LORA_APPLY_NO_PDL 0x2u
#define LORA_APPLY_Y_READY 0x4u

/*
 * Fused LoRA delta for n_proj projections that share the input x (q/k/v or
 * gate/up) [TGI 4, 5]:
 *   - prefill rows: SGMV over meta->seg_*;
 *   - decode rows: BGMV when r_slot <= LORA_BGMV_MAX_RANK, otherwise SGMV
 *     over the gather groups meta->perm / gseg_* [TGI 4].
 * Each projection p adds its delta into y[:, projs[p].out_off + (0..width));
 * the projections' column ranges must not overlap (LORA_ERR_SHAPE).
 * workspace [dev] at least lora_apply_workspace_bytes(n_rows, n_proj, r_slot)
 *           bytes, 256-byte aligned; its contents are scratch (the
 *           intermediate v: fp32, and bf16 hi/lo planes for the kernels
 *           whose expand runs on tensor cores; and the tensor-core
 *           expand's work-item counter), written only after the kernel
 *           enqueued just before the call has completed.  Calls that may
 *           run at the same time on the GPU need separate workspaces.
 * flags     LORA_APPLY_* above (0 = default ordering).
 * Errors (before anything is enqueued): LORA_ERR_INVALID_ARG (NULL projs,
 * meta, x or lora_ids; n_proj outside 1..LORA_MAX_PROJ), LORA_ERR_SHAPE (a
 * slice past ld_y, overlapping slices, ld_x < h_in), LORA_ERR_ALIGNMENT,
 * LORA_ERR_RANK_EXCEEDS_SLOT (r_slot > LORA_MAX_RANK), LORA_ERR_METADATA
 * (n_prefill outside [0, n_rows], missing segment or group tables),
 * LORA_ERR_WORKSPACE, LORA_ERR_CUDA (a launch failed; kernels enqueued
 * before it stay enqueued).  Device status: LORA_DEV_* above.
 */
lora_status_t lora_apply(lora_bf16_t* y, int ld_y, const lora_bf16_t* x, int ld_x, int h_in,
                         const lora_proj_t* projs, int n_proj, int r_slot, int n_slots,
                         const lora_meta_t* meta, void* workspace, size_t ws_bytes,
                         uint32_t flags, int32_t* dev_status, lora_stream_t stream);

/* Workspace bytes lora_apply needs for n_rows rows, n_proj projections of
 * slot rank r_slot; 0 for counts lora_apply rejects (a non-positive count,
 * n_proj > LORA_MAX_PROJ, r_slot > LORA_MAX_RANK). */
size_t lora_apply_workspace_bytes(int n_rows, int n_proj, int r_slot);

/* Size of the scratch array built into the library for lora_apply_noalloc. */
#define LORA_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * lora_apply for callers that cannot allocate device memory at call time
 * (an engine that has reserved nearly all free HBM for its KV cache, a
 * plug-in that may only use its host's memory pool, a loop that cannot
 * afford cudaMalloc's device synchronisation).  The source pages have no
 * counterpart to this entry point; it is a deployment convenience.
 * Same arguments and results as lora_apply, minus the workspace: lora_apply's
 * workspace (the intermediate v, fp32 and as bf16 hi/lo planes) lives in a
 * LORA_NOALLOC_SCRATCH_BYTES array compiled into the library, which every
 * GPU that loads the library holds until exit.
 *   - Returns LORA_ERR_WORKSPACE, before anything is enqueued, when
 *     lora_apply_workspace_bytes(meta->n_rows, n_proj, r_slot) exceeds
 *     LORA_NOALLOC_SCRATCH_BYTES (16 MiB: e.g. 16384 rows x 2 projections
 *     of slot rank 64).
 *   - The first call on a device looks up the array's device address on
 *     the current device (cudaGetSymbolAddress); make that first call
 *     before any stream capture.  LORA_ERR_CUDA if the lookup fails.  The
 *     address is kept for the life of the process: after a device reset
 *     (cudaDeviceReset, or a reset of the primary context) it may be stale,
 *     so do not call this entry point again on that device.
 *   - n_slots, r_slot and the row count are checked as lora_apply checks
 *     them before the size test, so a bad rank gives lora_apply's status.
 *   - No allocation of any kind happens on this path.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero); calls that may overlap on the
 *     GPU, e.g. on two streams, race on it.
 */
lora_status_t lora_apply_noalloc(lora_bf16_t* y, int ld_y, const lora_bf16_t* x, int ld_x, int h_in,
                                 const lora_proj_t* projs, int n_proj, int r_slot, int n_slots,
                                 const lora_meta_t* meta, uint32_t flags, int32_t* dev_status,
                                 lora_stream_t stream);

/*
 * The LoRA linear layer [MLS, direct answer: the base product runs once for
 * the whole batch and every row adds its own adapter's delta; TGI,
 * implementation: the LoRA layer adds the adapter output to the base
 * layer's output].  For every row t and every column c of projection p:
 *   y[t][off_p + c] = bf16_rne( sum_k x[t][k] W[off_p + c][k]
 *                               + sum_j B'_{p,id_t}[c][j] (A_{p,id_t} x_t)[j] )
 * one rounding of the fp32 sum (base rows, id -1: the base product alone).
 * y is written, not read.
 *   W      [dev] [n_out][ld_w] bf16: the projections' base weights stacked,
 *          rows [off_p, off_p + width_p) for projection p, where the
 *          projections tile [0, n_out) in order (off_0 = 0, off_{p+1} =
 *          off_p + width_p); 16-byte aligned, ld_w >= h_in, ld_w % 8 == 0
 *   other arguments as lora_apply (the same stores, metadata and
 *   workspace: lora_apply_workspace_bytes(n_rows, n_proj, r_slot)).
 * Limits: r_slot <= 64 when the batch has decode rows; up to
 * LORA_MAX_RANK for prefill-only batches whose r_slot is a multiple of 16
 * with n_proj * r_slot <= 256.  Per-row ids are read from meta->lora_ids,
 * which must name the same adapters as the segment and group tables.
 * Errors (before anything is enqueued): as lora_apply, plus LORA_ERR_SHAPE
 * when the projections do not tile [0, n_out) or ld_w < h_in, and
 * LORA_ERR_RANK_EXCEEDS_SLOT beyond the limits above.  Device status: rows
 * naming an id outside [-1, n_slots) keep the base product and set
 * LORA_DEV_SLOT_OUT_OF_RANGE; LORA_DEV_TIMEOUT as lora_apply.
 */
lora_status_t lora_linear(lora_bf16_t* y, int ld_y, const lora_bf16_t* x, int ld_x, int h_in,
                          const lora_bf16_t* W, int ld_w, const lora_proj_t* projs, int n_proj, int r_slot,
                          int n_slots, const lora_meta_t* meta, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, lora_stream_t stream);

/*
 * Merged weight for single-tenant serving [MLS, interviewer follow-ups:
 * merging W' = W + B A gives the same model]:
 *   W[o][k] <- bf16_rne(W[o][k] + sign * sum_j B[o][j] A[j][k])
 * sign = +1 folds the adapter into the base weight, -1 takes it out again
 * (W comes back to within one bf16 rounding per element; exactly when no
 * rounding happened).  The sum runs in fp32 over the slot rank (padding
 * ranks are zero).
 *   W      [dev] [out][ld_w] bf16, updated in place (16-byte aligned,
 *          ld_w >= h_in, both multiples of 8)
 *   A      [dev] [r_slot][h_in]: one adapter slot of the A store
 *          (the store pointer + slot * r_slot * h_in)
 *   B      [dev] [out][r_slot]: the same slot of the scaled B store
 * Errors (before anything is enqueued): LORA_ERR_INVALID_ARG (null pointer,
 * non-positive size, sign not +1 or -1), LORA_ERR_SHAPE (ld_w < h_in, more
 * than 4M rows), LORA_ERR_RANK_EXCEEDS_SLOT (r_slot > LORA_MAX_RANK),
 * LORA_ERR_ALIGNMENT, LORA_ERR_CUDA (launch).  No device-side failure is
 * possible: the kernel reads no indices.
 */
lora_status_t lora_merge(lora_bf16_t* W, int ld_w, int out, int h_in, const lora_bf16_t* A,
                         const lora_bf16_t* B, int r_slot, int sign, lora_stream_t stream);

/*
 * lora_merge over n weights in one launch (per 32 weights): W[i], ld_w[i],
 * out[i], h_in[i], A[i], B[i] as in lora_merge, all with the same r_slot
 * and sign (e.g. one adapter folded into every projection of a model).
 * The arrays are host memory; the pointers in them are device memory.
 * Same result, bit for bit, as n calls of lora_merge.  Errors (before
 * anything is enqueued): as lora_merge for any weight, LORA_ERR_INVALID_ARG
 * for n < 0 or a NULL array.
 */
lora_status_t lora_merge_batch(int n, lora_bf16_t* const* W, const int* ld_w, const int* out, const int* h_in,
                               const lora_bf16_t* const* A, const lora_bf16_t* const* B, int r_slot, int sign,
                               lora_stream_t stream);

/* ------------------------------------------------------------------ *
 *  Adapter slots: GPU slots fed from a host cache of prepared adapters
 * ------------------------------------------------------------------ */

/*
 * [VLLM step 2]: max_loras adapters live in GPU slots at once, up to
 * max_cpu_loras prepared adapters wait in host memory, and the slot rank is
 * the largest rank served; [VLLM, limits]: an adapter of higher rank cannot
 * load.  [TGI 3]: an adapter is prepared once -- scale folded into B, ranks
 * zero-padded to the slot rank -- before it is used.
 *
 * The manager owns a host cache of up to max_cpu prepared adapters in pinned
 * memory mapped into the device's address space (least recently used
 * evicted first) and assigns adapters to the n_slots slots of the caller's
 * device stores (least recently used slot reused first, never one the
 * current batch needs).  The adapters a batch loads are gathered from the
 * host cache into their slots by one kernel launch (per 64 pieces; a piece
 * is one projection's A or B) on the caller's stream: kernels enqueued on
 * that stream after lora_slots_acquire see them, kernels enqueued before it
 * have finished with the slots' old contents.  Use one stream for lora_slots_acquire and the kernels that read
 * the stores.  Not thread-safe: one manager per serving thread.
 *
 * Without device stores the manager only tracks the assignment (no device
 * memory, no copies): the policy on its own.
 */
typedef struct lora_slot_manager lora_slot_manager_t;

typedef struct {
    uint64_t registered;        /* adapters prepared into the host cache */
    uint64_t host_evictions;    /* cached adapters dropped to make room */
    uint64_t hits;              /* batch adapters already resident in a slot */
    uint64_t loads;             /* adapters copied into a slot */
    uint64_t slot_evictions;    /* resident adapters replaced by a load */
} lora_slot_stats_t;

/*
 * Creates a manager for n_proj projections (1..16) of input widths h_in[p]
 * (multiples of 8) and output widths width[p], with device stores
 * A_stores[p] [n_slots][r_slot][h_in[p]] and B_stores[p]
 * [n_slots][width[p]][r_slot] (both arrays NULL: policy only), and a host
 * cache of max_cpu adapters (max_cpu >= n_slots).  Errors:
 * LORA_ERR_INVALID_ARG, LORA_ERR_RANK_EXCEEDS_SLOT (r_slot > LORA_MAX_RANK),
 * LORA_ERR_ALIGNMENT (r_slot or an h_in not a multiple of 8, a store not
 * 16-byte aligned).
 */
lora_status_t lora_slots_create(int n_proj, const int* h_in, const int* width, lora_bf16_t* const* A_stores,
                                lora_bf16_t* const* B_stores, int n_slots, int r_slot, int max_cpu,
                                lora_slot_manager_t** out);
void lora_slots_destroy(lora_slot_manager_t* m);

/*
 * Prepares adapter `adapter_id` (>= 0) into the host cache: A[p] host bf16
 * [r][h_in[p]], B[p] host bf16 [width[p]][r] (peft orientation, unscaled),
 * scale alpha/r (alpha/sqrt(r) with use_rslora) folded into B with one
 * rounding, ranks padded to r_slot.  Re-registering an id replaces it (a
 * resident copy is reloaded at its next acquire).  A full cache first drops
 * its least recently used adapter that is not resident in a slot.
 * Errors, all before anything changes: LORA_ERR_INVALID_ARG,
 * LORA_ERR_RANK_EXCEEDS_SLOT (r > r_slot), LORA_ERR_SLOT_RANGE (cache full
 * of resident adapters), LORA_ERR_CUDA (pinned allocation).
 */
lora_status_t lora_slots_register(lora_slot_manager_t* m, int64_t adapter_id, const lora_bf16_t* const* A,
                                  const lora_bf16_t* const* B, int r, double alpha, int use_rslora);

/*
 * Maps a batch's adapter ids (n entries, -1 = base model) to slot ids in
 * slots_out (-1 stays -1), loading the adapters that are not resident.
 * Errors, before anything is enqueued or changed: LORA_ERR_INVALID_ARG (an
 * id neither -1 nor registered), LORA_ERR_SLOT_RANGE (more distinct adapters
 * than slots).  LORA_ERR_CUDA: the load could not be enqueued; the slots
 * meant for this batch's loads are left empty (resident adapters stay).
 */
lora_status_t lora_slots_acquire(lora_slot_manager_t* m, const int64_t* adapter_ids, int n, int32_t* slots_out,
                                 lora_stream_t stream);

/* Slot currently holding adapter_id, or -1. */
int lora_slots_slot_of(const lora_slot_manager_t* m, int64_t adapter_id);
lora_status_t lora_slots_stats(const lora_slot_manager_t* m, lora_slot_stats_t* out);

/* ------------------------------------------------------------------ *
 *  Host helpers (host pointers, synchronous)
 * ------------------------------------------------------------------ */

/*
 * Batch metadata [TGI 4; VLLM step 3]:
 *   (i) prefill segments = maximal runs of equal id over rows [0, n_prefill)
 *       in row order; runs of -1 are kept with slot -1;
 *  (ii) decode gather form = decode rows sorted by slot ascending, ties in
 *       row order, -1 rows last, one group per distinct id present; perm
 *       holds absolute row indices.
 * Capacities: seg_starts n_prefill+1, seg_slot n_prefill,
 * perm n_rows-n_prefill, gseg_starts n_slots+2, gseg_slot n_slots+1.
 * max_seg_len / max_gseg_len may be NULL.
 * Returns LORA_ERR_SLOT_RANGE if an id lies outside [-1, n_slots).
 */
lora_status_t lora_build_metadata(const int32_t* ids, int n_rows, int n_prefill, int n_slots,
                                  int32_t* seg_starts, int32_t* seg_slot, int* n_segs,
                                  int* max_seg_len, int32_t* perm, int32_t* gseg_starts,
                                  int32_t* gseg_slot, int* n_gsegs, int* max_gseg_len);

/*
 * Adapter store preparation [TGI 3]:
 *   s = alpha / r, or alpha / sqrt(r) when use_rslora (computed in double);
 *   B_slot[c][j] = bf16_rne(s * B[c][j]) for j < r, 0 for r <= j < r_slot;
 *   A_slot[j][i] = A[j][i] for j < r, 0 for r <= j < r_slot.
 * A [host] bf16 [r][h_in]; B [host] bf16 [out][r] (peft lora_A / lora_B);
 * A_slot_out [host] [r_slot][h_in]; B_slot_out [host] [out][r_slot].
 * Returns LORA_ERR_RANK_EXCEEDS_SLOT if r > r_slot [VLLM limits].
 */
lora_status_t lora_prepare_adapter(const lora_bf16_t* A, const lora_bf16_t* B, int r, int h_in,
                                   int out, double alpha, int use_rslora, int r_slot,
                                   lora_bf16_t* A_slot_out, lora_bf16_t* B_slot_out);

/* Slot rank for a set of adapter ranks: the largest rank [VLLM step 2],
 * rounded up to a multiple of 8 (the kernels' 128-bit vector of bf16). */
int lora_slot_rank(const int* ranks, int n);

/* Copies *dev_status to *out (host) on `stream` and waits for it. */
lora_status_t lora_read_device_status(const int32_t* dev_status, int32_t* out,
                                      lora_stream_t stream);

const char* lora_status_string(lora_status_t status);

/* Number of kernels this library has launched from the host since it was
 * loaded (a diagnostic; replays of a captured CUDA graph are not counted). */
uint64_t lora_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_GB300_H */
