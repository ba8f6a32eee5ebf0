// bgmv_grouped.cu -- decode-row LoRA delta in two launches: a grouped shrink
// that stores the fp32 intermediate v, then a grouped expand.
//
// TGI multi-LoRA page, "4. SGMV and BGMV at inference": decode tokens apply
// their own adapters; the rows arrive grouped by adapter (gather form of the
// batch metadata), a unit of work is (adapter, up to 16 of its rows), and
// each adapter's A and B' are streamed from HBM once per call.  This form
// serves the calls the one-launch kernel handles poorly: wide outputs and
// calls that stream many weight bytes, where the whole cost is moving A
// and B' and the launch overhead of a second kernel is small beside it.
//
// Grouped shrink: one CTA per (unit, block of 16 ranks) -- optionally a
// cluster of CTAs splitting K -- computes
//   v[t][j] = sum_k A_slot[j][k] x[t][k]      (fp32, mma.sync m16n8k16)
// for the unit's rows t, with the ranks as the mma M and the rows as N (a
// unit of <= 8 rows costs one mma per 16 ranks x 16 K).  Each stage brings
// 512 K-elements of every one of its 16 A rows and of the unit's x rows by
// 16-byte cp.async, a warp per 512 contiguous bytes, into padded shared
// rows (pitch 1040 bytes, so ldmatrix is conflict-free), four stages deep.
// (Bulk copies of 1 KB pieces reach well under half the bandwidth of this
// form on GB300; bulk copies pay off from about 4 KB, as in the expand
// below.)  Partial sums of the eight warps (and of the cluster's CTAs) are
// added in a fixed order: the result does not depend on timing.
//
// Grouped expand: one CTA per (unit, block of 256 output columns); each warp
// brings its 64 columns of B' (contiguous in [columns][r_slot] storage) with
// one bulk copy, requested as soon as the adapter slot is known (before the
// rows and the grid dependency resolve), loads the y pieces it will update
// while B' is in flight, and forms
//   d^T[col][t] = sum_j B'[col][j] (v_hi + v_lo)[t][j],   y <- bf16_rne(y + d)
// with v split into bf16 hi and lo parts (v itself is never rounded to one
// bf16; the split carries it to ~2^-17 relative).
//
// Ordering (programmatic dependent launch): both kernels read metadata and
// weights before griddepcontrol.wait.  The shrink reads x after it unless
// LORA_APPLY_X_READY, and always stores v after it (the previous call's
// expand may still be reading v); the expand reads v and y after it.
// Waits on mbarriers are bounded (0.2 s) and end in LORA_DEV_TIMEOUT.

#include <algorithm>
#include <climits>

#include "decode_common.cuh"
#include "launch.h"

namespace lora {

namespace {

using namespace dec;

// ---- unit lookup -----------------------------------------------------------

// Unit u of the grid.  Direct form (upg > 0): u = group * upg + sub, rows
// [gstarts[group] + 16 sub, ...): one round trip, no block-wide scan; a
// group whose bounds are not sane is reported by its first unit, and a
// table that does not cover [0, n_pos) by unit 0.  Scanned
// form (upg == 0): units are numbered over all groups by a prefix sum.
template <int NT, class Params>
__device__ __forceinline__ UnitInfo grouped_unit(const Params& p, int u, int grid_units)
{
    if (p.upg > 0) {
        UnitInfo ui;
        ui.g = u / p.upg;
        const int sub = u - ui.g * p.upg;
        const int s = __ldg(p.gstarts + ui.g), e = __ldg(p.gstarts + ui.g + 1);
        ui.slot = __ldg(p.gslot + ui.g);
        const bool sane = s >= 0 && e <= p.n_pos && s <= e && e - s <= p.upg * kRB;
        // the first unit also checks that the table covers [0, n_pos)
        const bool covers = u != 0 || (__ldg(p.gstarts) == 0 && __ldg(p.gstarts + p.n_groups) == p.n_pos);
        ui.bad = (!sane && sub == 0) || !covers;
        ui.pos0 = s + sub * kRB;
        ui.nrows = sane ? min(kRB, e - ui.pos0) : 0;
        ui.found = ui.nrows > 0;
        return ui;
    }
    UnitInfo ui = find_unit<NT>(p, u, nullptr, false, grid_units);
    if (!ui.found) ui.nrows = 0;
    return ui;
}

// Rows of the unit through perm (threads 0..15; no perm: the positions are
// the rows); false when one is out of range.
__device__ __forceinline__ bool unit_rows(const int32_t* perm, int pos0, int nrows, int n_rows, int* s_rows)
{
    bool bad = false;
    const int tid = threadIdx.x;
    if (tid < kRB) {
        int r = 0;
        if (tid < nrows) {
            r = perm ? __ldg(perm + pos0 + tid) : pos0 + tid;
            if (r < 0 || r >= n_rows) {
                bad = true;
                r = 0;
            }
        }
        s_rows[tid] = r;
    }
    return bad;
}

// Ids form (per-row adapter ids, no gather metadata: the standalone BGMV
// calls).  Unit u is the (u % subs)-th run of up to 16 rows, in row order,
// among the rows whose id is slot u / subs; its rows land in s_rows (rows
// past the unit's read 0).  One block-wide ordered compaction per NT ids,
// stopping once the run is complete.  Unit 0 reads every id and reports one
// outside [-1, n_slots) in bad (such a row matches no slot and is skipped).
// Every thread takes part; the answer is uniform across the CTA.
template <int NT>
__device__ UnitInfo ids_unit(const int32_t* ids, int n_pos, int n_slots, int u, int subs, int* s_rows)
{
    __shared__ int s_cnt[NT / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    UnitInfo ui;
    ui.slot = u / subs;
    ui.g = ui.slot;
    ui.pos0 = 0;
    const int lo = (u - ui.slot * subs) * kRB;
    int base = 0;   // matching rows in earlier rounds
    bool bad = false;
    for (int r0 = 0; r0 < n_pos && (u == 0 || base < lo + kRB); r0 += NT) {
        const int i = r0 + tid;
        const int id = i < n_pos ? __ldg(ids + i) : -1;
        bad |= id < -1 || id >= n_slots;
        const bool m = i < n_pos && id == ui.slot;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, m);
        if (lane == 0) s_cnt[warp] = __popc(bal);
        __syncthreads();
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) {
            const int c = s_cnt[w];
            if (w < warp) before += c;
            total += c;
        }
        const int rank = base + before + __popc(bal & ((1u << lane) - 1u));
        if (m && rank >= lo && rank < lo + kRB) s_rows[rank - lo] = i;
        base += total;
        __syncthreads();   // s_cnt is rewritten by the next round
    }
    ui.nrows = max(0, min(kRB, base - lo));
    ui.found = ui.nrows > 0;
    if (tid < kRB && tid >= ui.nrows) s_rows[tid] = 0;
    ui.bad = __syncthreads_or(bad) && u == 0;
    return ui;
}

// ---- grouped shrink ----------------------------------------------------------

constexpr int kGsThreads = 256;
constexpr int kGsWarps = kGsThreads / 32;
constexpr int kGsRanks = 16;                      // ranks per CTA: two mma n-tiles
constexpr int kGsKT = 512;                        // K elements per stage
constexpr int kGsPitch = kGsKT * 2 + 16;          // shared row pitch (bytes): 16 mod 128
constexpr int kGsStages = 4;

struct GsParams {
    ProjSet ps;
    const bf16_t* x;
    int ld_x;
    int h_in;
    bf16_t* vh;               // v = vh + vl: bf16 planes [n_rows][ld_p], projection p at p*r_pad64
    bf16_t* vl;
    int ld_p;
    int r_pad64;
    float* v;                 // or, when not null, fp32 v [n_rows][ld_v] (rank j at column j)
    int ld_v;
    const int32_t* perm;
    const int32_t* gstarts;
    const int32_t* gslot;
    int n_groups;
    int n_pos;
    int n_slots;
    int n_rows;
    int n_rb;                 // rank blocks per unit
    int upg;                  // direct unit form (units per group) or 0
    int xr;                   // x rows per stage buffer: >= rows of any unit, <= 16
    int kc;                   // K elements per cluster rank (multiple of kGsKT)
    int ks;                   // cluster size (CTAs splitting K)
    int x_ready;
    int late_trigger;         // dependents launch only once x may be read (see kShrinkTriggerLate)
    const int32_t* ids;       // ids form: per-row adapter ids instead of the gather metadata (or null)
    int id_subs;              // ids form: units per slot, ceil(n_pos / 16)
    int32_t* status;
};

__host__ inline size_t gs_smem_bytes(int xr)
{
    return static_cast<size_t>(kGsStages) * (kGsRanks + xr) * kGsPitch;
}

__global__ void __launch_bounds__(kGsThreads)
bgmv_group_shrink_kernel(GsParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sA = smem;                                            // [S][16][pitch]
    unsigned char* sX = smem + static_cast<size_t>(kGsStages) * kGsRanks * kGsPitch;   // [S][xr][pitch]
    float* red = reinterpret_cast<float*>(smem);   // [warps][16][16], after the last stage
    __shared__ __align__(16) float s_vp[kRB * kGsRanks];
    __shared__ int s_rows[kRB];

    if (!p.late_trigger) grid_dep_launch();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int crank = p.ks > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int cl = blockIdx.x / p.ks;
    const int unit = cl / p.n_rb, rb = cl - unit * p.n_rb;
    const int grid_units = static_cast<int>(gridDim.x) / (p.ks * p.n_rb);
    // uniform across the cluster
    const UnitInfo ui = p.ids ? ids_unit<kGsThreads>(p.ids, p.n_pos, p.n_slots, unit, p.id_subs, s_rows)
                              : grouped_unit<kGsThreads>(p, unit, grid_units);
    const int pos0 = ui.pos0, nrows = ui.nrows, slot = ui.slot;
    const bool flagger = rb == 0 && crank == 0 && tid == 0;
    if (ui.bad) {   // flagged, and a unit that was found is still done
        grid_dep_wait();
        if (flagger) flag(p.status, p.ids ? LORA_DEV_SLOT_OUT_OF_RANGE : LORA_DEV_BAD_SEGMENT);
    }
    if (nrows <= 0 || slot == -1) {
        if (blockIdx.x == 0) grid_dep_wait();
        return;
    }
    if (slot < -1 || slot >= p.n_slots) {
        grid_dep_wait();
        if (flagger) flag(p.status, LORA_DEV_SLOT_OUT_OF_RANGE);
        return;
    }
    if (nrows > p.xr) {   // a group longer than the metadata's longest
        grid_dep_wait();
        if (flagger) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }
    const int R = p.ps.n_proj * p.ps.r_slot, r_slot = p.ps.r_slot;
    const int j0 = rb * kGsRanks, nj = min(kGsRanks, R - j0);   // 8 or 16
    const int k_begin = crank * p.kc;
    const int k_end = min(p.h_in, k_begin + p.kc);
    const int n_kt = k_end > k_begin ? (k_end - k_begin + kGsKT - 1) / kGsKT : 0;

    // Copy plan: 64 threads per row piece of kGsKT elements (one 16-byte
    // chunk each, so a warp reads 512 contiguous bytes), rows r4, r4+4, ...
    // The source pointers stay fixed; a stage adds its K offset.  Chunks past
    // k_end, and x rows past the unit's, are zero-filled.
    const int c16 = tid & 63, r4 = tid >> 6;
    const bf16_t* a_src[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = r4 + 4 * i;
        a_src[i] = nullptr;
        if (row < nj) {
            int pj = 0, jj = j0 + row;
            while (jj >= r_slot) {
                jj -= r_slot;
                ++pj;
            }
            a_src[i] = p.ps.A[pj] + (static_cast<size_t>(slot) * r_slot + jj) * p.h_in + k_begin + c16 * 8;
        }
    }
    auto issue_A = [&](int kt, int b) {
        const int off = kt * kGsKT;
        const bool ok = k_begin + off + c16 * 8 < k_end;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = r4 + 4 * i;
            if (row < nj)
                cp_async16(smem_u32(sA + (b * kGsRanks + row) * kGsPitch + c16 * 16), ok ? a_src[i] + off : p.x, ok);
        }
    };
    // Weights first: A for the first stages is requested as soon as the
    // slot is known, before the rows are resolved and before the grid
    // dependency resolves.
#pragma unroll
    for (int st = 0; st < kGsStages; ++st) {
        if (st < n_kt) issue_A(st, st);
        cp_async_commit();
    }

    if (__syncthreads_or(p.ids ? false : unit_rows(p.perm, pos0, nrows, p.n_rows, s_rows))) {
        cp_async_wait<0>();   // no copy may land after the CTA has left
        grid_dep_wait();      // same rows in every CTA of the cluster: all leave here
        if (flagger) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }
    const bf16_t* x_src[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = r4 + 4 * i;
        x_src[i] = row < nrows ? p.x + static_cast<size_t>(s_rows[row]) * p.ld_x + k_begin + c16 * 8 : nullptr;
    }
    auto issue_X = [&](int kt, int b) {
        const int off = kt * kGsKT;
        const bool ok = k_begin + off + c16 * 8 < k_end;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = r4 + 4 * i;
            if (t < p.xr) {
                const bool v = ok && t < nrows;
                cp_async16(smem_u32(sX + (b * p.xr + t) * kGsPitch + c16 * 16), v ? x_src[i] + off : p.x, v);
            }
        }
    };
    // x follows the grid dependency unless the caller says x is ready.
    bool waited = false;
    if (!p.x_ready) {
        grid_dep_wait();
        waited = true;
    }
    if (p.late_trigger) grid_dep_launch();   // everything before this kernel is complete: x may be read
#pragma unroll
    for (int st = 0; st < kGsStages; ++st) {
        if (st < n_kt) issue_X(st, st);
        cp_async_commit();
    }

    // ---- K loop: warp w takes k-steps w, w+8, ... of each stage ----
    // Transposed tile: the 16 ranks fill the mma M, the unit's rows the N
    // (8 per n-tile), so units of <= 8 rows take one mma per k-step.
    //   d[nt][0..1] = (rank g, rows 8nt+2q, +1), d[nt][2..3] = (rank g+8, same rows)
    const int n_nt = (nrows + 7) / 8;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int mi = lane >> 3, mr = lane & 7;
    const int arow = (mi & 1) * 8 + mr;                // rank row of this lane's ldmatrix address
    const int l16 = lane & 15;
    for (int kt = 0; kt < n_kt; ++kt) {
        // groups so far: {A_0}..{A_S-1} {X_0}..{X_S-1}, then one per
        // iteration: stage kt is complete once at most S-1 groups are pending
        cp_async_wait<kGsStages - 1>();
        __syncthreads();
        const int b = kt % kGsStages;
        const int n_ks = (min(kGsKT, k_end - (k_begin + kt * kGsKT)) + 15) / 16;
        const unsigned char* xs = sX + b * p.xr * kGsPitch;
        const unsigned char* as = sA + b * kGsRanks * kGsPitch;
        for (int ks = warp; ks < n_ks; ks += kGsWarps) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(smem_u32(as + arow * kGsPitch + (ks * 16 + (mi >> 1) * 8) * 2), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                if (nt < n_nt) {
                    uint32_t b0, b1;
                    const int xrow = min(nt * 8 + (l16 & 7), p.xr - 1);   // rows past the unit's: never stored
                    ldmatrix_x2(smem_u32(xs + xrow * kGsPitch + (ks * 16 + (l16 >> 3) * 8) * 2), b0, b1);
                    mma_bf16_16816(acc[nt], a0, a1, a2, a3, b0, b1);
                }
            }
        }
        __syncthreads();   // every warp is done with buffer b
        if (kt + kGsStages < n_kt) {
            issue_A(kt + kGsStages, b);
            issue_X(kt + kGsStages, b);
        }
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- fixed-order reduction over the warps, then over the cluster ----
    {
        const int g = lane >> 2, q2 = (lane & 3) * 2;
        float* rw = red + warp * kRB * kGsRanks;   // [row t][rank j]
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int t = nt * 8 + q2;
            rw[t * kGsRanks + g] = acc[nt][0];
            rw[(t + 1) * kGsRanks + g] = acc[nt][1];
            rw[t * kGsRanks + g + 8] = acc[nt][2];
            rw[(t + 1) * kGsRanks + g + 8] = acc[nt][3];
        }
    }
    __syncthreads();
    {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kGsWarps; ++w) s += red[w * kRB * kGsRanks + tid];
        s_vp[tid] = s;   // kGsThreads == kRB * kGsRanks: element (tid / 16, tid % 16)
    }
    if (!waited) grid_dep_wait();   // v may still be read by the preceding grid
    const int t = tid >> 4, j = tid & 15;
    // v (fp32) is stored as it is, or split: vh = bf16(v), vl = bf16(v - vh), exact in fp32
    auto store_v = [&](float v) {
        const int jr = j0 + j, pj = jr / r_slot, jj = jr - pj * r_slot;
        if (p.v) {
            p.v[static_cast<size_t>(s_rows[t]) * p.ld_v + jr] = v;
            return;
        }
        const size_t off = static_cast<size_t>(s_rows[t]) * p.ld_p + pj * p.r_pad64 + jj;
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        p.vh[off] = __bfloat16_as_ushort(hi);
        p.vl[off] = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(hi)));
    };
    if (p.ks == 1) {
        if (t < nrows && j < nj) store_v(s_vp[tid]);
        return;
    }
    cluster_arrive();
    cluster_wait();
    if (t < nrows && j < nj && t % p.ks == crank) {   // CTA c stores rows c, c + ks, ...
        const uint32_t base = smem_u32(s_vp + tid);
        float s = 0.f;
        for (int c = 0; c < p.ks; ++c) {
            float f;
            asm("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(f) : "r"(map_rank(base, c)));
            s += f;
        }
        store_v(s);
    }
    cluster_arrive();   // peers may leave once everyone has read their partials
    cluster_wait();
}

// ---- grouped expand ----------------------------------------------------------

constexpr int kGxThreads = 128;
constexpr int kGxWarps = kGxThreads / 32;
constexpr int kGxCols = 256;                          // output columns per block
constexpr int kGxWarpCols = kGxCols / kGxWarps;       // 64: one bulk copy per warp
constexpr int kGxTiles = kGxWarpCols / 16;            // 16-column tiles per warp
constexpr int kGxLdD = 20;       // per-warp delta tile row stride (floats): conflict-free

struct GexParams {
    ProjSet ps;
    const bf16_t* vh;         // v = vh + vl: bf16 planes [n_rows][ld_p], projection p at p*r_pad64
    const bf16_t* vl;
    int ld_p;
    int r_pad64;
    const float* v;           // or, when not null, fp32 v [n_rows][ld_v], projection p at p*r_slot,
    int ld_v;                 //   split into the same hi/lo parts as it is read
    bf16_t* y;
    int ld_y;
    const int32_t* perm;
    const int32_t* gstarts;
    const int32_t* gslot;
    int n_groups;
    int n_pos;
    int n_slots;
    int n_rows;
    int n_blocks;             // column blocks per unit, over all projections
    int upg;                  // direct unit form (units per group) or 0
    const int32_t* ids;       // ids form: per-row adapter ids instead of the gather metadata (or null)
    int id_subs;              // ids form: units per slot, ceil(n_pos / 16)
    int32_t* status;
};

// Column block b -> projection and its first column.
__device__ __forceinline__ void block_proj(const ProjSet& ps, int b, int& pj, int& col0)
{
    pj = 0;
    int nb = (ps.width[0] + kGxCols - 1) / kGxCols;
    while (pj < ps.n_proj - 1 && b >= nb) {
        b -= nb;
        ++pj;
        nb = (ps.width[pj] + kGxCols - 1) / kGxCols;
    }
    col0 = b * kGxCols;
}

__device__ __forceinline__ uint4 lds128(const bf16_t* p)
{
    return *reinterpret_cast<const uint4*>(p);
}

__global__ void __launch_bounds__(kGxThreads, 5)
bgmv_group_expand_kernel(GexParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];   // B' block [ncols][r_slot]
    __shared__ __align__(16) float s_d[kGxWarps][kRB * kGxLdD];
    __shared__ __align__(8) uint64_t s_bar[kGxWarps];
    __shared__ int s_rows[kRB];
    const bf16_t* sB = reinterpret_cast<const bf16_t*>(smem);

    grid_dep_launch();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x / p.n_blocks;
    const int blk = blockIdx.x - unit * p.n_blocks;
    const UnitInfo ui = p.ids ? ids_unit<kGxThreads>(p.ids, p.n_pos, p.n_slots, unit, p.id_subs, s_rows)
                              : grouped_unit<kGxThreads>(p, unit, INT_MAX);   // unit count: checked by the shrink
    const int pos0 = ui.pos0, nrows = ui.nrows, slot = ui.slot;
    const bool bad = ui.bad;
    const int32_t bad_bit = p.ids ? LORA_DEV_SLOT_OUT_OF_RANGE : LORA_DEV_BAD_SEGMENT;
    const bool flagger = blk == 0 && tid == 0;   // one CTA per unit reports
    if (nrows <= 0 || slot == -1) {
        if (blockIdx.x == 0 || bad) grid_dep_wait();
        if (bad && flagger) flag(p.status, bad_bit);
        return;
    }
    if (slot < -1 || slot >= p.n_slots) {
        grid_dep_wait();
        if (flagger) flag(p.status, LORA_DEV_SLOT_OUT_OF_RANGE);
        return;
    }
    int pj, col0;
    block_proj(p.ps, blk, pj, col0);
    const int width = p.ps.width[pj];
    const int ncols = min(kGxCols, width - col0);          // a multiple of 8
    const int r_slot = p.ps.r_slot;
    const int wc0 = warp * kGxWarpCols;                    // this warp's first column in the block
    const int wcols = max(0, min(kGxWarpCols, ncols - wc0));
    if (wcols > 0 && lane == 0) {
        // Weights first, as soon as the slot is known: lane 0 owns the warp's
        // barrier (init, expect, copy), before the rows and the grid dependency.
        const unsigned bytes = static_cast<unsigned>(wcols * r_slot * sizeof(bf16_t));
        mbar_init(&s_bar[warp], 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        mbar_expect(&s_bar[warp], bytes);
        bulk_g2s(smem + sizeof(bf16_t) * wc0 * r_slot,
                 p.ps.B[pj] + (static_cast<size_t>(slot) * width + col0 + wc0) * r_slot, bytes, &s_bar[warp]);
    }
    __syncwarp();
    if (__syncthreads_or(p.ids ? false : unit_rows(p.perm, pos0, nrows, p.n_rows, s_rows))) {
        if (wcols > 0 && lane == 0) mbar_wait(&s_bar[warp], 0);   // let the block land before leaving (bounded)
        grid_dep_wait();
        if (flagger) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }

    grid_dep_wait();   // v is the preceding kernel's output; y may be too
    if (wcols == 0) return;

    // y pieces this lane updates (tile i, row lane/2, columns 8*(lane&1)..+7),
    // loaded now so they arrive together with B'
    const int yt = lane >> 1, yh = lane & 1;
    bf16_t* yrow = p.y + static_cast<size_t>(s_rows[yt]) * p.ld_y + p.ps.out_off[pj] + col0;
    uint4 yv[kGxTiles];
#pragma unroll
    for (int i = 0; i < kGxTiles; ++i) {
        const int c = wc0 + i * 16 + yh * 8;
        yv[i] = (yt < nrows && c < ncols) ? *reinterpret_cast<const uint4*>(yrow + c) : make_uint4(0, 0, 0, 0);
    }

    // v fragments (the mma B operand) straight from the hi/lo planes, n-tile
    // nt = rows 8nt..8nt+7: b0 <- v[t][k0..k0+1], b1 <- v[t][k0+2..k0+3],
    // k0 = 8(q+4h)+4e: one 8-byte load per plane.
    const int g = lane >> 2, q = lane & 3;
    const int n_nt = (nrows + 7) / 8;
    const int np = r_slot / 8;              // 16-byte pieces per B' row
    const int H = (np + 3) / 4;             // pieces per lane
    uint32_t bh[2][2][2][2], bl[2][2][2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = nt * 8 + g, k0 = 8 * (q + 4 * h) + 4 * e;
                uint2 hv = make_uint2(0, 0), lv = make_uint2(0, 0);
                if (nt < n_nt && t < nrows && k0 < r_slot) {
                    if (p.v) {
                        const float4 f = *reinterpret_cast<const float4*>(
                            p.v + static_cast<size_t>(s_rows[t]) * p.ld_v + pj * r_slot + k0);
                        split_hi_lo(f.x, f.y, hv.x, lv.x);
                        split_hi_lo(f.z, f.w, hv.y, lv.y);
                    } else {
                        const size_t off = static_cast<size_t>(s_rows[t]) * p.ld_p + pj * p.r_pad64 + k0;
                        hv = *reinterpret_cast<const uint2*>(p.vh + off);
                        lv = *reinterpret_cast<const uint2*>(p.vl + off);
                    }
                }
                bh[nt][h][e][0] = hv.x;
                bh[nt][h][e][1] = hv.y;
                bl[nt][h][e][0] = lv.x;
                bl[nt][h][e][1] = lv.y;
            }

    if (!mbar_wait(&s_bar[warp], 0)) {
        // This warp's block never landed: wait once more (bounded) so no copy
        // is in flight into shared memory when the CTA leaves, then report.
        mbar_wait(&s_bar[warp], 0);
        if (lane == 0) flag(p.status, LORA_DEV_TIMEOUT);
        return;
    }

    // Odd rows read their second piece first when a lane holds two (rows
    // 128 bytes apart would otherwise meet in the same banks).
    const int swap = (H == 2) ? (g & 1) : 0;
    float* sd = s_d[warp];
#pragma unroll
    for (int i = 0; i < kGxTiles; ++i) {
        const int m0 = wc0 + i * 16;
        if (m0 >= ncols) break;
        const int ca = m0 + g, cb = ca + 8;
        uint4 La[2], Lb[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int piece = q + 4 * (j ^ swap);
            const bool okp = (j ^ swap) < H && piece < np;
            La[j] = (okp && ca < ncols) ? lds128(sB + ca * r_slot + piece * 8) : make_uint4(0, 0, 0, 0);
            Lb[j] = (okp && cb < ncols) ? lds128(sB + cb * r_slot + piece * 8) : make_uint4(0, 0, 0, 0);
        }
        const uint4 Pa0 = swap ? La[1] : La[0], Pa1 = swap ? La[0] : La[1];
        const uint4 Pb0 = swap ? Lb[1] : Lb[0], Pb1 = swap ? Lb[0] : Lb[1];
        float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (h < H) {
                const uint4 A = h ? Pa1 : Pa0, B = h ? Pb1 : Pb0;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t a0 = e ? A.z : A.x, a2 = e ? A.w : A.y;
                    const uint32_t a1 = e ? B.z : B.x, a3 = e ? B.w : B.y;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        if (nt < n_nt) {
                            mma_bf16_16816(d[nt], a0, a1, a2, a3, bh[nt][h][e][0], bh[nt][h][e][1]);
                            mma_bf16_16816(d[nt], a0, a1, a2, a3, bl[nt][h][e][0], bl[nt][h][e][1]);
                        }
                    }
                }
            }
        }
        // d[nt]: (column g, rows 8nt+2q, +1) and (column g+8, same rows)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            if (nt < n_nt) {
                const int t = nt * 8 + 2 * q;
                sd[t * kGxLdD + g] = d[nt][0];
                sd[(t + 1) * kGxLdD + g] = d[nt][1];
                sd[t * kGxLdD + g + 8] = d[nt][2];
                sd[(t + 1) * kGxLdD + g + 8] = d[nt][3];
            }
        }
        __syncwarp();
        {
            const int c = m0 + yh * 8;
            if (yt < nrows && c < ncols) {
                const float4* dp = reinterpret_cast<const float4*>(sd + yt * kGxLdD + yh * 8);
                const float4 d0 = dp[0], d1 = dp[1];
                const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                *reinterpret_cast<uint4*>(yrow + c) = add_round8(yv[i], dd);
            }
        }
        __syncwarp();
    }
    if (bad && flagger) flag(p.status, bad_bit);
}

}  // namespace

namespace {

// Launch geometry shared by the grouped shrink and expand of one call.
struct GroupedPlan {
    int r_pad64, ld_p, form_upg, xr, pdl, n_sms;
    long long units;
    const int32_t* ids;   // ids form (per-row adapter ids), or null
    int id_subs;
};

cudaError_t grouped_plan(const ProjSet& ps, int n_groups, int n_pos, int max_group_len, unsigned flags,
                         GroupedPlan& g)
{
    static int configured_device = -1;
    static int n_sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(bgmv_group_shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(gs_smem_bytes(kRB)));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(bgmv_group_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(bf16_t) * kGxCols * 64));
        if (e != cudaSuccess) return e;
        e = prefer_max_shared(reinterpret_cast<const void*>(bgmv_group_shrink_kernel));
        if (e != cudaSuccess) return e;
        e = prefer_max_shared(reinterpret_cast<const void*>(bgmv_group_expand_kernel));
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    g.n_sms = n_sms;
    g.r_pad64 = (ps.r_slot + 63) / 64 * 64;
    g.ld_p = ps.n_proj * g.r_pad64;
    // Units: direct numbering (group, sub-unit) unless the longest group
    // makes that grid much larger than the scanned one.
    const long long upg = max_group_len > 0 ? (max_group_len + kRB - 1) / kRB : 0;
    const long long scanned_units = n_groups + n_pos / kRB;
    const long long direct_units = n_groups * upg;
    g.form_upg = (upg > 0 && direct_units <= 2 * scanned_units) ? static_cast<int>(upg) : 0;
    g.units = g.form_upg ? direct_units : scanned_units;
    if (!g.form_upg && max_group_len > 0) g.units = std::min(g.units, direct_units);
    g.xr = max_group_len > 0 ? std::min(kRB, max_group_len) : kRB;
    g.pdl = (flags & LORA_APPLY_NO_PDL) ? 0 : 1;
    return cudaSuccess;
}

// The ids form's plan: units are (slot, run of 16 rows), as many as the
// worst case (every row on one slot) needs.
cudaError_t grouped_plan_ids(const ProjSet& ps, const int32_t* ids, int n_rows, int n_slots, GroupedPlan& g)
{
    const int subs = (n_rows + kRB - 1) / kRB;
    const cudaError_t e = grouped_plan(ps, 1, n_rows, kRB, 0u, g);
    if (e != cudaSuccess) return e;
    g.form_upg = 0;
    g.units = static_cast<long long>(n_slots) * subs;
    g.xr = kRB;
    g.ids = ids;
    g.id_subs = subs;
    return cudaSuccess;
}

// v goes to the planes vh/vl, or as fp32 to v (ld_v) when v is not null.
cudaError_t grouped_shrink(const GroupedPlan& g, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                           const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                           int n_pos, int n_rows, int n_slots, unsigned flags, bf16_t* vh, bf16_t* vl,
                           float* v, int ld_v, int32_t* status, cudaStream_t stream)
{
    const int R = ps.n_proj * ps.r_slot;
    GsParams sp{};
    sp.ps = ps;
    sp.x = x;
    sp.ld_x = ld_x;
    sp.h_in = h_in;
    sp.vh = vh;
    sp.vl = vl;
    sp.v = v;
    sp.ld_v = ld_v;
    sp.ld_p = g.ld_p;
    sp.r_pad64 = g.r_pad64;
    sp.perm = perm;
    sp.gstarts = gstarts;
    sp.gslot = gslot;
    sp.n_groups = n_groups;
    sp.n_pos = n_pos;
    sp.n_slots = n_slots;
    sp.n_rows = n_rows;
    sp.n_rb = (R + kGsRanks - 1) / kGsRanks;
    sp.upg = g.form_upg;
    sp.xr = g.xr;
    // Split K over a cluster only when the (unit, rank block) CTAs would not
    // fill the GPU twice over, keeping at least two stages per CTA.
    int ks = 1;
    while (ks < 8 && g.units * sp.n_rb * ks < 2LL * g.n_sms && h_in / (ks * 2) >= 2 * kGsKT) ks *= 2;
    ks = env_int("LORA_GROUPED_KS", ks);
    sp.ks = ks;
    sp.kc = ((h_in + ks - 1) / ks + kGsKT - 1) / kGsKT * kGsKT;
    sp.x_ready = (flags & LORA_APPLY_X_READY) ? 1 : 0;
    sp.late_trigger = (flags & kShrinkTriggerLate) ? 1 : 0;
    sp.ids = g.ids;
    sp.id_subs = g.id_subs;
    sp.status = status;
    const long long n_shrink = g.units * sp.n_rb * ks;
    if (n_shrink > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_shrink));
    cfg.blockDim = dim3(kGsThreads);
    cfg.dynamicSmemBytes = gs_smem_bytes(g.xr);
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (ks > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = ks;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (g.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, bgmv_group_shrink_kernel, sp);
    note_launch();
    return e;
}

// v from the planes vh/vl, or as fp32 from v (ld_v) when v is not null.
cudaError_t grouped_expand(const GroupedPlan& g, bf16_t* y, int ld_y, const ProjSet& ps, const int32_t* perm,
                           const int32_t* gstarts, const int32_t* gslot, int n_groups, int n_pos, int n_rows,
                           int n_slots, const bf16_t* vh, const bf16_t* vl, const float* v, int ld_v,
                           int32_t* status, cudaStream_t stream)
{
    GexParams gp{};
    gp.ps = ps;
    gp.vh = vh;
    gp.vl = vl;
    gp.ld_p = g.ld_p;
    gp.r_pad64 = g.r_pad64;
    gp.v = v;
    gp.ld_v = ld_v;
    gp.y = y;
    gp.ld_y = ld_y;
    gp.perm = perm;
    gp.gstarts = gstarts;
    gp.gslot = gslot;
    gp.n_groups = n_groups;
    gp.n_pos = n_pos;
    gp.n_slots = n_slots;
    gp.n_rows = n_rows;
    for (int q = 0; q < ps.n_proj; ++q) gp.n_blocks += (ps.width[q] + kGxCols - 1) / kGxCols;
    gp.upg = g.form_upg;
    gp.ids = g.ids;
    gp.id_subs = g.id_subs;
    gp.status = status;
    const long long n_expand = g.units * gp.n_blocks;
    if (n_expand > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t gcfg = {};
    gcfg.gridDim = dim3(static_cast<unsigned>(n_expand));
    gcfg.blockDim = dim3(kGxThreads);
    gcfg.dynamicSmemBytes = sizeof(bf16_t) * kGxCols * ps.r_slot;   // <= 32 KB
    gcfg.stream = stream;
    cudaLaunchAttribute gattr;
    gattr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    gattr.val.programmaticStreamSerializationAllowed = 1;
    gcfg.attrs = &gattr;
    gcfg.numAttrs = g.pdl;
    const cudaError_t e = cudaLaunchKernelEx(&gcfg, bgmv_group_expand_kernel, gp);
    note_launch();
    return e;
}

}  // namespace

cudaError_t launch_bgmv_grouped_shrink(const bf16_t* x, int ld_x, int h_in, const ProjSet& ps, const int32_t* perm,
                                       const int32_t* gstarts, const int32_t* gslot, int n_groups, int n_pos,
                                       int max_group_len, int n_rows, int n_slots, unsigned flags, bf16_t* vh,
                                       bf16_t* vl, int32_t* status, cudaStream_t stream)
{
    if (n_pos <= 0 || n_groups <= 0) return cudaSuccess;
    if (!vh || !vl || ps.r_slot > 64 || ps.r_slot % 8 != 0) return cudaErrorInvalidValue;
    GroupedPlan g{};
    const cudaError_t e = grouped_plan(ps, n_groups, n_pos, max_group_len, flags, g);
    if (e != cudaSuccess) return e;
    return grouped_shrink(g, x, ld_x, h_in, ps, perm, gstarts, gslot, n_groups, n_pos, n_rows, n_slots, flags, vh,
                          vl, nullptr, 0, status, stream);
}

cudaError_t launch_bgmv_grouped(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                                const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                                int n_pos, int max_group_len, int n_rows, int n_slots, unsigned flags,
                                bf16_t* vh, bf16_t* vl, int32_t* status, cudaStream_t stream)
{
    if (n_pos <= 0 || n_groups <= 0) return cudaSuccess;
    if (!vh || !vl || ps.r_slot > 64 || ps.r_slot % 8 != 0) return cudaErrorInvalidValue;
    GroupedPlan g{};
    cudaError_t e = grouped_plan(ps, n_groups, n_pos, max_group_len, flags, g);
    if (e != cudaSuccess) return e;
    e = grouped_shrink(g, x, ld_x, h_in, ps, perm, gstarts, gslot, n_groups, n_pos, n_rows, n_slots, flags, vh, vl,
                       nullptr, 0, status, stream);
    if (e != cudaSuccess) return e;
    return grouped_expand(g, y, ld_y, ps, perm, gstarts, gslot, n_groups, n_pos, n_rows, n_slots, vh, vl, nullptr, 0,
                          status, stream);
}

cudaError_t launch_group_shrink_f32(float* v, int ld_v, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                                    const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                                    int n_pos, int max_group_len, int n_rows, int n_slots, int32_t* status,
                                    cudaStream_t stream)
{
    if (n_pos <= 0 || n_groups <= 0) return cudaSuccess;
    if (!v || ps.r_slot > 64 || ps.r_slot % 8 != 0) return cudaErrorInvalidValue;
    GroupedPlan g{};
    const cudaError_t e = grouped_plan(ps, n_groups, n_pos, max_group_len, 0u, g);
    if (e != cudaSuccess) return e;
    return grouped_shrink(g, x, ld_x, h_in, ps, perm, gstarts, gslot, n_groups, n_pos, n_rows, n_slots, 0u, nullptr,
                          nullptr, v, ld_v, status, stream);
}

// The ids form launches n_slots * ceil(n_rows / 16) units, most of them
// empty when the rows spread over the slots; past this many per call the
// per-row kernels serve instead.
constexpr long long kIdsMaxUnits = 1 << 16;

bool bgmv_ids_supported(int r_slot, int n_rows, int n_slots)
{
    const long long units = static_cast<long long>(n_slots) * ((n_rows + kRB - 1) / kRB);
    return r_slot <= 64 && r_slot % 8 == 0 && n_rows > 0 && units <= kIdsMaxUnits;
}

cudaError_t launch_bgmv_ids_shrink_f32(float* v, int ld_v, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                                       const int32_t* ids, int n_rows, int n_slots, int32_t* status,
                                       cudaStream_t stream)
{
    if (n_rows <= 0) return cudaSuccess;
    if (!v || !bgmv_ids_supported(ps.n_proj * ps.r_slot, n_rows, n_slots)) return cudaErrorInvalidValue;
    GroupedPlan g{};
    const cudaError_t e = grouped_plan_ids(ps, ids, n_rows, n_slots, g);
    if (e != cudaSuccess) return e;
    return grouped_shrink(g, x, ld_x, h_in, ps, nullptr, nullptr, nullptr, 0, n_rows, n_rows, n_slots, 0u, nullptr,
                          nullptr, v, ld_v, status, stream);
}

cudaError_t launch_bgmv_ids_expand_f32(bf16_t* y, int ld_y, const float* v, int ld_v, const ProjSet& ps,
                                       const int32_t* ids, int n_rows, int n_slots, int32_t* status,
                                       cudaStream_t stream)
{
    if (n_rows <= 0) return cudaSuccess;
    if (!v || !bgmv_ids_supported(ps.r_slot, n_rows, n_slots)) return cudaErrorInvalidValue;
    GroupedPlan g{};
    const cudaError_t e = grouped_plan_ids(ps, ids, n_rows, n_slots, g);
    if (e != cudaSuccess) return e;
    return grouped_expand(g, y, ld_y, ps, nullptr, nullptr, nullptr, 0, n_rows, n_rows, n_slots, nullptr, nullptr,
                          v, ld_v, status, stream);
}

cudaError_t launch_group_expand_f32(bf16_t* y, int ld_y, const float* v, int ld_v, const ProjSet& ps,
                                    const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                                    int n_pos, int max_group_len, int n_rows, int n_slots, int32_t* status,
                                    cudaStream_t stream)
{
    if (n_pos <= 0 || n_groups <= 0) return cudaSuccess;
    if (!v || ps.r_slot > 64 || ps.r_slot % 8 != 0) return cudaErrorInvalidValue;
    GroupedPlan g{};
    const cudaError_t e = grouped_plan(ps, n_groups, n_pos, max_group_len, 0u, g);
    if (e != cudaSuccess) return e;
    return grouped_expand(g, y, ld_y, ps, perm, gstarts, gslot, n_groups, n_pos, n_rows, n_slots, nullptr, nullptr,
                          v, ld_v, status, stream);
}

}  // namespace lora
