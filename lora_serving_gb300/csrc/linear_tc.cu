// linear_tc.cu -- the LoRA linear layer: the base projection of the whole
// batch with every row's adapter delta added to the same fp32 accumulator,
// rounded to bf16 once.
//
// Multi-LoRA serving note, "direct answer": the base product W x runs once
// for the whole batch and each row adds its own adapter's B(A x).  TGI
// multi-LoRA page, "implementation": the LoRA linear layer adds the adapter
// output to the base layer's output.  Here, for projection p of a group
// whose base weights are stacked row-wise in W (rows [off_p, off_p + w_p)
// are projection p's output columns):
//   y[t][off_p + c] = bf16_rne( sum_k x[t][k] W[off_p + c][k]
//                               + sum_j B'_{p,id_t}[c][j] v_{p,t}[j] )
// with v = A x from the shrink kernels, stored as bf16 planes v_hi + v_lo.
//
// Persistent tcgen05 GEMM, one CTA per SM, tiles of 256 rows x 256 output
// columns of one projection, visited in groups of kGroupM row tiles so that
// the x and W tiles in flight at once fit in L2.  A tile is two 128-row
// halves, each an M = 128 MMA into its own 256 columns of tensor memory,
// sharing every W box: 64 KB of operands per 1024 MMA cycles.  Per tile
// the K loop is ceil(h_in / 64) base steps (a 256-row x box and a W box)
// followed by ceil(r_slot / 64) LoRA steps (the half's v_hi and v_lo boxes
// and a box of B') per adapter of each half, into the half's accumulator:
// the delta is a K extension of the GEMM.  A half whose rows all carry one
// adapter (the common case inside a prefill segment) takes one extension;
// a half with up to four adapters (a segment boundary, base rows) takes one
// per adapter, the v rows of the other rows zeroed in shared memory by a
// mask warp first; with more adapters than that (decode rows) the epilogue
// adds each row's delta on the CUDA cores from the planes and B' before
// rounding.  The LoRA boxes of a tile are prefetched into L2 when the
// tile starts.
//   warp 0: TMA producer   warp 1: MMA issuer   warps 2..17: epilogue
//   warp 18: masks v in the LoRA steps of halves that mix adapters
// The accumulator fills all 512 tensor-memory columns, so a tile's MMAs
// start once the epilogue has read the previous tile out (a few percent of
// a tile's K loop).  Every wait is bounded (0.2 s); a timeout sets
// LORA_DEV_TIMEOUT and the CTA winds down, freeing its tensor memory.
//
// Batches of at most 128 rows with few column tiles split K instead: a
// cluster of up to 8 CTAs per tile (the largest size whose clusters are all
// resident at once), each streaming a slice of K (rank 0 also the LoRA
// steps); the fp32 partials meet in distributed shared memory and each CTA
// sums, adds per-row deltas, rounds and stores its share of the tile's
// columns.  Such a batch loads only its own rows of x.

#include <algorithm>

#include "launch.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace lora {

namespace {

using namespace tc;

constexpr int kLH = 128;                      // rows per MMA (one tensor-memory lane each)
constexpr int kLM = 2 * kLH;                  // rows per tile
constexpr int kLN = 256;                      // output columns per tile
constexpr int kLK = 64;                       // K elements per step (one 128-byte swizzled row)
constexpr int kLStages = 3;
constexpr int kABytes = kLM * 128;            // x box (256 rows); a v box uses the first half
constexpr int kBBytes = kLN * 128;            // W or B' box
constexpr int kHalfBytes = kLH * 128;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kLEpiWarps = 16;                // 4 per tensor-memory lane quarter, 64 columns each
constexpr int kLMaskWarp = 2 + kLEpiWarps;    // zeroes v rows of other adapters in masked LoRA steps
constexpr int kLThreads = 32 * (3 + kLEpiWarps);
constexpr int kGroupM = 16;                   // row tiles per raster group
constexpr int kPartPitch = kLN + 4;           // fp32 pitch of the split-K partial sums (conflict-free float4 rows)
constexpr int kMaxSplit = 8;                  // split-K cluster size, at most (portable)
constexpr int kSplitCacheTiles = 160;         // tile counts whose split-K choice is remembered

struct LinearParams {
    int n_proj, r_slot, r_pad64, n_slots, n_rows;
    int out_off[LORA_MAX_PROJ];
    int width[LORA_MAX_PROJ];
    int ntiles[LORA_MAX_PROJ];   // 256-column tiles per projection
    const bf16_t* B[LORA_MAX_PROJ];
    int n_tm, n_tn, n_tiles, n_kb, kbs;
    int cs;                      // split-K cluster size (1: persistent tiles)
    unsigned* tickets;           // persistent tiles in the dynamic order: the call's tile counter (zeroed
                                 // by the shrink before this kernel), or null for tiles c, c + G, ...
    int x_box_bytes;             // bytes of one x box (fewer rows when the batch is one short tile)
    const int32_t* ids;
    const bf16_t* vh;
    const bf16_t* vl;
    int ld_p;
    bf16_t* y;
    int ld_y;
    int32_t* status;
};

struct LTile {
    int m, p, col0, ncols;
};

// Tile t: groups of kGroupM row tiles, row tile fastest inside a group.
__device__ __forceinline__ LTile tile_of(const LinearParams& P, int t)
{
    const int per_group = kGroupM * P.n_tn;
    const int g = t / per_group, rem = t - g * per_group;
    const int m0 = g * kGroupM, gm = min(kGroupM, P.n_tm - m0);
    LTile T;
    T.m = m0 + rem % gm;
    int nt = rem / gm, p = 0;
    while (p < P.n_proj - 1 && nt >= P.ntiles[p]) {
        nt -= P.ntiles[p];
        ++p;
    }
    T.p = p;
    T.col0 = nt * kLN;
    T.ncols = min(kLN, P.width[p] - T.col0);
    return T;
}

constexpr int kMaxSlotsHalf = 4;   // adapters per half taken on the tensor cores

// How the delta of one 128-row half is formed.
enum HalfKind { kNone = 0, kUniform = 1, kMasked = 2, kRows = 3 };

// Plans half h of row tile m (whole warp; every warp that asks gets the
// same answer).  Each lane holds the ids of rows lane, lane+32, lane+64,
// lane+96 of the half (-1 past the last row).  The half's distinct valid
// adapters, in order of first claim, go to sl[]:
//   kNone     no row has an adapter;
//   kUniform  every row has the same adapter: one K extension;
//   kMasked   up to kMaxSlotsHalf adapters (a segment boundary, base rows):
//             one K extension per adapter, with the v rows of the other
//             rows zeroed in shared memory before the MMA;
//   kRows     more adapters than that (decode rows): the epilogue adds
//             each row's delta on the CUDA cores.
// Ids outside [-1, n_slots) take no delta (the epilogue flags them).
__device__ __forceinline__ int plan_half(const LinearParams& P, int m, int h, int* sl, int& nsl, int* myid)
{
    const int lane = threadIdx.x & 31;
    const int row0 = m * kLM + h * kLH, nr = min(kLH, P.n_rows - row0);
    unsigned open = 0;   // this lane's rows with a valid adapter not yet listed
    bool all_valid = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        myid[i] = r < nr ? __ldg(P.ids + row0 + r) : -1;
        const bool v = myid[i] >= 0 && myid[i] < P.n_slots;
        if (v) open |= 1u << i;
        if (r < nr && !v) all_valid = false;
    }
    all_valid = __all_sync(0xFFFFFFFFu, all_valid);
    nsl = 0;
    for (;;) {
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, open != 0);
        if (ball == 0) break;
        if (nsl == kMaxSlotsHalf) return kRows;
        int cand = -1;
#pragma unroll
        for (int i = 3; i >= 0; --i)
            if (open & (1u << i)) cand = myid[i];
        cand = __shfl_sync(0xFFFFFFFFu, cand, __ffs(ball) - 1);
        sl[nsl++] = cand;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (myid[i] == cand) open &= ~(1u << i);
    }
    if (nsl == 0) return kNone;
    return (nsl == 1 && all_valid) ? kUniform : kMasked;
}

// A tile's K steps: the base steps, then kbs LoRA steps for each adapter
// of each half planned onto the tensor cores (half 0 first).  A LoRA step
// carries the v_hi and v_lo boxes of the half (the A region) and one box
// of B' (the B region): two MMAs per K slice on the same B'.
struct Plan {
    int kind[2];
    int nsl[2];
    int sl[2][kMaxSlotsHalf];
    int myid[2][4];
    int live[2];   // the half has rows
    int kb_lo, nb; // base K blocks [kb_lo, kb_lo + nb)
    int n_ks;
    // The tile's plan; with split K (cluster size P.cs) this CTA takes the
    // K blocks of its cluster rank, and rank 0 alone the LoRA steps.
    __device__ __forceinline__ void make(const LinearParams& P, int m, int crank)
    {
        live[0] = 1;
        live[1] = m * kLM + kLH < P.n_rows;
        int n_ext = 0;
        for (int h = 0; h < 2; ++h) {
            kind[h] = plan_half(P, m, h, sl[h], nsl[h], myid[h]);
            if ((kind[h] == kUniform || kind[h] == kMasked) && crank == 0) n_ext += nsl[h];
            else nsl[h] = 0;
        }
        kb_lo = crank * P.n_kb / P.cs;
        nb = (crank + 1) * P.n_kb / P.cs - kb_lo;
        n_ks = nb + P.kbs * n_ext;
    }
    // LoRA step l (0-based after the base steps) -> half, adapter index, K block
    __device__ __forceinline__ void lora(const LinearParams& P, int l, int& h, int& j, int& kb) const
    {
        j = l / P.kbs;
        kb = l - j * P.kbs;
        h = 0;
        if (j >= nsl[0]) {
            j -= nsl[0];
            h = 1;
        }
    }
};

// L2 prefetches of a box (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p)
{
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// acc[c] += B'_{p,slot}[col0 + c] . (v_hi + v_lo)[row] for the 32 columns
// col0 .. col0 + 31 of projection p that lie inside its width.
__device__ __forceinline__ void add_row_delta(const LinearParams& P, int p, int slot, int row, int col0, float* acc)
{
    const size_t vo = static_cast<size_t>(row) * P.ld_p + p * P.r_pad64;
    const bf16_t* Bp = P.B[p] + (static_cast<size_t>(slot) * P.width[p] + col0) * P.r_slot;
    const int nc = min(32, P.width[p] - col0);
    for (int j8 = 0; j8 < P.r_slot; j8 += 8) {
        const uint4 h = __ldg(reinterpret_cast<const uint4*>(P.vh + vo + j8));
        const uint4 l = __ldg(reinterpret_cast<const uint4*>(P.vl + vo + j8));
        float v[8];
        v[0] = bf16_lo(h.x) + bf16_lo(l.x);
        v[1] = bf16_hi(h.x) + bf16_hi(l.x);
        v[2] = bf16_lo(h.y) + bf16_lo(l.y);
        v[3] = bf16_hi(h.y) + bf16_hi(l.y);
        v[4] = bf16_lo(h.z) + bf16_lo(l.z);
        v[5] = bf16_hi(h.z) + bf16_hi(l.z);
        v[6] = bf16_lo(h.w) + bf16_lo(l.w);
        v[7] = bf16_hi(h.w) + bf16_hi(l.w);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            if (c < nc) {
                const uint4 b = __ldg(reinterpret_cast<const uint4*>(Bp + static_cast<size_t>(c) * P.r_slot + j8));
                float s = acc[c];
                s = fmaf(bf16_lo(b.x), v[0], s);
                s = fmaf(bf16_hi(b.x), v[1], s);
                s = fmaf(bf16_lo(b.y), v[2], s);
                s = fmaf(bf16_hi(b.y), v[3], s);
                s = fmaf(bf16_lo(b.z), v[4], s);
                s = fmaf(bf16_hi(b.z), v[5], s);
                s = fmaf(bf16_lo(b.w), v[6], s);
                s = fmaf(bf16_hi(b.w), v[7], s);
                acc[c] = s;
            }
        }
    }
}

// acc[c] += B'_{p,slot}[col0 + c] . (v_hi + v_lo)[row] for 8 columns col0 .. col0 + 7
// (all inside the width: widths are multiples of 8).
__device__ __forceinline__ void add_row_delta8(const LinearParams& P, int p, int slot, int row, int col0, float* acc)
{
    const size_t vo = static_cast<size_t>(row) * P.ld_p + p * P.r_pad64;
    const bf16_t* Bp = P.B[p] + (static_cast<size_t>(slot) * P.width[p] + col0) * P.r_slot;
    for (int j8 = 0; j8 < P.r_slot; j8 += 8) {
        const uint4 h = __ldg(reinterpret_cast<const uint4*>(P.vh + vo + j8));
        const uint4 l = __ldg(reinterpret_cast<const uint4*>(P.vl + vo + j8));
        const float v[8] = {bf16_lo(h.x) + bf16_lo(l.x), bf16_hi(h.x) + bf16_hi(l.x), bf16_lo(h.y) + bf16_lo(l.y),
                            bf16_hi(h.y) + bf16_hi(l.y), bf16_lo(h.z) + bf16_lo(l.z), bf16_hi(h.z) + bf16_hi(l.z),
                            bf16_lo(h.w) + bf16_lo(l.w), bf16_hi(h.w) + bf16_hi(l.w)};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(Bp + static_cast<size_t>(c) * P.r_slot + j8));
            float s = acc[c];
            s = fmaf(bf16_lo(b.x), v[0], s);
            s = fmaf(bf16_hi(b.x), v[1], s);
            s = fmaf(bf16_lo(b.y), v[2], s);
            s = fmaf(bf16_hi(b.y), v[3], s);
            s = fmaf(bf16_lo(b.z), v[4], s);
            s = fmaf(bf16_hi(b.z), v[5], s);
            s = fmaf(bf16_lo(b.w), v[6], s);
            s = fmaf(bf16_hi(b.w), v[7], s);
            acc[c] = s;
        }
    }
}

// Rounds 32 accumulator columns to bf16 and stores those inside the width.
__device__ __forceinline__ void store_row32(bf16_t* yrow, int ncols_left, const float* acc)
{
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        if (c8 * 8 < ncols_left) {
            uint4 o;
            o.x = pack_bf16x2(acc[c8 * 8 + 0], acc[c8 * 8 + 1]);
            o.y = pack_bf16x2(acc[c8 * 8 + 2], acc[c8 * 8 + 3]);
            o.z = pack_bf16x2(acc[c8 * 8 + 4], acc[c8 * 8 + 5]);
            o.w = pack_bf16x2(acc[c8 * 8 + 6], acc[c8 * 8 + 7]);
            *reinterpret_cast<uint4*>(yrow + c8 * 8) = o;
        }
    }
}

// Split K, after the cluster barrier: the 8-column groups of this CTA's
// share of the tile summed over the cluster's partials (rank order), the
// per-row deltas of a half that mixes many adapters added, rounded, stored.
// Whole CTA (the plan's warp votes).
__device__ __noinline__ void splitk_reduce(const LinearParams& P, int t, int crank, float* part)
{
    const int tid = threadIdx.x;
    const LTile T = tile_of(P, t);
    Plan pl;
    pl.make(P, T.m, 0);
    const int n_g = (T.ncols + 7) / 8;   // 8-column groups of the tile
    const int g_lo = crank * n_g / P.cs, g_hi = (crank + 1) * n_g / P.cs;
    const int per_row = g_hi - g_lo;
    const uint32_t part_s = smem_u32(part);
    for (int it = tid; it < P.n_rows * per_row; it += kLThreads) {
        const int row = it / per_row, c0 = (g_lo + it - row * per_row) * 8;
        float acc[8] = {};
        for (int peer = 0; peer < P.cs; ++peer) {
            const uint32_t src = map_rank(part_s + 4u * static_cast<uint32_t>(row * kPartPitch + c0), peer);
            const float4 a = ld_dsmem_f4(src), b = ld_dsmem_f4(src + 16u);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        const int id = __ldg(P.ids + row);
        if (id >= 0 && id < P.n_slots) {
            if (pl.kind[0] == kRows) add_row_delta8(P, T.p, id, row, T.col0 + c0, acc);
        } else if (id != -1 && c0 == 0) {
            flag(P.status, LORA_DEV_SLOT_OUT_OF_RANGE);   // the row keeps its base value
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(P.y + static_cast<size_t>(row) * P.ld_y + P.out_off[T.p] + T.col0 + c0) = o;
    }
}

// The tiles a CTA takes: tiles c, c + G, ... (static order), or in the
// dynamic order the tiles numbered by the call's counter, so that CTAs that
// start late or run slow take fewer.  In the dynamic order the producer
// warp's lane 0 takes each tile's ticket one tile early and hands the tile
// numbers to the MMA, mask and epilogue warps through a queue of kLQD slots.
constexpr int kLQD = 8;
constexpr int kLTileReaders = 2 + kLEpiWarps;   // MMA warp, mask warp, epilogue warps
template <bool kDyn>
struct LTileSeq {
    int t_first, t_step, n_tiles;
    const LinearParams& P;
    long long* q_item;
    uint64_t* q_full;
    uint64_t* q_empty;
    volatile int* fail;
    unsigned ahead;   // producer lane 0: the next tile's ticket
    __device__ __forceinline__ LTileSeq(int tf, int ts, const LinearParams& pp, long long* qi, uint64_t* qf, uint64_t* qe,
                                        volatile int* f)
        : t_first(tf), t_step(ts), n_tiles(pp.n_tiles), P(pp), q_item(qi), q_full(qf), q_empty(qe), fail(f), ahead(0)
    {
    }
    // The warp's k-th tile, or -1 past the last (or on a timeout, with *fail
    // set).  Every lane of the warp calls it.
    __device__ __forceinline__ int get(int k, bool producer)
    {
        if constexpr (!kDyn) {
            const long long t = t_first + static_cast<long long>(k) * t_step;
            return t < n_tiles ? static_cast<int>(t) : -1;
        } else {
            const int lane = threadIdx.x & 31, slot = k % kLQD;
            int t = -1;
            if (producer) {
                if (lane == 0) {
                    if (k >= kLQD && !mbar_wait_spin(&q_empty[slot], ((k / kLQD) - 1) & 1)) {
                        *fail = 1;   // the tile numbers stop here: every reader's wait runs out
                    } else {
                        const unsigned tk = *fail ? 0xFFFFFFFFu : (k == 0 ? atomicAdd(P.tickets, 1u) : ahead);
                        t = static_cast<long long>(tk) < n_tiles ? static_cast<int>(tk) : -1;
                        if (t >= 0) ahead = atomicAdd(P.tickets, 1u);
                        q_item[slot] = t;
                        mbar_arrive(&q_full[slot]);
                    }
                }
                return __shfl_sync(0xFFFFFFFFu, t, 0);
            }
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&q_full[slot], (k / kLQD) & 1));
            if (!ok) {
                *fail = 1;
                return -1;
            }
            t = static_cast<int>(q_item[slot]);
            __syncwarp();   // every lane has read the slot before it is freed
            if (lane == 0) mbar_arrive(&q_empty[slot]);
            return t;
        }
    }
};

template <bool kDyn>
__global__ void __launch_bounds__(kLThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                 const __grid_constant__ CUtensorMap mvh, const __grid_constant__ CUtensorMap mvl,
                 const __grid_constant__ CUtensorMap mb0, const __grid_constant__ CUtensorMap mb1,
                 const __grid_constant__ CUtensorMap mb2, const __grid_constant__ CUtensorMap mb3, LinearParams P)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kLStages], empty[kLStages], mask_req[kLStages], masked[kLStages];
    __shared__ __align__(8) uint64_t acc_full, acc_empty;
    __shared__ __align__(8) uint64_t q_full[kLQD], q_empty[kLQD];
    __shared__ long long q_item[kLQD];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t* ring = align1024(smem_raw);
    const CUtensorMap* bmap[4] = {&mb0, &mb1, &mb2, &mb3};

    if (warp == 0) tmem_alloc(&s_tmem, 2 * kLN);
    if (tid == 0) {
        for (int s = 0; s < kLStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);   // released by the MMA commit of the stage's last read
            mbar_init(&mask_req[s], 1);  // the MMA asks for a masked LoRA step's v rows to be zeroed
            mbar_init(&masked[s], 1);    // ... and they are
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, kLEpiWarps);
        for (int j = 0; j < kLQD; ++j) {
            mbar_init(&q_full[j], 1);
            mbar_init(&q_empty[j], kLTileReaders);
        }
        mbar_init_fence();
        s_fail = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // persistent: tiles blockIdx.x, + gridDim.x, ...; split K: the cluster's one tile
    const int crank = P.cs > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int t_first = P.cs > 1 ? static_cast<int>(blockIdx.x) / P.cs : static_cast<int>(blockIdx.x);
    const int t_step = P.cs > 1 ? P.n_tiles : static_cast<int>(gridDim.x);
    LTileSeq<kDyn> seq(t_first, t_step, P, q_item, q_full, q_empty, &s_fail);
    float* part = reinterpret_cast<float*>(ring);   // split K: this CTA's partial sums, after its K loop

    if (warp == 0) {   // ---- producer (lane 0 issues; the warp plans each tile) ----
        int it = 0;
        for (int kk = 0; !s_fail; ++kk) {
            const int t = seq.get(kk, true);
            if (t < 0) break;
            const LTile T = tile_of(P, t);
            Plan pl;
            pl.make(P, T.m, crank);
            if (lane == 0) {
                // the LoRA boxes come after the whole base K loop: start them
                // towards L2 now so that those steps do not wait on DRAM
                for (int l = 0; l < pl.n_ks - pl.nb; ++l) {
                    int h, j, kb;
                    pl.lora(P, l, h, j, kb);
                    tma_prefetch_3d(&mvh, kb * kLK, T.p, T.m * kLM + h * kLH);
                    tma_prefetch_3d(&mvl, kb * kLK, T.p, T.m * kLM + h * kLH);
                    tma_prefetch_2d(bmap[T.p], kb * kLK, pl.sl[h][j] * P.width[T.p] + T.col0);
                }
                for (int k = 0; k < pl.n_ks; ++k, ++it) {
                    const int s = it % kLStages;
                    if (it >= kLStages && !mbar_wait_spin(&empty[s], ((it / kLStages) - 1) & 1)) {
                        s_fail = 1;
                        break;
                    }
                    uint8_t* a = ring + s * kStageBytes;
                    uint8_t* b = a + kABytes;
                    if (k < pl.nb) {
                        const int kc = (pl.kb_lo + k) * kLK;
                        mbar_expect_tx(&full[s], P.x_box_bytes + kBBytes);
                        tma_load_2d(a, &mx, kc, T.m * kLM, &full[s]);
                        tma_load_2d(b, &mw, kc, P.out_off[T.p] + T.col0, &full[s]);
                    } else {
                        int h, j, kb;
                        pl.lora(P, k - pl.nb, h, j, kb);
                        mbar_expect_tx(&full[s], kStageBytes);
                        tma_load_3d(a, &mvh, kb * kLK, T.p, T.m * kLM + h * kLH, &full[s]);
                        tma_load_3d(a + kHalfBytes, &mvl, kb * kLK, T.p, T.m * kLM + h * kLH, &full[s]);
                        tma_load_2d(b, bmap[T.p], kb * kLK, pl.sl[h][j] * P.width[T.p] + T.col0, &full[s]);
                    }
                }
            }
            it = __shfl_sync(0xFFFFFFFFu, it, 0);
            __syncwarp();
        }
    } else if (warp == 1) {   // ---- MMA issuer ----
        int it = 0, ti = 0, ok = 1;
        int mc[kLStages] = {};   // masked steps seen per stage (the phase of masked[s])
        for (int kk = 0; ok && !s_fail; ++kk, ++ti) {
            const int t = seq.get(kk, false);
            if (t < 0) break;
            const LTile T = tile_of(P, t);
            Plan pl;
            pl.make(P, T.m, crank);
            if (lane == 0) {
                const uint32_t idesc = idesc_bf16_f32(kLH, (T.ncols + 15) / 16 * 16);
                const bool live1 = pl.live[1];
                if (ti >= 1 && !mbar_wait_spin(&acc_empty, (ti - 1) & 1)) ok = 0;
                tc_fence_after();
                for (int k = 0; ok && k < pl.n_ks; ++k, ++it) {
                    const int s = it % kLStages;
                    if (!mbar_wait_spin(&full[s], (it / kLStages) & 1)) {
                        ok = 0;
                        break;
                    }
                    const uint32_t as = smem_u32(ring + s * kStageBytes), bs = as + kABytes;
                    if (k < pl.nb) {
                        tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < kLK / 16; ++ks)
                            mma_bf16(tmem, sdesc_sw128(as + ks * 32), sdesc_sw128(bs + ks * 32), idesc, k > 0 || ks > 0);
                        if (live1) {
#pragma unroll
                            for (int ks = 0; ks < kLK / 16; ++ks)
                                mma_bf16(tmem + kLN, sdesc_sw128(as + kHalfBytes + ks * 32), sdesc_sw128(bs + ks * 32),
                                         idesc, k > 0 || ks > 0);
                        }
                    } else {
                        int h, j, kb;
                        pl.lora(P, k - pl.nb, h, j, kb);
                        if (pl.kind[h] == kMasked) {
                            // the mask warp zeroes the other adapters' rows of this v box first;
                            // requests and replies alternate, so each stage's phases pair up
                            mbar_arrive(&mask_req[s]);
                            if (!mbar_wait_spin(&masked[s], (mc[s]++) & 1)) {
                                ok = 0;
                                break;
                            }
                        }
                        tc_fence_after();
                        for (int plane = 0; plane < 2; ++plane) {   // v_hi, then v_lo, on the same B'
#pragma unroll
                            for (int ks = 0; ks < kLK / 16; ++ks)
                                mma_bf16(tmem + h * kLN, sdesc_sw128(as + plane * kHalfBytes + ks * 32),
                                         sdesc_sw128(bs + ks * 32), idesc, true);
                        }
                    }
                    mma_commit(&empty[s]);   // the stage is free once these MMAs have read it
                }
                if (ok) mma_commit(&acc_full);
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            it = __shfl_sync(0xFFFFFFFFu, it, 0);
        }
        if (!ok) s_fail = 1;
    } else if (warp == kLMaskWarp) {   // ---- v masking for halves that mix adapters ----
        int it = 0, ok = 1;
        int mr[kLStages] = {};   // requests served per stage (the phase of mask_req[s])
        for (int kk = 0; ok && !s_fail; ++kk) {
            const int t = seq.get(kk, false);
            if (t < 0) break;
            const LTile T = tile_of(P, t);
            Plan pl;
            pl.make(P, T.m, crank);
            for (int k = pl.nb; ok && k < pl.n_ks; ++k) {
                const int step = it + k, s = step % kLStages;
                int h, j, kb;
                pl.lora(P, k - pl.nb, h, j, kb);
                if (pl.kind[h] != kMasked) continue;
                // the request comes after the stage has landed and before it can be
                // refilled, so the stage's fill phase is exactly this step's
                if (lane == 0 && (!mbar_wait_spin(&mask_req[s], (mr[s]++) & 1) ||
                                  !mbar_wait_spin(&full[s], (step / kLStages) & 1)))
                    ok = 0;
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok) break;
                uint8_t* vbox = ring + s * kStageBytes;   // v_hi box, then the v_lo box
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (pl.myid[h][i] != pl.sl[h][j]) {
#pragma unroll
                        for (int plane = 0; plane < 2; ++plane) {
                            uint4* row = reinterpret_cast<uint4*>(vbox + plane * kHalfBytes + (lane + 32 * i) * 128);
#pragma unroll
                            for (int c = 0; c < 8; ++c) row[c] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_async_smem();   // the tensor cores read what these generic stores wrote
                __syncwarp();
                if (lane == 0) mbar_arrive(&masked[s]);
            }
            it += pl.n_ks;
        }
        if (!ok) s_fail = 1;
    } else {   // ---- epilogue ----
        const int e = warp - 2;
        const int quarter = warp & 3;        // tensor-memory lanes this warp may read
        const int cs = (e >> 2) * 64;        // its 64 columns of the tile
        int ti = 0;
        for (int kk = 0;; ++kk, ++ti) {
            const int t = seq.get(kk, false);
            if (t < 0) break;
            const LTile T = tile_of(P, t);
            Plan pl;
            pl.make(P, T.m, crank);
            if (s_fail || !mbar_wait(&acc_full, ti & 1)) {
                s_fail = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + cs;
            if (P.cs > 1) {
                // split K (at most 128 rows: half 0): the partial sums go to
                // shared memory, where the cluster adds them up below
                float* prow = part + (quarter * 32 + lane) * kPartPitch + cs;
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    float d[32];
                    tmem_ld32(tbase + q * 32, d);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(prow + q * 32 + 4 * i) =
                            make_float4(d[4 * i], d[4 * i + 1], d[4 * i + 2], d[4 * i + 3]);
                }
                continue;
            }
            if (pl.kind[0] != kRows && pl.kind[1] != kRows) {
                // no per-row delta: read the warp's four 32-column pieces,
                // round them into registers, hand the accumulator back to the
                // MMA at once, then store
                uint32_t pk[4][16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int g = 0; g < 2; ++g) {   // 16 columns per read keeps the registers in bounds
                        float d[16];
                        tmem_ld16(tbase + (q >> 1) * kLN + (q & 1) * 32 + g * 16, d);
#pragma unroll
                        for (int i = 0; i < 8; ++i) pk[q][8 * g + i] = pack_bf16x2(d[2 * i], d[2 * i + 1]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int h = q >> 1, c0 = cs + (q & 1) * 32;
                    const int row = T.m * kLM + h * kLH + quarter * 32 + lane;
                    if (row < P.n_rows && c0 < T.ncols) {
                        const int id = quarter == 0 ? pl.myid[h][0] : quarter == 1 ? pl.myid[h][1]
                                     : quarter == 2 ? pl.myid[h][2] : pl.myid[h][3];
                        if ((id < -1 || id >= P.n_slots) && (q & 1) == 0 && c0 == 0)
                            flag(P.status, LORA_DEV_SLOT_OUT_OF_RANGE);   // the row keeps its base value
                        uint4* yp = reinterpret_cast<uint4*>(P.y + static_cast<size_t>(row) * P.ld_y + P.out_off[T.p] +
                                                             T.col0 + c0);
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8)
                            if (c8 * 8 < T.ncols - c0)
                                yp[c8] = make_uint4(pk[q][4 * c8], pk[q][4 * c8 + 1], pk[q][4 * c8 + 2], pk[q][4 * c8 + 3]);
                    }
                }
                continue;
            }
            // a half adds per-row deltas on the CUDA cores: 32 accumulator
            // columns at a time (half h, piece c): read, add the row's delta,
            // round and store; the accumulator goes back after the last read
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                const int h = q >> 1, c0 = cs + (q & 1) * 32;
                float d[32];
                tmem_ld32(tbase + h * kLN + (q & 1) * 32, d);
                if (q == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty);
                }
                const int row = T.m * kLM + h * kLH + quarter * 32 + lane;
                if (row < P.n_rows && c0 < T.ncols) {
                    const int id = pl.myid[h][quarter];   // the id of this lane's row (row = quarter * 32 + lane)
                    if (id >= 0 && id < P.n_slots) {
                        if (pl.kind[h] == kRows) add_row_delta(P, T.p, id, row, T.col0 + c0, d);
                    } else if (id != -1 && (q & 1) == 0 && c0 == 0) {
                        flag(P.status, LORA_DEV_SLOT_OUT_OF_RANGE);   // the row keeps its base value
                    }
                    store_row32(P.y + static_cast<size_t>(row) * P.ld_y + P.out_off[T.p] + T.col0 + c0,
                                T.ncols - c0, d);
                }
            }
        }
    }
    __syncthreads();
    if (P.cs > 1) {
        // ---- split K: sum the cluster's partials, add per-row deltas, round, store ----
        // Every thread of every CTA of the cluster meets both barriers (a CTA
        // that timed out still takes part; its status flag tells the caller).
        cluster_arrive();
        cluster_wait();
        splitk_reduce(P, t_first, crank, part);
        cluster_arrive();   // the peers have read this CTA's partials
        cluster_wait();
    }
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 2 * kLN);
    if (tid == 0 && s_fail) flag(P.status, LORA_DEV_TIMEOUT);
}

}  // namespace

size_t linear_tc_smem() { return static_cast<size_t>(kLStages) * kStageBytes + 1024; }

cudaError_t launch_linear_tc(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const bf16_t* W, int ld_w,
                             int n_out, const ProjSet& ps, const bf16_t* vh, const bf16_t* vl,
                             const int32_t* ids, int n_rows, int n_slots, int32_t* status, cudaStream_t stream,
                             unsigned* tickets)
{
    if (n_rows <= 0) return cudaSuccess;
    LinearParams P{};
    P.n_proj = ps.n_proj;
    P.r_slot = ps.r_slot;
    P.r_pad64 = (ps.r_slot + kLK - 1) / kLK * kLK;
    P.kbs = P.r_pad64 / kLK;
    P.ld_p = ps.n_proj * P.r_pad64;
    P.n_slots = n_slots;
    P.n_rows = n_rows;
    P.ids = ids;
    P.vh = vh;
    P.vl = vl;
    P.y = y;
    P.ld_y = ld_y;
    P.status = status;
    P.n_kb = (h_in + kLK - 1) / kLK;
    P.n_tm = (n_rows + kLM - 1) / kLM;
    // A batch of one row tile loads only its rows of x (rounded up to 8):
    // the other rows of the A operand are left over from earlier steps and
    // only feed accumulator rows that are never stored.
    const int x_rows = P.n_tm == 1 ? std::min(kLM, (n_rows + 7) / 8 * 8) : kLM;
    P.x_box_bytes = x_rows * 128;
    CUtensorMap mx, mw, mvh, mvl, mb[4];
    if (!encode_tmap_bf16(&mx, x, n_rows, h_in, ld_x, x_rows, kLK, true) ||
        !encode_tmap_bf16(&mw, W, n_out, h_in, ld_w, kLN, kLK, true) ||
        !encode_tmap_bf16_3d(&mvh, vh, ps.r_slot, ps.n_proj, n_rows, P.r_pad64, P.ld_p, kLK, kLH) ||
        !encode_tmap_bf16_3d(&mvl, vl, ps.r_slot, ps.n_proj, n_rows, P.r_pad64, P.ld_p, kLK, kLH))
        return cudaErrorInvalidValue;
    for (int q = 0; q < 4; ++q) {
        const int src = q < ps.n_proj ? q : 0;
        if (!encode_tmap_bf16(&mb[q], ps.B[src], static_cast<uint64_t>(n_slots) * ps.width[src], ps.r_slot,
                              ps.r_slot, kLN, kLK, true))
            return cudaErrorInvalidValue;
        if (q < ps.n_proj) {
            P.out_off[q] = ps.out_off[q];
            P.width[q] = ps.width[q];
            P.B[q] = ps.B[q];
            P.ntiles[q] = (ps.width[q] + kLN - 1) / kLN;
            P.n_tn += P.ntiles[q];
        }
    }
    const long long n_tiles = static_cast<long long>(P.n_tm) * P.n_tn;
    if (n_tiles > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    P.n_tiles = static_cast<int>(n_tiles);

    static int configured_device = -1, n_sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        for (const void* fn : {reinterpret_cast<const void*>(linear_tc_kernel<false>),
                               reinterpret_cast<const void*>(linear_tc_kernel<true>)}) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(linear_tc_smem()));
            if (e != cudaSuccess) return e;
            e = prefer_max_shared(fn);
            if (e != cudaSuccess) return e;
        }
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    // Few rows (one half of one row tile) and few column tiles: split K over
    // a cluster per tile so that the weight streams through most SMs.
    // The largest cluster for which every tile's cluster is resident at once
    // (clusters must fit inside a GPC, so fewer than n_sms / cs may be).
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kLThreads);
    cfg.dynamicSmemBytes = linear_tc_smem();
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    // (the answer depends only on the tile count and the K blocks: kept per
    // device in a small table, so repeated calls skip the occupancy queries)
    static int split_dev = -1;
    static signed char split_cache[kSplitCacheTiles][kMaxSplit + 1];
    if (split_dev != dev) {
        for (auto& row : split_cache)
            for (auto& c : row) c = -1;
        split_dev = dev;
    }
    int cs = 1;
    if (P.n_tm == 1 && n_rows <= kLH && 2 * P.n_tiles <= n_sms) {
        const int c_max = std::min(kMaxSplit, P.n_kb);
        signed char* cached = P.n_tiles < kSplitCacheTiles ? &split_cache[P.n_tiles][c_max] : nullptr;
        if (cached && *cached >= 0) {
            cs = *cached;
        } else {
            for (int c = c_max; c >= 2 && cs == 1; --c) {
                attr.val.clusterDim.x = c;
                cfg.gridDim = dim3(static_cast<unsigned>(P.n_tiles * c));
                cfg.attrs = &attr;
                cfg.numAttrs = 1;
                int active = 0;
                if (cudaOccupancyMaxActiveClusters(&active, linear_tc_kernel<false>, &cfg) == cudaSuccess &&
                    active >= P.n_tiles)
                    cs = c;
            }
            (void)cudaGetLastError();
            if (cached) *cached = static_cast<signed char>(cs);
        }
    }
    cs = std::max(1, std::min({env_int("LORA_LINEAR_SPLIT", cs), kMaxSplit, P.n_kb}));
    if (n_rows > kLH || P.n_tm != 1) cs = 1;
    P.cs = cs;
    // persistent tiles in the dynamic order when the call's counter is given
    // (its shrink zeroes it); split K keeps one tile per cluster
    P.tickets = cs == 1 && env_int("LORA_LINEAR_DYNAMIC", 1) != 0 ? tickets : nullptr;
    cfg.gridDim = dim3(static_cast<unsigned>(cs > 1 ? P.n_tiles * cs
                                                    : std::min<long long>(env_int("LORA_LINEAR_GRID", n_sms), n_tiles)));
    attr.val.clusterDim.x = cs;
    cfg.attrs = &attr;
    cfg.numAttrs = cs > 1 ? 1 : 0;
    e = P.tickets != nullptr
            ? cudaLaunchKernelEx(&cfg, linear_tc_kernel<true>, mx, mw, mvh, mvl, mb[0], mb[1], mb[2], mb[3], P)
            : cudaLaunchKernelEx(&cfg, linear_tc_kernel<false>, mx, mw, mvh, mvl, mb[0], mb[1], mb[2], mb[3], P);
    note_launch();
    return e;
}

}  // namespace lora
