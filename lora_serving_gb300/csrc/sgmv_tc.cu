// sgmv_tc.cu -- SGMV on the 5th-generation tensor cores (tcgen05) for long
// prefill segments.
//
// TGI multi-LoRA page, "4. SGMV and BGMV at inference": prefill rows come in
// variable-length segments that share one adapter, so each segment's shrink
// and expand are dense contractions:
//   shrink  V[rows, 0:R]      = X[rows, :] . A_slot^T          (R = n_proj * r_slot)
//   expand  Y[rows, off + c] += V[rows, p-slice] . B'_slot,p^T
// Both run as 128-row tiles of one segment: TMA brings 128-byte-swizzled
// bf16 tiles into shared memory, one thread issues tcgen05.mma with the fp32
// accumulator in tensor memory, and the epilogue reads it back with
// tcgen05.ld.  Rows of a tile past the segment's end are computed but never
// written (they belong to the next segment or to no one).
//
// The intermediate never becomes a single bf16: the shrink writes it either
// as fp32 (the lora_sgmv_shrink entry point) or as two bf16 planes
// hi = bf16(v), lo = bf16(v - hi) (inside lora_apply), and the expand
// multiplies both planes by B', carrying v to ~2^-17 relative.
//
// Every mbarrier wait is bounded (0.2 s); a timeout sets LORA_DEV_TIMEOUT,
// skips the rest of the tile and still frees the tensor memory.  The shrink
// then stores a zero intermediate for the tile's rows (so the expand adds
// nothing to them) and the expand writes nothing; before a CTA leaves, its
// producer waits (bounded) for every copy it issued, so no copy into the
// CTA's shared memory is still in flight when the CTA's resources go back.

#include <algorithm>
#include <cstdlib>

#include "launch.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace lora {

namespace {

using namespace tc;

constexpr int kTileM = 128;
constexpr int kKB = 64;                 // K elements per 128-byte swizzled row
constexpr int kBoxBytes = kTileM * 128; // one 128-row x 64-element box
constexpr int kShrinkThreads = 128;
constexpr int kExpandN = 128;           // output columns per expand tile

struct TileInfo {
    int found, slot, row0, nrows, bad;
};

// Tile u of the segments' 128-row tiles (segments with slot -1 have none).
// One parallel round trip over the segment table when it fits the block,
// a serial scan otherwise.  Malformed entries (bounds outside [0, n_pos))
// contribute no tiles and set bad, as does a table that does not cover
// [0, n_pos).
template <int kThreads>
__device__ TileInfo find_tile(const int32_t* seg_starts, const int32_t* seg_slot, int n_segs, int n_pos, int u)
{
    __shared__ int s_warp[kThreads / 32];
    __shared__ TileInfo s_info;
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_info.found = 0;
        // the table must cover [0, n_pos): its first entry 0, its last n_pos
        s_bad = n_segs > 0 && (__ldg(seg_starts) != 0 || __ldg(seg_starts + n_segs) != n_pos);
    }
    if (n_segs <= kThreads) {
        int s = 0, e = 0, sl = -1, n = 0;
        bool bad = false;
        if (tid < n_segs) {
            s = __ldg(seg_starts + tid);
            e = __ldg(seg_starts + tid + 1);
            sl = __ldg(seg_slot + tid);
            const bool sane = s >= 0 && e <= n_pos && s <= e;
            bad = !sane;
            n = (sane && sl >= 0) ? (e - s + kTileM - 1) / kTileM : 0;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += s_warp[w];
        incl += before;
        const int excl = incl - n;
        if (bad) atomicOr(&s_bad, 1);
        if (tid < n_segs && u >= excl && u < incl) {
            TileInfo t;
            t.found = 1;
            t.slot = sl;
            t.row0 = s + (u - excl) * kTileM;
            t.nrows = min(kTileM, e - t.row0);
            t.bad = 0;
            s_info = t;
        }
        __syncthreads();
    } else {
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            bool bad = false;
            for (int i = 0; i < n_segs; ++i) {
                const int s = __ldg(seg_starts + i), e = __ldg(seg_starts + i + 1), sl = __ldg(seg_slot + i);
                const bool sane = s >= 0 && e <= n_pos && s <= e;
                bad |= !sane;
                const int n = (sane && sl >= 0) ? (e - s + kTileM - 1) / kTileM : 0;
                if (u < acc + n) {
                    s_info.found = 1;
                    s_info.slot = sl;
                    s_info.row0 = s + (u - acc) * kTileM;
                    s_info.nrows = min(kTileM, e - s_info.row0);
                    break;
                }
                acc += n;
            }
            s_bad |= bad;
        }
        __syncthreads();
    }
    TileInfo r = s_info;
    r.bad = s_bad;
    return r;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p)
{
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// ------------------------------------------------------------- shrink ----

struct ShrinkTcParams {
    int n_proj, r_slot, R, h_in, n_slots;
    const int32_t* seg_starts;
    const int32_t* seg_slot;
    int n_segs, n_pos, n_rows;
    int stages;
    int kps;             // K blocks per ring stage (1 or 2: a row's adjacent 128-byte pieces fetched together)
    int mode;            // 0: fp32 v [n_rows][ld_v]; 1: bf16 hi/lo planes [n_rows][ld_p]
    float* v;
    int ld_v;
    bf16_t* vh;
    bf16_t* vl;
    int ld_p;            // plane row length: n_proj * r_pad64
    int r_pad64;         // r_slot rounded up to 64 (plane columns per projection)
    int ks;              // CTAs per row tile (a cluster), each a slice of K
    int x_ready;         // x is not written by the preceding kernel: read it before the wait
    unsigned stall_tx;   // test hook: extra bytes expected on the first stage (0 normally)
    unsigned* tickets;   // the work counter of the kernel that follows in the call (expand or linear), zeroed here (or null)
    int32_t* status;
};

// Rows of v for one tile row r (16 columns from c, fp32) -> the output form.
__device__ __forceinline__ void store_v16(const ShrinkTcParams& p, size_t row, int c, const float* v)
{
    if (p.mode == 0) {
        float4* dst = reinterpret_cast<float4*>(p.v + row * p.ld_v + c);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        return;
    }
    const int q = c / p.r_slot, jj = c - q * p.r_slot;
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
        hi[i] = *reinterpret_cast<const uint32_t*>(&h);
        lo[i] = *reinterpret_cast<const uint32_t*>(&l);
    }
    const size_t off = row * p.ld_p + q * p.r_pad64 + jj;
    uint4* dh = reinterpret_cast<uint4*>(p.vh + off);
    uint4* dl = reinterpret_cast<uint4*>(p.vl + off);
    dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
}

// Zeroes the planes' columns past r_slot in one row (the expand's K runs to r_pad64).
__device__ __forceinline__ void zero_plane_padding(const ShrinkTcParams& p, size_t row)
{
    for (int q = 0; q < p.n_proj; ++q)
        for (int jj = p.r_slot; jj < p.r_pad64; jj += 8) {
            const size_t off = row * p.ld_p + q * p.r_pad64 + jj;
            *reinterpret_cast<uint4*>(p.vh + off) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(p.vl + off) = make_uint4(0, 0, 0, 0);
        }
}

__global__ void __launch_bounds__(kShrinkThreads, 1)
sgmv_shrink_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap ma0,
                      const __grid_constant__ CUtensorMap ma1, const __grid_constant__ CUtensorMap ma2,
                      const __grid_constant__ CUtensorMap ma3, ShrinkTcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[8], empty[8], done;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // With ks > 1 a cluster of ks CTAs shares a row tile, CTA c reducing K
    // blocks [c n_kb / ks, (c+1) n_kb / ks); the fp32 partial accumulators
    // meet in distributed shared memory and are summed in a fixed order.
    //
    // Under programmatic dependent launch the segment table and A are read
    // at once, x too when it is ready (LORA_APPLY_X_READY); everything this
    // grid writes (v, the planes, status) waits for the preceding grid, and
    // every CTA waits before it leaves, so this grid never completes before
    // that one.
    grid_dep_launch();
    const int crank = p.ks > 1 ? static_cast<int>(cluster_rank()) : 0;
    const TileInfo ti = find_tile<kShrinkThreads>(p.seg_starts, p.seg_slot, p.n_segs, p.n_pos, blockIdx.x / p.ks);
    // Block 0 zeroes the counter the kernel after this one takes its work
    // from (after the grid dependency: no kernel before this one still uses
    // it), on every path, also when the call has no adapter tile at all.
    if (!ti.found) {
        grid_dep_wait();
        if (p.tickets != nullptr && blockIdx.x == 0 && tid == 0) *p.tickets = 0u;
        if (ti.bad && blockIdx.x == 0 && tid == 0) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }
    if (ti.slot >= p.n_slots || ti.slot < -1) {
        grid_dep_wait();
        if (p.tickets != nullptr && blockIdx.x == 0 && tid == 0) *p.tickets = 0u;
        if (tid == 0 && crank == 0) flag(p.status, LORA_DEV_SLOT_OUT_OF_RANGE);
        return;
    }
    const CUtensorMap* amap[4] = {&ma0, &ma1, &ma2, &ma3};
    const int S = p.stages, KPS = p.kps;
    const int sub_bytes = kBoxBytes + p.R * 128;   // one K block: the x box, then one A box per projection
    const int stage_bytes = KPS * sub_bytes;
    uint8_t* base = align1024(smem_raw);
    const int n_kb_all = (p.h_in + kKB - 1) / kKB;
    const int kb0 = crank * n_kb_all / p.ks;
    const int n_kb = (crank + 1) * n_kb_all / p.ks - kb0;   // >= 1: the launcher keeps ks <= n_kb_all
    const int n_st = (n_kb + KPS - 1) / KPS;                 // ring stages this CTA fills

    uint32_t ncols = 32;   // accumulator columns: a power of two >= R
    while (ncols < static_cast<uint32_t>(p.R)) ncols <<= 1;
    if (warp == 0) tmem_alloc(&s_tmem, ncols);
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        mbar_init_fence();
        s_fail = 0;
        tma_prefetch_desc(&mx);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    if (!p.x_ready) grid_dep_wait();   // x may be the preceding kernel's output

    if (warp == 0 && lane == 0) {
        // producer: per K block an X box + one A box per projection, KPS
        // K blocks to a stage
        int issued = 0;
        for (int i = 0; i < n_st; ++i) {
            const int s = i % S;
            // a stage is re-armed only once the MMAs have consumed it (its
            // previous phase complete)
            if (i >= S && !mbar_wait_spin(&empty[s], ((i / S) - 1) & 1)) {
                s_fail = 1;
                break;
            }
            uint8_t* st = base + s * stage_bytes;
            const int nkb = min(KPS, n_kb - i * KPS);
            mbar_expect_tx(&full[s], nkb * sub_bytes + (i == 0 ? p.stall_tx : 0u));
            for (int j = 0; j < nkb; ++j) {
                const int k = (kb0 + i * KPS + j) * kKB;
                uint8_t* sb = st + j * sub_bytes;
                tma_load_2d(sb, &mx, k, ti.row0, &full[s]);
                for (int q = 0; q < p.n_proj; ++q)
                    tma_load_2d(sb + kBoxBytes + q * p.r_slot * 128, amap[q], k, ti.slot * p.r_slot, &full[s]);
            }
            issued = i + 1;
        }
        // Every copy issued has landed before the CTA moves on (after a normal
        // run the MMA thread has already seen each of these phases complete).
        for (int i = issued > S ? issued - S : 0; i < issued; ++i)
            if (!mbar_wait(&full[i % S], (i / S) & 1)) s_fail = 1;
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: 4 x (128 x R x 16) per K block, accumulating in TMEM
        const uint32_t idesc = idesc_bf16_f32(kTileM, p.R);
        bool ok = true;
        for (int i = 0; i < n_st && ok; ++i) {
            const int s = i % S;
            if (!mbar_wait_spin(&full[s], (i / S) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int nkb = min(KPS, n_kb - i * KPS);
            for (int j = 0; j < nkb; ++j) {
                const uint32_t sb = smem_u32(base + s * stage_bytes + j * sub_bytes);
#pragma unroll
                for (int ks = 0; ks < kKB / 16; ++ks)
                    mma_bf16(tmem, sdesc_sw128(sb + ks * 32), sdesc_sw128(sb + kBoxBytes + ks * 32), idesc,
                             (i | j | ks) != 0);
            }
            mma_commit(&empty[s]);   // frees the stage once these MMAs have read it
        }
        if (!ok) s_fail = 1;
        mma_commit(&done);
    }
    __syncwarp();

    // ---- epilogue: TMEM row (lane) -> v ----
    // A tile whose copies or MMAs did not complete stores a zero intermediate
    // for its rows (the expand then adds nothing to them) and reports the
    // timeout; s_fail is final once every thread has passed the barrier
    // below (the producer and MMA threads have left their loops).
    bool ok = mbar_wait(&done, 0);
    tc_fence_after();
    ok = __syncthreads_and(ok && !s_fail);
    grid_dep_wait();   // the preceding kernel may still read the buffers written below
    if (p.tickets != nullptr && blockIdx.x == 0 && tid == 0) *p.tickets = 0u;   // (as above)
    const int r = warp * 32 + lane;   // tile row = TMEM lane
    if (p.ks == 1) {
        const bool row_ok = r < ti.nrows;
        const size_t row = static_cast<size_t>(ti.row0 + r);
        for (int c = 0; c < p.R; c += 16) {
            float v[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
            if (!ok)
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
            if (row_ok) store_v16(p, row, c, v);
        }
        if (p.mode == 1 && row_ok && p.r_pad64 > p.r_slot) zero_plane_padding(p, row);
    } else {
        // partial accumulator -> shared memory (over the consumed ring), row
        // pitch R + 4 floats: 16-byte stores from 8 consecutive rows meet no
        // bank twice
        float* red = reinterpret_cast<float*>(base);
        const int pitch = p.R + 4;
        for (int c = 0; c < p.R; c += 16) {
            float v[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
            float4* dst = reinterpret_cast<float4*>(red + r * pitch + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        if (tid == 0) s_fail = ok ? 0 : 1;   // this CTA's partials are valid unless it failed
        __syncthreads();
        cluster_arrive();
        cluster_wait();
        // a peer whose copies timed out has no valid partials: the whole
        // tile then gets a zero intermediate
        for (int peer = 0; peer < p.ks; ++peer) {
            int f;
            asm volatile("ld.shared::cluster.b32 %0, [%1];\n"
                         : "=r"(f)
                         : "r"(map_rank(smem_u32(const_cast<int*>(&s_fail)), peer))
                         : "memory");
            if (f) ok = false;
        }
        // CTA c sums rows [c * 128 / ks, (c + 1) * 128 / ks) over the cluster,
        // 16 columns per item, peers in rank order
        const int r_lo = crank * kTileM / p.ks, r_hi = (crank + 1) * kTileM / p.ks;
        const int per_row = p.R / 16;
        const uint32_t red_s = smem_u32(red);
        for (int it = tid; it < (r_hi - r_lo) * per_row; it += kShrinkThreads) {
            const int rr = r_lo + it / per_row, c = (it - (it / per_row) * per_row) * 16;
            float v[16] = {};
            for (int peer = 0; peer < p.ks; ++peer) {
                const uint32_t src = map_rank(red_s + 4u * static_cast<uint32_t>(rr * pitch + c), peer);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 f = ld_dsmem_f4(src + 16u * i);
                    v[4 * i] += f.x;
                    v[4 * i + 1] += f.y;
                    v[4 * i + 2] += f.z;
                    v[4 * i + 3] += f.w;
                }
            }
            if (!ok)
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
            if (rr < ti.nrows) store_v16(p, static_cast<size_t>(ti.row0 + rr), c, v);
        }
        if (p.mode == 1 && p.r_pad64 > p.r_slot)
            for (int rr = r_lo + tid; rr < min(r_hi, ti.nrows); rr += kShrinkThreads)
                zero_plane_padding(p, static_cast<size_t>(ti.row0 + rr));
        cluster_arrive();   // peers may leave once everyone has read their partials
        cluster_wait();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, ncols);
    if (tid == 0 && !ok) flag(p.status, LORA_DEV_TIMEOUT);
    if (tid == 0 && ti.bad && blockIdx.x == 0) flag(p.status, LORA_DEV_BAD_SEGMENT);
}

// ------------------------------------------------------------- expand ----
//
// Persistent: one CTA per SM walks work items -- (projection q, chunk of up
// to p.chunk 128-column output tiles, 128-row tile u of the segments) -- taken
// round-robin (item c, c + G, c + 2G, ... for CTA c of G), ordered with the
// row tile fastest, so at any moment the CTAs work on the same chunk of B'
// for different row tiles and B' is read from HBM about once.  The TMA ring
// keeps streaming across items: no CTA pays a start-up and a drain per item.
// The row tiles of a CTA's items are resolved once, at its start, into a
// shared-memory table.  The v_hi / v_lo slice of an item (row tile,
// projection) is loaded once into one of two buffers (one when r_pad64 > 64),
// so the next item's slice loads while the current one's tiles finish.  A
// tile's B' boxes (from L2) go through a two-stage ring that the MMA's
// completion frees; its y tile (from HBM) through a ring of up to kStagesY
// stages, each held from its load until the store has read it back, which
// is why the two do not share stages.  The fp32 accumulator is
// double-buffered in tensor memory, so the epilogue of tile i (TMEM ->
// registers, + y from shared memory, round) overlaps the loads and MMAs of
// tile i+1, and a store warp writes finished tiles back, so that no
// epilogue warp waits on a store.
//   warp 0: TMA producer   warp 1: MMA issuer   warps 2..17: epilogue
//   warp 18: TMA store

constexpr int kStagesY = 5;        // y ring stages, at most (the launcher picks 2 to 5)
constexpr int kEpiWarps = 16;       // 4 per TMEM lane quarter, 32 columns each
constexpr int kStoreWarpE = 2 + kEpiWarps;
constexpr int kExpandThreadsP = 32 * (kStoreWarpE + 1);
constexpr int kChunkMax = 16;       // output tiles per work item, at most
constexpr int kMaxItems = 64;       // work items per CTA in the static order (the launcher sizes the grid)
constexpr int kMaxRt = 1024;        // row tiles a CTA can table (the dynamic order needs all of them)
constexpr int kQD = 8;              // work-item queue depth (dynamic order)

struct ExpandTcParams {
    int n_proj, r_slot, r_pad64, n_slots;
    int out_off[LORA_MAX_PROJ];
    int width[LORA_MAX_PROJ];
    int col_tiles[LORA_MAX_PROJ];   // ceil(width / 128) per projection
    int chunks[LORA_MAX_PROJ];      // ceil(col_tiles / chunk) per projection
    int n_chunks;                   // sum of chunks
    int chunk;                      // output tiles per work item
    const int32_t* seg_starts;
    const int32_t* seg_slot;
    int n_segs, n_pos, n_rows;
    bf16_t* y;
    int ld_y;
    int stages;                     // y ring stages (<= kStagesY)
    int vbufs;                      // v slice buffers (1 or 2)
    unsigned stall_tx;              // test hook: extra bytes expected on the first B' stage (0 normally)
    unsigned* tickets;              // dynamic order: the call's work-item counter (zeroed by the shrink)
    int dyn;                        // 1: items taken from tickets; 0: item c + k G for CTA c
    int table_bytes;                // the row-tile table at the start of dynamic shared memory
    int32_t* status;
};

struct RowTile {
    int slot, row0, nrows;
};

// Work items in the dynamic order: the producer takes each item's number
// from the call's counter (one atomic per item) and passes it through a
// queue of kQD slots; the MMA thread, every epilogue warp and the store
// thread read the items in the same order.  An item number past the last
// item ends the sequence.
struct ItemQueue {
    long long* item;
    uint64_t* full;    // the producer's arrival
    uint64_t* empty;   // one arrival per reader
};
constexpr int kItemReaders = 2 + kEpiWarps;   // MMA thread, epilogue warps, store thread
enum ItemRole { kRoleProducer, kRoleThread, kRoleWarp };

// Walks this CTA's tiles: item k (static order: global item c + k * G;
// dynamic order: the k-th item taken), tile ct of the item's projection.
// Divides once per item, never per tile.  kDyn and kRole are compile-time,
// so the static order carries none of the queue's state.
template <bool kDyn, int kRole>
struct TileIter {
    int k, q, ct, ct_end, rix;   // rix: the item's entry of the row-tile table
    unsigned ahead;              // producer, dynamic order: the next item's ticket, taken one item early
    const ExpandTcParams& p;
    int n_rt;
    long long n_all;
    ItemQueue Q;
    volatile int* fail;
    __device__ __forceinline__ TileIter(const ExpandTcParams& pp, int nrt, long long nall, const ItemQueue& qq,
                                        volatile int* f)
        : k(0), q(0), ct(0), ct_end(0), rix(0), ahead(0), p(pp), n_rt(nrt), n_all(nall), Q(qq), fail(f)
    {
    }
    // item k's number, or -1 past the end (or on a timeout, with *fail set)
    __device__ __forceinline__ long long take()
    {
        if constexpr (!kDyn) {
            const long long it = blockIdx.x + static_cast<long long>(k) * gridDim.x;
            return it < n_all ? it : -1;
        } else {
            const int slot = k % kQD;
            long long it;
            if constexpr (kRole == kRoleProducer) {
                if (k >= kQD && !mbar_wait_spin(&Q.empty[slot], ((k / kQD) - 1) & 1)) {
                    *fail = 1;
                    return -1;
                }
                // this item's ticket was taken one item earlier, so the atomic's
                // round trip overlaps the previous item's loads; the next one is
                // requested now
                const unsigned t = *fail ? 0xFFFFFFFFu : (k == 0 ? atomicAdd(p.tickets, 1u) : ahead);
                it = static_cast<long long>(t) < n_all ? static_cast<long long>(t) : -1;
                if (it >= 0) ahead = atomicAdd(p.tickets, 1u);
                Q.item[slot] = it;
                mbar_arrive(&Q.full[slot]);
                return it;
            } else {
                const bool ok = kRole == kRoleThread ? mbar_wait_spin(&Q.full[slot], (k / kQD) & 1)
                                                     : mbar_wait(&Q.full[slot], (k / kQD) & 1);
                if (!ok) {
                    *fail = 1;
                    return -1;
                }
                it = Q.item[slot];
                if constexpr (kRole == kRoleWarp) __syncwarp();   // every lane has read the slot before it is freed
                if (kRole == kRoleThread || (threadIdx.x & 31) == 0) mbar_arrive(&Q.empty[slot]);
                return it;
            }
        }
    }
    __device__ __forceinline__ bool item()
    {
        const long long it = take();
        if (it < 0) return false;
        int ch = static_cast<int>(it / n_rt);   // chunk index over all projections
        if constexpr (kDyn) rix = static_cast<int>(it - static_cast<long long>(ch) * n_rt);
        else rix = k;
        q = 0;
        while (q < p.n_proj - 1 && ch >= p.chunks[q]) {
            ch -= p.chunks[q];
            ++q;
        }
        ct = ch * p.chunk;
        ct_end = min(ct + p.chunk, p.col_tiles[q]);
        return true;
    }
    __device__ __forceinline__ bool init()
    {
        k = 0;
        return item();
    }
    // false once past the CTA's last item
    __device__ __forceinline__ bool next()
    {
        if (++ct < ct_end) return true;
        ++k;
        return item();
    }
};

// Row tile u of item it (row tile fastest).
__device__ __forceinline__ int item_row_tile(long long it, int n_rt) { return static_cast<int>(it % n_rt); }

// One block-wide pass over the segment table, kExpandThreadsP segments per
// round: row tiles per segment (slot -1 and malformed segments have none)
// and their prefix sums.  With fill, the segment holding the row tile of
// each of this CTA's n_items items writes s_rt[item] (static order), or
// every segment writes s_rt[u] for each of its row tiles u (dynamic order).
// Returns the total number of row tiles.  Every thread of the block takes
// part.
__device__ int scan_row_tiles(const ExpandTcParams& p, bool fill, int n_rt, int n_items, RowTile* s_rt, int* s_warp,
                              int* s_bad)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int base = 0;
    for (int g0 = 0; g0 < p.n_segs; g0 += kExpandThreadsP) {
        const int gi = g0 + tid;
        int n = 0, s = 0, e = 0, sl = -1;
        if (gi < p.n_segs) {
            s = __ldg(p.seg_starts + gi);
            e = __ldg(p.seg_starts + gi + 1);
            sl = __ldg(p.seg_slot + gi);
            const bool sane = s >= 0 && e <= p.n_pos && s <= e;
            if (!sane) atomicOr(s_bad, 1);
            n = (sane && sl >= 0) ? (e - s + kTileM - 1) / kTileM : 0;
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
        for (int w = 0; w < kExpandThreadsP / 32; ++w) {
            if (w < warp) before += s_warp[w];
            total += s_warp[w];
        }
        if (fill && n > 0 && p.dyn) {
            const int excl = base + before + (incl - n);   // row tiles before this segment
            const int cap = p.table_bytes / static_cast<int>(sizeof(RowTile));   // entries the table holds
            for (int j = 0; j < n && excl + j < cap; ++j) {
                RowTile rt;
                rt.slot = sl;
                rt.row0 = s + j * kTileM;
                rt.nrows = min(kTileM, e - rt.row0);
                s_rt[excl + j] = rt;
            }
        } else if (fill && n > 0) {
            const int excl = base + before + (incl - n);   // row tiles before this segment
            for (int kk = 0; kk < n_items; ++kk) {
                const int u = item_row_tile(blockIdx.x + static_cast<long long>(kk) * gridDim.x, n_rt);
                if (u >= excl && u < excl + n) {
                    RowTile rt;
                    rt.slot = sl;
                    rt.row0 = s + (u - excl) * kTileM;
                    rt.nrows = min(kTileM, e - rt.row0);
                    s_rt[kk] = rt;
                }
            }
        }
        base += total;
        __syncthreads();   // s_warp is rewritten by the next round
    }
    return base;
}

template <bool kDyn>
__global__ void __launch_bounds__(kExpandThreadsP, 1)
sgmv_expand_tc_kernel(const __grid_constant__ CUtensorMap mvh, const __grid_constant__ CUtensorMap mvl,
                      const __grid_constant__ CUtensorMap my, const __grid_constant__ CUtensorMap mb0,
                      const __grid_constant__ CUtensorMap mb1, const __grid_constant__ CUtensorMap mb2,
                      const __grid_constant__ CUtensorMap mb3, ExpandTcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t yfull[kStagesY], yempty[kStagesY], epi_done[kStagesY];
    __shared__ __align__(8) uint64_t bfull[2], bempty[2], acc_full[2], acc_empty[2], v_full[2], v_empty[2], mma_done;
    __shared__ __align__(8) uint64_t q_full[kQD], q_empty[kQD];
    __shared__ long long q_item[kQD];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_fail;
    __shared__ int s_warp[kExpandThreadsP / 32];
    __shared__ int s_bad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // row tiles: of this CTA's items (static order) or all of them (dynamic)
    RowTile* s_rt = reinterpret_cast<RowTile*>(smem_raw);

    // ---- this CTA's items and their row tiles ----
    // Under programmatic dependent launch the segment table is read at once;
    // v and y are touched only after the preceding grid has completed, and
    // every CTA waits before it leaves.
    grid_dep_launch();
    if (tid == 0)   // the table must cover [0, n_pos): its first entry 0, its last n_pos
        s_bad = p.n_segs > 0 && (__ldg(p.seg_starts) != 0 || __ldg(p.seg_starts + p.n_segs) != p.n_pos);
    __syncthreads();
    const int n_rt = scan_row_tiles(p, false, 1, 0, s_rt, s_warp, &s_bad);
    const long long n_all = static_cast<long long>(n_rt) * p.n_chunks;
    // static order: this CTA's item count; dynamic order: every CTA takes part
    // while the row tiles fit the table (the launcher's bound makes sure)
    const int n_items = p.dyn ? (n_all > 0 ? 1 : 0)
                              : (n_all > blockIdx.x ? static_cast<int>((n_all - 1 - blockIdx.x) / gridDim.x + 1) : 0);
    // (a segment table whose tiles outnumber the launcher's bound, possible
    // only for overlapping segments, is flagged and left alone)
    if (n_items <= 0 || n_items > kMaxItems || (p.dyn && n_rt > p.table_bytes / static_cast<int>(sizeof(RowTile)))) {
        grid_dep_wait();
        if (tid == 0 && (n_items > 0 || (blockIdx.x == 0 && s_bad))) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }
    scan_row_tiles(p, true, n_rt, n_items, s_rt, s_warp, &s_bad);
    const int n_table = p.dyn ? n_rt : n_items;
    for (int i = tid; i < n_table; i += kExpandThreadsP)
        if (s_rt[i].slot >= p.n_slots || s_rt[i].slot < -1) atomicOr(&s_bad, 2);
    __syncthreads();
    grid_dep_wait();
    if (tid == 0 && blockIdx.x == 0 && (s_bad & 1)) flag(p.status, LORA_DEV_BAD_SEGMENT);
    if (s_bad & 2) {   // a slot out of range: flag it, leave this CTA's tiles alone
        if (tid == 0) flag(p.status, LORA_DEV_SLOT_OUT_OF_RANGE);
        return;
    }

    const CUtensorMap* bmap[4] = {&mb0, &mb1, &mb2, &mb3};
    const int kbs = p.r_pad64 / kKB;                         // K blocks per plane
    const int S = p.stages;                                  // y ring depth (shared memory permitting)
    const int VB = p.vbufs;                                  // v slice buffers
    const int bstage_bytes = kbs * kBoxBytes;                // B' of one tile
    const int ystage_bytes = 2 * kBoxBytes;                  // one y tile: two 64-column boxes
    const int vbuf_bytes = 2 * kbs * kBoxBytes;              // v_hi boxes, then v_lo boxes
    uint8_t* vbufs = align1024(smem_raw + p.table_bytes);    // VB x [v_hi | v_lo]
    uint8_t* bring = vbufs + VB * vbuf_bytes;                // 2 x B'
    uint8_t* yring = bring + 2 * bstage_bytes;               // S x y

    if (warp == 0) tmem_alloc(&s_tmem, 2 * kExpandN);
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&yfull[s], 1);
            mbar_init(&yempty[s], 1);                 // the store warp
            mbar_init(&epi_done[s], kEpiWarps / 2);   // the team that took the tile
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bfull[a], 1);
            mbar_init(&bempty[a], 1);                 // the MMA thread's commit
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], kEpiWarps / 2);
            mbar_init(&v_full[a], 1);
            mbar_init(&v_empty[a], 1);
        }
        mbar_init(&mma_done, 1);
        for (int j = 0; j < kQD; ++j) {
            mbar_init(&q_full[j], 1);
            mbar_init(&q_empty[j], kItemReaders);
        }
        mbar_init_fence();
        s_fail = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const ItemQueue Q{q_item, q_full, q_empty};

    if (warp == 0) {
        if (lane == 0) {   // ---- producer ----
            TileIter<kDyn, kRoleProducer> tr(p, n_rt, n_all, Q, &s_fail);
            bool more = tr.init();
            int k_prev = -1;
            int y_issued = 0, b_issued = 0, v_issued = 0;   // stages and v slices armed so far
            for (int i = 0; more && !s_fail; ++i) {
                const RowTile rt = s_rt[tr.rix];
                if (tr.k != k_prev) {   // a new item: its v slice into buffer k % VB
                    k_prev = tr.k;
                    const int vb = tr.k % VB;
                    if (tr.k >= VB && !mbar_wait_spin(&v_empty[vb], ((tr.k / VB) - 1) & 1)) {
                        s_fail = 1;
                        break;
                    }
                    uint8_t* vh = vbufs + vb * vbuf_bytes;
                    mbar_expect_tx(&v_full[vb], vbuf_bytes);
                    for (int kb = 0; kb < kbs; ++kb) {
                        tma_load_2d(vh + kb * kBoxBytes, &mvh, tr.q * p.r_pad64 + kb * kKB, rt.row0, &v_full[vb]);
                        tma_load_2d(vh + (kbs + kb) * kBoxBytes, &mvl, tr.q * p.r_pad64 + kb * kKB, rt.row0,
                                    &v_full[vb]);
                    }
                    v_issued = tr.k + 1;
                }
                const int col0 = tr.ct * kExpandN;
                // B' of the tile into B' stage i % 2
                const int b = i & 1;
                if (i >= 2 && !mbar_wait_spin(&bempty[b], ((i >> 1) - 1) & 1)) {
                    s_fail = 1;
                    break;
                }
                // The epilogue releases a stage after a failure too (setting
                // s_fail first): re-arm it only while nothing has failed, so a
                // stage whose previous phase never completed is never armed again.
                if (s_fail) break;
                uint8_t* bs = bring + b * bstage_bytes;
                mbar_expect_tx(&bfull[b], bstage_bytes + (i == 0 ? p.stall_tx : 0u));
                for (int kb = 0; kb < kbs; ++kb)
                    tma_load_2d(bs + kb * kBoxBytes, bmap[tr.q], kb * kKB, rt.slot * p.width[tr.q] + col0, &bfull[b]);
                b_issued = i + 1;
                // the y tile into y stage i % S
                const int s = i % S;
                if (i >= S && !mbar_wait_spin(&yempty[s], ((i / S) - 1) & 1)) {
                    s_fail = 1;
                    break;
                }
                if (s_fail) break;
                uint8_t* ys = yring + s * ystage_bytes;
                mbar_expect_tx(&yfull[s], ystage_bytes);
                const int ycol = p.out_off[tr.q] + col0;
                tma_load_2d(ys, &my, ycol, rt.row0, &yfull[s]);
                tma_load_2d(ys + kBoxBytes, &my, ycol + kKB, rt.row0, &yfull[s]);
                y_issued = i + 1;
                more = tr.next();
            }
            // Every copy issued has landed before the CTA moves on (after a
            // normal run the consumers have seen each of these phases complete).
            for (int i = y_issued > S ? y_issued - S : 0; i < y_issued; ++i)
                if (!mbar_wait(&yfull[i % S], (i / S) & 1)) s_fail = 1;
            for (int i = b_issued > 2 ? b_issued - 2 : 0; i < b_issued; ++i)
                if (!mbar_wait(&bfull[i & 1], (i >> 1) & 1)) s_fail = 1;
            for (int k = v_issued > VB ? v_issued - VB : 0; k < v_issued; ++k)
                if (!mbar_wait(&v_full[k % VB], (k / VB) & 1)) s_fail = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---- MMA issuer ----
            const uint32_t idesc = idesc_bf16_f32(kTileM, kExpandN);
            bool ok = true;
            TileIter<kDyn, kRoleThread> tr(p, n_rt, n_all, Q, &s_fail);
            bool more = tr.init();
            int k_prev = -1;
            for (int i = 0; more && ok && !s_fail; ++i) {
                const int k = tr.k;
                if (k != k_prev) {
                    k_prev = k;
                    if (!mbar_wait_spin(&v_full[k % VB], (k / VB) & 1)) { ok = false; break; }
                }
                const int b = i & 1, a = i & 1;
                if (i >= 2 && !mbar_wait_spin(&acc_empty[a], ((i >> 1) - 1) & 1)) { ok = false; break; }
                if (!mbar_wait_spin(&bfull[b], (i >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t bs = smem_u32(bring + b * bstage_bytes);
                const uint32_t vs = smem_u32(vbufs + (k % VB) * vbuf_bytes);
                const uint32_t d = tmem + a * kExpandN;
                int n = 0;
                for (int plane = 0; plane < 2; ++plane)
                    for (int kb = 0; kb < kbs; ++kb) {
                        const uint32_t av = vs + (plane * kbs + kb) * kBoxBytes;
#pragma unroll
                        for (int ks = 0; ks < kKB / 16; ++ks, ++n)
                            mma_bf16(d, sdesc_sw128(av + ks * 32), sdesc_sw128(bs + kb * kBoxBytes + ks * 32),
                                     idesc, n != 0);
                    }
                mma_commit(&acc_full[a]);
                mma_commit(&bempty[b]);   // B' stage b is free once these MMAs are done
                more = tr.next();
                if (!more || tr.k != k) mma_commit(&v_empty[k % VB]);   // the item's slice is free after these
            }
            if (!ok) s_fail = 1;
            // the tensor memory is freed only after every MMA issued has completed
            mma_commit(&mma_done);
            if (!mbar_wait(&mma_done, 0)) s_fail = 1;
        }
    } else if (warp < kStoreWarpE) {   // ---- epilogue warps ----
        // Two teams of 8 warps take alternate tiles (team t: tiles i = t, t+2,
        // ..., accumulator t), so two tiles' epilogues are in flight at once.
        // Within a team, 2 warps per TMEM lane quarter, 64 columns each.
        const int e = warp - 2;
        const int team = e >> 3, w8 = e & 7;
        const int quarter = warp & 3;       // TMEM lanes this warp may read
        const int hc = w8 >> 2;             // which 64-column half of the tile (one y box)
        const int r = quarter * 32 + lane;  // tile row
        // Every warp of a team runs every one of the team's iterations and
        // arrives on its barriers whatever happened (after a timeout it only
        // skips work), so no wait is left without its arrivals.
        TileIter<kDyn, kRoleWarp> tr(p, n_rt, n_all, Q, &s_fail);
        bool more = tr.init();
        if (team == 1 && more) more = tr.next();
        for (int i = team; more; i += 2) {
            const RowTile rt = s_rt[tr.rix];
            const int s = i % S, a = team;
            bool ok = !s_fail && mbar_wait(&acc_full[a], (i >> 1) & 1);
            ok = ok && mbar_wait(&yfull[s], (i / S) & 1);   // the staged y tile (TMA-written) is visible here
            if (!ok) s_fail = 1;
            tc_fence_after();
            const uint32_t tcol = tmem + a * kExpandN + (static_cast<uint32_t>(quarter * 32) << 16) + hc * kKB;
            uint8_t* ybox = yring + s * ystage_bytes + hc * kBoxBytes;
            uint8_t* sy = ybox + r * 128;
            const int tile_col0 = tr.ct * kExpandN;
            const int col0 = tile_col0 + hc * kKB;
            const int cols_left = p.width[tr.q] - col0;
            // whole tile inside the segment's rows and the projection's columns:
            // results go back into the staged tile and leave by TMA bulk stores
            const bool whole = rt.nrows == kTileM && tile_col0 + kExpandN <= p.width[tr.q];
            const bool mine = ok && r < rt.nrows;
            bf16_t* yrow_g = p.y + static_cast<size_t>(rt.row0 + min(r, rt.nrows - 1)) * p.ld_y + p.out_off[tr.q];
            // 32 accumulator columns at a time, so registers are left for the
            // four 16-byte pieces of y in flight
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float d[32];
                tmem_ld32(tcol + half * 32, d);
                if (half == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[a]);   // accumulator a may be overwritten now
                }
                if (mine) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int chunk = half * 4 + c4;
                        if (chunk * 8 >= cols_left) continue;
                        uint4* slot8 = reinterpret_cast<uint4*>(sy + ((chunk ^ (r & 7)) << 4));
                        const uint4 res = add_round8(*slot8, d + c4 * 8);
                        if (whole) *slot8 = res;
                        else *reinterpret_cast<uint4*>(yrow_g + col0 + chunk * 8) = res;
                    }
                }
            }
            fence_async_smem();   // the TMA store reads what these threads wrote
            __syncwarp();
            if (lane == 0) mbar_arrive(&epi_done[s]);   // this warp is done with y stage s
            more = tr.next() && tr.next();
        }
    } else if (lane == 0) {   // ---- store: finished whole tiles back to y, then the stage is free ----
        TileIter<kDyn, kRoleThread> tr(p, n_rt, n_all, Q, &s_fail);
        bool more = tr.init();
        for (int i = 0; more; ++i) {
            const RowTile rt = s_rt[tr.rix];
            const int s = i % S;
            if (!s_fail && !mbar_wait(&epi_done[s], (i / S) & 1)) s_fail = 1;
            const int tile_col0 = tr.ct * kExpandN;
            const bool whole = rt.nrows == kTileM && tile_col0 + kExpandN <= p.width[tr.q];
            if (whole && !s_fail) {
                uint8_t* y0 = yring + s * ystage_bytes;
                tma_store_2d(&my, p.out_off[tr.q] + tile_col0, rt.row0, y0);
                tma_store_2d(&my, p.out_off[tr.q] + tile_col0 + kKB, rt.row0, y0 + kBoxBytes);
                bulk_commit();
                bulk_wait_read();   // the stage may be refilled once the stores have read it
            }
            mbar_arrive(&yempty[s]);
            more = tr.next();
        }
        bulk_wait_all();
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 2 * kExpandN);
    if (tid == 0 && s_fail) flag(p.status, LORA_DEV_TIMEOUT);
}

}  // namespace

bool sgmv_tc_supported(int n_proj, int r_slot, int h_in)
{
    return r_slot % 16 == 0 && r_slot <= LORA_MAX_RANK && n_proj * r_slot <= 256 && h_in >= kKB;
}

size_t sgmv_tc_plane_bytes(int n_rows, int n_proj, int r_slot)
{
    const int r_pad64 = (r_slot + kKB - 1) / kKB * kKB;
    return 2 * static_cast<size_t>(n_rows) * n_proj * r_pad64 * sizeof(bf16_t);
}

namespace {

size_t shrink_smem(int stages, int R, int kps = 1)
{
    return static_cast<size_t>(stages) * kps * (kBoxBytes + R * 128) + 1024;
}

// Four stages, two CTAs per SM where they fit in shared memory; where one
// CTA is alone on its SM anyway (wide rank stacks), as many stages as that
// SM holds, since the CTA's bytes in flight are then all the SM has.
int shrink_stages(int R, int kps)
{
    constexpr size_t kTwoPerSm = 113 * 1024, kOnePerSm = 225 * 1024;
    int s = 4;
    if (shrink_smem(4, R) > kTwoPerSm)
        while (s < 8 && shrink_smem(s + 1, R) <= kOnePerSm) ++s;
    // the same bytes in flight when a stage holds kps K blocks
    s = std::max(2, (s + kps - 1) / kps);
    while (s > 2 && shrink_smem(s, R, kps) > kOnePerSm) --s;
    int e = std::max(2, std::min(8, env_int("LORA_TC_SHRINK_STAGES", s)));
    while (e > 2 && shrink_smem(e, R, kps) > kOnePerSm) --e;
    return e;
}

// Raises the kernel's dynamic shared-memory limit to at least smem on the
// current device (the limit excludes the kernel's static shared memory).
bool configure_once(const void* fn, size_t smem, int& configured_device, size_t& configured_bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (configured_device == dev && configured_bytes >= smem) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return false;
    if (prefer_max_shared(fn) != cudaSuccess) return false;
    configured_device = dev;
    configured_bytes = smem;
    return true;
}

// Output tiles per expand CTA (LORA_TC_TILES_PER_CTA overrides; tuning aid).

}  // namespace

cudaError_t launch_sgmv_shrink_tc(float* v, int ld_v, bf16_t* vh, bf16_t* vl, const bf16_t* x, int ld_x, int h_in,
                                  const ProjSet& ps, const int32_t* seg_starts, const int32_t* seg_slot, int n_segs,
                                  int n_pos, int n_rows, int n_slots, unsigned flags, int32_t* status,
                                  cudaStream_t stream, unsigned* tickets)
{
    if (n_pos <= 0 || n_segs <= 0) return cudaSuccess;
    const int R = ps.n_proj * ps.r_slot;
    CUtensorMap mx, ma[4];
    if (!encode_tmap_bf16(&mx, x, n_rows, h_in, ld_x, kTileM, kKB, true)) return cudaErrorInvalidValue;
    for (int q = 0; q < 4; ++q) {
        const int src = q < ps.n_proj ? q : 0;
        if (!encode_tmap_bf16(&ma[q], ps.A[src], static_cast<uint64_t>(n_slots) * ps.r_slot, h_in, h_in,
                              ps.r_slot, kKB, true))
            return cudaErrorInvalidValue;
    }
    ShrinkTcParams p{};
    p.n_proj = ps.n_proj;
    p.r_slot = ps.r_slot;
    p.R = R;
    p.h_in = h_in;
    p.n_slots = n_slots;
    p.seg_starts = seg_starts;
    p.seg_slot = seg_slot;
    p.n_segs = n_segs;
    p.n_pos = n_pos;
    p.n_rows = n_rows;
    // Two K blocks to a stage: each x row's two adjacent 128-byte pieces are
    // requested together (Mistral-7B prefill: 1.432 against 1.444 ms per
    // step on one box; the mixed batch 3.678 against 3.706 ms).
    p.kps = std::max(1, std::min(2, env_int("LORA_TC_SHRINK_KPS", 2)));
    p.stages = shrink_stages(R, p.kps);
    p.mode = v ? 0 : 1;
    p.v = v;
    p.ld_v = ld_v;
    p.vh = vh;
    p.vl = vl;
    p.r_pad64 = (ps.r_slot + kKB - 1) / kKB * kKB;
    p.ld_p = ps.n_proj * p.r_pad64;
    p.x_ready = (flags & LORA_APPLY_X_READY) ? 1 : 0;
    p.stall_tx = test_stall_bytes(kStallShrinkTc);
    p.tickets = tickets;
    p.status = status;
    // Few row tiles: split K over a cluster of ks CTAs per tile so that the
    // grid covers the SMs (each CTA keeps at least two K blocks).
    static int n_sms = 0, sms_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidValue;
    if (sms_device != dev) {
        if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cudaErrorInvalidValue;
        sms_device = dev;
    }
    const int tiles = (n_pos + kTileM - 1) / kTileM + n_segs;   // upper bound
    const int n_kb = (h_in + kKB - 1) / kKB;
    int ks = 1;
    while (ks < 8 && static_cast<long long>(tiles) * ks < n_sms && n_kb >= 4 * ks) ks *= 2;
    p.ks = std::max(1, std::min(env_int("LORA_TC_SHRINK_KS", ks), n_kb));
    // the cluster's partials reuse the ring: 128 rows x (R + 4) fp32
    const size_t red = p.ks > 1 ? static_cast<size_t>(kTileM) * (R + 4) * sizeof(float) + 1024 : 0;
    const size_t smem = std::max(shrink_smem(p.stages, R, p.kps), red);
    static int configured = -1;
    static size_t configured_bytes = 0;
    if (!configure_once(reinterpret_cast<const void*>(sgmv_shrink_tc_kernel), smem, configured, configured_bytes))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * p.ks));
    cfg.blockDim = dim3(kShrinkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & LORA_APPLY_NO_PDL) ? 1 : 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, sgmv_shrink_tc_kernel, mx, ma[0], ma[1], ma[2], ma[3], p);
    note_launch();
    return e;
}

cudaError_t launch_sgmv_expand_tc(bf16_t* y, int ld_y, const bf16_t* vh, const bf16_t* vl, const ProjSet& ps,
                                  const int32_t* seg_starts, const int32_t* seg_slot, int n_segs, int n_pos,
                                  int n_rows, int n_slots, unsigned flags, int32_t* status, cudaStream_t stream,
                                  unsigned* tickets)
{
    if (n_pos <= 0 || n_segs <= 0) return cudaSuccess;
    const int r_pad64 = (ps.r_slot + kKB - 1) / kKB * kKB;
    const int ld_p = ps.n_proj * r_pad64;
    CUtensorMap mvh, mvl, my, mb[4];
    if (!encode_tmap_bf16(&mvh, vh, n_rows, ld_p, ld_p, kTileM, kKB, true) ||
        !encode_tmap_bf16(&mvl, vl, n_rows, ld_p, ld_p, kTileM, kKB, true) ||
        !encode_tmap_bf16(&my, y, n_rows, ld_y, ld_y, kTileM, kKB, true))
        return cudaErrorInvalidValue;
    static int n_sms = 0, sms_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidValue;
    if (sms_device != dev) {
        if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cudaErrorInvalidValue;
        sms_device = dev;
    }
    ExpandTcParams p{};
    int tiles_per_row = 0;
    for (int q = 0; q < ps.n_proj; ++q) tiles_per_row += (ps.width[q] + kExpandN - 1) / kExpandN;
    // Work items of up to 16 output tiles; fewer for small calls, so that
    // every SM gets about three items and the last ones end together.
    const long long rt_bound = (n_pos + kTileM - 1) / kTileM + static_cast<long long>(n_segs);
    p.chunk = static_cast<int>(std::max(4LL, std::min<long long>(kChunkMax, rt_bound * tiles_per_row / (3LL * n_sms))));
    p.chunk = std::max(1, env_int("LORA_TC_EXPAND_CHUNK", p.chunk));
    for (int q = 0; q < 4; ++q) {
        const int src = q < ps.n_proj ? q : 0;
        if (!encode_tmap_bf16(&mb[q], ps.B[src], static_cast<uint64_t>(n_slots) * ps.width[src], ps.r_slot,
                              ps.r_slot, kExpandN, kKB, true))
            return cudaErrorInvalidValue;
        if (q < ps.n_proj) {
            p.out_off[q] = ps.out_off[q];
            p.width[q] = ps.width[q];
            p.col_tiles[q] = (ps.width[q] + kExpandN - 1) / kExpandN;
            p.chunks[q] = (p.col_tiles[q] + p.chunk - 1) / p.chunk;
            p.n_chunks += p.chunks[q];
        }
    }
    p.n_proj = ps.n_proj;
    p.r_slot = ps.r_slot;
    p.r_pad64 = r_pad64;
    p.n_slots = n_slots;
    p.seg_starts = seg_starts;
    p.seg_slot = seg_slot;
    p.n_segs = n_segs;
    p.n_pos = n_pos;
    p.n_rows = n_rows;
    p.y = y;
    p.ld_y = ld_y;
    p.stall_tx = test_stall_bytes(kStallExpandTc);
    p.status = status;
    // Dynamic order (work items taken from the call's counter, so that CTAs
    // that start late or run slow take fewer) for large work items, while
    // every row tile fits the table; the static round-robin order otherwise.
    // Measured on one box: Mistral-7B prefill (16-tile items) 1.427 ->
    // 1.409 ms per step; the mixed batch (4-tile items) 3.70 -> 3.81 ms, where
    // each item's hand-off costs more than the balance gains.
    // LORA_TC_EXPAND_DYNAMIC: 0 never, 2 for every size the table allows.
    const int dyn_env = env_int("LORA_TC_EXPAND_DYNAMIC", 1);
    p.tickets = tickets;
    p.dyn = tickets != nullptr && rt_bound <= kMaxRt && dyn_env != 0 && (dyn_env == 2 || p.chunk >= 8);
    const int kbs = r_pad64 / kKB;
    // The row-tile table, then the rings: r_pad64 = 64: five y stages and one
    // v slice buffer, or four and two; r_pad64 = 128: fewer.  Large work items
    // (8 or more tiles) pay the v-slice load of one buffer rarely and gain
    // from the deeper ring; small ones keep the second buffer.  The deepest
    // form that fits beside the table and the kernel's own shared memory.
    const int table_entries = p.dyn ? static_cast<int>(rt_bound) : kMaxItems;
    p.table_bytes = (table_entries * static_cast<int>(sizeof(RowTile)) + 15) / 16 * 16;
    auto* kernel = p.dyn ? sgmv_expand_tc_kernel<true> : sgmv_expand_tc_kernel<false>;
    static size_t static_smem[2] = {0, 0}, smem_optin = 0;
    static int smem_device = -1;
    if (smem_device != dev) {
        cudaFuncAttributes fa0{}, fa1{};
        int optin = 0;
        if (cudaFuncGetAttributes(&fa0, sgmv_expand_tc_kernel<false>) != cudaSuccess ||
            cudaFuncGetAttributes(&fa1, sgmv_expand_tc_kernel<true>) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return cudaErrorInvalidValue;
        static_smem[0] = fa0.sharedSizeBytes;
        static_smem[1] = fa1.sharedSizeBytes;
        smem_optin = static_cast<size_t>(optin);
        smem_device = dev;
    }
    const size_t own_smem = static_smem[p.dyn ? 1 : 0];
    auto smem_of = [&](int st, int vb) {
        return static_cast<size_t>(p.table_bytes) + 1024 +
               static_cast<size_t>(vb * 2 * kbs + 2 * kbs + 2 * st) * kBoxBytes;
    };
    static const int kBig[][2] = {{5, 1}, {4, 1}, {3, 1}, {2, 1}};
    static const int kSmall[][2] = {{4, 2}, {3, 2}, {4, 1}, {3, 1}, {2, 1}};
    const bool big = p.chunk >= 8;
    const int n_forms = big ? 4 : 5;
    int stages = 2, vbufs = 1;
    const int st_env = env_int("LORA_TC_EXPAND_STAGES", 0);
    for (int f = 0; f < n_forms; ++f) {
        const int st = big ? kBig[f][0] : kSmall[f][0], vb = big ? kBig[f][1] : kSmall[f][1];
        if (kbs != 1 && vb != 1) continue;
        if (st_env > 0 && st != st_env) continue;
        if (own_smem + smem_of(st, vb) <= smem_optin) {
            stages = st;
            vbufs = vb;
            break;
        }
    }
    p.stages = stages;
    p.vbufs = vbufs;
    const size_t smem = smem_of(stages, vbufs);
    if (own_smem + smem > smem_optin) return cudaErrorInvalidValue;
    static int configured = -1;
    static size_t configured_bytes = 0;
    static int configured_dyn = -1;
    static size_t configured_bytes_dyn = 0;
    if (!(p.dyn ? configure_once(reinterpret_cast<const void*>(kernel), smem, configured_dyn, configured_bytes_dyn)
                : configure_once(reinterpret_cast<const void*>(kernel), smem, configured, configured_bytes)))
        return cudaErrorInvalidValue;
    // One CTA per SM (the shared memory allows no more), and enough CTAs that
    // none takes more than kMaxItems items.
    const long long items_bound = rt_bound * p.n_chunks;
    long long grid = env_int("LORA_TC_EXPAND_GRID", n_sms);
    if (!p.dyn) grid = std::max(grid, (items_bound + kMaxItems - 1) / kMaxItems);   // at most kMaxItems items per CTA
    grid = std::min(grid, items_bound);
    if (grid > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kExpandThreadsP);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = (flags & LORA_APPLY_NO_PDL) ? 0 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, mvh, mvl, my, mb[0], mb[1], mb[2], mb[3], p);
    note_launch();
    return e;
}

}  // namespace lora
