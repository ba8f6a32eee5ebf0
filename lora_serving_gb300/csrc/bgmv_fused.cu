// bgmv_fused.cu -- decode-row LoRA delta in one launch (the BGMV route of
// lora_apply): shrink, reduction of the fp32 intermediate and expand.
//
// TGI multi-LoRA page, "4. SGMV and BGMV at inference": decode tokens take
// BGMV, each token applying its own adapter.  Here the decode rows arrive
// grouped by adapter (the gather form of the batch metadata), so a unit of
// work is (adapter, up to 16 of its rows), and every adapter's weights are
// streamed from HBM once per call instead of once per token.
//
// Per unit, a thread-block cluster of CS CTAs splits the shrink's K = h_in:
//   CTA c computes partial v_c[t][j] = sum_{k in chunk c} A[j][k] x[t][k]
//   with mma.sync m16n8k16 (bf16 in, fp32 out: 16 rows x 8 ranks tiles).
// The partials meet in distributed shared memory: after a cluster barrier
// every CTA sums v = sum_c v_c in a fixed order (deterministic, fp32).  The
// expand of the CTA's own output columns runs on the tensor cores as well:
// v is split into v_hi = bf16(v) and v_lo = bf16(v - v_hi), so
//   d[t][col] = sum_j B'[col][j] (v_hi + v_lo)[t][j]
// carries v to ~2^-17 relative (v itself is never rounded to one bf16), and
// the last step is y[t][off_p + col] = bf16_rne(y + d).
//
// Data movement: A and x stream through a two-stage cp.async pipeline
// (16-byte copies, half a warp per 256-byte row piece); the CTA's slice of
// B' arrives by one bulk copy per projection (cp.async.bulk, completion
// counted on an mbarrier).  Waits on the mbarrier are bounded (0.2 s); a
// copy that does not land sets LORA_DEV_TIMEOUT and the CTA leaves its
// rows unwritten, while still taking part in every cluster barrier.
//
// Calls that stream many weights, or outputs wider than the clusters can
// expand in two tiles, take the two-launch form instead (bgmv_grouped.cu).
//
// Ordering (programmatic dependent launch): metadata and weights are read
// before griddepcontrol.wait, so they stream in while the preceding kernel
// on the stream is still running, and the CTA's y lines are prefetched into
// L2.  With LORA_APPLY_X_READY the shrink, the cluster reduction and the
// delta are formed before the wait as well, and only the read-modify-write
// of y follows it.

#include <cstdlib>

#include "decode_common.cuh"
#include "launch.h"

namespace lora {

namespace {

using namespace dec;

constexpr int kKT = 128;           // K elements per pipeline stage
constexpr int kPad = 8;            // bf16 padding per smem row: conflict-free ldmatrix
constexpr int kLds = kKT + kPad;
constexpr int kMaxStages = 3;      // K stages in flight: 2, or 3 for small calls whose K slice is 3 stages
constexpr int kMaxChunks = 128;    // output chunks (8 columns) per expand tile, at most
constexpr int kPartChunks = 64;    // column parts keep a CTA's chunks within two tiles of this
constexpr int kTileBBytes = 32768; // B' bytes per expand tile, at most
constexpr int kPermStage = 4096;   // decode positions staged in smem with the group table
constexpr int kBSlack = 32;        // zeroed bf16 after B' so padded-K fragments stay finite
constexpr int kDPad = 8;           // fp32 padding per delta-tile row: rows 8 banks apart

struct FusedParams {
    ProjSet ps;
    const bf16_t* x;
    int ld_x;
    int h_in;
    bf16_t* y;
    int ld_y;
    const int32_t* perm;      // absolute rows, grouped by slot
    const int32_t* gstarts;   // [n_groups+1] over positions of perm
    const int32_t* gslot;     // [n_groups]
    int n_groups;
    int n_pos;                // positions covered by perm
    int n_slots;
    int n_rows;
    int kc;                   // K elements per cluster rank (multiple of 16)
    int n_parts;              // column parts per unit
    int cs;                   // cluster size
    int nch_tile;             // chunks per expand tile (<= kMaxChunks, B' <= kTileBBytes)
    int r_pad;                // r_slot rounded up to 16 (expand mma K)
    int x_ready;              // x may be read before the grid dependency resolves
    int y_ready;              // y may be updated before it resolves
    unsigned stall_tx;        // test hook: extra bytes expected on the first B' tile (0 normally)
    int32_t* status;
};

// Output chunk (8 columns) -> projection and column within it.
__device__ __forceinline__ void chunk_proj(const ProjSet& ps, int ch, int& p, int& col0)
{
    p = 0;
    while (p < ps.n_proj - 1 && ch >= (ps.width[p] >> 3)) {
        ch -= ps.width[p] >> 3;
        ++p;
    }
    col0 = ch << 3;
}

struct SmemLayout {
    size_t a, x, vpart, vfull, b, perm, total;
};

__host__ __device__ inline size_t align128(size_t v) { return (v + 127) / 128 * 128; }

// sD (the delta tile, fp32) overlays the K stages of A and x: it is written
// only after every stage has been consumed.  Keeping the overlay tight lets
// three CTAs of a 3B-shaped q/k/v call (80 chunks, rank 16) share an SM.
__host__ __device__ inline SmemLayout smem_layout(int R, int r_slot, int nch_tile, int n_pos, int stages)
{
    SmemLayout L;
    const size_t sa = align128(sizeof(bf16_t) * stages * R * kLds);
    const size_t sx = align128(sizeof(bf16_t) * stages * kRB * kLds);
    const size_t sd = align128(sizeof(float) * kRB * (nch_tile * 8 + kDPad));
    L.a = 0;
    L.x = sa;
    L.vpart = sa + sx > sd ? sa + sx : sd;
    L.vfull = L.vpart + align128(sizeof(float) * kRB * R);
    L.b = L.vfull + align128(sizeof(float) * kRB * R);
    // the B' tile, and after the delta is formed, the y pieces being updated
    const size_t sb = sizeof(bf16_t) * (nch_tile * 8 * r_slot + kBSlack), sy = 16 * kRB * nch_tile;
    L.perm = L.b + align128(sb > sy ? sb : sy);
    L.total = L.perm + (n_pos <= kPermStage ? sizeof(int) * n_pos : 0);
    return L;
}

// kThreads = 256 for small calls, whose time is the chain of dependent
// latencies of each CTA; 128 for calls whose grid exceeds the resident
// slots, which more CTAs in flight serve better.  Registers are held to 64
// per thread (1024 threads per SM): in a chain of calls the next call's
// CTAs then find room beside the running ones (shared memory permitting:
// four CTAs of a 48 KB o-projection call), without spilling.
template <int kThreads, int kStages>
__global__ void __launch_bounds__(kThreads, 1024 / kThreads)
bgmv_fused_kernel(FusedParams p)
{
    constexpr int kWarps = kThreads / 32;
    constexpr int kTilesPerWarp = 16 / kWarps;   // shrink n-tiles of 8 ranks per warp (R <= 128)
    extern __shared__ __align__(128) unsigned char smem[];
    const int R = p.ps.n_proj * p.ps.r_slot;
    const int r_slot = p.ps.r_slot;
    const int r_pad = p.r_pad;
    const SmemLayout L = smem_layout(R, r_slot, p.nch_tile, p.n_pos, kStages);
    bf16_t* sA = reinterpret_cast<bf16_t*>(smem + L.a);        // [kStages][R][kLds]
    float* sD = reinterpret_cast<float*>(smem + L.a);          // [kRB][nch_tile*8 + kDPad], after the shrink
    bf16_t* sX = reinterpret_cast<bf16_t*>(smem + L.x);        // [kStages][kRB][kLds]
    float* vpart = reinterpret_cast<float*>(smem + L.vpart);   // [kRB][R]
    float* vfull = reinterpret_cast<float*>(smem + L.vfull);   // [kRB][R]
    bf16_t* sB = reinterpret_cast<bf16_t*>(smem + L.b);        // [nch_tile*8][r_slot] + slack
    int* s_perm = reinterpret_cast<int*>(smem + L.perm);
    __shared__ __align__(8) uint64_t s_barB;
    __shared__ int s_rows[kRB];
    __shared__ int s_cp[kMaxChunks];      // chunk -> projection
    __shared__ int s_ccol[kMaxChunks];    // chunk -> first column within its projection

    grid_dep_launch();

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int crank = static_cast<int>(cluster_rank());
    const int cluster = blockIdx.x / p.cs;
    const int unit = cluster / p.n_parts;
    const int part = cluster - unit * p.n_parts;
    const bool stage_perm = p.n_pos <= kPermStage;

    // Exits: CTA 0 of the grid always waits for the preceding grid before it
    // leaves, so this grid never completes before that one (stream order
    // stays transitive under PDL); status flags are written only after a
    // wait.  Clusters without work leave at once and free their SM slots.
    if (tid == 0) {   // the B' barrier, initialised while the group table is in flight
        mbar_init(&s_barB, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    const int grid_units = static_cast<int>(gridDim.x) / (p.cs * p.n_parts);
    const UnitInfo ui = find_unit<kThreads>(p, unit, s_perm, stage_perm, grid_units);   // uniform across the cluster
    const bool bad_group = ui.bad;
    const int pos0 = ui.pos0, nrows = ui.nrows, slot = ui.slot;
    if (!ui.found || slot == -1) {              // nothing to do (or base-only rows)
        if (blockIdx.x == 0 || bad_group) grid_dep_wait();
        if (bad_group && crank == 0 && part == 0 && tid == 0) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }
    if (slot < -1 || slot >= p.n_slots) {
        grid_dep_wait();
        if (crank == 0 && part == 0 && tid == 0) flag(p.status, LORA_DEV_SLOT_OUT_OF_RANGE);
        return;
    }
    // ---- this CTA's K range and output chunks ----
    const int k_begin = crank * p.kc;
    const int k_end = min(p.h_in, k_begin + p.kc);
    const int n_kt = k_end > k_begin ? (k_end - k_begin + kKT - 1) / kKT : 0;
    int total_ch = 0;
    for (int q = 0; q < p.ps.n_proj; ++q) total_ch += p.ps.width[q] >> 3;
    const int q_idx = part * p.cs + crank, q_n = p.n_parts * p.cs;
    // total_ch * q_n < 2^31: the launcher takes at most 2^24 chunks, q_n <= 128
    const int ch_begin = (total_ch * q_idx) / q_n;
    const int ch_end = (total_ch * (q_idx + 1)) / q_n;
    const int tile0_end = min(ch_end, ch_begin + p.nch_tile);

    auto map_chunks = [&](int c0, int c1) {
        for (int ci = tid; ci < c1 - c0; ci += kThreads) {
            int pj, col0;
            chunk_proj(p.ps, c0 + ci, pj, col0);
            s_cp[ci] = pj;
            s_ccol[ci] = col0;
        }
    };
    // Bytes of B' for chunks [c0, c1): 8 columns x r_slot each.
    auto b_bytes = [&](int c0, int c1) { return static_cast<unsigned>((c1 - c0) * 8 * r_slot * sizeof(bf16_t)); };
    // The expected bytes, then one bulk copy per projection segment of
    // chunks [c0, c1), all from thread 0 (no barrier needed between them).
    auto copy_B = [&](int c0, int c1, uint64_t* bar, unsigned extra) {
        if (tid == 0) {
            mbar_expect(bar, b_bytes(c0, c1) + extra);
            int pc0 = 0;
            for (int q = 0; q < p.ps.n_proj; ++q) {
                const int pc1 = pc0 + (p.ps.width[q] >> 3);
                const int s = max(c0, pc0), e = min(c1, pc1);
                if (s < e) {
                    const bf16_t* src = p.ps.B[q] + (static_cast<size_t>(slot) * p.ps.width[q] + (s - pc0) * 8) * r_slot;
                    bulk_g2s(sB + static_cast<size_t>(s - c0) * 8 * r_slot, src, b_bytes(s, e), bar);
                }
                pc0 = pc1;
            }
        }
    };
    // A rows (weights) for stage kt into buffer buf, 16 bytes per cp.async;
    // columns past k_end are zero-filled.
    auto copy_A = [&](int kt, int buf) {
        const int k0 = k_begin + kt * kKT;
        for (int i = tid; i < R * (kKT / 8); i += kThreads) {
            const int j = i / (kKT / 8), u = i - j * (kKT / 8);
            const int k = k0 + u * 8;
            const int pj = j / r_slot, jj = j - pj * r_slot;
            const bool ok = k < k_end;
            const bf16_t* src = p.ps.A[pj] + (static_cast<size_t>(slot) * r_slot + jj) * p.h_in + (ok ? k : 0);
            cp_async16(smem_u32(sA + (buf * R + j) * kLds + u * 8), src, ok);
        }
    };
    // x rows (gathered through perm); rows past nrows and columns past k_end are zero-filled.
    auto copy_X = [&](int kt, int buf) {
        const int k0 = k_begin + kt * kKT;
        for (int i = tid; i < kRB * (kKT / 8); i += kThreads) {
            const int t = i / (kKT / 8), u = i - t * (kKT / 8);
            const int k = k0 + u * 8;
            const bool ok = t < nrows && k < k_end;
            const bf16_t* src = p.x + (ok ? static_cast<size_t>(s_rows[t]) * p.ld_x + k : 0);
            cp_async16(smem_u32(sX + (buf * kRB + t) * kLds + u * 8), src, ok);
        }
    };

    // ---- weights first, as soon as the slot is known: they depend neither
    // on the rows nor on the preceding kernel ----
    if (ch_end > ch_begin) copy_B(ch_begin, tile0_end, &s_barB, p.stall_tx);
#pragma unroll
    for (int st = 0; st < kStages; ++st) {
        if (st < n_kt) copy_A(st, st);
        cp_async_commit();
    }

    // ---- rows, zero slack, chunk map ----
    bool bad_row = false;
    if (tid < kRB) {
        int r = 0;
        if (tid < nrows) {
            r = stage_perm ? s_perm[pos0 + tid] : __ldg(p.perm + pos0 + tid);
            if (r < 0 || r >= p.n_rows) { bad_row = true; r = 0; }
        }
        s_rows[tid] = r;
    }
    for (int i = tid; i < kBSlack / 8; i += kThreads)
        reinterpret_cast<uint4*>(sB + p.nch_tile * 8 * r_slot)[i] = make_uint4(0, 0, 0, 0);
    map_chunks(ch_begin, tile0_end);
    if (__syncthreads_or(bad_row)) {
        // A malformed permutation: flag it and leave this unit's rows alone.
        // Every CTA of the cluster reads the same entries, so all return here,
        // once the copies already issued have landed (bounded wait for B').
        cp_async_wait<0>();
        if (tid == 0 && ch_end > ch_begin) mbar_wait(&s_barB, 0);
        grid_dep_wait();
        if (tid == 0 && crank == 0 && part == 0) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }
    // The first tile's y lines go into L2 now: their addresses do not depend
    // on the preceding kernel and L2 is coherent with its writes, so the
    // read-modify-write after the grid dependency finds them there.  One
    // request per 128-byte line of each row (a 16-byte piece never spans two).
    {
        const int nch0 = tile0_end - ch_begin;
        for (int i = tid; i < nrows * nch0; i += kThreads) {
            const int t = i / nch0, ci = i - t * nch0;
            const bf16_t* yp = p.y + static_cast<size_t>(s_rows[t]) * p.ld_y + p.ps.out_off[s_cp[ci]] + s_ccol[ci];
            if (ci == 0 || (reinterpret_cast<uintptr_t>(yp) & 127) == 0) prefetch_l2(yp);
        }
    }

    bool waited = false;
    if (!p.x_ready) {
        grid_dep_wait();
        waited = true;
    }
#pragma unroll
    for (int st = 0; st < kStages; ++st) {
        if (st < n_kt) copy_X(st, st);
        cp_async_commit();
    }

    // ---- shrink: 16 rows x R ranks x this CTA's K range on tensor cores ----
    const int n_tiles = R / 8;                  // 8 ranks per mma tile; <= 16
    float acc[kTilesPerWarp][4] = {};
    for (int kt = 0; kt < n_kt; ++kt) {
        // groups so far: {A_0} {A_1} {X_0} {X_1}, then one per iteration;
        // stage kt is complete once at most one group is pending
        cp_async_wait<kStages - 1>();
        __syncthreads();
        const int buf = kt % kStages;
        const bf16_t* xs = sX + buf * kRB * kLds;
        const bf16_t* as = sA + buf * R * kLds;
#pragma unroll
        for (int ks = 0; ks < kKT / 16; ++ks) {
            const int mi = lane >> 3, mr = lane & 7;
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(smem_u32(xs + ((mi & 1) * 8 + mr) * kLds + ks * 16 + (mi >> 1) * 8), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < kTilesPerWarp; ++nt) {
                const int tile = warp + nt * kWarps;
                if (tile < n_tiles) {
                    uint32_t b0, b1;
                    const int l = lane & 15;
                    ldmatrix_x2(smem_u32(as + (tile * 8 + (l & 7)) * kLds + ks * 16 + (l >> 3) * 8), b0, b1);
                    mma_bf16_16816(acc[nt], a0, a1, a2, a3, b0, b1);
                }
            }
        }
        __syncthreads();                        // every warp is done with this buffer
        if (kt + kStages < n_kt) {              // refill it with stage kt + kStages
            copy_A(kt + kStages, buf);
            copy_X(kt + kStages, buf);
        }
        cp_async_commit();
    }
    cp_async_wait<0>();
    {
        const int gr = lane >> 2, q2 = (lane & 3) * 2;
#pragma unroll
        for (int nt = 0; nt < kTilesPerWarp; ++nt) {
            const int tile = warp + nt * kWarps;
            if (tile < n_tiles) {
                const int j = tile * 8 + q2;
                vpart[gr * R + j] = acc[nt][0];
                vpart[gr * R + j + 1] = acc[nt][1];
                vpart[(gr + 8) * R + j] = acc[nt][2];
                vpart[(gr + 8) * R + j + 1] = acc[nt][3];
            }
        }
    }
    __syncthreads();

    // ---- cluster reduction of the fp32 partials through DSMEM ----
    // (the shrink's copies are cp.async, whose waits always complete: every
    // peer's partials are valid here)
    cluster_arrive();
    cluster_wait();
    {
        // 16-byte pieces (R is a multiple of 8): with R <= 64 every thread
        // has at most one piece, so the peers' loads make one round trip;
        // eight peers' loads in flight at a time, summed in rank order.
        const int n4 = kRB * R / 4;   // all 16 rows: rows past nrows sum to zero
        const uint32_t base = smem_u32(vpart);
        for (int i = tid; i < n4; i += kThreads) {
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = 0; c0 < p.cs; c0 += 8) {
                float4 part4[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (c0 + c < p.cs) part4[c] = ld_dsmem_f4(map_rank(base + i * 16, c0 + c));
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if (c0 + c < p.cs) {
                        if (c0 + c == 0) {
                            s = part4[0];
                        } else {
                            s.x += part4[c].x;
                            s.y += part4[c].y;
                            s.z += part4[c].z;
                            s.w += part4[c].w;
                        }
                    }
                }
            }
            reinterpret_cast<float4*>(vfull)[i] = s;
        }
    }
    cluster_arrive();   // this CTA no longer reads its peers' partials
    bool failed = false;
    if (ch_end > ch_begin && !mbar_wait(&s_barB, 0)) failed = true;   // B' of the first tile
    failed = __syncthreads_or(failed);

    // ---- expand on tensor cores (16 rows x 8 columns per chunk), delta to sD ----
    const int gr = lane >> 2, q2 = (lane & 3) * 2;
    unsigned b_phase = 1;
    for (int c0 = ch_begin; c0 < ch_end; c0 += p.nch_tile) {
        const int c1 = min(ch_end, c0 + p.nch_tile);
        const int nch = c1 - c0;
        // After a timeout the barrier's phase never completed: it is not armed
        // again, and this CTA's remaining tiles are left alone (failed is
        // uniform across the CTA here).
        if (failed) break;
        if (c0 != ch_begin) {                   // later tiles: fresh chunk map and B'
            __syncthreads();
            map_chunks(c0, c1);
            fence_proxy_async();
            __syncthreads();
            copy_B(c0, c1, &s_barB, 0u);
            if (!mbar_wait(&s_barB, b_phase)) failed = true;
            b_phase ^= 1u;
            failed = __syncthreads_or(failed);
        }
        int cur_p = -1;
        uint32_t ahi[4][4], alo[4][4];   // v fragments of the current projection (r_pad <= 64)
        for (int ci = warp; ci < nch; ci += kWarps) {
            const int pj = s_cp[ci];
            if (pj != cur_p) {
                cur_p = pj;
                const float* vp = vfull + pj * r_slot;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (kk * 16 >= r_pad) break;   // K steps past the slot rank are never used
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        // a0: (row g, k 2q..), a1: (row g+8, k 2q..), a2: (row g, k 2q+8..), a3: (row g+8, k 2q+8..)
                        const int row = gr + (h & 1) * 8;
                        const int k = kk * 16 + q2 + (h >> 1) * 8;
                        float v0 = 0.f, v1 = 0.f;
                        if (k < r_slot) {
                            v0 = vp[row * R + k];
                            v1 = vp[row * R + k + 1];
                        }
                        split_hi_lo(v0, v1, ahi[kk][h], alo[kk][h]);
                    }
                }
            }
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const bf16_t* bc = sB + ci * 8 * r_slot;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (kk * 16 < r_pad) {
                    uint32_t b0, b1;
                    const int l = lane & 15;
                    ldmatrix_x2(smem_u32(bc + (l & 7) * r_slot + kk * 16 + (l >> 3) * 8), b0, b1);
                    mma_bf16_16816(d, ahi[kk][0], ahi[kk][1], ahi[kk][2], ahi[kk][3], b0, b1);
                    mma_bf16_16816(d, alo[kk][0], alo[kk][1], alo[kk][2], alo[kk][3], b0, b1);
                }
            }
            // d: (row g, cols 2q, 2q+1) and (row g+8, same cols) of chunk ci
            const int ld_d = nch * 8 + kDPad;
            *reinterpret_cast<float2*>(sD + gr * ld_d + ci * 8 + q2) = make_float2(d[0], d[1]);
            *reinterpret_cast<float2*>(sD + (gr + 8) * ld_d + ci * 8 + q2) = make_float2(d[2], d[3]);
        }
        __syncthreads();
        if (!waited && !p.y_ready) {
            grid_dep_wait();   // y may be the preceding kernel's output
            waited = true;
        }
        // ---- read-modify-write of y: 16-byte pieces, coalesced along each row.
        // All of a thread's pieces are requested at once (cp.async into the
        // B' region, free once the delta is formed): one round trip. ----
        if (!failed) {
            uint4* sY = reinterpret_cast<uint4*>(sB);
            for (int i = tid; i < nrows * nch; i += kThreads) {
                const int t = i / nch, ci = i - t * nch;
                cp_async16(smem_u32(sY + i),
                           p.y + static_cast<size_t>(s_rows[t]) * p.ld_y + p.ps.out_off[s_cp[ci]] + s_ccol[ci], true);
            }
            cp_async_commit();
            cp_async_wait<0>();   // each thread reads back only its own pieces
            for (int i = tid; i < nrows * nch; i += kThreads) {
                const int t = i / nch, ci = i - t * nch;
                const float4* dp = reinterpret_cast<const float4*>(sD + t * (nch * 8 + kDPad) + ci * 8);
                const float4 d0 = dp[0], d1 = dp[1];
                const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                *reinterpret_cast<uint4*>(p.y + static_cast<size_t>(s_rows[t]) * p.ld_y + p.ps.out_off[s_cp[ci]] +
                                          s_ccol[ci]) = add_round8(sY[i], dd);
            }
        }
    }
    // With LORA_APPLY_Y_READY only CTA 0 (and CTAs with a flag to write) wait
    // here: enough to keep this grid from completing before the preceding one.
    if (!waited && (blockIdx.x == 0 || bad_group || failed)) grid_dep_wait();
    if (tid == 0) {
        if (bad_group && crank == 0 && part == 0) flag(p.status, LORA_DEV_BAD_SEGMENT);
        if (failed) flag(p.status, LORA_DEV_TIMEOUT);
    }
    cluster_wait();     // peers are done reading this CTA's partials
}

// Cluster size of the one-launch form: split K over up to 8 CTAs while each
// keeps >= one stage (8 measured faster than 16 on the 3B decode shapes:
// smaller grids let more consecutive calls be resident at once under PDL);
// 16 for long K.
int fused_cluster_size(int h_in)
{
    int cs = 1;
    const int cs_max = h_in >= 8192 ? 16 : 8;
    while (cs < cs_max && h_in / (cs * 2) >= kKT) cs *= 2;
    return env_int("LORA_FUSED_CS", cs);
}

int total_chunks(const ProjSet& ps)
{
    int total_ch = 0;
    for (int q = 0; q < ps.n_proj; ++q) total_ch += ps.width[q] / 8;
    return total_ch;
}

// Column parts per unit (more clusters, each recomputing the shrink from
// L2) so that each CTA expands at most two tiles of kPartChunks chunks.
int fused_parts(int total_ch, int cs)
{
    int parts = 1;
    while (parts < 8 && (total_ch + cs * parts - 1) / (cs * parts) > 2 * kPartChunks) parts *= 2;
    return env_int("LORA_FUSED_PARTS", parts);
}

}  // namespace

bool fused_decode_supported(int n_proj, int r_slot)
{
    // <= 2 rank tiles of 8 per warp in the shrink; <= 4 K steps of 16 in the expand
    return r_slot <= 64 && n_proj * r_slot <= 2 * 8 * 8 && r_slot % 8 == 0;
}

bool decode_two_launch(const ProjSet& ps, int h_in, int n_groups)
{
    const int forced = env_int("LORA_DECODE_TWO_LAUNCH", -1);
    if (forced >= 0) return forced != 0;
    // Outputs wider than one launch's clusters expand in two tiles, and calls
    // that stream many weights: the one-launch form keeps two K stages in
    // flight per CTA and expands in the same CTAs, the two-launch form
    // streams A and B' in long runs from many small CTAs.
    const int total_ch = total_chunks(ps);
    if (fused_parts(total_ch, fused_cluster_size(h_in)) > 1) return true;
    const double weight_bytes = static_cast<double>(n_groups) * sizeof(bf16_t) *
                                (static_cast<double>(ps.n_proj) * ps.r_slot * h_in + 8.0 * total_ch * ps.r_slot);
    return weight_bytes >= 32.0 * (1 << 20);
}

cudaError_t launch_bgmv_fused(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                              const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                              int n_pos, int max_group_len, int n_rows, int n_slots, unsigned flags,
                              int32_t* status, cudaStream_t stream)
{
    if (n_pos <= 0 || n_groups <= 0) return cudaSuccess;
    if (total_chunks(ps) > (1 << 24)) return cudaErrorInvalidValue;   // > 128M output columns
    const int R = ps.n_proj * ps.r_slot;
    static int configured_device = -1;
    static int n_sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        for (auto fn : {bgmv_fused_kernel<128, 2>, bgmv_fused_kernel<256, 2>, bgmv_fused_kernel<256, 3>}) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
            if (e != cudaSuccess) return e;
            e = prefer_max_shared(reinterpret_cast<const void*>(fn));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int cs = fused_cluster_size(h_in);
    // Units of <= 16 rows: at most ceil(longest group / 16) per group.
    int max_units = n_groups + n_pos / kRB;
    if (max_group_len > 0) max_units = min(max_units, n_groups * ((max_group_len + kRB - 1) / kRB));
    const int total_ch = total_chunks(ps);
    const int parts = fused_parts(total_ch, cs);
    const int per_cta = (total_ch + cs * parts - 1) / (cs * parts);
    const long long n_ctas = static_cast<long long>(max_units) * parts * cs;
    const int threads = env_int("LORA_FUSED_THREADS", n_ctas > 2LL * n_sms ? 128 : 256) == 128 ? 128 : 256;
    // Small calls (256 threads): one tile when the B' slice fits, since a
    // second tile would put its B' copy and delta behind the grid
    // dependency.  Large grids (128 threads): tiles of kPartChunks, so four
    // CTAs' shared memory fits on an SM.
    const int tile_cap = threads == 256 ? min(kMaxChunks, kTileBBytes / (16 * ps.r_slot)) : kPartChunks;
    const int nch_tile = min(tile_cap, max(1, per_cta));
    const int kc = ((h_in + cs - 1) / cs + 15) / 16 * 16;
    // Two K stages in flight.  Three (the whole K slice of a 3B-shaped call
    // in one round trip) shorten one call alone a little, but the larger
    // shared-memory footprint lets fewer CTAs of consecutive calls overlap
    // (LORA_FUSED_STAGES=3 selects it for small calls).
    const int n_kt = (kc + kKT - 1) / kKT;
    const int stages = env_int("LORA_FUSED_STAGES", 2) == kMaxStages && threads == 256 && n_kt <= kMaxStages
                           ? kMaxStages : 2;

    FusedParams p{};
    p.ps = ps;
    p.x = x;
    p.ld_x = ld_x;
    p.h_in = h_in;
    p.y = y;
    p.ld_y = ld_y;
    p.perm = perm;
    p.gstarts = gstarts;
    p.gslot = gslot;
    p.n_groups = n_groups;
    p.n_pos = n_pos;
    p.n_slots = n_slots;
    p.n_rows = n_rows;
    p.kc = kc;
    p.n_parts = parts;
    p.cs = cs;
    p.nch_tile = nch_tile;
    p.r_pad = (ps.r_slot + 15) / 16 * 16;
    p.x_ready = (flags & LORA_APPLY_X_READY) ? 1 : 0;
    p.y_ready = (flags & LORA_APPLY_Y_READY) ? 1 : 0;
    p.stall_tx = test_stall_bytes(kStallFusedDecode);
    p.status = status;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_ctas));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem_layout(R, ps.r_slot, nch_tile, n_pos, stages).total;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = cs;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
    if (!(flags & LORA_APPLY_NO_PDL)) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    e = threads == 128  ? cudaLaunchKernelEx(&cfg, bgmv_fused_kernel<128, 2>, p)
        : stages == 2   ? cudaLaunchKernelEx(&cfg, bgmv_fused_kernel<256, 2>, p)
                        : cudaLaunchKernelEx(&cfg, bgmv_fused_kernel<256, 3>, p);
    note_launch();
    return e;
}

}  // namespace lora
