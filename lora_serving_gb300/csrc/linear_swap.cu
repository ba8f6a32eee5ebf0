// linear_swap.cu -- the LoRA linear layer for decode-sized batches (at most
// 64 rows): the base projection with every row's adapter delta in the same
// fp32 accumulator, rounded to bf16 once.
//
// Multi-LoRA serving note, "direct answer": the base product W x runs once
// for the whole batch and each row adds its own adapter's B(A x); TGI
// multi-LoRA page, "implementation": the LoRA linear layer adds the adapter
// output to the base layer's output.  For projection p (rows [off_p, off_p +
// w_p) of the stacked W) and every row t of the batch:
//   y[t][off_p + c] = bf16_rne( sum_k W[off_p + c][k] x[t][k]
//                               + sum_j B'_{p,id_t}[c][j] v_{p,t}[j] )
// with v = A x from the shrink kernels, stored as bf16 planes v_hi + v_lo.
//
// With few rows the weights are the bytes, so the tile is turned around:
// 128 output columns (W rows) form the MMA's M operand and the batch rows
// its N (tensor memory holds 128 x N fp32), and W streams through every SM
// once.  A cluster of cs CTAs shares a column tile, each taking a slice of
// K.  The delta is a K extension of the same accumulator: for each adapter
// slot present in the batch (shared out round-robin over the cluster), one
// step brings that slot's B' box (128 columns x 64 ranks) and the v_hi and
// v_lo boxes of projection p for all rows; the MMA warp zeroes the v rows of
// rows that name another adapter (whole 128-byte rows of the swizzled
// boxes) before it issues B' x v_hi^T and B' x v_lo^T.  The fp32 partials
// are stored transposed ([row][column]) in shared memory and meet over
// distributed shared memory: each CTA sums its share of the columns over
// the cluster in rank order, rounds, and writes whole 16-byte pieces of y.
//   warp 0: TMA producer   warp 1: masks v and issues the MMAs
//   warps 2..5: read the accumulator out
// Under programmatic dependent launch the base steps (x, W) run while the
// shrink that produces v finishes; the adapter steps, y and the status word
// follow the grid dependency.
// Every wait is bounded (0.2 s); a timeout sets LORA_DEV_TIMEOUT, the CTA
// writes nothing, its producer lets every copy it issued land, and the
// tensor memory is freed.

#include <algorithm>

#include "launch.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace lora {

namespace {

using namespace tc;

constexpr int kSwM = 128;                    // output columns per tile (tensor-memory lanes)
constexpr int kSwK = 64;                     // K elements per step (one 128-byte swizzled row)
constexpr int kSwMaxN = 64;                  // batch rows, at most
constexpr int kSwStages = 3;                 // 97 KB: two CTAs per SM
constexpr int kSwABytes = kSwM * 128;        // W or B' box
constexpr int kSwBBytes = kSwMaxN * 128;     // x, v_hi or v_lo box (room for 64 rows)
constexpr int kSwStageBytes = kSwABytes + 2 * kSwBBytes;
constexpr int kSwThreads = 192;              // 6 warps
constexpr int kSwMaxSplit = 8;
constexpr int kSwRedPitch = kSwM + 4;        // fp32 pitch of the transposed partial
constexpr int kScanBar = 1;                  // named barrier: warp 1's group scan -> the producer's adapter steps

struct SwapParams {
    int n_proj, r_slot, n_slots, n_rows, n_pad;   // n_pad: rows rounded up to 16 (the MMA N)
    int h_in, n_kb;
    int out_off[LORA_MAX_PROJ];
    int width[LORA_MAX_PROJ];
    int ntiles[LORA_MAX_PROJ];   // 128-column tiles per projection
    int w_row[LORA_MAX_PROJ];    // first W row of projection p
    int cs;                      // cluster size (K split)
    const int32_t* ids;
    bf16_t* y;
    int ld_y;
    int32_t* status;
};

// Column tile -> projection and its first column.
__device__ __forceinline__ void swap_tile(const SwapParams& P, int tile, int& p, int& col0)
{
    p = 0;
    while (p < P.n_proj - 1 && tile >= P.ntiles[p]) {
        tile -= P.ntiles[p];
        ++p;
    }
    col0 = tile * kSwM;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* ptr)
{
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ptr) + 1023) & ~static_cast<uintptr_t>(1023));
}

__global__ void __launch_bounds__(kSwThreads, 1)
linear_swap_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                   const __grid_constant__ CUtensorMap mvh, const __grid_constant__ CUtensorMap mvl,
                   const __grid_constant__ CUtensorMap mb0, const __grid_constant__ CUtensorMap mb1,
                   const __grid_constant__ CUtensorMap mb2, const __grid_constant__ CUtensorMap mb3, SwapParams P)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kSwStages], empty[kSwStages], done, recv_bar;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_fail;
    __shared__ int s_slot[kSwMaxN];                 // this CTA's adapter slots (LoRA steps)
    __shared__ unsigned long long s_mask[kSwMaxN];  // rows of each of them
    __shared__ int s_ngroups, s_badid;
    __shared__ int s_peer_fail[kSwMaxSplit];        // the cluster's failure flags, written by each CTA
    // Programmatic dependent launch: x, W, B' and the ids are read at once
    // (none is written by the shrink before this kernel), the base steps
    // run while the shrink finishes; v, y and the status word wait for it.
    grid_dep_launch();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int crank = P.cs > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int tile = blockIdx.x / P.cs;
    int p, col0;
    swap_tile(P, tile, p, col0);
    const int ncols = min(kSwM, P.width[p] - col0);
    const CUtensorMap* bmap = p == 0 ? &mb0 : p == 1 ? &mb1 : p == 2 ? &mb2 : &mb3;   // projection p's B' store
    uint8_t* ring = align1024(smem_raw);

    // K blocks of this CTA; adapter slots present in the batch, in order of
    // first appearance, the g-th taken by cluster rank g % cs
    const int kb0 = crank * P.n_kb / P.cs;
    const int n_base = (crank + 1) * P.n_kb / P.cs - kb0;
    // tile columns [c_lo, c_hi) are summed over the cluster by this CTA: 8
    // columns (one 16-byte piece of y) at a time, the 16 pieces shared out
    // as evenly as cs allows
    const int c_lo = crank * (kSwM / 8) / P.cs * 8, c_hi = (crank + 1) * (kSwM / 8) / P.cs * 8;
    const int n_own = c_hi - c_lo;
    const uint32_t b_bytes = static_cast<uint32_t>(P.n_pad) * 128;

    // ---- producer (warp 0, lane 0): the base steps (W box + x box) at
    // once, the first ring's worth before the tensor memory is allocated;
    // then, once warp 1 has scanned the groups, the LoRA steps (B' box + v
    // boxes) ----
    int issued = 0;
    auto issue = [&](int i) -> bool {
        const int s = i % kSwStages;
        if (i >= kSwStages && !mbar_wait_spin(&empty[s], ((i / kSwStages) - 1) & 1)) return false;
        uint8_t* st = ring + s * kSwStageBytes;
        if (i < n_base) {
            const int k = (kb0 + i) * kSwK;
            mbar_expect_tx(&full[s], kSwABytes + b_bytes);
            tma_load_2d(st, &mw, k, P.w_row[p] + col0, &full[s]);
            tma_load_2d(st + kSwABytes, &mx, k, 0, &full[s]);
        } else {
            if (i == n_base) grid_dep_wait();   // v is the preceding kernel's output
            const int g = i - n_base;
            mbar_expect_tx(&full[s], kSwABytes + 2 * b_bytes);
            tma_load_2d(st, bmap, 0, s_slot[g] * P.width[p] + col0, &full[s]);
            tma_load_3d(st + kSwABytes, &mvh, 0, p, 0, &full[s]);
            tma_load_3d(st + kSwABytes + kSwBBytes, &mvl, 0, p, 0, &full[s]);
        }
        issued = i + 1;
        return true;
    };
    if (tid == 0) {
        for (int s = 0; s < kSwStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        mbar_init(&recv_bar, 1);
        mbar_init_fence();
        // the partials of this CTA's columns, from every CTA of the cluster
        if (P.cs > 1) mbar_expect_tx(&recv_bar, static_cast<unsigned>(P.cs * n_own * P.n_pad) * 4u);
        s_fail = 0;
        for (int i = 0; i < min(n_base, kSwStages); ++i) issue(i);   // no wait: the ring is empty
    }
    if (warp == 0) tmem_alloc(&s_tmem, kSwMaxN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        bool ok = true;
        if (lane == 0)
            for (int i = issued; i < n_base && ok && !s_fail; ++i) ok = issue(i);
        __syncwarp();
        // warp 1 has arrived after its group scan (it does not wait here: it
        // goes on to consume the base steps)
        named_barrier(kScanBar, 64);
        if (lane == 0) {
            const int n_steps = n_base + s_ngroups;
            for (int i = n_base; i < n_steps && ok && !s_fail; ++i) ok = issue(i);
            if (!ok) s_fail = 1;
            // every copy issued lands before the CTA moves on
            for (int i = issued > kSwStages ? issued - kSwStages : 0; i < issued; ++i)
                if (!mbar_wait(&full[i % kSwStages], (i / kSwStages) & 1)) s_fail = 1;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- group scan: lanes own rows lane and lane + 32; a row opens a
        // group if its slot is valid and no earlier row names it; group g
        // (in order of first appearance) goes to cluster rank g % cs, with
        // the mask of every row that names its slot ----
        {
            int idv[2];
            bool first[2], bad = false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int t = lane + 32 * h;
                idv[h] = t < P.n_rows ? __ldg(P.ids + t) : -1;
                bad |= t < P.n_rows && (idv[h] < -1 || idv[h] >= P.n_slots);
            }
            // rows of each half naming the same slot as this lane's row
            unsigned same[2][2];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    unsigned m = 0;
                    for (int u = 0; u < 32; ++u) m |= (__shfl_sync(0xFFFFFFFFu, idv[hh], u) == idv[h]) ? (1u << u) : 0u;
                    same[h][hh] = m;
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const bool valid = idv[h] >= 0 && idv[h] < P.n_slots;
                const unsigned long long m = static_cast<unsigned long long>(same[h][0]) |
                                             (static_cast<unsigned long long>(same[h][1]) << 32);
                const int t = lane + 32 * h;
                first[h] = valid && (m & ((1ull << t) - 1ull)) == 0;
            }
            const unsigned long long F = static_cast<unsigned long long>(__ballot_sync(0xFFFFFFFFu, first[0])) |
                                         (static_cast<unsigned long long>(__ballot_sync(0xFFFFFFFFu, first[1])) << 32);
            const bool any_bad = __any_sync(0xFFFFFFFFu, bad);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int t = lane + 32 * h;
                if (!first[h]) continue;
                const int g = __popcll(F & ((1ull << t) - 1ull));
                if (g % P.cs != crank) continue;
                const unsigned long long rows_mask = (static_cast<unsigned long long>(same[h][0]) |
                                                      (static_cast<unsigned long long>(same[h][1]) << 32)) &
                                                     (P.n_rows >= 64 ? ~0ull : ((1ull << P.n_rows) - 1ull));
                s_slot[g / P.cs] = idv[h];
                s_mask[g / P.cs] = rows_mask;
            }
            if (lane == 0) {
                const int G = __popcll(F);
                s_ngroups = G > crank ? (G - crank + P.cs - 1) / P.cs : 0;
                s_badid = any_bad ? 1 : 0;
            }
            __syncwarp();
        }
        named_barrier_arrive(kScanBar, 64);   // the producer may issue the adapter steps
        // ---- MMA warp: masks the v boxes of a LoRA step, lane 0 issues ----
        const uint32_t idesc = idesc_bf16_f32(kSwM, P.n_pad);
        const int n_steps = n_base + s_ngroups;
        bool ok = true, acc = false;
        for (int i = 0; i < n_steps && ok; ++i) {
            const int s = i % kSwStages;
            // lane 0 waits for the stage; the warp follows its answer together
            int landed = 1;
            if (lane == 0) landed = mbar_wait_spin(&full[s], (i / kSwStages) & 1) ? 1 : 0;
            landed = __shfl_sync(0xFFFFFFFFu, landed, 0);
            __syncwarp();
            if (!landed) {
                ok = false;
                break;
            }
            uint8_t* st = ring + s * kSwStageBytes;
            if (i >= n_base) {
                // zero the 128-byte rows of rows that name another adapter
                // (the swizzle permutes 16-byte pieces within a row only)
                const unsigned long long m = s_mask[i - n_base];
                for (int t = lane; t < P.n_pad; t += 32)
                    if (!((m >> t) & 1ull)) {
                        uint4* rh = reinterpret_cast<uint4*>(st + kSwABytes + t * 128);
                        uint4* rl = reinterpret_cast<uint4*>(st + kSwABytes + kSwBBytes + t * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            rh[c] = make_uint4(0, 0, 0, 0);
                            rl[c] = make_uint4(0, 0, 0, 0);
                        }
                    }
                fence_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                tc_fence_after();
                const uint32_t a = smem_u32(st), b1 = a + kSwABytes, b2 = b1 + kSwBBytes;
                const int planes = i < n_base ? 1 : 2;
                for (int pl = 0; pl < planes; ++pl)
#pragma unroll
                    for (int ks = 0; ks < kSwK / 16; ++ks) {
                        mma_bf16(tmem, sdesc_sw128(a + ks * 32), sdesc_sw128((pl ? b2 : b1) + ks * 32), idesc, acc);
                        acc = true;
                    }
                mma_commit(&empty[s]);   // frees the stage once these MMAs have read it
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (!ok) s_fail = 1;
            mma_commit(&done);
        }
        __syncwarp();
    }

    // ---- epilogue: each column's fp32 partial (accumulator lane = column,
    // accumulator column = row) goes to the CTA that sums that column over
    // the cluster; it lands in that CTA's ring, idle once the cluster
    // barrier below has passed ----
    bool ok = mbar_wait(&done, 0);
    tc_fence_after();
    ok = __syncthreads_and(ok && !s_fail);
    const bool has_steps = n_base + s_ngroups > 0;   // an accumulator with no MMA is left unwritten
    if (tid == 0 && !ok) s_fail = 1;
    __syncthreads();
    // this CTA's failure flag into every peer's s_peer_fail[crank]: the
    // cluster barrier publishes them, so the check below reads local memory
    if (tid < P.cs) {
        if (P.cs > 1)
            st_dsmem_u32(map_rank(smem_u32(&s_peer_fail[crank]), tid), s_fail);
        else
            s_peer_fail[0] = s_fail;
    }
    if (P.cs > 1) {
        cluster_arrive();
        cluster_wait();
    }
    // receive buffer of every CTA: [source rank][own column][row] fp32
    float* recv = reinterpret_cast<float*>(ring);
    if (warp >= 2) {
        const int quarter = warp & 3;               // the tensor-memory lanes this warp may read
        const int c = quarter * 32 + lane;          // tile column
        int r = 0;                                  // the CTA that sums column c
        while (r + 1 < P.cs && c >= (r + 1) * (kSwM / 8) / P.cs * 8) ++r;
        const int lo_r = r * (kSwM / 8) / P.cs * 8, n_r = (r + 1) * (kSwM / 8) / P.cs * 8 - lo_r;
        const int off = (crank * n_r + (c - lo_r)) * P.n_pad;
        const uint32_t dst = P.cs > 1 ? map_rank(smem_u32(recv + off), r) : 0u;
        const uint32_t bar = P.cs > 1 ? map_rank(smem_u32(&recv_bar), r) : 0u;
        for (int j0 = 0; j0 < P.n_pad; j0 += 16) {
            float d[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + j0, d);
#pragma unroll
            for (int j = 0; j < 16; ++j) d[j] = (has_steps && ok) ? d[j] : 0.f;
            if (P.cs > 1) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    st_async_f4(dst + 4u * static_cast<uint32_t>(j0 + 4 * q4), d[4 * q4], d[4 * q4 + 1], d[4 * q4 + 2],
                                d[4 * q4 + 3], bar);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) recv[off + j0 + j] = d[j];
            }
        }
    }
    grid_dep_wait();   // y and the status word are touched only after the preceding grid has completed
    bool got = true;
    if (P.cs > 1)
        got = mbar_wait(&recv_bar, 0);
    else
        __syncthreads();
    // a failed peer has no valid partial: then nothing of the tile is written
    bool all_ok = got;
    for (int r = 0; r < P.cs; ++r)
        if (s_peer_fail[r]) all_ok = false;
    // rows fastest across the threads (conflict-free reads of recv); the
    // sources are summed in rank order
    const int per_row = n_own / 8;
    for (int it = tid; it < P.n_rows * per_row; it += kSwThreads) {
        const int piece = it / P.n_rows, t = it - piece * P.n_rows;
        const int lc = piece * 8;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int src = 0; src < P.cs; ++src) {
            const float* rp = recv + (src * n_own + lc) * P.n_pad + t;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] += rp[e * P.n_pad];
        }
        if (all_ok && c_lo + lc < ncols) {
            uint4 o;
            o.x = pack_bf16x2(v[0], v[1]);
            o.y = pack_bf16x2(v[2], v[3]);
            o.z = pack_bf16x2(v[4], v[5]);
            o.w = pack_bf16x2(v[6], v[7]);
            *reinterpret_cast<uint4*>(P.y + static_cast<size_t>(t) * P.ld_y + P.out_off[p] + col0 + c_lo + lc) = o;
        }
    }
    // no peer reads this CTA's memory, and every write into it has landed
    // (the receive barrier): the CTA may leave without a second cluster barrier
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kSwMaxN);
    if (tid == 0) {
        if (!all_ok && s_fail) flag(P.status, LORA_DEV_TIMEOUT);
        if (!got) flag(P.status, LORA_DEV_TIMEOUT);
        if (s_badid && tile == 0 && crank == 0) flag(P.status, LORA_DEV_SLOT_OUT_OF_RANGE);
    }
}

size_t swap_smem() { return static_cast<size_t>(kSwStages) * kSwStageBytes + 1024; }

}  // namespace

bool linear_swap_supported(int n_rows, int r_slot) { return n_rows >= 1 && n_rows <= kSwMaxN && r_slot <= kSwK; }

cudaError_t launch_linear_swap(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const bf16_t* W, int ld_w,
                               int n_out, const ProjSet& ps, const bf16_t* vh, const bf16_t* vl, const int32_t* ids,
                               int n_rows, int n_slots, int32_t* status, cudaStream_t stream)
{
    if (n_rows <= 0) return cudaSuccess;
    if (!linear_swap_supported(n_rows, ps.r_slot)) return cudaErrorInvalidValue;
    SwapParams P{};
    P.n_proj = ps.n_proj;
    P.r_slot = ps.r_slot;
    P.n_slots = n_slots;
    P.n_rows = n_rows;
    P.n_pad = (n_rows + 15) / 16 * 16;
    P.h_in = h_in;
    P.n_kb = (h_in + kSwK - 1) / kSwK;
    P.ids = ids;
    P.y = y;
    P.ld_y = ld_y;
    P.status = status;
    const int ld_p = ps.n_proj * ((ps.r_slot + kSwK - 1) / kSwK * kSwK);
    CUtensorMap mx, mw, mvh, mvl, mb[4];
    // boxes of n_pad rows: rows past the batch read as zero
    if (!encode_tmap_bf16(&mx, x, n_rows, h_in, ld_x, P.n_pad, kSwK, true) ||
        !encode_tmap_bf16(&mw, W, n_out, h_in, ld_w, kSwM, kSwK, true) ||
        !encode_tmap_bf16_3d(&mvh, vh, ps.r_slot, ps.n_proj, n_rows, kSwK, ld_p, kSwK, P.n_pad) ||
        !encode_tmap_bf16_3d(&mvl, vl, ps.r_slot, ps.n_proj, n_rows, kSwK, ld_p, kSwK, P.n_pad))
        return cudaErrorInvalidValue;
    int n_ct = 0, w_row = 0;
    for (int q = 0; q < 4; ++q) {
        const int src = q < ps.n_proj ? q : 0;
        if (!encode_tmap_bf16(&mb[q], ps.B[src], static_cast<uint64_t>(n_slots) * ps.width[src], ps.r_slot, ps.r_slot,
                              kSwM, kSwK, true))
            return cudaErrorInvalidValue;
        if (q < ps.n_proj) {
            P.out_off[q] = ps.out_off[q];
            P.width[q] = ps.width[q];
            P.ntiles[q] = (ps.width[q] + kSwM - 1) / kSwM;
            P.w_row[q] = w_row;
            w_row += ps.width[q];
            n_ct += P.ntiles[q];
        }
    }
    static int configured_device = -1, n_sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(linear_swap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(swap_smem()));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(linear_swap_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        e = prefer_max_shared(reinterpret_cast<const void*>(linear_swap_kernel));
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    // Split K so the column tiles' clusters cover the SMs (two CTAs fit on
    // an SM), each CTA keeping at least two K blocks.  (One CTA per SM with
    // a six-stage ring, splits of 3 and 6 filling the SMs once, was slower:
    // 57 against 43 us per Llama-3.2-3B decode layer.)
    int cs = 1;
    while (cs < kSwMaxSplit && static_cast<long long>(n_ct) * cs < n_sms && P.n_kb >= 4 * cs) cs *= 2;
    cs = std::max(1, std::min({env_int("LORA_SWAP_SPLIT", cs), kSwMaxSplit, P.n_kb}));
    P.cs = cs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_ct * cs));
    cfg.blockDim = dim3(kSwThreads);
    cfg.dynamicSmemBytes = swap_smem();
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, linear_swap_kernel, mx, mw, mvh, mvl, mb[0], mb[1], mb[2], mb[3], P);
    note_launch();
    return e;
}

}  // namespace lora
