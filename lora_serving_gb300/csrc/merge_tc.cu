// merge_tc.cu -- merge / unmerge on the 5th-generation tensor cores, for slot
// ranks up to 64.
//
// Multi-LoRA serving note, "interviewer follow-ups": merging W' = W + B A
// gives the same model as the base plus the adapter's delta.  Here
//   W[o][k] <- bf16_rne(W[o][k] + sign * sum_j B'[o][j] A[j][k])
// in place, the sum in fp32 over the slot rank (padding ranks are zero).
//
// A persistent kernel, one CTA per SM.  The tiles (128 x 128 of W) are
// ordered weight by weight, and within a weight row block by row block, each
// row block's column strips in order; CTA b takes tiles b, b + G, b + 2G, ...
// (G CTAs), so at any moment the CTAs work on neighbouring tiles.  Per tile,
// TMA brings the W tile (two 128 x 64 boxes, from HBM) into a four-stage W
// ring, and B' rows o0..o0+127 (one box: the MMA's A operand, K-major) with
// A[0:64][k0:k0+128] (two boxes; both from L2) into a two-stage operand
// ring.  The MMA's B operand is A^T, which two warps build from the staged A
// in the K-major swizzled layout.  tcgen05.mma forms D = B' A (M = 128,
// N = 128, K = 64) into one of two tensor-memory accumulators, and its
// completion frees the operand stage.  Eight epilogue warps add sign * D into
// the staged W tile in place with one rounding; a store warp writes the tile
// back by TMA and frees the W stage once the store has read it.  The W ring
// is what bounds the rate: a stage is held from its load through the store,
// so the operands, which are done much sooner, live in their own ring.
//   warp 0: TMA producer   warp 1: MMA issuer   warps 2-3: transpose A
//   warps 4-11: epilogue (tensor-memory lane quarter = warp % 4; warps 4-7
//               the tile's first 64 columns, 8-11 the second)
//   warp 12: TMA store
// HBM-bound: W is read and written once; A and B' come from L2.  Every wait
// is bounded (0.2 s).  On a timeout the CTA sets its failure flag and
// stores nothing more; its producer lets every copy it issued land, and the
// tensor memory is freed once the MMAs issued have completed.

#include <algorithm>

#include "launch.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace lora {

namespace {

using namespace tc;

constexpr int kGm = 128;                     // W rows per tile (MMA M)
constexpr int kGn = 128;                     // W columns per tile (MMA N)
constexpr int kGk = 64;                      // ranks (MMA K): slot ranks up to 64
constexpr int kGWStages = 4;                 // W ring (HBM): held until the store has read the tile
constexpr int kGOStages = 2;                 // operand ring (L2): held until the MMAs are done
constexpr int kGBox = 128 * 128;             // a 128-row x 64-element swizzled box: 16 KB
constexpr int kGABox = 64 * 128;             // a 64-rank x 64-column box of A: 8 KB
constexpr int kGWBytes = 2 * kGBox;          // W tile: two boxes
constexpr int kGOBytes = kGBox + 2 * kGABox; // B' box + A (two boxes)
constexpr int kGAtBytes = kGn * 128;         // A^T: 128 rows x 64 ranks
constexpr int kGEpiWarps = 8;
constexpr int kGStoreWarp = 4 + kGEpiWarps;
constexpr int kGThreads = 32 * (kGStoreWarp + 1);
constexpr int kGMaxW = 32;                   // weights per launch

struct MergeTcWeight {
    int h_in;
    int col_tiles;
    long long first;                         // first tile of this weight in the launch
};

struct MergeTcParams {
    MergeTcWeight w[kGMaxW];
    int n;
    long long n_tiles;
    float sign;
};

// Per weight: W [out][ld_w], A [r_slot][h_in], B' [out][r_slot].
struct MergeTcMaps {
    CUtensorMap m[3 * kGMaxW];
};

// Tile t of the launch -> weight q (advanced from its previous value: the
// tiles a CTA visits increase), row tile and column strip.
__device__ __forceinline__ void merge_tile_of(const MergeTcParams& P, long long t, int& q, int& rt, int& strip)
{
    while (q + 1 < P.n && t >= P.w[q + 1].first) ++q;
    const long long local = t - P.w[q].first;
    const int ct = P.w[q].col_tiles;
    if (local < 0x7FFFFFFFll) {
        rt = static_cast<int>(local) / ct;
        strip = static_cast<int>(local) - rt * ct;
    } else {
        rt = static_cast<int>(local / ct);
        strip = static_cast<int>(local - static_cast<long long>(rt) * ct);
    }
}

// w8 <- bf16_rne(w8 + sign * d) for 8 packed bf16 values (sign = +-1: the
// product is exact, so the fused form rounds once like the sum).
__device__ __forceinline__ uint4 fma_round8(const uint4& w, float sign, const float* d)
{
    uint4 o;
    o.x = pack_bf16x2(fmaf(sign, d[0], bf16_lo(w.x)), fmaf(sign, d[1], bf16_hi(w.x)));
    o.y = pack_bf16x2(fmaf(sign, d[2], bf16_lo(w.y)), fmaf(sign, d[3], bf16_hi(w.y)));
    o.z = pack_bf16x2(fmaf(sign, d[4], bf16_lo(w.z)), fmaf(sign, d[5], bf16_hi(w.z)));
    o.w = pack_bf16x2(fmaf(sign, d[6], bf16_lo(w.w)), fmaf(sign, d[7], bf16_hi(w.w)));
    return o;
}

__global__ void __launch_bounds__(kGThreads, 1)
merge_tc_kernel(const __grid_constant__ MergeTcMaps maps, const __grid_constant__ MergeTcParams P)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t wfull[kGWStages], wempty[kGWStages], epi_done[kGWStages];
    __shared__ __align__(8) uint64_t ofull[kGOStages], op_free[kGOStages], at_full[kGOStages];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // W ring (stage: W box 0 | W box 1), operand ring (stage: B' box | A box 0 |
    // A box 1), A^T buffers; tile i uses W stage i % 4 and operand stage,
    // A^T buffer and accumulator i % 2
    uint8_t* wring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t* oring = wring + kGWStages * kGWBytes;
    uint8_t* at = oring + kGOStages * kGOBytes;

    // this CTA's tiles: blockIdx.x + i * gridDim.x, i < n_my
    const long long G = gridDim.x;
    const int n_my = static_cast<int>((P.n_tiles - blockIdx.x + G - 1) / G);

    if (tid == 0) {
        for (int s = 0; s < kGWStages; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], 1);               // the store warp
            mbar_init(&epi_done[s], kGEpiWarps);    // one arrival per epilogue warp
        }
        for (int b = 0; b < kGOStages; ++b) {
            mbar_init(&ofull[b], 1);
            mbar_init(&op_free[b], 1);    // the MMA thread's commit: operand stage and A^T buffer free
            mbar_init(&at_full[b], 2);    // one per transpose warp
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kGEpiWarps);
        }
        mbar_init(&mma_done, 1);
        mbar_init_fence();
        s_fail = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 2 * kGn);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        if (lane == 0) {   // ---- producer ----
            int q = 0, o_issued = 0, w_issued = 0;
            for (int i = 0; i < n_my && !s_fail; ++i) {
                int rt, strip;
                merge_tile_of(P, blockIdx.x + i * G, q, rt, strip);
                const CUtensorMap* mW = &maps.m[3 * q];
                const bool two = strip * kGn + 64 < P.w[q].h_in;   // the second 64-column half holds columns
                const int b = i & 1, sw = i % kGWStages;
                // operands (L2): B' rows of the row tile, A columns of the strip
                if (i >= kGOStages && !mbar_wait_spin(&op_free[b], ((i >> 1) - 1) & 1)) {
                    s_fail = 1;
                    break;
                }
                if (s_fail) break;   // a stage released after a failure is not armed again
                uint8_t* so = oring + b * kGOBytes;
                mbar_expect_tx(&ofull[b], kGBox + (two ? 2 : 1) * kGABox);
                tma_load_2d(so, mW + 2, 0, rt * kGm, &ofull[b]);
                tma_load_2d(so + kGBox, mW + 1, strip * kGn, 0, &ofull[b]);
                if (two) tma_load_2d(so + kGBox + kGABox, mW + 1, strip * kGn + 64, 0, &ofull[b]);
                o_issued = i + 1;
                // the W tile (HBM)
                if (i >= kGWStages && !mbar_wait_spin(&wempty[sw], ((i / kGWStages) - 1) & 1)) {
                    s_fail = 1;
                    break;
                }
                if (s_fail) break;
                uint8_t* st = wring + sw * kGWBytes;
                mbar_expect_tx(&wfull[sw], (two ? 2 : 1) * kGBox);
                tma_load_2d(st, mW, strip * kGn, rt * kGm, &wfull[sw]);
                if (two) tma_load_2d(st + kGBox, mW, strip * kGn + 64, rt * kGm, &wfull[sw]);
                w_issued = i + 1;
            }
            // every copy issued lands before the CTA moves on
            for (int i = w_issued > kGWStages ? w_issued - kGWStages : 0; i < w_issued; ++i)
                if (!mbar_wait(&wfull[i % kGWStages], (i / kGWStages) & 1)) s_fail = 1;
            for (int i = o_issued > kGOStages ? o_issued - kGOStages : 0; i < o_issued; ++i)
                if (!mbar_wait(&ofull[i & 1], (i >> 1) & 1)) s_fail = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---- MMA issuer ----
            const uint32_t idesc = idesc_bf16_f32(kGm, kGn);
            bool ok = true;
            for (int i = 0; i < n_my && !s_fail; ++i) {
                const int a = i & 1;
                if (!mbar_wait_spin(&at_full[a], (i >> 1) & 1)) { ok = false; break; }
                if (i >= 2 && !mbar_wait_spin(&acc_empty[a], ((i >> 1) - 1) & 1)) { ok = false; break; }
                if (!mbar_wait_spin(&ofull[a], (i >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t b_rows = smem_u32(oring + a * kGOBytes);   // B' (M x K)
                const uint32_t a_t = smem_u32(at + a * kGAtBytes);        // A^T (N x K)
#pragma unroll
                for (int ks = 0; ks < kGk / 16; ++ks)
                    mma_bf16(tmem + a * kGn, sdesc_sw128(b_rows + ks * 32), sdesc_sw128(a_t + ks * 32), idesc,
                             ks != 0);
                mma_commit(&acc_full[a]);
                mma_commit(&op_free[a]);   // operand stage a and A^T buffer a are free once these MMAs are done
            }
            if (!ok) s_fail = 1;
            // the tensor memory is freed only after every MMA issued has completed
            mma_commit(&mma_done);
            if (!mbar_wait(&mma_done, 0)) s_fail = 1;
        }
    } else if (warp < 4) {
        // ---- transpose: staged A [64 ranks][128 columns] (two boxes) -> A^T
        // [128 columns][64 ranks].  Both are 128-byte-swizzled: element (row,
        // e) of a 128-byte-row tile sits at row * 128 + ((e / 8) ^ (row % 8)) * 16
        // + (e % 8) * 2.  Warp tw takes columns tw*64 .. tw*64+63 (box tw); lane
        // l the column pair 2l, 2l+1 of it: one 32-bit word per rank holds both,
        // and the 32 lanes' words fall in 32 distinct banks. ----
        const int tw = warp - 2;
        const int kk = 2 * lane, n0 = tw * 64 + kk;
        for (int i = 0; i < n_my && !s_fail; ++i) {
            const int b = i & 1;
            bool ready = mbar_wait(&ofull[b], (i >> 1) & 1);
            if (ready && i >= 2) ready = mbar_wait(&op_free[b], ((i >> 1) - 1) & 1);
            if (!__all_sync(0xFFFFFFFFu, ready)) {
                s_fail = 1;
                break;
            }
            const uint8_t* src = oring + b * kGOBytes + kGBox + tw * kGABox;
            uint8_t* dst = at + b * kGAtBytes;
#pragma unroll 1
            for (int c = 0; c < kGk / 8; ++c) {   // ranks 8c .. 8c+7
                uint32_t w[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    w[jj] = *reinterpret_cast<const uint32_t*>(src + (c * 8 + jj) * 128 + (((kk >> 3) ^ jj) << 4) +
                                                               (kk & 7) * 2);
                const uint4 even = make_uint4(__byte_perm(w[0], w[1], 0x5410), __byte_perm(w[2], w[3], 0x5410),
                                              __byte_perm(w[4], w[5], 0x5410), __byte_perm(w[6], w[7], 0x5410));
                const uint4 odd = make_uint4(__byte_perm(w[0], w[1], 0x7632), __byte_perm(w[2], w[3], 0x7632),
                                             __byte_perm(w[4], w[5], 0x7632), __byte_perm(w[6], w[7], 0x7632));
                *reinterpret_cast<uint4*>(dst + n0 * 128 + ((c ^ (n0 & 7)) << 4)) = even;
                *reinterpret_cast<uint4*>(dst + (n0 + 1) * 128 + ((c ^ ((n0 + 1) & 7)) << 4)) = odd;
            }
            fence_async_smem();   // the MMA (async proxy) reads what these threads wrote
            __syncwarp();
            if (lane == 0) mbar_arrive(&at_full[b]);
        }
    } else if (warp < kGStoreWarp) {
        // ---- epilogue: W half-tile += sign * D, one rounding, in the staged box ----
        const int quarter = warp & 3, half = (warp - 4) >> 2;
        const int r = quarter * 32 + lane;   // tile row = tensor-memory lane
        for (int i = 0; i < n_my; ++i) {
            const int sw = i % kGWStages, a = i & 1;
            bool ok = !s_fail && mbar_wait(&acc_full[a], (i >> 1) & 1);
            ok = ok && mbar_wait(&wfull[sw], (i / kGWStages) & 1);   // the W tile (TMA-written) is visible here
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) s_fail = 1;
            tc_fence_after();
            uint8_t* row = wring + sw * kGWBytes + half * kGBox + r * 128;   // W box `half`, row r
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float d[32];
                tmem_ld32(tmem + a * kGn + (static_cast<uint32_t>(quarter * 32) << 16) + half * 64 + c0, d);
                if (ok) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int cc = (c0 >> 3) + u;   // 16-byte chunk of the row within the box
                        uint4* p = reinterpret_cast<uint4*>(row + ((cc ^ (r & 7)) << 4));
                        *p = fma_round8(*p, P.sign, d + u * 8);
                    }
                }
            }
            fence_async_smem();   // the TMA store reads what these threads wrote
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[a]);   // the accumulator may be overwritten
                mbar_arrive(&epi_done[sw]);   // this half of the tile may be stored
            }
        }
    } else if (lane == 0) {
        // ---- store: the finished tile back to W, then the stage is free ----
        int q = 0;
        for (int i = 0; i < n_my; ++i) {
            int rt, strip;
            merge_tile_of(P, blockIdx.x + i * G, q, rt, strip);
            const int sw = i % kGWStages;
            if (!s_fail && !mbar_wait(&epi_done[sw], (i / kGWStages) & 1)) s_fail = 1;
            if (!s_fail) {
                const CUtensorMap* mW = &maps.m[3 * q];
                uint8_t* st = wring + sw * kGWBytes;
                tma_store_2d(mW, strip * kGn, rt * kGm, st);
                if (strip * kGn + 64 < P.w[q].h_in) tma_store_2d(mW, strip * kGn + 64, rt * kGm, st + kGBox);
                bulk_commit();
                bulk_wait_read();   // the stage may be refilled once the store has read it
            }
            mbar_arrive(&wempty[sw]);
        }
        bulk_wait_all();
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 2 * kGn);
}

constexpr size_t kGSmem = static_cast<size_t>(kGWStages) * kGWBytes + kGOStages * (kGOBytes + kGAtBytes) + 1024;

}  // namespace

bool merge_tc_supported(int r_slot) { return r_slot <= kGk; }

cudaError_t launch_merge_tc(int n, bf16_t* const* W, const int* ld_w, const int* out, const int* h_in,
                            const bf16_t* const* A, const bf16_t* const* B, int r_slot, int sign, cudaStream_t stream)
{
    if (r_slot > kGk) return cudaErrorInvalidValue;
    static int configured_device = -1, n_sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(merge_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGSmem));
        if (e != cudaSuccess) return e;
        e = prefer_max_shared(reinterpret_cast<const void*>(merge_tc_kernel));
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    for (int i0 = 0; i0 < n; i0 += kGMaxW) {
        const int nw = std::min(kGMaxW, n - i0);
        // boxes: W 128 rows x 64 columns; A 64 ranks x 64 columns and B' 128 rows x
        // 64 ranks, ranks past r_slot reading as zero
        MergeTcMaps maps;
        MergeTcParams P{};
        P.n = nw;
        P.sign = sign > 0 ? 1.f : -1.f;
        long long tiles = 0;
        for (int q = 0; q < nw; ++q) {
            const int i = i0 + q;
            if (!encode_tmap_bf16(&maps.m[3 * q], W[i], out[i], h_in[i], ld_w[i], kGm, 64, true) ||
                !encode_tmap_bf16(&maps.m[3 * q + 1], A[i], r_slot, h_in[i], h_in[i], 64, 64, true) ||
                !encode_tmap_bf16(&maps.m[3 * q + 2], B[i], out[i], r_slot, r_slot, kGm, 64, true))
                return cudaErrorInvalidValue;
            P.w[q].h_in = h_in[i];
            P.w[q].col_tiles = (h_in[i] + kGn - 1) / kGn;
            P.w[q].first = tiles;
            tiles += static_cast<long long>((out[i] + kGm - 1) / kGm) * P.w[q].col_tiles;
        }
        P.n_tiles = tiles;
        if (tiles <= 0) continue;
        const unsigned grid = static_cast<unsigned>(std::min<long long>(tiles, std::max(1, n_sms)));
        merge_tc_kernel<<<grid, kGThreads, kGSmem, stream>>>(maps, P);
        note_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace lora
