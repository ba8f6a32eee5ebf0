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
// Persistent tcgen05 GEMM, one CTA per SM, tiles of 128 rows x 256 output
// columns of one projection, visited in groups of kGroupM row tiles so that
// the x and W tiles in flight at once fit in L2.  Per tile the K loop is
// ceil(h_in / 64) base steps (an x box and a W box) followed, when every row
// of the tile carries the same adapter (the common case inside a prefill
// segment), by 2 * ceil(r_slot / 64) LoRA steps (a v_hi or v_lo box and a
// box of B') into the same accumulator: the delta is a K extension of the
// GEMM.  In tiles whose rows mix adapters (segment boundaries, decode rows)
// the epilogue adds each row's delta on the CUDA cores from the planes and
// B' before rounding.
//   warp 0: TMA producer   warp 1: MMA issuer   warps 2..17: epilogue
// The fp32 accumulator is double-buffered in tensor memory (2 x 256
// columns), so the epilogue of one tile overlaps the K loop of the next.
// Every wait is bounded (0.2 s); a timeout sets LORA_DEV_TIMEOUT and the
// CTA winds down, freeing its tensor memory.

#include <algorithm>

#include "launch.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace lora {

namespace {

using namespace tc;

constexpr int kLM = 128;                      // rows per tile
constexpr int kLN = 256;                      // output columns per tile
constexpr int kLK = 64;                       // K elements per step (one 128-byte swizzled row)
constexpr int kLStages = 4;
constexpr int kABytes = kLM * 128;            // x or v box
constexpr int kBBytes = kLN * 128;            // W or B' box
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kLEpiWarps = 16;                // 4 per tensor-memory lane quarter, 64 columns each
constexpr int kLThreads = 32 * (2 + kLEpiWarps);
constexpr int kGroupM = 16;                   // row tiles per raster group

struct LinearParams {
    int n_proj, r_slot, r_pad64, n_slots, n_rows;
    int out_off[LORA_MAX_PROJ];
    int width[LORA_MAX_PROJ];
    int ntiles[LORA_MAX_PROJ];   // 256-column tiles per projection
    const bf16_t* B[LORA_MAX_PROJ];
    int n_tm, n_tn, n_tiles, n_kb, kbs;
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

// The adapter slot shared by every row of row tile m, or -1 when the rows
// mix adapters, include base rows or name an id outside [0, n_slots).
// Whole warp; the answer is the same in every warp that asks.
__device__ __forceinline__ int uniform_slot(const LinearParams& P, int m)
{
    const int lane = threadIdx.x & 31;
    const int row0 = m * kLM, nr = min(kLM, P.n_rows - row0);
    const int first = __ldg(P.ids + row0);
    bool same = true;
    for (int i = lane; i < nr; i += 32) same &= __ldg(P.ids + row0 + i) == first;
    same = __all_sync(0xFFFFFFFFu, same);
    return (same && first >= 0 && first < P.n_slots) ? first : -1;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
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

__global__ void __launch_bounds__(kLThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                 const __grid_constant__ CUtensorMap mvh, const __grid_constant__ CUtensorMap mvl,
                 const __grid_constant__ CUtensorMap mb0, const __grid_constant__ CUtensorMap mb1,
                 const __grid_constant__ CUtensorMap mb2, const __grid_constant__ CUtensorMap mb3, LinearParams P)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kLStages], empty[kLStages], acc_full[2], acc_empty[2];
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
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], kLEpiWarps);
        }
        mbar_init_fence();
        s_fail = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {   // ---- producer (lane 0 issues; the warp decides each tile's kind) ----
        int it = 0;
        for (int t = blockIdx.x; t < P.n_tiles && !s_fail; t += gridDim.x) {
            const LTile T = tile_of(P, t);
            const int us = uniform_slot(P, T.m);
            const int n_ks = P.n_kb + (us >= 0 ? 2 * P.kbs : 0);
            if (lane == 0) {
                for (int k = 0; k < n_ks; ++k, ++it) {
                    const int s = it % kLStages;
                    if (it >= kLStages && !mbar_wait(&empty[s], ((it / kLStages) - 1) & 1)) {
                        s_fail = 1;
                        break;
                    }
                    uint8_t* a = ring + s * kStageBytes;
                    uint8_t* b = a + kABytes;
                    mbar_expect_tx(&full[s], kStageBytes);
                    if (k < P.n_kb) {
                        tma_load_2d(a, &mx, k * kLK, T.m * kLM, &full[s]);
                        tma_load_2d(b, &mw, k * kLK, P.out_off[T.p] + T.col0, &full[s]);
                    } else {
                        const int l = k - P.n_kb, plane = l / P.kbs, kb = l - plane * P.kbs;
                        tma_load_3d(a, plane ? &mvl : &mvh, kb * kLK, T.p, T.m * kLM, &full[s]);
                        tma_load_2d(b, bmap[T.p], kb * kLK, us * P.width[T.p] + T.col0, &full[s]);
                    }
                }
            }
            it = __shfl_sync(0xFFFFFFFFu, it, 0);
            __syncwarp();
        }
    } else if (warp == 1) {   // ---- MMA issuer ----
        int it = 0, ti = 0, ok = 1;
        for (int t = blockIdx.x; ok && t < P.n_tiles && !s_fail; t += gridDim.x, ++ti) {
            const LTile T = tile_of(P, t);
            const int us = uniform_slot(P, T.m);
            const int n_ks = P.n_kb + (us >= 0 ? 2 * P.kbs : 0);
            if (lane == 0) {
                const int a = ti & 1;
                const uint32_t idesc = idesc_bf16_f32(kLM, (T.ncols + 15) / 16 * 16);
                if (ti >= 2 && !mbar_wait(&acc_empty[a], ((ti >> 1) - 1) & 1)) ok = 0;
                tc_fence_after();
                const uint32_t d = tmem + a * kLN;
                for (int k = 0; ok && k < n_ks; ++k, ++it) {
                    const int s = it % kLStages;
                    if (!mbar_wait(&full[s], (it / kLStages) & 1)) {
                        ok = 0;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t as = smem_u32(ring + s * kStageBytes), bs = as + kABytes;
#pragma unroll
                    for (int ks = 0; ks < kLK / 16; ++ks)
                        mma_bf16(d, sdesc_sw128(as + ks * 32), sdesc_sw128(bs + ks * 32), idesc, k > 0 || ks > 0);
                    mma_commit(&empty[s]);   // the stage is free once these MMAs have read it
                }
                if (ok) mma_commit(&acc_full[a]);
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            it = __shfl_sync(0xFFFFFFFFu, it, 0);
        }
        if (!ok) s_fail = 1;
    } else {   // ---- epilogue ----
        const int e = warp - 2;
        const int quarter = warp & 3;        // tensor-memory lanes this warp may read
        const int cs = (e >> 2) * 64;        // its 64 columns of the tile
        const int r = quarter * 32 + lane;   // its row of the tile
        int ti = 0;
        for (int t = blockIdx.x; t < P.n_tiles; t += gridDim.x, ++ti) {
            const LTile T = tile_of(P, t);
            const int us = uniform_slot(P, T.m);
            const int a = ti & 1;
            if (s_fail || !mbar_wait(&acc_full[a], (ti >> 1) & 1)) {
                s_fail = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tcol = tmem + a * kLN + (static_cast<uint32_t>(quarter * 32) << 16) + cs;
            const int row = T.m * kLM + r;
            const bool live = row < P.n_rows;
            int id = -1;
            if (live && us < 0) {
                id = __ldg(P.ids + row);
                if (id < -1 || id >= P.n_slots) {
                    flag(P.status, LORA_DEV_SLOT_OUT_OF_RANGE);   // the row keeps its base value
                    id = -1;
                }
            }
            bf16_t* yrow = P.y + static_cast<size_t>(min(row, P.n_rows - 1)) * P.ld_y + P.out_off[T.p] + T.col0;
            // 32 accumulator columns at a time; the accumulator is handed back
            // to the MMA after the second read (it is next needed two tiles on)
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float d[32];
                tmem_ld32(tcol + h * 32, d);
                if (h == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[a]);
                }
                const int c0 = cs + h * 32;   // first column of this piece in the tile
                if (live && c0 < T.ncols) {
                    // rows that mix adapters add their own delta here
                    if (id >= 0) add_row_delta(P, T.p, id, row, T.col0 + c0, d);
                    store_row32(yrow + c0, T.ncols - c0, d);
                }
            }
        }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 2 * kLN);
    if (tid == 0 && s_fail) flag(P.status, LORA_DEV_TIMEOUT);
}

}  // namespace

size_t linear_tc_smem() { return static_cast<size_t>(kLStages) * kStageBytes + 1024; }

cudaError_t launch_linear_tc(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const bf16_t* W, int ld_w,
                             int n_out, const ProjSet& ps, const bf16_t* vh, const bf16_t* vl,
                             const int32_t* ids, int n_rows, int n_slots, int32_t* status, cudaStream_t stream)
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
    CUtensorMap mx, mw, mvh, mvl, mb[4];
    if (!encode_tmap_bf16(&mx, x, n_rows, h_in, ld_x, kLM, kLK, true) ||
        !encode_tmap_bf16(&mw, W, n_out, h_in, ld_w, kLN, kLK, true) ||
        !encode_tmap_bf16_3d(&mvh, vh, ps.r_slot, ps.n_proj, n_rows, P.r_pad64, P.ld_p, kLK, kLM) ||
        !encode_tmap_bf16_3d(&mvl, vl, ps.r_slot, ps.n_proj, n_rows, P.r_pad64, P.ld_p, kLK, kLM))
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
        e = cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(linear_tc_smem()));
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int grid = static_cast<int>(std::min<long long>(env_int("LORA_LINEAR_GRID", n_sms), n_tiles));
    linear_tc_kernel<<<grid, kLThreads, linear_tc_smem(), stream>>>(mx, mw, mvh, mvl, mb[0], mb[1], mb[2], mb[3],
                                                                    P);
    note_launch();
    return cudaGetLastError();
}

}  // namespace lora
