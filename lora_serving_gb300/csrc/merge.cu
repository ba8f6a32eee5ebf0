// merge.cu -- fold one adapter into (or out of) a base weight, for serving a
// single tenant at the base model's cost.
//
// Multi-LoRA serving note, "interviewer follow-ups": merging W' = W + B A
// gives the same model as the base plus the adapter's delta.  Here
//   W[o][k] <- bf16_rne(W[o][k] + sign * sum_j B'[o][j] A[j][k]),
// sign = +1 (merge) or -1 (unmerge), B' the folded store (scale applied),
// the sum in fp32 over the slot rank (padding ranks are zero).
//
// Slot ranks up to 64 take the tensor-memory kernel of merge_tc.cu; the
// kernels here serve larger ranks (and LORA_MERGE_TC=0).
//
// One CTA per 128 x 128 tile of W: its 128 rows of B' and 128 columns of A
// arrive by 16-byte cp.async, then the tile itself (a second group, needed
// only by the epilogue, so it lands while the MMAs run); warp w forms rows
// 16w..16w+15 of B'A on the tensor cores (mma.sync m16n8k16, fp32
// accumulate; A enters as the col-major operand through transposing
// ldmatrix); each thread adds its accumulator fragments into the staged
// tile and rounds once; the tile leaves by coalesced 16-byte stores.
// HBM-bound: W is read and written once, A and B' come from L2 after their
// first use.

#include <algorithm>

#include "decode_common.cuh"
#include "launch.h"

namespace lora {

namespace {

using namespace dec;

constexpr int kMRows = 128;                // W rows per CTA
constexpr int kMCols = 128;                // W columns per CTA
constexpr int kMThreads = 256;             // 8 warps, 16 rows each
constexpr int kMPitch = kMCols + 8;        // bf16 pitch of the W and A tiles (conflict-free ldmatrix)
constexpr int kMaxMergeWeights = 32;       // weights per batch launch

__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];\n"
                 : "=r"(r0), "=r"(r1) : "r"(addr));
}

// One weight to merge: W [out][ld_w], its adapter slot's A [r_slot][h_in]
// and B' [out][r_slot].
struct MergeWeight {
    bf16_t* W;
    const bf16_t* A;
    const bf16_t* B;
    int ld_w, out, h_in;
    int col_tiles;       // ceil(h_in / 128)
    long long first;     // first tile of this weight in the batch's tile order
};

struct MergeParams {
    MergeWeight w[kMaxMergeWeights];
    int n;               // weights
    long long n_tiles;   // all weights' tiles
    int r_slot, r_pad;   // r_pad: r_slot rounded up to 16 (the mma K)
    float sign;
};

// W[o0 .. o0+127][k0 .. k0+127] += sign * B'A, one rounding.  Whole CTA;
// the caller synchronises before smem is reused.
__device__ __forceinline__ void merge_tile(const MergeWeight& m, const MergeParams& p, int o0, int k0,
                                           unsigned char* smem)
{
    const int bp_pitch = p.r_pad + 8;
    bf16_t* sW = reinterpret_cast<bf16_t*>(smem);                       // [kMRows][kMPitch]
    bf16_t* sB = sW + kMRows * kMPitch;                                 // [kMRows][r_pad + 8]
    bf16_t* sA = sB + kMRows * bp_pitch;                                // [r_pad][kMPitch]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- stage B' rows and A columns (the MMA's operands), then the W tile
    // (needed only by the epilogue); zero outside the matrices ----
    const int bch = p.r_pad / 8;
    for (int i = tid; i < kMRows * bch; i += kMThreads) {
        const int r = i / bch, c = (i % bch) * 8;
        const bool ok = o0 + r < m.out && c < p.r_slot;
        cp_async16(smem_u32(sB + r * bp_pitch + c),
                   ok ? static_cast<const void*>(m.B + static_cast<size_t>(o0 + r) * p.r_slot + c) : m.B, ok);
    }
    for (int i = tid; i < p.r_pad * (kMCols / 8); i += kMThreads) {
        const int j = i / (kMCols / 8), c = (i % (kMCols / 8)) * 8;
        const bool ok = j < p.r_slot && k0 + c < m.h_in;
        cp_async16(smem_u32(sA + j * kMPitch + c),
                   ok ? static_cast<const void*>(m.A + static_cast<size_t>(j) * m.h_in + k0 + c) : m.A, ok);
    }
    cp_async_commit();
    for (int i = tid; i < kMRows * (kMCols / 8); i += kMThreads) {
        const int r = i / (kMCols / 8), c = (i % (kMCols / 8)) * 8;
        const bool ok = o0 + r < m.out && k0 + c < m.h_in;
        cp_async16(smem_u32(sW + r * kMPitch + c),
                   ok ? static_cast<const void*>(m.W + static_cast<size_t>(o0 + r) * m.ld_w + k0 + c) : m.W, ok);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    // ---- B'A for rows 16w..16w+15, all 128 columns (16 n-tiles of 8) ----
    float acc[16][4] = {};
    const int mi = lane >> 3, mr = lane & 7, l16 = lane & 15;
    for (int kk = 0; kk < p.r_pad; kk += 16) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(smem_u32(sB + (warp * 16 + (mi & 1) * 8 + mr) * bp_pitch + kk + (mi >> 1) * 8), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            uint32_t b0, b1;
            ldmatrix_x2_trans(smem_u32(sA + (kk + l16) * kMPitch + nt * 8), b0, b1);
            mma_bf16_16816(acc[nt], a0, a1, a2, a3, b0, b1);
        }
    }

    cp_async_wait<0>();
    __syncthreads();

    // ---- W += sign * B'A at the fragment positions, one rounding ----
    const int g = lane >> 2, q2 = (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t* w2 = reinterpret_cast<uint32_t*>(sW + (warp * 16 + g + h * 8) * kMPitch + nt * 8 + q2);
            const uint32_t old = *w2;
            *w2 = pack_bf16x2(bf16_lo(old) + p.sign * acc[nt][2 * h], bf16_hi(old) + p.sign * acc[nt][2 * h + 1]);
        }
    }
    __syncthreads();
    for (int i = tid; i < kMRows * (kMCols / 8); i += kMThreads) {
        const int r = i / (kMCols / 8), c = (i % (kMCols / 8)) * 8;
        if (o0 + r < m.out && k0 + c < m.h_in)
            *reinterpret_cast<uint4*>(m.W + static_cast<size_t>(o0 + r) * m.ld_w + k0 + c) =
                *reinterpret_cast<const uint4*>(sW + r * kMPitch + c);
    }
}

// One weight: one CTA per tile (blockIdx.x = column block, blockIdx.y = row block).
__global__ void __launch_bounds__(kMThreads)
merge_kernel(const __grid_constant__ MergeParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    merge_tile(p.w[0], p, blockIdx.y * kMRows, blockIdx.x * kMCols, smem);
}

// Tile t of the batch: its weight (q advances monotonically) and its corner.
__device__ __forceinline__ void locate_tile(const MergeParams& p, long long t, int& q, int& o0, int& k0)
{
    while (q + 1 < p.n && t >= p.w[q + 1].first) ++q;
    const MergeWeight& m = p.w[q];
    const long long local = t - m.first;
    const int rb = static_cast<int>(local / m.col_tiles);
    o0 = rb * kMRows;
    k0 = static_cast<int>(local - static_cast<long long>(rb) * m.col_tiles) * kMCols;
}

// One 128-byte line of a W tile per thread (128 rows x 2 lines) into L2.
__device__ __forceinline__ void prefetch_tile_l2(const MergeWeight& m, int o0, int k0)
{
    const int r = threadIdx.x >> 1, c = k0 + (threadIdx.x & 1) * 64;
    if (o0 + r < m.out && c < m.h_in)
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(m.W + static_cast<size_t>(o0 + r) * m.ld_w + c));
}

// Several weights in one launch: the CTAs walk the weights' tiles in order
// (tile c, c + gridDim.x, ...), so no weight leaves a partial last wave and
// there is one launch for all.  Within a weight, column block fastest: the
// CTAs in flight together share B' rows and read neighbouring A columns.
// Each CTA requests its next tile's W into L2 before it works on the current
// one, so the HBM reads of the next tile overlap this tile's compute and
// stores instead of following them.  Three CTAs per SM (shared memory
// allows three at slot rank 64), registers held to match.
__global__ void __launch_bounds__(kMThreads, 3)
merge_batch_kernel(const __grid_constant__ MergeParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    static_assert(kMThreads == 2 * kMRows && kMCols * sizeof(bf16_t) == 2 * 128, "one L2 line per thread");
    int q = 0, qn = 0, o0 = 0, k0 = 0;
    if (blockIdx.x < p.n_tiles) locate_tile(p, blockIdx.x, qn, o0, k0);
    for (long long t = blockIdx.x; t < p.n_tiles; t += gridDim.x) {
        q = qn;
        const int to0 = o0, tk0 = k0;
        if (t + gridDim.x < p.n_tiles) {
            locate_tile(p, t + gridDim.x, qn, o0, k0);
            prefetch_tile_l2(p.w[qn], o0, k0);
        }
        merge_tile(p.w[q], p, to0, tk0, smem);
        __syncthreads();   // the next tile reuses the staging buffers
    }
}

size_t merge_smem(int r_pad)
{
    return sizeof(bf16_t) * (static_cast<size_t>(kMRows) * kMPitch + static_cast<size_t>(kMRows) * (r_pad + 8) +
                             static_cast<size_t>(r_pad) * kMPitch);
}

}  // namespace

namespace {

cudaError_t configure_merge(int& n_sms)
{
    static int configured_device = -1, sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        const int max_smem = static_cast<int>(merge_smem((LORA_MAX_RANK + 15) / 16 * 16));
        e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(merge_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (e != cudaSuccess) return e;
        e = prefer_max_shared(reinterpret_cast<const void*>(merge_kernel));
        if (e != cudaSuccess) return e;
        e = prefer_max_shared(reinterpret_cast<const void*>(merge_batch_kernel));
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    n_sms = sms;
    return cudaSuccess;
}

}  // namespace

// Slot ranks up to 64 take the tensor-memory kernel (merge_tc.cu) unless
// LORA_MERGE_TC=0; larger ranks take the kernels above.
static bool use_merge_tc(int r_slot) { return merge_tc_supported(r_slot) && env_int("LORA_MERGE_TC", 1) != 0; }

cudaError_t launch_merge(bf16_t* W, int ld_w, int out, int h_in, const bf16_t* A, const bf16_t* B, int r_slot,
                         int sign, cudaStream_t stream)
{
    if (use_merge_tc(r_slot)) return launch_merge_tc(1, &W, &ld_w, &out, &h_in, &A, &B, r_slot, sign, stream);
    MergeParams p{};
    p.n = 1;
    p.w[0] = MergeWeight{W, A, B, ld_w, out, h_in, (h_in + kMCols - 1) / kMCols, 0};
    p.r_slot = r_slot;
    p.r_pad = (r_slot + 15) / 16 * 16;
    p.sign = sign > 0 ? 1.f : -1.f;
    int n_sms = 0;
    const cudaError_t e = configure_merge(n_sms);
    if (e != cudaSuccess) return e;
    const dim3 grid((h_in + kMCols - 1) / kMCols, (out + kMRows - 1) / kMRows);
    merge_kernel<<<grid, kMThreads, merge_smem(p.r_pad), stream>>>(p);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_merge_batch(int n, bf16_t* const* W, const int* ld_w, const int* out, const int* h_in,
                               const bf16_t* const* A, const bf16_t* const* B, int r_slot, int sign,
                               cudaStream_t stream)
{
    if (use_merge_tc(r_slot)) return launch_merge_tc(n, W, ld_w, out, h_in, A, B, r_slot, sign, stream);
    int n_sms = 0;
    cudaError_t e = configure_merge(n_sms);
    if (e != cudaSuccess) return e;
    const size_t smem = merge_smem((r_slot + 15) / 16 * 16);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, merge_batch_kernel, kMThreads, smem);
    if (e != cudaSuccess) return e;
    for (int i0 = 0; i0 < n; i0 += kMaxMergeWeights) {
        MergeParams p{};
        p.n = std::min(kMaxMergeWeights, n - i0);
        p.r_slot = r_slot;
        p.r_pad = (r_slot + 15) / 16 * 16;
        p.sign = sign > 0 ? 1.f : -1.f;
        long long tiles = 0;
        for (int q = 0; q < p.n; ++q) {
            const int i = i0 + q;
            const int ct = (h_in[i] + kMCols - 1) / kMCols;
            p.w[q] = MergeWeight{W[i], A[i], B[i], ld_w[i], out[i], h_in[i], ct, tiles};
            tiles += static_cast<long long>(ct) * ((out[i] + kMRows - 1) / kMRows);
        }
        p.n_tiles = tiles;
        const long long grid = std::min<long long>(tiles, static_cast<long long>(std::max(1, per_sm)) * n_sms);
        if (grid <= 0) continue;
        merge_batch_kernel<<<static_cast<unsigned>(grid), kMThreads, smem, stream>>>(p);
        note_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace lora
