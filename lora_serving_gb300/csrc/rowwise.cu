// rowwise.cu -- CUDA-core shrink and expand, one position (row) per CTA.
//
// These are the general kernels behind lora_bgmv_* and lora_sgmv_* for any
// row map (per-token ids, contiguous segments or gathered segments):
//   shrink  v = A_slot x        (TGI page, "4. SGMV and BGMV": the rank-r
//                                intermediate; fp32 accumulation, never
//                                rounded to bf16)
//   expand  y = bf16(y + B'_slot v)   on the projection's output slice
//                                     (TGI page, "5. tensor parallelism":
//                                      uneven q/k/v slices)
// Loads are 128-bit (8 bf16) and coalesced across the warp; x is staged in
// shared memory once per row and reused by every rank of the CTA.  A second
// grid dimension splits a row's work over several CTAs (blocks of ranks for
// the shrink, blocks of output columns for the expand), so that a decode
// batch of a few dozen rows still covers every SM; the adapter rows a
// position reads are shared by the positions of the same adapter through L2.

#include <algorithm>

#include "launch.h"

namespace lora {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
shrink_rowwise_kernel(float* __restrict__ v, int ld_v, const bf16_t* __restrict__ x, int ld_x,
                      int h_in, ProjSet ps, RowMap map, int32_t* status)
{
    extern __shared__ uint4 xs[];
    int row, slot;
    if (!resolve(map, blockIdx.x, row, slot, status)) return;
    const int nv = h_in >> 3;
    const uint4* xg = reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * ld_x);
    for (int i = threadIdx.x; i < nv; i += kThreads) xs[i] = __ldg(xg + i);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = ps.n_proj * ps.r_slot;
    // ranks [j0, j1) of this CTA's block
    const int per = (R + gridDim.y - 1) / gridDim.y;
    const int j0 = blockIdx.y * per, j1 = min(R, j0 + per);
    for (int j = j0 + warp; j < j1; j += kThreads / 32) {
        const int pj = j / ps.r_slot, jj = j - pj * ps.r_slot;
        const uint4* a = reinterpret_cast<const uint4*>(
            ps.A[pj] + (static_cast<size_t>(slot) * ps.r_slot + jj) * h_in);
        float acc = 0.f;
        for (int i = lane; i < nv; i += 32) acc = dot8(__ldg(a + i), xs[i], acc);
        acc = warp_sum(acc);
        if (lane == 0) v[static_cast<size_t>(row) * ld_v + j] = acc;
    }
}

__global__ void __launch_bounds__(kThreads)
expand_rowwise_kernel(bf16_t* __restrict__ y, int ld_y, const float* __restrict__ v, int ld_v,
                      ProjSet ps, RowMap map, int32_t* status)
{
    __shared__ float vs[LORA_MAX_PROJ * LORA_MAX_RANK];
    int row, slot;
    if (!resolve(map, blockIdx.x, row, slot, status)) return;
    const int R = ps.n_proj * ps.r_slot;
    for (int i = threadIdx.x; i < R; i += kThreads) vs[i] = v[static_cast<size_t>(row) * ld_v + i];
    __syncthreads();

    int total = 0;
    for (int p = 0; p < ps.n_proj; ++p) total += ps.width[p] >> 3;
    bf16_t* yrow = y + static_cast<size_t>(row) * ld_y;
    for (int c = blockIdx.y * kThreads + threadIdx.x; c < total; c += kThreads * gridDim.y) {
        int p = 0, q = c;
        while (q >= (ps.width[p] >> 3)) { q -= ps.width[p] >> 3; ++p; }
        const int col0 = q << 3;
        const bf16_t* b = ps.B[p] + (static_cast<size_t>(slot) * ps.width[p] + col0) * ps.r_slot;
        const float* vp = vs + p * ps.r_slot;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int jj = 0; jj < ps.r_slot; jj += 8) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[e] = dot8f(__ldg(reinterpret_cast<const uint4*>(b + e * ps.r_slot + jj)), vp + jj, acc[e]);
        }
        uint4* yp = reinterpret_cast<uint4*>(yrow + ps.out_off[p] + col0);
        *yp = add_round8(*yp, acc);
    }
}

// Multiprocessors of the current device (queried once per device).
int sm_count()
{
    static int n_sms = 0, sms_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (sms_device != dev) {
        if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 152;
        sms_device = dev;
    }
    return n_sms;
}

}  // namespace

cudaError_t launch_shrink_rowwise(float* v, int ld_v, const bf16_t* x, int ld_x, int h_in,
                                  const ProjSet& ps, const RowMap& map, int32_t* status,
                                  cudaStream_t stream)
{
    if (map.n_pos <= 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(h_in) * sizeof(bf16_t);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(shrink_rowwise_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        e = prefer_max_shared(reinterpret_cast<const void*>(shrink_rowwise_kernel));
        if (e != cudaSuccess) return e;
        e = prefer_max_shared(reinterpret_cast<const void*>(expand_rowwise_kernel));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // Rank blocks of at least 8 ranks (one per warp), enough of them that
    // the grid covers the SMs about twice.
    const int R = ps.n_proj * ps.r_slot;
    const int want = (2 * sm_count() + map.n_pos - 1) / map.n_pos;
    const int blocks = std::max(1, std::min(want, (R + 7) / 8));
    shrink_rowwise_kernel<<<dim3(map.n_pos, blocks), kThreads, smem, stream>>>(v, ld_v, x, ld_x, h_in, ps, map,
                                                                               status);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_expand_rowwise(bf16_t* y, int ld_y, const float* v, int ld_v,
                                  const ProjSet& ps, const RowMap& map, int32_t* status,
                                  cudaStream_t stream)
{
    if (map.n_pos <= 0) return cudaSuccess;
    // Column blocks of kThreads 8-column chunks, enough that the grid covers
    // the SMs about twice.
    int total = 0;
    for (int p = 0; p < ps.n_proj; ++p) total += ps.width[p] >> 3;
    const int want = (2 * sm_count() + map.n_pos - 1) / map.n_pos;
    const int blocks = std::max(1, std::min(want, (total + kThreads - 1) / kThreads));
    expand_rowwise_kernel<<<dim3(map.n_pos, blocks), kThreads, 0, stream>>>(y, ld_y, v, ld_v, ps, map, status);
    note_launch();
    return cudaGetLastError();
}

}  // namespace lora
