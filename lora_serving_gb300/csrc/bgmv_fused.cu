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
// Data movement: rows of A, x and the CTA's slice of B' arrive by bulk
// asynchronous copies (cp.async.bulk, completion counted on mbarriers), so
// a CTA issues a few hundred large copies instead of thousands of 16-byte
// requests.  Waits on the mbarriers are bounded (0.2 s); a copy that does
// not land sets LORA_DEV_TIMEOUT and the CTA leaves its rows unwritten,
// while still taking part in every cluster barrier.
//
// Ordering (programmatic dependent launch): metadata and weights are read
// before griddepcontrol.wait, so they stream in while the preceding kernel
// on the stream is still running.  With LORA_APPLY_X_READY the shrink, the
// cluster reduction and the delta are formed before the wait as well, and
// only the read-modify-write of y follows it.

#include <cstdlib>

#include "launch.h"

namespace lora {

namespace {

constexpr int kRB = 16;            // rows per unit (the mma M)
constexpr int kKT = 128;           // K elements per pipeline stage
constexpr int kPad = 8;            // bf16 padding per smem row: conflict-free ldmatrix
constexpr int kLds = kKT + kPad;
constexpr int kStages = 2;         // K stages of the one-launch form
constexpr int kStagesShrink = 4;   // K stages of the shrink-only form
constexpr double kSplitWeightBytes = 32.0 * (1 << 20);   // two launches from this many weight bytes per call
constexpr int kMaxChunks = 64;     // output chunks (8 columns) per expand tile
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPermStage = 4096;   // decode positions staged in smem with the group table
constexpr int kBSlack = 32;        // zeroed bf16 after B' so padded-K fragments stay finite
constexpr unsigned long long kTimeoutNs = 200000000ull;

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
    int nch_tile;             // chunks per expand tile (<= kMaxChunks)
    int r_pad;                // r_slot rounded up to 16 (expand mma K)
    int x_ready;              // x may be read before the grid dependency resolves
    int y_ready;              // y may be updated before it resolves
    float* v_out;             // shrink only: fp32 v rows go here, no expand
    int ld_v;
    int32_t* status;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long gtime()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on an mbarrier phase: false after kTimeoutNs without it.
__device__ __noinline__ bool mbar_wait(uint64_t* bar, unsigned parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = gtime();
    while (!mbar_try_wait(bar, parity))
        if (gtime() - t0 > kTimeoutNs) return false;
    return true;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid)
{
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t map_rank(uint32_t local_addr, uint32_t rank)
{
    uint32_t remote;
    asm("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}
// Plain (non-volatile) DSMEM load: ordering against the partials' writes is
// given by the cluster barrier, so independent loads may be issued together.
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t remote)
{
    float2 v;
    asm("ld.shared::cluster.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(remote));
    return v;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// v (two fp32 values) -> packed bf16 hi pair and bf16 lo pair (v ~= hi + lo).
__device__ __forceinline__ void split_hi_lo(float a, float b, uint32_t& hi, uint32_t& lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // .x = a (low half)
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Units of a group: ceil(len / 16), or 0 (and bad) when its bounds fall
// outside [0, n_pos) -- so perm is never read out of range.
__device__ __forceinline__ int group_units(int s, int e, int n_pos, bool& bad)
{
    const bool sane = s >= 0 && e <= n_pos && s <= e;
    bad |= !sane;
    return sane ? (e - s + kRB - 1) / kRB : 0;
}

struct UnitInfo {
    int g, pos0, nrows, slot, found, bad;
};

// Unit u -> (group, first position, rows, slot).  Every thread of the CTA
// takes part and the answer is uniform across the CTA (and across a
// cluster, whose CTAs all map to the same unit).  The group table is read
// NT groups per round trip (one group per thread, block-wide prefix sum),
// together with the permutation when it fits in s_perm.
template <int NT, class Params>
__device__ __forceinline__ UnitInfo find_unit(const Params& p, int u, int* s_perm, bool stage_perm)
{
    __shared__ int s_warp[NT / 32];
    __shared__ UnitInfo s_info;
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_info.found = 0;
        s_bad = 0;
    }
    if (stage_perm)
        for (int i = tid; i < p.n_pos; i += NT) s_perm[i] = __ldg(p.perm + i);
    int base = 0;   // units in the groups of earlier rounds
    for (int g0 = 0; g0 < p.n_groups; g0 += NT) {
        const int gi = g0 + tid;
        int s = 0, e = 0, sl = -1;
        bool bad = false;
        int n = 0;
        if (gi < p.n_groups) {
            s = __ldg(p.gstarts + gi);
            e = __ldg(p.gstarts + gi + 1);
            sl = __ldg(p.gslot + gi);
            n = group_units(s, e, p.n_pos, bad);
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
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) {
            const int c = s_warp[w];
            if (w < warp) before += c;
            total += c;
        }
        incl += base + before;
        const int excl = incl - n;
        if (bad) atomicOr(&s_bad, 1);
        if (gi < p.n_groups && u >= excl && u < incl) {
            UnitInfo info;
            info.g = gi;
            info.pos0 = s + (u - excl) * kRB;
            info.nrows = min(kRB, e - info.pos0);
            info.slot = sl;
            info.found = 1;
            info.bad = 0;
            s_info = info;
        }
        base += total;
        __syncthreads();   // s_warp is rewritten by the next round
    }
    if (p.n_groups <= 0) __syncthreads();
    UnitInfo r = s_info;
    r.bad = s_bad;
    return r;
}

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

// sA (the K stages) and sD (the delta tile, fp32) share the first region:
// sD is written only after every stage has been consumed.
__host__ __device__ inline SmemLayout smem_layout(int R, int r_slot, int nch_tile, int n_pos, int stages)
{
    SmemLayout L;
    const size_t sa = sizeof(bf16_t) * stages * R * kLds;
    const size_t sd = sizeof(float) * kRB * nch_tile * 8;
    L.a = 0;
    L.x = align128(sa > sd ? sa : sd);
    L.vpart = L.x + align128(sizeof(bf16_t) * stages * kRB * kLds);
    L.vfull = L.vpart + align128(sizeof(float) * kRB * R);
    L.b = L.vfull + align128(sizeof(float) * kRB * R);
    L.perm = L.b + align128(sizeof(bf16_t) * (nch_tile * 8 * r_slot + kBSlack));
    L.total = L.perm + (n_pos <= kPermStage ? sizeof(int) * n_pos : 0);
    return L;
}

template <int S>   // K stages in flight
__global__ void __launch_bounds__(kThreads, 2)
bgmv_fused_kernel(FusedParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int R = p.ps.n_proj * p.ps.r_slot;
    const int r_slot = p.ps.r_slot;
    const int r_pad = p.r_pad;
    const SmemLayout L = smem_layout(R, r_slot, p.nch_tile, p.n_pos, S);
    bf16_t* sA = reinterpret_cast<bf16_t*>(smem + L.a);        // [S][R][kLds]
    float* sD = reinterpret_cast<float*>(smem + L.a);          // [kRB][nch_tile*8], after the shrink
    bf16_t* sX = reinterpret_cast<bf16_t*>(smem + L.x);        // [S][kRB][kLds]
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
    const UnitInfo ui = find_unit<kThreads>(p, unit, s_perm, stage_perm);   // uniform across the cluster
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
    bool bad_row = false;
    if (tid < kRB) {
        int r = 0;
        if (tid < nrows) {
            r = stage_perm ? s_perm[pos0 + tid] : __ldg(p.perm + pos0 + tid);
            if (r < 0 || r >= p.n_rows) { bad_row = true; r = 0; }
        }
        s_rows[tid] = r;
    }

    // ---- this CTA's K range and output chunks ----
    const int k_begin = crank * p.kc;
    const int k_end = min(p.h_in, k_begin + p.kc);
    const int n_kt = k_end > k_begin ? (k_end - k_begin + kKT - 1) / kKT : 0;
    int total_ch = 0;   // none in the shrink-only form
    if (!p.v_out)
        for (int q = 0; q < p.ps.n_proj; ++q) total_ch += p.ps.width[q] >> 3;
    const int q_idx = part * p.cs + crank, q_n = p.n_parts * p.cs;
    const int ch_begin = static_cast<int>((static_cast<long long>(total_ch) * q_idx) / q_n);
    const int ch_end = static_cast<int>((static_cast<long long>(total_ch) * (q_idx + 1)) / q_n);
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
    // One bulk copy per projection segment of chunks [c0, c1), issued by threads 0..n_proj-1.
    auto copy_B = [&](int c0, int c1, uint64_t* bar) {
        if (tid < p.ps.n_proj) {
            int pc0 = 0;
            for (int q = 0; q < tid; ++q) pc0 += p.ps.width[q] >> 3;
            const int pc1 = pc0 + (p.ps.width[tid] >> 3);
            const int s = max(c0, pc0), e = min(c1, pc1);
            if (s < e) {
                const bf16_t* src = p.ps.B[tid] + (static_cast<size_t>(slot) * p.ps.width[tid] + (s - pc0) * 8) * r_slot;
                bulk_g2s(sB + static_cast<size_t>(s - c0) * 8 * r_slot, src, b_bytes(s, e), bar);
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

    // ---- set-up: barrier, zero slack, chunk map ----
    if (tid == 0) {
        mbar_init(&s_barB, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    for (int i = tid; i < kBSlack / 8; i += kThreads)
        reinterpret_cast<uint4*>(sB + p.nch_tile * 8 * r_slot)[i] = make_uint4(0, 0, 0, 0);
    map_chunks(ch_begin, tile0_end);
    if (__syncthreads_or(bad_row)) {
        // A malformed permutation: flag it and leave this unit's rows alone.
        // Every CTA of the cluster reads the same entries, so all return here.
        grid_dep_wait();
        if (tid == 0 && crank == 0 && part == 0) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }

    // ---- weights first: they do not depend on the preceding kernel ----
    if (ch_end > ch_begin) {
        if (tid == 0) mbar_expect(&s_barB, b_bytes(ch_begin, tile0_end));
        __syncthreads();
        copy_B(ch_begin, tile0_end, &s_barB);
    }
#pragma unroll
    for (int st = 0; st < S; ++st) {
        if (st < n_kt) copy_A(st, st);
        cp_async_commit();
    }

    bool waited = false;
    if (!p.x_ready) {
        grid_dep_wait();
        waited = true;
    }
#pragma unroll
    for (int st = 0; st < S; ++st) {
        if (st < n_kt) copy_X(st, st);
        cp_async_commit();
    }

    // ---- shrink: 16 rows x R ranks x this CTA's K range on tensor cores ----
    const int n_tiles = R / 8;                  // 8 ranks per mma tile; <= 16
    bool failed = false;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int kt = 0; kt < n_kt; ++kt) {
        // groups so far: {A_0}..{A_S-1} {X_0}..{X_S-1}, then one per
        // iteration; stage kt is complete once at most S-1 groups are pending
        cp_async_wait<S - 1>();
        __syncthreads();
        const int buf = kt % S;
        const bf16_t* xs = sX + buf * kRB * kLds;
        const bf16_t* as = sA + buf * R * kLds;
#pragma unroll
        for (int ks = 0; ks < kKT / 16; ++ks) {
            const int mi = lane >> 3, mr = lane & 7;
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(smem_u32(xs + ((mi & 1) * 8 + mr) * kLds + ks * 16 + (mi >> 1) * 8), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tile = warp + nt * 8;
                if (tile < n_tiles) {
                    uint32_t b0, b1;
                    const int l = lane & 15;
                    ldmatrix_x2(smem_u32(as + (tile * 8 + (l & 7)) * kLds + ks * 16 + (l >> 3) * 8), b0, b1);
                    mma_bf16_16816(acc[nt], a0, a1, a2, a3, b0, b1);
                }
            }
        }
        __syncthreads();                        // every warp is done with this buffer
        if (kt + S < n_kt) {                    // refill it with stage kt + S
            copy_A(kt + S, buf);
            copy_X(kt + S, buf);
        }
        cp_async_commit();
    }
    cp_async_wait<0>();
    {
        const int gr = lane >> 2, q2 = (lane & 3) * 2;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int tile = warp + nt * 8;
            if (tile < n_tiles) {
                const int j = tile * 8 + q2;
                vpart[gr * R + j] = acc[nt][0];
                vpart[gr * R + j + 1] = acc[nt][1];
                vpart[(gr + 8) * R + j] = acc[nt][2];
                vpart[(gr + 8) * R + j + 1] = acc[nt][3];
            }
        }
    }
    __shared__ int s_cta_fail, s_any_fail;
    failed = __syncthreads_or(failed);
    if (tid == 0) s_cta_fail = failed ? 1 : 0;
    __syncthreads();

    // ---- cluster reduction of the fp32 partials through DSMEM ----
    cluster_arrive();
    cluster_wait();
    if (tid == 0) {   // a peer whose copies timed out has no valid partials
        int any = 0;
        for (int c = 0; c < p.cs; ++c) {
            int f;
            asm("ld.shared::cluster.b32 %0, [%1];\n" : "=r"(f) : "r"(map_rank(smem_u32(&s_cta_fail), c)));
            any |= f;
        }
        s_any_fail = any;
    }
    if (p.v_out) {
        // Shrink only: the cluster's CTAs share the reduction of the unit's
        // rows and store v (fp32) for the grouped expand that follows.  The
        // store waits for the preceding grid, which may still read v.
        __syncthreads();                        // s_any_fail
        if (!waited) {
            grid_dep_wait();
            waited = true;
        }
        const bool ok = s_any_fail == 0;
        const int n2 = nrows * R / 2;
        const uint32_t base = smem_u32(vpart);
        for (int i = crank * kThreads + tid; i < n2; i += kThreads * p.cs) {
            float2 part2[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (c < p.cs) part2[c] = ld_dsmem_f2(map_rank(base + i * 8, c));
            float2 s = part2[0];
#pragma unroll
            for (int c = 1; c < 16; ++c) {
                if (c < p.cs) {
                    s.x += part2[c].x;
                    s.y += part2[c].y;
                }
            }
            const int t = (2 * i) / R, j = 2 * i - t * R;
            if (ok) *reinterpret_cast<float2*>(p.v_out + static_cast<size_t>(s_rows[t]) * p.ld_v + j) = s;
        }
    } else {
        const int n2 = kRB * R / 2;   // all 16 rows: rows past nrows sum to zero
        const uint32_t base = smem_u32(vpart);
        for (int i = tid; i < n2; i += kThreads) {
            float2 part2[16];         // all peers' loads in flight, then a fixed-order sum
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (c < p.cs) part2[c] = ld_dsmem_f2(map_rank(base + i * 8, c));
            float2 s = part2[0];
#pragma unroll
            for (int c = 1; c < 16; ++c) {
                if (c < p.cs) {
                    s.x += part2[c].x;
                    s.y += part2[c].y;
                }
            }
            reinterpret_cast<float2*>(vfull)[i] = s;
        }
    }
    cluster_arrive();   // this CTA no longer reads its peers' partials
    __syncthreads();
    failed = s_any_fail != 0;
    if (ch_end > ch_begin && !mbar_wait(&s_barB, 0)) failed = true;   // B' of the first tile
    failed = __syncthreads_or(failed);

    // ---- expand on tensor cores (16 rows x 8 columns per chunk), delta to sD ----
    const int gr = lane >> 2, q2 = (lane & 3) * 2;
    unsigned b_phase = 1;
    for (int c0 = ch_begin; c0 < ch_end; c0 += p.nch_tile) {
        const int c1 = min(ch_end, c0 + p.nch_tile);
        const int nch = c1 - c0;
        if (c0 != ch_begin) {                   // later tiles: fresh chunk map and B'
            __syncthreads();
            map_chunks(c0, c1);
            fence_proxy_async();
            if (tid == 0) mbar_expect(&s_barB, b_bytes(c0, c1));
            __syncthreads();
            copy_B(c0, c1, &s_barB);
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
            const int ld_d = nch * 8;
            *reinterpret_cast<float2*>(sD + gr * ld_d + ci * 8 + q2) = make_float2(d[0], d[1]);
            *reinterpret_cast<float2*>(sD + (gr + 8) * ld_d + ci * 8 + q2) = make_float2(d[2], d[3]);
        }
        __syncthreads();
        if (!waited && !p.y_ready) {
            grid_dep_wait();   // y may be the preceding kernel's output
            waited = true;
        }
        // ---- read-modify-write of y: 16-byte pieces, coalesced along each row ----
        if (!failed) {
            constexpr int kPairs = kRB * kMaxChunks / kThreads;
            uint4 yo[kPairs];
#pragma unroll
            for (int q = 0; q < kPairs; ++q) {
                const int i = tid + q * kThreads;
                if (i < nrows * nch) {
                    const int t = i / nch, ci = i - t * nch;
                    yo[q] = *reinterpret_cast<const uint4*>(p.y + static_cast<size_t>(s_rows[t]) * p.ld_y +
                                                            p.ps.out_off[s_cp[ci]] + s_ccol[ci]);
                }
            }
#pragma unroll
            for (int q = 0; q < kPairs; ++q) {
                const int i = tid + q * kThreads;
                if (i < nrows * nch) {
                    const int t = i / nch, ci = i - t * nch;
                    const float4* dp = reinterpret_cast<const float4*>(sD + t * nch * 8 + ci * 8);
                    const float4 d0 = dp[0], d1 = dp[1];
                    const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                    *reinterpret_cast<uint4*>(p.y + static_cast<size_t>(s_rows[t]) * p.ld_y +
                                              p.ps.out_off[s_cp[ci]] + s_ccol[ci]) = add_round8(yo[q], dd);
                }
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

// ---- grouped expand (second half of the two-launch form) --------------------
//
// Wide outputs (more columns than one cluster expands in two tiles) take
// two launches: the kernel above in its shrink-only form stores fp32 v per
// decode row, then this kernel streams B' in blocks of kGxCols columns,
// one CTA per (unit, block), many CTAs per SM.  A block of B'[slot] is
// contiguous ([columns][r_slot] bf16): each warp's 64 columns land in
// shared memory with one bulk copy, issued before the grid dependency
// resolves, and the warp proceeds as soon as its own part has arrived.
// The y pieces the warp will update are loaded while B' is in flight, so a
// CTA waits on memory twice, not once per tile.
//
// Tensor-core form (mma.sync m16n8k16, fp32 accumulate), transposed so the
// columns fill M and the rows N: d^T[col][t] = sum_j B'[col][j] v[t][j],
// 16 columns x 8 rows per tile, v split into bf16 hi + lo as above.  K is
// permuted: in step (h, e) lane quad q carries ranks 8(q + 4h) + 4e + 0..3
// of both operands, so each lane reads whole 16-byte pieces of a B' row.

constexpr int kGxThreads = 128;
constexpr int kGxWarps = kGxThreads / 32;
constexpr int kGxCols = 256;                          // output columns per block
constexpr int kGxWarpCols = kGxCols / kGxWarps;       // 64: one bulk copy per warp
constexpr int kGxTiles = kGxWarpCols / 16;            // 16-column tiles per warp
constexpr int kGxLdD = 20;       // per-warp delta tile row stride (floats): conflict-free

struct GexParams {
    ProjSet ps;
    const float* v;           // [n_rows][ld_v] fp32, projection p at p*r_slot
    int ld_v;
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
    int upg;                  // > 0: unit = group * upg + sub (direct form); 0: scanned
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
    int pos0, nrows, slot;
    bool bad;
    if (p.upg > 0) {
        // Direct form: the unit names its group; all threads read the same
        // three words (one round trip, no block-wide scan).
        const int g = unit / p.upg, sub = unit - g * p.upg;
        const int s = __ldg(p.gstarts + g), e = __ldg(p.gstarts + g + 1);
        slot = __ldg(p.gslot + g);
        const bool sane = s >= 0 && e <= p.n_pos && s <= e && e - s <= p.upg * kRB;
        bad = !sane && sub == 0;
        pos0 = s + sub * kRB;
        nrows = sane ? min(kRB, e - pos0) : 0;
    } else {
        const UnitInfo ui = find_unit<kGxThreads>(p, unit, nullptr, false);
        bad = ui.bad;
        pos0 = ui.pos0;
        nrows = ui.found ? ui.nrows : 0;
        slot = ui.slot;
    }
    const bool flagger = blk == 0 && tid == 0;   // one CTA per unit reports
    if (nrows <= 0 || slot == -1) {
        if (blockIdx.x == 0 || bad) grid_dep_wait();
        if (bad && flagger) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }
    if (slot < -1 || slot >= p.n_slots) {
        grid_dep_wait();
        if (flagger) flag(p.status, LORA_DEV_SLOT_OUT_OF_RANGE);
        return;
    }
    bool bad_row = false;
    if (tid < kRB) {
        int r = 0;
        if (tid < nrows) {
            r = __ldg(p.perm + pos0 + tid);
            if (r < 0 || r >= p.n_rows) {
                bad_row = true;
                r = 0;
            }
        }
        s_rows[tid] = r;
    }
    if (tid < kGxWarps) mbar_init(&s_bar[tid], 1);
    if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    if (__syncthreads_or(bad_row)) {
        grid_dep_wait();
        if (flagger) flag(p.status, LORA_DEV_BAD_SEGMENT);
        return;
    }

    int pj, col0;
    block_proj(p.ps, blk, pj, col0);
    const int width = p.ps.width[pj];
    const int ncols = min(kGxCols, width - col0);          // a multiple of 8
    const int r_slot = p.ps.r_slot;
    const int wc0 = warp * kGxWarpCols;                    // this warp's first column in the block
    const int wcols = max(0, min(kGxWarpCols, ncols - wc0));
    if (wcols > 0 && lane == 0) {   // weights first: they do not depend on the preceding kernel
        const unsigned bytes = static_cast<unsigned>(wcols * r_slot * sizeof(bf16_t));
        mbar_expect(&s_bar[warp], bytes);
        bulk_g2s(smem + sizeof(bf16_t) * wc0 * r_slot,
                 p.ps.B[pj] + (static_cast<size_t>(slot) * width + col0 + wc0) * r_slot, bytes, &s_bar[warp]);
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

    // v fragments (the mma B operand), n-tile nt = rows 8nt..8nt+7:
    // b0 <- v[t][k0], v[t][k0+1]; b1 <- v[t][k0+2], v[t][k0+3], k0 = 8(q+4h)+4e.
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
                float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
                if (nt < n_nt && t < nrows && k0 < r_slot)
                    vv = *reinterpret_cast<const float4*>(p.v + static_cast<size_t>(s_rows[t]) * p.ld_v +
                                                          pj * r_slot + k0);
                split_hi_lo(vv.x, vv.y, bh[nt][h][e][0], bl[nt][h][e][0]);
                split_hi_lo(vv.z, vv.w, bh[nt][h][e][1], bl[nt][h][e][1]);
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
    if (bad && flagger) flag(p.status, LORA_DEV_BAD_SEGMENT);
}

int env_int(const char* name, int dflt)
{
    const char* e = std::getenv(name);
    return (e && *e) ? std::atoi(e) : dflt;
}

}  // namespace

bool fused_decode_supported(int n_proj, int r_slot)
{
    // <= 2 rank tiles of 8 per warp in the shrink; <= 4 K steps of 16 in the expand
    return r_slot <= 64 && n_proj * r_slot <= 2 * 8 * 8 && r_slot % 8 == 0;
}

cudaError_t launch_bgmv_fused(bf16_t* y, int ld_y, const bf16_t* x, int ld_x, int h_in, const ProjSet& ps,
                              const int32_t* perm, const int32_t* gstarts, const int32_t* gslot, int n_groups,
                              int n_pos, int max_group_len, int n_rows, int n_slots, unsigned flags,
                              float* v_ws, int32_t* status, cudaStream_t stream)
{
    if (n_pos <= 0 || n_groups <= 0) return cudaSuccess;
    const int R = ps.n_proj * ps.r_slot;
    static int configured_device = -1;
    static int n_sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        for (auto fn : {bgmv_fused_kernel<kStages>, bgmv_fused_kernel<kStagesShrink>}) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    // Cluster size: split K over up to 8 CTAs while each keeps >= one stage
    // (8 measured faster than 16 on the 3B decode shapes: smaller grids let
    // more consecutive calls be resident at once under PDL); 16 for long K.
    int cs = 1;
    const int cs_max = h_in >= 8192 ? 16 : 8;
    while (cs < cs_max && h_in / (cs * 2) >= kKT) cs *= 2;
    const int cs_env = env_int("LORA_FUSED_CS", 0);
    if (cs_env > 0) cs = cs_env;
    // Units of <= 16 rows: at most ceil(longest group / 16) per group.
    int max_units = n_groups + n_pos / kRB;
    if (max_group_len > 0) max_units = min(max_units, n_groups * ((max_group_len + kRB - 1) / kRB));
    int total_ch = 0;
    for (int q = 0; q < ps.n_proj; ++q) total_ch += ps.width[q] / 8;
    // Column parts per unit (more clusters, each recomputing the shrink from
    // L2): one for the decode shapes here; wide outputs get enough parts that
    // each CTA expands at most two tiles of kMaxChunks chunks.
    int parts = 1;
    while (parts < 8 && (total_ch + cs * parts - 1) / (cs * parts) > 2 * kMaxChunks) parts *= 2;
    // Wider than that (and with a workspace for v): two launches, the
    // shrink-only form of this kernel and the grouped expand.
    // So do calls that stream many weights (the one-launch form keeps only
    // two K stages in flight per CTA and expands in the same CTAs).
    const double weight_bytes =
        static_cast<double>(n_groups) * sizeof(bf16_t) * (static_cast<double>(R) * h_in + 8.0 * total_ch * ps.r_slot);
    int split = env_int("LORA_FUSED_SPLIT", -1);
    if (split < 0) split = (parts > 1 || weight_bytes >= kSplitWeightBytes) ? 1 : 0;
    if (!v_ws) split = 0;
    if (split) {
        // The shrink-only clusters only need to cover the SMs once: fewer
        // CTAs per unit each stream a longer K range through more stages.
        parts = 1;
        cs = 1;
        while (cs < 16 && static_cast<long long>(max_units) * cs < n_sms && h_in / (cs * 2) >= kKT) cs *= 2;
        if (cs_env > 0) cs = cs_env;
    }
    parts = env_int("LORA_FUSED_PARTS", parts);
    const int per_cta = (total_ch + cs * parts - 1) / (cs * parts);
    const int nch_tile = split ? 1 : min(kMaxChunks, max(1, per_cta));

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
    p.kc = ((h_in + cs - 1) / cs + 15) / 16 * 16;
    p.n_parts = parts;
    p.cs = cs;
    p.nch_tile = nch_tile;
    p.r_pad = (ps.r_slot + 15) / 16 * 16;
    p.x_ready = (flags & LORA_APPLY_X_READY) ? 1 : 0;
    p.y_ready = (flags & LORA_APPLY_Y_READY) ? 1 : 0;
    p.v_out = split ? v_ws : nullptr;
    p.ld_v = R;
    p.status = status;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(max_units * parts * cs));
    cfg.blockDim = dim3(kThreads);
    const int stages = (split && env_int("LORA_SHRINK_STAGES", kStagesShrink) == kStagesShrink) ? kStagesShrink
                                                                                                : kStages;
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
    e = stages == kStagesShrink ? cudaLaunchKernelEx(&cfg, bgmv_fused_kernel<kStagesShrink>, p)
                                : cudaLaunchKernelEx(&cfg, bgmv_fused_kernel<kStages>, p);
    note_launch();
    if (e != cudaSuccess || !split) return e;

    GexParams gp{};
    gp.ps = ps;
    gp.v = v_ws;
    gp.ld_v = R;
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
    gp.status = status;
    // Direct unit numbering (group, sub-unit) unless the longest group makes
    // that grid much larger than the scanned one.
    const long long upg = max_group_len > 0 ? (max_group_len + kRB - 1) / kRB : 0;
    const long long scanned_units = n_groups + n_pos / kRB;
    gp.upg = (upg > 0 && n_groups * upg <= 2 * scanned_units) ? static_cast<int>(upg) : 0;
    const long long units = gp.upg ? n_groups * upg : max_units;
    const long long n_ctas = units * gp.n_blocks;
    if (n_ctas > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t gcfg = {};
    gcfg.gridDim = dim3(static_cast<unsigned>(n_ctas));
    gcfg.blockDim = dim3(kGxThreads);
    gcfg.dynamicSmemBytes = sizeof(bf16_t) * kGxCols * ps.r_slot;   // <= 32 KB
    gcfg.stream = stream;
    cudaLaunchAttribute gattr;
    gattr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    gattr.val.programmaticStreamSerializationAllowed = 1;
    gcfg.attrs = &gattr;
    gcfg.numAttrs = (flags & LORA_APPLY_NO_PDL) ? 0 : 1;
    e = cudaLaunchKernelEx(&gcfg, bgmv_group_expand_kernel, gp);
    note_launch();
    return e;
}

}  // namespace lora
