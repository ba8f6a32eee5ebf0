// host.cpp -- host-side parts of the C ABI: adapter store preparation, the
// batch metadata builder, slot-rank selection and status strings.
//
// Sources: TGI multi-LoRA page, "implementation 3. weight preprocessing"
// (scale folded into lora_B, rank padded), "4. SGMV and BGMV" (segments);
// vLLM offline per-request LoRA page, step 2 (slot rank = largest rank),
// step 3 (None = base model) and "limits" (reject bad input up front).

#include <cmath>
#include <cstring>
#include <vector>

#include "lora.h"

namespace {

// Round a double to bf16, nearest-even, in one step, working on the bits of
// the binary64 value: keep the top 8 significant bits of the 53-bit
// significand (fewer below the bf16 normal range, where the spacing is
// fixed at 2^-133) and round on the dropped bits.
uint16_t bf16_from_double(double x)
{
    uint64_t u;
    std::memcpy(&u, &x, sizeof u);
    const uint16_t sign = static_cast<uint16_t>((u >> 48) & 0x8000u);
    const uint64_t mag = u & 0x7FFFFFFFFFFFFFFFull;
    if (mag > 0x7FF0000000000000ull) return 0x7FC0;         // NaN
    if (mag == 0x7FF0000000000000ull) return sign | 0x7F80; // inf
    const int biased = static_cast<int>(mag >> 52);
    if (biased == 0) return sign;  // binary64 subnormal: far below bf16's range
    const int e = biased - 1023;   // value = sig * 2^(e-52)
    const uint64_t sig = (1ull << 52) | (mag & ((1ull << 52) - 1));
    const bool normal = e >= -126;
    const int drop = normal ? 45 : 45 + (-126 - e);
    if (drop > 54) return sign;    // below half of the smallest subnormal
    uint64_t kept = sig >> drop;
    const uint64_t rem = sig & ((1ull << drop) - 1);
    const uint64_t half = 1ull << (drop - 1);
    if (rem > half || (rem == half && (kept & 1))) ++kept;
    if (!normal) return sign | static_cast<uint16_t>(kept);  // 128 = smallest normal
    int be = e + 127;
    if (kept == 256) { kept = 128; ++be; }
    if (be >= 255) return sign | 0x7F80;
    return sign | static_cast<uint16_t>((be << 7) | (kept & 0x7F));
}

double bf16_value(uint16_t b)
{
    uint32_t w = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &w, sizeof f);
    return static_cast<double>(f);
}

}  // namespace

extern "C" {

const char* lora_status_string(lora_status_t s)
{
    switch (s) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG: null pointer, negative size or bad count";
    case LORA_ERR_SHAPE: return "LORA_ERR_SHAPE: leading dimension too small or slice outside the row";
    case LORA_ERR_RANK_EXCEEDS_SLOT: return "LORA_ERR_RANK_EXCEEDS_SLOT: rank larger than the slot rank";
    case LORA_ERR_SLOT_RANGE: return "LORA_ERR_SLOT_RANGE: adapter id outside [-1, n_slots)";
    case LORA_ERR_ALIGNMENT: return "LORA_ERR_ALIGNMENT: pointer or size breaks the 16-byte rule";
    case LORA_ERR_METADATA: return "LORA_ERR_METADATA: segment table inconsistent with the rows";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE: workspace missing or too small";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA: a CUDA call failed";
    }
    return "LORA_ERR_UNKNOWN";
}

int lora_slot_rank(const int* ranks, int n)
{
    if (!ranks || n <= 0) return 0;
    int m = 0;
    for (int i = 0; i < n; ++i) {
        if (ranks[i] <= 0) return 0;
        if (ranks[i] > m) m = ranks[i];
    }
    return (m + 7) / 8 * 8;
}

lora_status_t lora_prepare_adapter(const lora_bf16_t* A, const lora_bf16_t* B, int r, int h_in,
                                   int out, double alpha, int use_rslora, int r_slot,
                                   lora_bf16_t* A_slot_out, lora_bf16_t* B_slot_out)
{
    if (!A || !B || !A_slot_out || !B_slot_out) return LORA_ERR_INVALID_ARG;
    if (r <= 0 || h_in <= 0 || out <= 0 || r_slot <= 0) return LORA_ERR_INVALID_ARG;
    if (r > r_slot || r_slot > LORA_MAX_RANK) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (r_slot % 8 != 0) return LORA_ERR_ALIGNMENT;
    const double s = use_rslora ? alpha / std::sqrt(static_cast<double>(r))
                                : alpha / static_cast<double>(r);
    for (int j = 0; j < r_slot; ++j) {
        lora_bf16_t* dst = A_slot_out + static_cast<size_t>(j) * h_in;
        if (j < r)
            std::memcpy(dst, A + static_cast<size_t>(j) * h_in, sizeof(lora_bf16_t) * h_in);
        else
            std::memset(dst, 0, sizeof(lora_bf16_t) * h_in);
    }
    for (int c = 0; c < out; ++c) {
        const lora_bf16_t* src = B + static_cast<size_t>(c) * r;
        lora_bf16_t* dst = B_slot_out + static_cast<size_t>(c) * r_slot;
        for (int j = 0; j < r_slot; ++j)
            dst[j] = j < r ? bf16_from_double(s * bf16_value(src[j])) : lora_bf16_t(0);
    }
    return LORA_OK;
}

lora_status_t lora_build_metadata(const int32_t* ids, int n_rows, int n_prefill, int n_slots,
                                  int32_t* seg_starts, int32_t* seg_slot, int* n_segs,
                                  int* max_seg_len, int32_t* perm, int32_t* gseg_starts,
                                  int32_t* gseg_slot, int* n_gsegs, int* max_gseg_len)
{
    if (n_rows < 0 || n_prefill < 0 || n_prefill > n_rows || n_slots <= 0)
        return LORA_ERR_INVALID_ARG;
    if ((n_rows > 0 && !ids) || !seg_starts || !n_segs || !gseg_starts || !n_gsegs)
        return LORA_ERR_INVALID_ARG;
    if ((n_prefill > 0 && !seg_slot) || (n_rows > n_prefill && (!perm || !gseg_slot)))
        return LORA_ERR_INVALID_ARG;
    for (int t = 0; t < n_rows; ++t)
        if (ids[t] < -1 || ids[t] >= n_slots) return LORA_ERR_SLOT_RANGE;

    // (i) prefill: one segment per maximal run of equal ids.
    int S = 0, longest = 0;
    for (int t = 0; t < n_prefill; ++t) {
        if (t == 0 || ids[t] != ids[t - 1]) {
            if (S > 0 && t - seg_starts[S - 1] > longest) longest = t - seg_starts[S - 1];
            seg_starts[S] = t;
            seg_slot[S] = ids[t];
            ++S;
        }
    }
    if (S > 0 && n_prefill - seg_starts[S - 1] > longest) longest = n_prefill - seg_starts[S - 1];
    seg_starts[S] = n_prefill;
    *n_segs = S;
    if (max_seg_len) *max_seg_len = longest;

    // (ii) decode: counting sort by key (slot, with -1 mapped after the last
    // slot), stable in row order.
    const int D = n_rows - n_prefill;
    std::vector<int> count(static_cast<size_t>(n_slots) + 2, 0);
    for (int t = n_prefill; t < n_rows; ++t) {
        const int key = ids[t] < 0 ? n_slots : ids[t];
        ++count[key + 1];
    }
    std::vector<int> next(static_cast<size_t>(n_slots) + 1, 0);
    int run = 0;
    for (int k = 0; k <= n_slots; ++k) { next[k] = run; run += count[k + 1]; }
    int G = 0, biggest = 0;
    for (int k = 0; k <= n_slots; ++k) {
        const int c = count[k + 1];
        if (c == 0) continue;
        gseg_starts[G] = next[k];
        gseg_slot[G] = k == n_slots ? -1 : k;
        if (c > biggest) biggest = c;
        ++G;
    }
    gseg_starts[G] = D;
    for (int t = n_prefill; t < n_rows; ++t) {
        const int key = ids[t] < 0 ? n_slots : ids[t];
        perm[next[key]++] = t;
    }
    *n_gsegs = G;
    if (max_gseg_len) *max_gseg_len = biggest;
    return LORA_OK;
}

}  // extern "C"
