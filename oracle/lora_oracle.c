/*
 * lora_oracle.c -- plain, slow, fp64 CPU oracle for the multi-LoRA delta.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * legs of the benchmark (its host baseline and its reference arm) may load
 * this library.  It shares no code,
 * header, table or helper with the CUDA library under lora_serving_gb300/,
 * and it must never sit on the product path.
 *
 * Sources (page title, section):
 *   [MLS]  "Multi-LoRA serving: one base, many adapters" (interview note),
 *          sections "direct answer" and "interviewer follow-ups".
 *   [TGI]  "Text Generation Inference multi-LoRA adapter serving in
 *          practice: LORA_ADAPTERS config and SGMV/BGMV kernels",
 *          section "implementation 3. weight preprocessing" and
 *          "4. SGMV and BGMV at inference".
 *   [VLLM] "How vLLM attaches a different LoRA adapter per request in
 *          offline inference", steps 2 and 3.
 *
 * What is computed (plain definition, no blocking or reordering):
 *   For a row t whose adapter slot is k >= 0 and a projection with output
 *   slice [off, off+w):
 *       s_k   = alpha_k / r_k, or alpha_k / sqrt(r_k) with rsLoRA   [TGI 3]
 *       B'_k  = bf16_rne(s_k * B_k)      (scale folded into lora_B) [TGI 3]
 *       v     = A_k x_t                  (rank-r intermediate)      [MLS]
 *       delta = B'_k v                                              [MLS]
 *       y[t, off+j] = bf16_rne(y_in[t, off+j] + delta[j])
 *   Rows whose id is -1 run the base model only: y is left untouched
 *   [VLLM step 3, "None" entries].  A is stored [r][h_in] and B [out][r],
 *   the peft orientation of Delta W = B A with B in R^{d x r}, A in R^{r x k}
 *   [MLS].  All arithmetic is in double; the only roundings are the two
 *   bf16 roundings named above.
 *
 * Metadata (segments and gather form), the reading used where the pages
 * are silent:
 *   - prefill segments: maximal runs of equal id in row order over
 *     [0, n_prefill) ("variable-length segments", [TGI 4]); runs of -1 are
 *     kept as segments whose slot is -1.
 *   - gather form of the decode rows [n_prefill, n_rows): rows sorted by
 *     slot ascending, ties kept in row order, rows with id -1 last; one
 *     group per distinct id present.
 *
 * Parity pins: every function below is checked by the CPU tests against
 * closed forms, brute force, the merged-weight identity and invariants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- bf16 <-> double ------------------------------------------------ */

/* A bf16 value is the upper 16 bits of an IEEE binary32 value. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16, ties to even, in ONE rounding.
 * bf16 keeps 8 significant bits and the binary32 exponent range:
 * for |a| in [2^(e-1), 2^e) the spacing of bf16 values is 2^(e-8); below
 * the smallest normal 2^-126 the spacing is fixed at 2^-133.  Scaling by a
 * power of two is exact, and nearbyint() rounds to nearest-even in the
 * default rounding mode.
 */
uint16_t oracle_double_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    int q_exp = e - 8;
    if (q_exp < -133)
        q_exp = -133;
    double q = nearbyint(ldexp(a, -q_exp));
    double r = ldexp(q, q_exp);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80; /* rounds past the largest finite bf16 */
    float f = (float)r;      /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

void oracle_bf16_to_double_array(const uint16_t* src, double* dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_bf16_to_double(src[i]);
}

void oracle_double_to_bf16_array(const double* src, uint16_t* dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_double_to_bf16(src[i]);
}

/* ---- scaling and folding  [TGI 3] ------------------------------------ */

/* lora_alpha / r, or lora_alpha / r**0.5 when rsLoRA is enabled. */
double oracle_scale(double alpha, int r, int use_rslora)
{
    return use_rslora ? alpha / sqrt((double)r) : alpha / (double)r;
}

/* B'[j][c] = bf16_rne(s * B[j][c]) for a B of shape [out][r]. */
void oracle_fold_B(const uint16_t* B, int out, int r, double s, uint16_t* Bp)
{
    for (int64_t i = 0; i < (int64_t)out * r; ++i)
        Bp[i] = oracle_double_to_bf16(s * oracle_bf16_to_double(B[i]));
}

/* ---- metadata builder ------------------------------------------------ */

/*
 * Returns 0 on success, 1 if an id is outside [-1, n_slots), 2 if the row
 * counts are inconsistent.  Capacities: seg_starts n_prefill+1,
 * seg_slot n_prefill, perm n_rows-n_prefill, gseg_starts n_slots+2,
 * gseg_slot n_slots+1.
 */
int oracle_build_metadata(const int32_t* ids, int n_rows, int n_prefill, int n_slots,
                          int32_t* seg_starts, int32_t* seg_slot, int* n_segs,
                          int32_t* perm, int32_t* gseg_starts, int32_t* gseg_slot,
                          int* n_gsegs)
{
    if (n_rows < 0 || n_prefill < 0 || n_prefill > n_rows || n_slots <= 0)
        return 2;
    for (int t = 0; t < n_rows; ++t)
        if (ids[t] < -1 || ids[t] >= n_slots)
            return 1;

    /* (i) maximal runs of equal id over the prefill rows */
    int S = 0;
    int t = 0;
    while (t < n_prefill) {
        int u = t;
        while (u < n_prefill && ids[u] == ids[t])
            ++u;
        seg_starts[S] = t;
        seg_slot[S] = ids[t];
        ++S;
        t = u;
    }
    seg_starts[S] = n_prefill;
    *n_segs = S;

    /* (ii) decode rows grouped by slot: 0, 1, ..., n_slots-1, then -1 */
    int G = 0;
    int pos = 0;
    for (int k = 0; k <= n_slots; ++k) {
        int want = (k == n_slots) ? -1 : k;
        int first = pos;
        for (int row = n_prefill; row < n_rows; ++row)
            if (ids[row] == want)
                perm[pos++] = row;
        if (pos > first) {
            gseg_starts[G] = first;
            gseg_slot[G] = want;
            ++G;
        }
    }
    gseg_starts[G] = pos;
    *n_gsegs = G;
    return 0;
}

/* ---- the delta ------------------------------------------------------- */

/*
 * Adapters are passed as one flat buffer per matrix plus a per-slot
 * element offset.  Slot k holds A_k as [rp_k][h_in] and B_k as [w][rp_k],
 * where rp_k is the stored rank (the true rank r_k, or a zero-padded
 * rank when checking padding invariance).  scale[k] is s_k.
 */

/* v[t][j] = sum_i A_k[j][i] * x[t][i], j < rp_k; other entries zero. */
void oracle_shrink(int n_rows, const int32_t* ids, const uint16_t* x, int64_t ld_x, int h_in,
                   const int* rp, const uint16_t* A_cat, const int64_t* A_off,
                   double* v, int64_t ld_v, int v_cols)
{
    for (int t = 0; t < n_rows; ++t) {
        double* vt = v + (int64_t)t * ld_v;
        for (int j = 0; j < v_cols; ++j)
            vt[j] = 0.0;
        int k = ids[t];
        if (k < 0)
            continue;
        const uint16_t* A = A_cat + A_off[k];
        const uint16_t* xt = x + (int64_t)t * ld_x;
        for (int j = 0; j < rp[k]; ++j) {
            double acc = 0.0;
            for (int i = 0; i < h_in; ++i)
                acc += oracle_bf16_to_double(A[(int64_t)j * h_in + i]) * oracle_bf16_to_double(xt[i]);
            vt[j] = acc;
        }
    }
}

/* d[t][c] = sum_j B'_k[c][j] * v[t][j] with B'_k = bf16_rne(s_k * B_k).
 * Each slot used by some row is folded once, on first use. */
static void expand_rows(int n_rows, const int32_t* ids, const double* v, int64_t ld_v,
                        int w, const int* rp, const double* scale,
                        const uint16_t* B_cat, const int64_t* B_off,
                        double* d, int64_t ld_d)
{
    int n_slots = 0;
    for (int t = 0; t < n_rows; ++t)
        if (ids[t] + 1 > n_slots)
            n_slots = ids[t] + 1;
    uint16_t** folded = (uint16_t**)calloc((size_t)(n_slots > 0 ? n_slots : 1), sizeof(uint16_t*));
    for (int t = 0; t < n_rows; ++t) {
        double* dt = d + (int64_t)t * ld_d;
        for (int c = 0; c < w; ++c)
            dt[c] = 0.0;
        int k = ids[t];
        if (k < 0)
            continue;
        if (!folded[k]) {
            folded[k] = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)w * (size_t)(rp[k] > 0 ? rp[k] : 1));
            oracle_fold_B(B_cat + B_off[k], w, rp[k], scale[k], folded[k]);
        }
        const uint16_t* Bp = folded[k];
        const double* vt = v + (int64_t)t * ld_v;
        for (int c = 0; c < w; ++c) {
            double acc = 0.0;
            for (int j = 0; j < rp[k]; ++j)
                acc += oracle_bf16_to_double(Bp[(int64_t)c * rp[k] + j]) * vt[j];
            dt[c] = acc;
        }
    }
    for (int k = 0; k < n_slots; ++k)
        free(folded[k]);
    free(folded);
}

/* The unrounded fp64 delta d[t][0:w] of one projection (zero for base rows). */
void oracle_delta(int n_rows, const int32_t* ids, const uint16_t* x, int64_t ld_x, int h_in,
                  int w, const int* rp, const double* scale,
                  const uint16_t* A_cat, const int64_t* A_off,
                  const uint16_t* B_cat, const int64_t* B_off,
                  double* d, int64_t ld_d)
{
    int rmax = 0;
    for (int t = 0; t < n_rows; ++t)
        if (ids[t] >= 0 && rp[ids[t]] > rmax)
            rmax = rp[ids[t]];
    int64_t ld_v = rmax > 0 ? rmax : 1;
    double* v = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1) * (size_t)ld_v);
    oracle_shrink(n_rows, ids, x, ld_x, h_in, rp, A_cat, A_off, v, ld_v, rmax);
    expand_rows(n_rows, ids, v, ld_v, w, rp, scale, B_cat, B_off, d, ld_d);
    free(v);
}

/* y[t][off+c] = bf16_rne(y[t][off+c] + d[t][c]) for rows with id >= 0. */
static void add_round(int n_rows, const int32_t* ids, const double* d, int64_t ld_d,
                      uint16_t* y, int64_t ld_y, int off, int w)
{
    for (int t = 0; t < n_rows; ++t) {
        if (ids[t] < 0)
            continue;
        uint16_t* yt = y + (int64_t)t * ld_y + off;
        const double* dt = d + (int64_t)t * ld_d;
        for (int c = 0; c < w; ++c)
            yt[c] = oracle_double_to_bf16(oracle_bf16_to_double(yt[c]) + dt[c]);
    }
}

/* One projection of the LoRA delta applied in place to y (bf16 bits). */
void oracle_apply_projection(int n_rows, const int32_t* ids, const uint16_t* x, int64_t ld_x, int h_in,
                             uint16_t* y, int64_t ld_y, int off, int w,
                             const int* rp, const double* scale,
                             const uint16_t* A_cat, const int64_t* A_off,
                             const uint16_t* B_cat, const int64_t* B_off)
{
    double* d = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1) * (size_t)(w > 0 ? w : 1));
    oracle_delta(n_rows, ids, x, ld_x, h_in, w, rp, scale, A_cat, A_off, B_cat, B_off, d, w);
    add_round(n_rows, ids, d, w, y, ld_y, off, w);
    free(d);
}

/* The expand step alone: y[t][off+c] = bf16_rne(y + sum_j B'_k[c][j] v[t][j]). */
void oracle_expand(int n_rows, const int32_t* ids, const double* v, int64_t ld_v,
                   uint16_t* y, int64_t ld_y, int off, int w,
                   const int* rp, const double* scale,
                   const uint16_t* B_cat, const int64_t* B_off)
{
    double* d = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1) * (size_t)(w > 0 ? w : 1));
    expand_rows(n_rows, ids, v, ld_v, w, rp, scale, B_cat, B_off, d, w);
    add_round(n_rows, ids, d, w, y, ld_y, off, w);
    free(d);
}

/*
 * One projection of the LoRA linear layer ([MLS], direct answer: the base
 * product runs once for the whole batch and each row adds its own adapter's
 * delta; [TGI], implementation: the LoRA layer adds the adapter output to
 * the base layer's output):
 *     y[t][off+c] = bf16_rne( sum_k x[t][k] W[c][k] + d[t][c] )
 * with d the delta of oracle_delta (zero for base rows), the sum in double
 * and ONE rounding.  W holds this projection's base weight as [w][ld_w];
 * y_in is not read.
 */
void oracle_linear_projection(int n_rows, const int32_t* ids, const uint16_t* x, int64_t ld_x, int h_in,
                              const uint16_t* W, int64_t ld_w, uint16_t* y, int64_t ld_y, int off, int w,
                              const int* rp, const double* scale,
                              const uint16_t* A_cat, const int64_t* A_off,
                              const uint16_t* B_cat, const int64_t* B_off)
{
    double* d = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1) * (size_t)(w > 0 ? w : 1));
    oracle_delta(n_rows, ids, x, ld_x, h_in, w, rp, scale, A_cat, A_off, B_cat, B_off, d, w);
    for (int t = 0; t < n_rows; ++t) {
        const uint16_t* xt = x + (int64_t)t * ld_x;
        for (int c = 0; c < w; ++c) {
            const uint16_t* Wc = W + (int64_t)c * ld_w;
            double base = 0.0;
            for (int k = 0; k < h_in; ++k)
                base += oracle_bf16_to_double(xt[k]) * oracle_bf16_to_double(Wc[k]);
            y[(int64_t)t * ld_y + off + c] = oracle_double_to_bf16(base + d[(int64_t)t * w + c]);
        }
    }
    free(d);
}

/*
 * Merged weight for single-tenant serving ([MLS], interviewer follow-ups:
 * W' = W + B A gives the same model as the base plus the adapter's delta):
 *     W'[o][k] = bf16_rne(W[o][k] + sign * sum_{j < r} B'[o][j] A[j][k])
 * with sign = +1 (merge) or -1 (unmerge), the sum over the true rank r in
 * double, and one rounding.  W is [out][ld_w], A [r][ld_a], B' [out][ld_b].
 */
void oracle_merge(const uint16_t* W, int64_t ld_w, int out, int h_in, const uint16_t* A, int64_t ld_a,
                  const uint16_t* Bp, int64_t ld_b, int r, int sign, uint16_t* W_out)
{
    for (int o = 0; o < out; ++o) {
        for (int k = 0; k < h_in; ++k) {
            double d = 0.0;
            for (int j = 0; j < r; ++j)
                d += oracle_bf16_to_double(Bp[(int64_t)o * ld_b + j]) * oracle_bf16_to_double(A[(int64_t)j * ld_a + k]);
            W_out[(int64_t)o * ld_w + k] =
                oracle_double_to_bf16(oracle_bf16_to_double(W[(int64_t)o * ld_w + k]) + (double)sign * d);
        }
    }
}
