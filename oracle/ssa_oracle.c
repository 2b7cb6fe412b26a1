/*
 * ssa_oracle.c -- plain, slow CPU restatement of Stratified Sparse Attention
 * single-token decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; it exists so that tests, the package's smoke check and the
 * benchmark's CPU-baseline leg can compare the CUDA library against an
 * independent statement of the method.  It shares no code, header, table or
 * constant generator with the CUDA sources.
 *
 * Sources (cited by page title and section):
 *  [SSA]  "Stratified Sparse Attention speeds up decoding 2.96x on a 1M
 *         context" (news.hamidun.com), sections "Where sparse attention
 *         loses quality" and "How SSA splits the cache into strata": tokens
 *         with high estimates are read deterministically, the rest of the
 *         cache is sampled with probability proportional to an approximate
 *         attention estimate, and each sampled token is corrected by its
 *         inclusion probability so that the mass outside the chosen set is
 *         recovered.  Top-k, top-p and top-k+sampling hybrids are special
 *         cases.
 *  [FASA] "FASA: Frequency-Aware Sparse Attention" (gist.science 2602.03152),
 *         technical summary, section 3 (Method): Stage 1 "Token Importance
 *         Prediction" scores every token from a fixed, pre-calibrated subset
 *         of dominant RoPE frequency chunks only; Stage 2 "Focused Attention
 *         Computation" runs full-precision attention over the selected
 *         tokens only, at their original positions.
 *  [S2O]  "S2O: early stopping for sparse attention via online permutation"
 *         (gist.science 2602.22575), technical summary, Method section 3
 *         (kernel): the online-softmax state (m, l, acc); Method section 2
 *         (early stop): blocks are processed in descending estimated
 *         importance, the marginal gain of each processed block is tracked,
 *         and the computation ends once that gain falls below a preset
 *         threshold tau relative to the accumulated score.
 *  [Philox] J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
 *         Random Numbers: As Easy as 1, 2, 3", SC'11: the Philox-4x32
 *         counter-based generator (round function, multipliers and Weyl key
 *         schedule), 10 rounds.
 *
 * Readings where the pages are silent:
 *  - score: s_i = fl32(scale * max_g sum_j q[g][S_ch[j]] * Ks[i][j]), the
 *    dot products taken in double from exact bf16 inputs;
 *  - the deterministic stratum T is the top-k under the total order
 *    (orderkey(s) descending, index ascending);
 *  - the reference point m of the exponentials (p does not depend on it)
 *    is the lower edge of the bucket of the k-th element of that order (the
 *    largest s when k == 0), the bucket being the set of binary32 values
 *    sharing the top 12 bits of the order key (sign, exponent and top three
 *    mantissa bits); m is the smallest value of that bucket, so that
 *    s_(k) - m < |s_(k)| / 8 and every remainder term is at most
 *    exp(|s_(k)| / 8);
 *  - e_j = fl32(exp(fl32(s_j - m))) for j in R (the complement of T);
 *  - Z = sum over R of e_j, summed EXACTLY (every fp32 value is an integer
 *    multiple of 2^-149, so the sum is an exact big integer) and rounded to
 *    the nearest fp32 (ties to even);
 *  - p_j = min(1, fl32(fl32(B * e_j) / Z)); p_j = 1 if B is +inf; p_j = 0
 *    if Z == 0; p = 1 on T;
 *  - u_j = (x0 >> 8) * 2^-24 with x0 the first word of
 *    Philox4x32-10(key = (seed lo, seed hi), counter = (j, h_kv, b, 0));
 *    j in R is selected iff u_j < p_j (fp32 compare);
 *  - attention over the selected rows with logit
 *    scale * q.K_i - log p_i, in double; lse = log of the corrected
 *    denominator.
 *  - early stop (S2O section 2 applied to the selected rows of one unit):
 *    the rows are ordered by orderkey(s) descending, ties by position in
 *    the list; block b is rows [b * block, (b + 1) * block) of that order;
 *    for each query head g, after block b the gain D_g(b) is the block's
 *    share of the corrected softmax denominator and L_g(b) the denominator
 *    over blocks 0..b (both at a common reference point), and the step stops
 *    after the first block b with D_g(b) < tau * L_g(b) for every head g
 *    (block b included; block 0 is always processed; tau = 0 never stops).
 *    The output is the corrected attention over the processed blocks.
 *
 * Parity pins for every function here live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NONFINITE 6
#define ORACLE_ERR_OVERFLOW 5

/* ------------------------------------------------------------------ */
/* bit helpers                                                         */
/* ------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* bf16 is the top half of an IEEE binary32: widening is exact. */
static double bf16_value(uint16_t h) { return (double)f32_from_bits(((uint32_t)h) << 16); }

/* Order-preserving map from binary32 to uint32: x < y (as reals, with
 * -0 below +0) iff key(x) < key(y).  Negative numbers are bit-inverted,
 * non-negative numbers get the sign bit set. */
uint32_t oracle_orderkey(float x)
{
    uint32_t u = bits_from_f32(x);
    if (u & 0x80000000u) return ~u;
    return u | 0x80000000u;
}

/* Inverse of oracle_orderkey. */
static float value_of_orderkey(uint32_t key)
{
    return f32_from_bits((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

/* The smallest binary32 value whose order key shares the top 12 bits with
 * that of x (the lower edge of x's bucket). */
float oracle_bucket_floor(float x)
{
    return value_of_orderkey(oracle_orderkey(x) & 0xFFF00000u);
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10, from the SC'11 definition                            */
/* ------------------------------------------------------------------ */

/* One Philox-4x32 round: two 32x32->64 products of the even words with
 * the two round multipliers; the high halves are xored with the odd words
 * and the round key, and the words are permuted. */
static void philox_round(uint32_t x[4], const uint32_t k[2])
{
    const uint64_t prod_a = (uint64_t)0xD2511F53u * (uint64_t)x[0];
    const uint64_t prod_b = (uint64_t)0xCD9E8D57u * (uint64_t)x[2];
    const uint32_t a_hi = (uint32_t)(prod_a >> 32), a_lo = (uint32_t)prod_a;
    const uint32_t b_hi = (uint32_t)(prod_b >> 32), b_lo = (uint32_t)prod_b;
    uint32_t y[4];
    y[0] = b_hi ^ x[1] ^ k[0];
    y[1] = b_lo;
    y[2] = a_hi ^ x[3] ^ k[1];
    y[3] = a_lo;
    memcpy(x, y, sizeof y);
}

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {           /* Weyl sequence key schedule */
            k[0] += 0x9E3779B9u;   /* golden ratio */
            k[1] += 0xBB67AE85u;   /* sqrt(3) - 1 */
        }
        philox_round(x, k);
    }
    memcpy(out, x, sizeof x);
}

/* The uniform for token j of unit (b, h_kv): the top 24 bits of the first
 * output word, scaled into [0, 1) -- exact in binary32. */
float oracle_uniform(uint64_t seed, int64_t j, int32_t h_kv, int32_t b)
{
    uint32_t ctr[4] = {(uint32_t)j, (uint32_t)h_kv, (uint32_t)b, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return (float)(out[0] >> 8) * (1.0f / 16777216.0f);
}

/* ------------------------------------------------------------------ */
/* exact sum of non-negative binary32 values                           */
/* ------------------------------------------------------------------ */

/* A non-negative binary32 x equals M * 2^(sh - 149) with M < 2^24 an
 * integer, so x * 2^149 is the integer M << sh.  We keep the running sum
 * of those integers in 10 little-endian 32-bit limbs (320 bits); 2^31
 * terms of at most 2^128 * 2^149 each stay below 2^309. */
#define EXACT_LIMBS 10
typedef struct { uint32_t limb[EXACT_LIMBS]; } exact_sum;

static void exact_add(exact_sum* z, float x)
{
    uint32_t u = bits_from_f32(x);
    uint32_t expo = (u >> 23) & 0xffu;
    uint32_t mant = u & 0x7fffffu;
    int shift = 0;
    if (expo != 0) { mant |= 0x800000u; shift = (int)expo - 1; }
    if (mant == 0) return;
    int at = shift / 32;
    uint64_t piece = (uint64_t)mant << (shift % 32);
    uint64_t carry = 0;
    for (int i = at; i < EXACT_LIMBS; ++i) {
        uint64_t add = (i == at) ? (piece & 0xffffffffu) : (i == at + 1 ? (piece >> 32) : 0);
        uint64_t s = (uint64_t)z->limb[i] + add + carry;
        z->limb[i] = (uint32_t)s;
        carry = s >> 32;
        if (i > at + 1 && carry == 0) break;
    }
}

/* Round (sum * 2^-149) to the nearest binary32, ties to even. */
static float exact_to_f32(const exact_sum* z)
{
    int top = -1;
    for (int i = EXACT_LIMBS - 1; i >= 0 && top < 0; --i)
        if (z->limb[i])
            for (int b = 31; b >= 0; --b)
                if ((z->limb[i] >> b) & 1u) { top = 32 * i + b; break; }
    if (top < 0) return 0.0f;
#define BIT(n) ((n) >= 0 ? ((z->limb[(n) / 32] >> ((n) % 32)) & 1u) : 0u)
    if (top < 24) {                      /* fits in 24 bits: exact */
        uint32_t v = 0;
        for (int b = top; b >= 0; --b) v = (v << 1) | BIT(b);
        return ldexpf((float)v, -149);
    }
    uint32_t mant = 0;
    for (int b = top; b > top - 24; --b) mant = (mant << 1) | BIT(b);
    uint32_t guard = BIT(top - 24);
    uint32_t sticky = 0;
    for (int b = top - 25; b >= 0; --b) sticky |= BIT(b);
#undef BIT
    if (guard && (sticky || (mant & 1u))) {
        mant += 1;
        if (mant == (1u << 24)) { mant >>= 1; top += 1; }
    }
    return ldexpf((float)mant, top - 23 - 149);
}

/* Exposed for the oracle's own pins: exact fp32-rounded sum of n values. */
float oracle_exact_sum_f32(const float* x, int64_t n)
{
    exact_sum z;
    memset(&z, 0, sizeof z);
    for (int64_t i = 0; i < n; ++i) exact_add(&z, x[i]);
    return exact_to_f32(&z);
}

/* ------------------------------------------------------------------ */
/* key summary (append-time gather of the dominant channels)           */
/* ------------------------------------------------------------------ */

/* [FASA] section 3, Stage 1: the dominant chunks are fixed per head; the
 * summary holds, for every cached key, only the channels S_ch[h_kv][0..d_sel). */
void oracle_pack_summary(const uint16_t* K, const int32_t* sel_ch, uint16_t* Ks,
                         int32_t Bt, int32_t Hkv, int32_t d, int32_t d_sel, int64_t N,
                         int64_t kv_sb, int64_t kv_sh, int64_t ks_sb, int64_t ks_sh)
{
    for (int32_t b = 0; b < Bt; ++b)
        for (int32_t h = 0; h < Hkv; ++h)
            for (int64_t i = 0; i < N; ++i)
                for (int32_t j = 0; j < d_sel; ++j)
                    Ks[b * ks_sb + h * ks_sh + i * d_sel + j] =
                        K[b * kv_sb + h * kv_sh + i * d + sel_ch[h * d_sel + j]];
}

/* ------------------------------------------------------------------ */
/* stage 1: approximate score                                          */
/* ------------------------------------------------------------------ */

/* [FASA] section 3, Stage 1 (online scoring from the dominant chunks only);
 * [SSA] "How SSA splits the cache into strata" (approximate estimates).
 * The query heads of one GQA group share the KV head; their estimates are
 * combined by max.  s_hat is [Bt][Hkv][N]. */
void oracle_score(const uint16_t* q, const uint16_t* Ks, const int32_t* sel_ch,
                  int32_t Bt, int32_t Hq, int32_t Hkv, int32_t d, int32_t d_sel, int64_t N,
                  int64_t ks_sb, int64_t ks_sh, float scale, float* s_hat)
{
    const int32_t G = Hq / Hkv;
    const int64_t units = (int64_t)Bt * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int32_t b = (int32_t)(unit / Hkv), h = (int32_t)(unit % Hkv);
        double* qs = (double*)malloc(sizeof(double) * (size_t)G * (size_t)d_sel);
        for (int32_t g = 0; g < G; ++g)
            for (int32_t j = 0; j < d_sel; ++j)
                qs[g * d_sel + j] = bf16_value(q[((int64_t)b * Hq + (int64_t)h * G + g) * d +
                                                 sel_ch[h * d_sel + j]]);
        const uint16_t* kb = Ks + b * ks_sb + h * ks_sh;
        float* out = s_hat + unit * N;
        for (int64_t i = 0; i < N; ++i) {
            double best = -INFINITY;
            for (int32_t g = 0; g < G; ++g) {
                double dot = 0.0;
                for (int32_t j = 0; j < d_sel; ++j)
                    dot += qs[g * d_sel + j] * bf16_value(kb[i * d_sel + j]);
                if (dot > best) best = dot;
            }
            out[i] = (float)((double)scale * best);
        }
        free(qs);
    }
}

/* ------------------------------------------------------------------ */
/* stage 2: stratified selection for one (b, h_kv) unit                 */
/* ------------------------------------------------------------------ */

typedef struct { uint32_t key; int32_t idx; } ranked;

/* total order: key descending, then index ascending */
static int ranked_cmp(const void* pa, const void* pb)
{
    const ranked* a = (const ranked*)pa;
    const ranked* b = (const ranked*)pb;
    if (a->key != b->key) return a->key > b->key ? -1 : 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

/* [SSA] "How SSA splits the cache into strata": T = the k tokens with the
 * highest estimates (read deterministically); every other token j is kept
 * with probability p_j proportional to its approximate attention
 * exp(s_j - m), scaled so that the expected number of samples is the budget
 * B (before clipping at one); the draw is Poisson (independent per token).
 * Output: the selected indices in ascending order with their p (1 on T).
 * Returns the count, or -1 on non-finite input, -2 when the list would
 * exceed cap.  m_out / z_out report m and the rounded normaliser; p_all
 * (may be NULL) receives p for every token.
 *
 * m_mode chooses the reference point m of the exponentials, which the
 * method leaves free (p is the same for every m in exact arithmetic):
 * 0 = the lower edge of the 12-bit order-key bucket of the k-th score (the
 * reading the library follows), 1 = the k-th score itself.  The oracle's
 * pins compare the two readings. */
int64_t oracle_select_unit_m(const float* s, int64_t N, int64_t top_k, float budget,
                             uint64_t seed, int32_t b, int32_t h_kv,
                             int32_t* idx, float* p, int64_t cap,
                             float* m_out, float* z_out, float* p_all, int32_t m_mode)
{
    for (int64_t i = 0; i < N; ++i)
        if (!isfinite(s[i])) return -1;
    if (m_out) *m_out = 0.0f;
    if (z_out) *z_out = 0.0f;
    if (N == 0) return 0;
    int64_t k = top_k < N ? top_k : N;

    ranked* order = (ranked*)malloc(sizeof(ranked) * (size_t)N);
    for (int64_t i = 0; i < N; ++i) { order[i].key = oracle_orderkey(s[i]); order[i].idx = (int32_t)i; }
    qsort(order, (size_t)N, sizeof(ranked), ranked_cmp);

    /* in_T[i] = 1 for the top-k stratum */
    unsigned char* in_T = (unsigned char*)calloc((size_t)N, 1);
    for (int64_t r = 0; r < k; ++r) in_T[order[r].idx] = 1;
    const float s_k = s[order[(k > 0 ? k : 1) - 1].idx];   /* the k-th score (the largest if k = 0) */
    const float m = (m_mode == 1) ? s_k : oracle_bucket_floor(s_k);

    /* normaliser over the remainder, summed exactly */
    float* e = (float*)malloc(sizeof(float) * (size_t)N);
    exact_sum zsum;
    memset(&zsum, 0, sizeof zsum);
    for (int64_t j = 0; j < N; ++j) {
        if (in_T[j]) { e[j] = 0.0f; continue; }
        const float diff = s[j] - m;                  /* binary32 subtraction */
        e[j] = (float)exp((double)diff);              /* correctly rounded in practice */
        exact_add(&zsum, e[j]);
    }
    const float Z = exact_to_f32(&zsum);
    if (m_out) *m_out = m;
    if (z_out) *z_out = Z;

    int64_t count = 0;
    int overflow = 0;
    for (int64_t j = 0; j < N; ++j) {
        float pj;
        if (in_T[j]) {
            pj = 1.0f;
            if (p_all) p_all[j] = 1.0f;
        } else {
            if (isinf(budget)) pj = 1.0f;
            else if (Z == 0.0f) pj = 0.0f;
            else {
                const float t = budget * e[j];         /* binary32 product */
                const float ratio = t / Z;             /* binary32 quotient */
                pj = ratio < 1.0f ? ratio : 1.0f;
            }
            if (p_all) p_all[j] = pj;
            const float u = oracle_uniform(seed, j, h_kv, b);
            if (!(u < pj)) continue;
        }
        if (count < cap) { idx[count] = (int32_t)j; p[count] = pj; }
        else overflow = 1;
        ++count;
    }
    free(e); free(in_T); free(order);
    return overflow ? -2 : count;
}

/* The selection with the library's reading of m (bucket edge). */
int64_t oracle_select_unit(const float* s, int64_t N, int64_t top_k, float budget,
                           uint64_t seed, int32_t b, int32_t h_kv,
                           int32_t* idx, float* p, int64_t cap,
                           float* m_out, float* z_out, float* p_all)
{
    return oracle_select_unit_m(s, N, top_k, budget, seed, b, h_kv, idx, p, cap, m_out, z_out, p_all, 0);
}

/* ------------------------------------------------------------------ */
/* stage 3: attention over the selected rows with the inclusion weight  */
/* ------------------------------------------------------------------ */

/* [FASA] section 3, Stage 2: full-precision attention over the selected
 * tokens only; [SSA] strata section: the inclusion correction 1/p_i is
 * applied to both the numerator and the denominator, i.e. folded into the
 * logit as -log p_i.  [S2O] Method section 3: (m, l, acc) state -- the
 * oracle uses the plain two-pass form (max, then sums) in double.
 * out[g][:] and lse[g] for the G query heads of one unit. */
void oracle_attend_unit(const uint16_t* q_heads /* [G][d] */, const uint16_t* Kb, const uint16_t* Vb,
                        int32_t G, int32_t d, const int32_t* idx, const float* p, int64_t count,
                        float scale, float* out /* [G][d] */, float* lse /* [G] */)
{
    double* logit = (double*)malloc(sizeof(double) * (size_t)(count > 0 ? count : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    for (int32_t g = 0; g < G; ++g) {
        if (count == 0) {
            for (int32_t c = 0; c < d; ++c) out[g * d + c] = 0.0f;
            lse[g] = -INFINITY;
            continue;
        }
        double mx = -INFINITY;
        for (int64_t r = 0; r < count; ++r) {
            const uint16_t* kr = Kb + (int64_t)idx[r] * d;
            double dot = 0.0;
            for (int32_t c = 0; c < d; ++c) dot += bf16_value(q_heads[g * d + c]) * bf16_value(kr[c]);
            logit[r] = (double)scale * dot - log((double)p[r]);
            if (logit[r] > mx) mx = logit[r];
        }
        double den = 0.0;
        for (int32_t c = 0; c < d; ++c) acc[c] = 0.0;
        for (int64_t r = 0; r < count; ++r) {
            const double w = exp(logit[r] - mx);
            const uint16_t* vr = Vb + (int64_t)idx[r] * d;
            den += w;
            for (int32_t c = 0; c < d; ++c) acc[c] += w * bf16_value(vr[c]);
        }
        for (int32_t c = 0; c < d; ++c) out[g * d + c] = (float)(acc[c] / den);
        lse[g] = (float)(mx + log(den));
    }
    free(acc); free(logit);
}

/* Attention over the selected rows with S2O-style early stopping (see the
 * reading in the header).  s [count]: the rows' estimated scores, giving the
 * order.  ratio_out [ceil(count / block)] (may be NULL) receives, for every
 * block b of the order, max over g of D_g(b) / L_g(b) as if no block had
 * been skipped.  force_blocks >= 0 processes exactly that many blocks
 * (clamped to the number of blocks) instead of applying tau.  Returns the
 * number of blocks processed. */
typedef struct { uint32_t key; int64_t pos; } es_order_t;

static int es_order_cmp(const void* a, const void* b)
{
    const es_order_t* x = (const es_order_t*)a;
    const es_order_t* y = (const es_order_t*)b;
    if (x->key != y->key) return x->key > y->key ? -1 : 1;   /* key descending */
    return x->pos < y->pos ? -1 : (x->pos > y->pos ? 1 : 0); /* then position ascending */
}

int64_t oracle_attend_unit_early_stop(const uint16_t* q_heads /* [G][d] */, const uint16_t* Kb, const uint16_t* Vb,
                                      int32_t G, int32_t d, const int32_t* idx, const float* p, const float* s,
                                      int64_t count, float scale, float tau, int64_t block, int64_t force_blocks,
                                      float* out /* [G][d] */, float* lse /* [G] */, float* ratio_out)
{
    const int64_t nb = count > 0 ? (count + block - 1) / block : 0;
    es_order_t* ord = (es_order_t*)malloc(sizeof(es_order_t) * (size_t)(count > 0 ? count : 1));
    double* logit = (double*)malloc(sizeof(double) * (size_t)(count > 0 ? count : 1) * (size_t)G);
    double* M = (double*)malloc(sizeof(double) * (size_t)G);
    double* L = (double*)malloc(sizeof(double) * (size_t)G);
    double* acc = (double*)malloc(sizeof(double) * (size_t)G * (size_t)d);
    for (int64_t i = 0; i < count; ++i) { ord[i].key = oracle_orderkey(s[i]); ord[i].pos = i; }
    qsort(ord, (size_t)count, sizeof(es_order_t), es_order_cmp);
    /* the corrected logits of every row, in the order */
    for (int64_t r = 0; r < count; ++r) {
        const int64_t i = ord[r].pos;
        const uint16_t* kr = Kb + (int64_t)idx[i] * d;
        for (int32_t g = 0; g < G; ++g) {
            double dot = 0.0;
            for (int32_t c = 0; c < d; ++c) dot += bf16_value(q_heads[g * d + c]) * bf16_value(kr[c]);
            logit[r * G + g] = (double)scale * dot - log((double)p[i]);
        }
    }
    /* the gain ratio of every block, as if none were skipped */
    for (int32_t g = 0; g < G; ++g) { M[g] = -INFINITY; L[g] = 0.0; }
    int64_t used = -1;
    for (int64_t b = 0; b < nb; ++b) {
        const int64_t r0 = b * block, r1 = (r0 + block < count) ? r0 + block : count;
        double worst = 0.0;
        for (int32_t g = 0; g < G; ++g) {
            double mb = -INFINITY;
            for (int64_t r = r0; r < r1; ++r) if (logit[r * G + g] > mb) mb = logit[r * G + g];
            const double mn = mb > M[g] ? mb : M[g];
            double D = 0.0;
            for (int64_t r = r0; r < r1; ++r) D += exp(logit[r * G + g] - mn);
            const double Ln = (M[g] == -INFINITY ? 0.0 : L[g] * exp(M[g] - mn)) + D;
            const double ratio = Ln > 0.0 ? D / Ln : 0.0;
            if (ratio > worst) worst = ratio;
            M[g] = mn;
            L[g] = Ln;
        }
        if (ratio_out) ratio_out[b] = (float)worst;
        if (used < 0 && force_blocks < 0 && worst < (double)tau) used = b + 1;
    }
    if (force_blocks >= 0) used = force_blocks < nb ? force_blocks : nb;
    if (used < 0) used = nb;
    /* the corrected attention over the first `used` blocks */
    const int64_t rows = used * block < count ? used * block : count;
    for (int32_t g = 0; g < G; ++g) {
        if (rows == 0) {
            for (int32_t c = 0; c < d; ++c) out[g * d + c] = 0.0f;
            lse[g] = -INFINITY;
            continue;
        }
        double mx = -INFINITY;
        for (int64_t r = 0; r < rows; ++r) if (logit[r * G + g] > mx) mx = logit[r * G + g];
        double den = 0.0;
        for (int32_t c = 0; c < d; ++c) acc[c] = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
            const double w = exp(logit[r * G + g] - mx);
            const uint16_t* vr = Vb + (int64_t)idx[ord[r].pos] * d;
            den += w;
            for (int32_t c = 0; c < d; ++c) acc[c] += w * bf16_value(vr[c]);
        }
        for (int32_t c = 0; c < d; ++c) out[g * d + c] = (float)(acc[c] / den);
        lse[g] = (float)(mx + log(den));
    }
    free(acc); free(L); free(M); free(logit); free(ord);
    return used;
}

/* ------------------------------------------------------------------ */
/* the whole decode step                                               */
/* ------------------------------------------------------------------ */

/* score -> select -> attend for every unit.  Optional outputs (may be
 * NULL): s_hat [Bt][Hkv][N], idx/p [Bt][Hkv][cap], count [Bt][Hkv],
 * m/Z [Bt][Hkv].  Returns ORACLE_OK or an error code. */
int oracle_decode(const uint16_t* q, const uint16_t* K, const uint16_t* V, const uint16_t* Ks,
                  const int32_t* sel_ch, int32_t Bt, int32_t Hq, int32_t Hkv, int32_t d,
                  int32_t d_sel, int64_t N, int64_t kv_sb, int64_t kv_sh, int64_t ks_sb,
                  int64_t ks_sh, int64_t top_k, float budget, uint64_t seed, float scale,
                  float* out, float* lse, float* s_hat_out, int32_t* idx_out, float* p_out,
                  int64_t* count_out, int64_t cap, float* m_out, float* z_out)
{
    if (Bt < 0 || Hkv <= 0 || Hq % Hkv != 0 || N < 0 || top_k < 0 || !(budget >= 0.0f))
        return ORACLE_ERR_ARG;
    const int32_t G = Hq / Hkv;
    const int64_t units = (int64_t)Bt * Hkv;
    float* s_hat = s_hat_out ? s_hat_out : (float*)malloc(sizeof(float) * (size_t)(units * N + 1));
    oracle_score(q, Ks, sel_ch, Bt, Hq, Hkv, d, d_sel, N, ks_sb, ks_sh, scale, s_hat);
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int32_t b = (int32_t)(unit / Hkv), h = (int32_t)(unit % Hkv);
        const int64_t lcap = cap > 0 ? cap : N;
        int32_t* idx = idx_out ? idx_out + unit * cap : (int32_t*)malloc(sizeof(int32_t) * (size_t)(lcap + 1));
        float* p = p_out ? p_out + unit * cap : (float*)malloc(sizeof(float) * (size_t)(lcap + 1));
        float m = 0.0f, Z = 0.0f;
        int64_t cnt = oracle_select_unit(s_hat + unit * N, N, top_k, budget, seed, b, h,
                                         idx, p, lcap, &m, &Z, NULL);
        if (cnt < 0) {
#pragma omp critical
            status = (cnt == -1) ? ORACLE_ERR_NONFINITE : ORACLE_ERR_OVERFLOW;
            cnt = 0;
        }
        if (count_out) count_out[unit] = cnt;
        if (m_out) m_out[unit] = m;
        if (z_out) z_out[unit] = Z;
        const int64_t head0 = (int64_t)b * Hq + (int64_t)h * G;
        oracle_attend_unit(q + head0 * d, K + b * kv_sb + h * kv_sh, V + b * kv_sb + h * kv_sh,
                           G, d, idx, p, cnt, scale, out + head0 * d, lse + head0);
        if (!idx_out) free(idx);
        if (!p_out) free(p);
    }
    if (!s_hat_out) free(s_hat);
    return status;
}

/* Dense softmax attention over all N rows (no selection, no weights): the
 * limit every special case is compared against. */
void oracle_dense_attention(const uint16_t* q, const uint16_t* K, const uint16_t* V,
                            int32_t Bt, int32_t Hq, int32_t Hkv, int32_t d, int64_t N,
                            int64_t kv_sb, int64_t kv_sh, float scale, float* out, float* lse)
{
    const int32_t G = Hq / Hkv;
    const int64_t units = (int64_t)Bt * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int32_t b = (int32_t)(unit / Hkv), h = (int32_t)(unit % Hkv);
        int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N + 1));
        float* p = (float*)malloc(sizeof(float) * (size_t)(N + 1));
        for (int64_t i = 0; i < N; ++i) { idx[i] = (int32_t)i; p[i] = 1.0f; }
        const int64_t head0 = (int64_t)b * Hq + (int64_t)h * G;
        oracle_attend_unit(q + head0 * d, K + b * kv_sb + h * kv_sh, V + b * kv_sb + h * kv_sh,
                           G, d, idx, p, N, scale, out + head0 * d, lse + head0);
        free(idx); free(p);
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the number of host threads later calls use (n >= 1); returns the count now in force. */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
