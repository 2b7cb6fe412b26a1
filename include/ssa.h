/*
 * ssa.h -- libssa: Stratified Sparse Attention single-token decode on one
 * B300 (sm_103a).  Plain C ABI: raw pointers, sizes and a CUDA stream; no
 * framework types.
 *
 * One decode step for every (batch b, KV head h_kv) "unit" has three parts
 * (sources cited by page title and section):
 *
 *  (a) score  -- an approximate score s_i for every cached token i from the
 *      key summary: a fixed per-KV-head subset of d_sel channels S_ch,
 *      stored contiguously at append time ("FASA: Frequency-Aware Sparse
 *      Attention", section 3, Stage 1 "Token Importance Prediction": online
 *      scoring from the pre-calibrated dominant frequency chunks only).
 *      The G query heads of a GQA group are combined by max:
 *          s_i = fl32(scale * max_g sum_j q_g[S_ch[j]] * Ks[i][j]).
 *  (b) select -- ("Stratified Sparse Attention speeds up decoding 2.96x on a
 *      1M context", section "How SSA splits the cache into strata") the
 *      top-k tokens by s (ties to the lower index) are taken
 *      deterministically (stratum T); every other token j (the remainder R)
 *      is drawn independently with inclusion probability
 *          p_j = min(1, B * exp(s_j - m) / sum_{l in R} exp(s_l - m)),
 *      computed in fp32 as min(1, fl32(fl32(B * e_j) / Z)) with
 *      e_j = fl32(expf(fl32(s_j - m))) and Z the sum over R of e_j (summed
 *      with compensated arithmetic in a fixed order, rounded once); p does
 *      not depend on m, which is the lower edge of the 12-bit order-key
 *      bucket holding the k-th largest s (the largest when k = 0); using
 *      the uniform
 *          u_j = (x0 >> 8) * 2^-24,  x0 = word 0 of Philox4x32-10 with
 *          key (seed & 0xffffffff, seed >> 32), counter (j, h_kv, b, 0)
 *      (Salmon et al., SC'11); j is selected iff u_j < p_j.  p = 1 on T.
 *  (c) attend -- exact softmax attention over the selected rows at their
 *      original positions ("FASA", section 3, Stage 2 "Focused Attention
 *      Computation"), with the inclusion correction 1/p_i folded into the
 *      logit as -log p_i so that numerator and denominator are both
 *      corrected (SSA strata section: the correction recovers the attention
 *      mass outside the chosen set); split across CTAs and merged through
 *      the online-softmax state (m, l, acc) ("S2O", technical summary,
 *      Method section 3).
 *
 * Layouts (row-major, element strides; bf16 values are passed as their raw
 * 16-bit patterns, type ssa_bf16):
 *   q      [batch][n_q_heads][head_dim]                     contiguous
 *   K, V   [batch][n_kv_heads][ctx_len][head_dim]           token stride head_dim,
 *          batch / head strides kv_stride_b / kv_stride_h
 *   Ks     [batch][n_kv_heads][ctx_len][d_sel]              token stride d_sel,
 *          batch / head strides ks_stride_b / ks_stride_h
 *   sel_ch [n_kv_heads][d_sel] int32 channel ids in [0, head_dim)
 *   s_hat  [batch][n_kv_heads][ctx_len] fp32                contiguous
 *   idx, p [batch][n_kv_heads][list_cap]  selected token ids (ascending) and
 *          their inclusion probabilities; count [batch][n_kv_heads] int32
 *   out    [batch][n_q_heads][head_dim] fp32;  lse [batch][n_q_heads] fp32
 *          (natural log of the corrected softmax denominator; -inf and a
 *          zero output when nothing is selected)
 * Query head g of KV head h_kv is q head h_kv * G + g, G = n_q_heads / n_kv_heads.
 *
 * Supported: head_dim in {64, 128}; d_sel in {16, 32} (d_sel <= head_dim);
 * G in {1, 2, 4, 8}; 0 <= ctx_len <= 2^31 - 4097; top_k >= 0; budget >= 0 or +inf
 * (+inf: every token is kept with p = 1, i.e. dense attention).
 * Alignment: q, K, V, Ks and the workspace must be 16-byte aligned (the
 * workspace 256-byte aligned) and kv/ks strides multiples of 8 elements.
 *
 * K, V and Ks may be NULL when ctx_len == 0 (nothing is read).
 *
 * Memory tiers ("FASA: Frequency-Aware Sparse Attention", section 3,
 * Variants, FASA-M: the dominant-channel summary stays in GPU memory while
 * the full K and V rows are offloaded to host memory and fetched for the
 * selected tokens only): K and V may be pinned host memory mapped into the
 * device's address space at the same address (cudaHostAlloc /
 * cudaHostRegister on a device with unified addressing); the step then
 * gathers the selected rows over the host link and streams the summary from
 * HBM as usual.  q, Ks, the workspace and the outputs must be device memory.
 * Pageable host memory (and any pointer the device cannot read) is refused
 * with SSA_ERR_INVALID_ARG before anything is launched.
 *
 * Memory and ownership: every buffer, the workspace included, is allocated
 * and owned by the caller.  Device pointers unless stated otherwise.  The
 * library allocates no device memory (ssa_decode_static's built-in array,
 * below, is part of the loaded module).  The results of a call depend only
 * on its arguments: the workspace needs no initialisation (each call resets
 * what it uses) and carries nothing from one call to the next, apart from
 * the device status word at its start, which collects flags until
 * ssa_get_device_status reads and clears it (clear a new workspace once,
 * with that call or by zeroing it, before reading flags).  What the
 * library does keep, per process, is launch bookkeeping that never changes
 * a result: the kernels' raised shared-memory limits and occupancy queries
 * (per kernel and device), the driver entry point that encodes tensor maps,
 * and the device address of ssa_decode_static's array (per CUDA context).
 * Calls on different streams need different workspaces.
 *
 * Errors: every entry point validates its arguments on the host and returns
 * a status before launching anything.  All launches are asynchronous on the
 * given stream.  Problems only the device can see (a non-finite score, a
 * list longer than list_cap, an index out of range, a wait that timed out)
 * set bits in a status word inside the workspace; ssa_get_device_status()
 * synchronises the stream, reads and clears them.
 */
#ifndef LIBSSA_SSA_H
#define LIBSSA_SSA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t ssa_bf16; /* raw bfloat16 bit pattern */

typedef enum {
    SSA_OK = 0,
    SSA_ERR_INVALID_ARG = 1,     /* null pointer, bad size, bad stride, bad scalar */
    SSA_ERR_UNSUPPORTED = 2,     /* head_dim / d_sel / group size not built */
    SSA_ERR_WORKSPACE = 3,       /* workspace too small or misaligned */
    SSA_ERR_CUDA = 4,            /* a CUDA runtime call failed (no device, launch error) */
    SSA_ERR_OVERFLOW = 5,        /* device: a unit selected more than list_cap rows */
    SSA_ERR_NONFINITE = 6,       /* device: a score was NaN or infinite */
    SSA_ERR_DEVICE_TIMEOUT = 7,  /* device: an asynchronous copy did not arrive in time */
    SSA_ERR_BAD_INDEX = 8        /* device: a selected index or summary channel out of range */
} ssa_status;

/* The strata of a step ("Stratified Sparse Attention speeds up decoding 2.96x
 * on a 1M context", sections "Where sparse attention loses quality" and "How
 * SSA splits the cache into strata": pure top-k, top-p and hybrids of a
 * deterministic stratum with sampling are special cases of the strata). */
typedef enum {
    SSA_STRATA_SSA = 0,      /* top-k stratum; the remainder R drawn with p_j = min(1, B e_j / Z),
                                e_j = exp(s_j - m) (the method; ssa_decode / ssa_select) */
    SSA_STRATA_UNIFORM = 1,  /* top-k stratum; every remainder token drawn with the same
                                p = min(1, fl32(B / fl32(N - min(k, N)))) (1 for B = +inf):
                                the top-k + uniform-sampling hybrid */
    SSA_STRATA_TOP_P = 2     /* top-p stratum: the fewest tokens, in the top-k order, whose share
                                of the softmax of s over all N tokens reaches top_p (none for
                                top_p <= 0, all for top_p >= 1); the remainder drawn as in
                                SSA_STRATA_SSA with k = that size.  The shares are summed from
                                fp32 expf terms in exact fixed point (63 fractional bits), so a
                                size can differ by one from an exact computation only where the
                                top_p falls within a few fp32 roundings of a token's boundary */
} ssa_strata;

/* Device status bits (ssa_get_device_status). */
#define SSA_DEV_NONFINITE 0x1u
#define SSA_DEV_OVERFLOW 0x2u
#define SSA_DEV_TIMEOUT 0x4u
#define SSA_DEV_BAD_INDEX 0x8u

typedef struct {
    int32_t batch;        /* B_t >= 0 */
    int32_t n_q_heads;    /* H_q, a multiple of n_kv_heads */
    int32_t n_kv_heads;   /* H_kv >= 1 */
    int32_t head_dim;     /* d: 64 or 128 */
    int32_t d_sel;        /* summary channels: 16 or 32 */
    int32_t reserved;     /* must be 0 */
    int64_t ctx_len;      /* N: cached tokens, all visible */
    int64_t kv_stride_b;  /* K/V elements between batches (>= n_kv_heads*kv_stride_h) */
    int64_t kv_stride_h;  /* K/V elements between KV heads (>= ctx_len*head_dim) */
    int64_t ks_stride_b;  /* Ks elements between batches */
    int64_t ks_stride_h;  /* Ks elements between KV heads (>= ctx_len*d_sel) */
} ssa_shape;

/* Human-readable name of a status code (static string). */
const char* ssa_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int ssa_version(void);

/* Bytes of device workspace every entry point below needs for this shape
 * (about 22 bytes per cached token plus 32 KB per unit: scores, candidate
 * and selection lists sized for the worst case, 16-bit Philox prefixes,
 * histograms).
 * Independent of the stream, the device, the strides and list_cap (kept for
 * symmetry with the calls that take a list capacity); the four stride fields
 * may all be 0 (the paged cache's shape).  0 on invalid input. */
size_t ssa_workspace_bytes(const ssa_shape* shape, int64_t list_cap);

/* Append-time key summary (step a0): Ks[b][h][i][j] = K[b][h][i][sel_ch[h][j]]
 * for all i < ctx_len.  An out-of-range channel sets SSA_DEV_BAD_INDEX (the
 * channel is clamped).  Not part of the timed step. */
ssa_status ssa_pack_summary(const ssa_bf16* K, const int32_t* sel_ch, ssa_bf16* Ks,
                            void* ws, size_t ws_bytes, const ssa_shape* shape,
                            cudaStream_t stream);

/* Append step, the step just before the decode path ("FASA: Frequency-Aware
 * Sparse Attention", section 3, Stage 1: the dominant channels of a token's
 * key are stored contiguously when the token is appended):
 *   K[b][h][pos][:] = k_new[b][h][:],   V[b][h][pos][:] = v_new[b][h][:],
 *   Ks[b][h][pos][j] = k_new[b][h][sel_ch[h][j]]   for j < d_sel.
 * k_new, v_new: [batch][n_kv_heads][head_dim], contiguous, 16-byte aligned;
 * K, V, Ks: the cache in the layouts above, ctx_len being its capacity in
 * tokens; 0 <= pos < ctx_len (else SSA_ERR_INVALID_ARG).  Only row pos is
 * written.  An out-of-range channel sets SSA_DEV_BAD_INDEX (the channel is
 * clamped).  ws holds only the device status word here. */
ssa_status ssa_append(const ssa_bf16* k_new, const ssa_bf16* v_new, const int32_t* sel_ch, int64_t pos,
                      ssa_bf16* K, ssa_bf16* V, ssa_bf16* Ks, void* ws, size_t ws_bytes,
                      const ssa_shape* shape, cudaStream_t stream);

/* Worst-case list length per unit: ctx_len (every cached token selected, as
 * when top_k >= ctx_len or budget = +inf).  A list_cap of at least this
 * never overflows.  Strides as in ssa_workspace_bytes.  0 on invalid input. */
size_t ssa_select_capacity(const ssa_shape* shape);

/* Step (a): s_hat[b][h][i] for every token ("FASA: Frequency-Aware Sparse
 * Attention", section 3, Stage 1 "Token Importance Prediction": each token
 * scored from the dominant channels only; the query heads of a GQA group
 * combined by max). */
ssa_status ssa_score(const ssa_bf16* q, const ssa_bf16* Ks, const int32_t* sel_ch, float scale,
                     float* s_hat, void* ws, size_t ws_bytes, const ssa_shape* shape,
                     cudaStream_t stream);

/* Step (b): stratified selection from given scores ("Stratified Sparse
 * Attention speeds up decoding 2.96x on a 1M context", section "How SSA
 * splits the cache into strata": the top-k tokens read deterministically,
 * the rest sampled with probability proportional to the approximate
 * attention exp(s), each kept token carrying its inclusion probability p).
 * Writes idx / p (the
 * first count[u] entries of each unit's row of length list_cap, ascending
 * token order) and count.  A unit whose count exceeds list_cap keeps the
 * first list_cap entries and sets SSA_DEV_OVERFLOW; count still holds the
 * true number. */
ssa_status ssa_select(const float* s_hat, int64_t top_k, float budget, uint64_t seed,
                      int32_t* idx, float* p, int32_t* count, int64_t list_cap,
                      void* ws, size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream);

/* ssa_select with a choice of strata (ssa_strata; top_p is read for
 * SSA_STRATA_TOP_P only, top_k for the others).  The same Philox uniforms
 * decide every draw.  An unknown strata or a negative or NaN top_p is
 * SSA_ERR_INVALID_ARG. */
ssa_status ssa_select_strata(const float* s_hat, int strata, int64_t top_k, float top_p, float budget,
                             uint64_t seed, int32_t* idx, float* p, int32_t* count, int64_t list_cap,
                             void* ws, size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream);

/* Step (c): corrected attention over given selections (rows idx[u][0..min(count[u],
 * list_cap)) with probabilities p > 0): softmax over the logits
 * scale * q.K_i - log p_i ("FASA", section 3, Stage 2 "Focused Attention
 * Computation": exact attention over the selected rows at their original
 * positions; SSA strata section: each kept token corrected by its inclusion
 * probability, numerator and denominator alike).  An index outside
 * [0, ctx_len) or a p outside (0, 1] sets SSA_DEV_BAD_INDEX and the entry is
 * skipped. */
ssa_status ssa_attend(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V,
                      const int32_t* idx, const float* p, const int32_t* count, int64_t list_cap,
                      float scale, float* out, float* lse,
                      void* ws, size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream);

/* Step (c) with S2O-style early stopping ("S2O: early stopping for sparse
 * attention via online permutation", technical summary, Method section 2:
 * blocks processed in descending estimated importance, the marginal gain of
 * each tracked, the computation ended once that gain falls below a preset
 * threshold tau relative to the accumulated score).  Each unit's rows
 * (idx / p / count as in ssa_attend, idx ascending as ssa_select writes
 * them) are ordered by their scores s_hat[b][h][idx] ([batch][n_kv_heads]
 * [ctx_len], e.g. from ssa_score) descending, ties by list position, and
 * attended in blocks of 128 rows of that order; after block b the gain of
 * head g is the block's share D_g(b) of the corrected softmax denominator
 * L_g(b) over blocks 0..b, and the step stops after the first block with
 * D_g(b) < tau * L_g(b) for every head g of the unit (block 0 is always
 * kept; tau = 0 keeps every block, i.e. ssa_attend's result up to the
 * summation order; tau > 1 keeps block 0 only).  out / lse are the corrected
 * attention over the kept blocks; blocks_opt [batch][n_kv_heads] (may be
 * NULL) receives the number of blocks kept.  The blocks are attended in
 * parallel (each CTA of the unit a run of them) and the gain test is applied
 * when their partial results are merged, so every selected row is read; the
 * test decides which blocks enter the result.  A unit's list holds at most
 * 32768 rows here: a longer one keeps its first 32768 entries and sets
 * SSA_DEV_OVERFLOW.  tau must be >= 0 (+inf allowed). */
ssa_status ssa_attend_early_stop(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V,
                                 const int32_t* idx, const float* p, const int32_t* count, int64_t list_cap,
                                 const float* s_hat, float tau, float scale, float* out, float* lse,
                                 int32_t* blocks_opt, void* ws, size_t ws_bytes, const ssa_shape* shape,
                                 cudaStream_t stream);

/* The whole step, (a) -> (b) -> (c) ("Stratified Sparse Attention speeds up
 * decoding 2.96x on a 1M context": estimate, stratify, sample, correct; the
 * arguments follow its problem statement: query, KV cache, k, budget B,
 * seed), enqueued on `stream` as a chain of three kernels: initialise;
 * score (streams the key summary); and the unit kernel, whose CTAs per unit
 * select, decide and attend, then merge their partial results.  Each after
 * the first is a programmatic dependent launch.  s_hat_opt, idx_opt,
 * p_opt, count_opt may be NULL; when given they receive the intermediate
 * results (idx_opt / p_opt need list_cap entries per unit and are given
 * together).  A step that selects every token (top_k >= ctx_len or
 * budget = +inf) skips the selection (and the score kernel when s_hat_opt
 * is NULL). */
ssa_status ssa_decode(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V,
                      const ssa_bf16* Ks, const int32_t* sel_ch, int64_t top_k, float budget,
                      uint64_t seed, float scale, float* out, float* lse,
                      float* s_hat_opt, int32_t* idx_opt, float* p_opt, int32_t* count_opt,
                      int64_t list_cap, void* ws, size_t ws_bytes, const ssa_shape* shape,
                      cudaStream_t stream);

/* ssa_decode with a choice of strata (as ssa_select_strata); the attention
 * corrects every kept token by its p whatever the strata. */
ssa_status ssa_decode_strata(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V,
                             const ssa_bf16* Ks, const int32_t* sel_ch, int strata, int64_t top_k,
                             float top_p, float budget, uint64_t seed, float scale, float* out, float* lse,
                             float* s_hat_opt, int32_t* idx_opt, float* p_opt, int32_t* count_opt,
                             int64_t list_cap, void* ws, size_t ws_bytes, const ssa_shape* shape,
                             cudaStream_t stream);

/* The whole step with the early-stopping attention of ssa_attend_early_stop
 * in place of step (c): scores and selection as ssa_decode, then each unit's
 * selected rows (the top-k stratum and the drawn remainder, each with its
 * p) ordered by score and attended block by block until the gain test with
 * tau stops it.  blocks_opt as in ssa_attend_early_stop. */
ssa_status ssa_decode_early_stop(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V,
                                 const ssa_bf16* Ks, const int32_t* sel_ch, int64_t top_k, float budget,
                                 uint64_t seed, float scale, float tau, float* out, float* lse,
                                 int32_t* blocks_opt, void* ws, size_t ws_bytes, const ssa_shape* shape,
                                 cudaStream_t stream);

/* Append and decode in one chain: the new token (k_new, v_new, as in
 * ssa_append) is written at position ctx_len - 1 of K, V and Ks by the
 * chain's first kernel, and the step then attends over all ctx_len tokens,
 * the new one included.  ctx_len >= 1.  Same results as ssa_append followed
 * by ssa_decode, without the extra launch. */
ssa_status ssa_decode_append(const ssa_bf16* q, const ssa_bf16* k_new, const ssa_bf16* v_new,
                             ssa_bf16* K, ssa_bf16* V, ssa_bf16* Ks, const int32_t* sel_ch,
                             int64_t top_k, float budget, uint64_t seed, float scale,
                             float* out, float* lse, void* ws, size_t ws_bytes,
                             const ssa_shape* shape, cudaStream_t stream);

/* ssa_decode with the step's query read from, and its result written to,
 * HOST memory, all on `stream`; the caller synchronises.  When q_host,
 * out_host and lse_host are pinned and mapped into the device's address
 * space (cudaHostAlloc / cudaHostRegister with unified addressing), the
 * kernels read q and write out / lse there directly and no copy is enqueued;
 * otherwise (pageable buffers) q is copied to a staging area inside the
 * workspace, the step runs, and out / lse are copied back.  The KV cache
 * (K, V, Ks, sel_ch) stays where it is (see the memory tiers above). */
ssa_status ssa_decode_host(const ssa_bf16* q_host, const ssa_bf16* K, const ssa_bf16* V,
                           const ssa_bf16* Ks, const int32_t* sel_ch, int64_t top_k, float budget,
                           uint64_t seed, float scale, float* out_host, float* lse_host,
                           void* ws, size_t ws_bytes, const ssa_shape* shape,
                           cudaStream_t stream);

/* A paged, variable-length KV cache (the serving layout): K, V and Ks live in
 * page pools shared by the batch's sequences,
 *   K_pool, V_pool [num_pages][n_kv_heads][page_size][head_dim]
 *   Ks_pool        [num_pages][n_kv_heads][page_size][d_sel]
 * (contiguous, 16-byte aligned), and token t of sequence b is slot
 * t % page_size of page block_table[b][t / page_size].  Sequence b holds
 * seq_lens[b] tokens, 0 <= seq_lens[b] <= shape.ctx_len; shape.ctx_len bounds
 * every sequence (the workspace, the score rows and the list capacity are
 * sized by it) and must not exceed max_pages * page_size.  The block-table
 * entries of the pages a sequence's tokens fall in must be page ids in
 * [0, num_pages); the others are not read.  block_table and seq_lens are
 * device memory, read by the kernels, so they may be updated on the stream
 * between steps without a host round trip. */
typedef struct {
    int32_t page_size;           /* tokens per page: a power of two, 16 <= page_size <= 2^20 */
    int32_t max_pages;           /* entries per sequence in block_table (>= 1) */
    int64_t num_pages;           /* pages in each pool; num_pages * page_size < 2^31 */
    const int32_t* block_table;  /* [batch][max_pages] page ids */
    const int32_t* seq_lens;     /* [batch] tokens per sequence */
} ssa_paged_kv;

/* The whole step over a paged, variable-length cache (ssa_paged_kv): every
 * unit (b, h_kv) gets the step of ssa_decode over its own seq_lens[b] tokens
 * (the same scores, strata and Philox draws -- counters (j, h_kv, b, 0) with
 * j the token's position in its sequence -- and attention; Z is summed over
 * the plan's tiles of ctx_len, so it can differ from a contiguous call with
 * ctx_len = seq_lens[b] in its last bits).  With every seq_lens[b] equal to
 * ctx_len the results equal ssa_decode's on the same data bit for bit.  A unit with
 * top_k >= seq_lens[b] keeps all its tokens with p = 1; an empty sequence
 * gives zero outputs and lse = -inf.  shape's four stride fields must be 0
 * (the pools' layout is fixed above).  When k_new and v_new are given
 * ([batch][n_kv_heads][head_dim], as in ssa_append) the chain's first
 * kernel first writes the new token at position seq_lens[b] - 1 of every
 * non-empty sequence (its K, V and Ks rows, in its page), so seq_lens
 * already counts it; else they are NULL.  s_hat_opt [batch][n_kv_heads]
 * [ctx_len] receives the scores of positions < seq_lens[b] (the rest of each
 * row is not written); idx_opt / p_opt / count_opt as in ssa_decode, with
 * token positions within the sequence.  A length outside [0, ctx_len] or a
 * page id outside [0, num_pages) sets SSA_DEV_BAD_INDEX (the length is
 * clamped, the page replaced by page 0: no access leaves the pools).  K and
 * V pools may be pinned host memory (the memory tiers above). */
ssa_status ssa_decode_paged(const ssa_bf16* q, const ssa_bf16* k_new, const ssa_bf16* v_new, ssa_bf16* K_pool,
                            ssa_bf16* V_pool, ssa_bf16* Ks_pool, const ssa_paged_kv* pages,
                            const int32_t* sel_ch, int64_t top_k, float budget, uint64_t seed, float scale,
                            float* out, float* lse, float* s_hat_opt, int32_t* idx_opt, float* p_opt,
                            int32_t* count_opt, int64_t list_cap, void* ws, size_t ws_bytes,
                            const ssa_shape* shape, cudaStream_t stream);

/* Size of the library's built-in scratch array used by ssa_decode_static. */
#define SSA_STATIC_SCRATCH_BYTES (64u << 20)

/* ssa_decode for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this is a deployment convenience, not part of the
 * method.)  Some callers own no allocator: an inference engine that reserves
 * all HBM for its KV cache when it starts and forbids allocation inside the
 * decode loop, or a plugin interface that hands over inputs and outputs but
 * no workspace.  For them this entry point takes the same inputs and
 * outputs as ssa_decode but no workspace: its scratch is one static array of
 * SSA_STATIC_SCRATCH_BYTES (64 MiB) inside the library, which every GPU that
 * loads the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   - The first call in a CUDA context (with that context current) looks
 *     up the array's device address once and remembers it for that context;
 *     make that first call before any stream capture.  A context created
 *     anew (after cudaDeviceReset, say) looks it up again.
 *   - Shapes whose scratch (ssa_workspace_bytes(shape, 0)) exceeds the array
 *     are rejected with SSA_ERR_WORKSPACE before anything is enqueued.
 *   - All calls share the one array and it keeps the previous call's
 *     contents; each call clears the status word it needs.  Calls that
 *     overlap on the GPU (different streams, or different host threads on
 *     the same device) race on the array: serialise them.
 *   - device_flags (device memory, may be NULL) receives this call's device
 *     status bits (SSA_DEV_*), written on `stream` after the step. */
ssa_status ssa_decode_static(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V,
                             const ssa_bf16* Ks, const int32_t* sel_ch, int64_t top_k, float budget,
                             uint64_t seed, float scale, float* out, float* lse,
                             uint32_t* device_flags, const ssa_shape* shape, cudaStream_t stream);

/* Synchronises `stream`, ORs the device status bits (SSA_DEV_*) into
 * *flags_out (may be NULL), clears them, and returns the status code of the
 * most serious one (SSA_OK if none). */
ssa_status ssa_get_device_status(void* ws, cudaStream_t stream, uint32_t* flags_out);

/* Launch geometry the library would use for a shape on the current device:
 * CTAs of the (persistent) score kernel, selection tiles per unit, and
 * attention CTAs per unit.  Any output pointer may be NULL.  For tests and
 * tuning. */
ssa_status ssa_query_plan(const ssa_shape* shape, int32_t* score_ctas, int32_t* tiles_per_unit,
                          int32_t* attend_ctas_per_unit);

#ifdef __cplusplus
}
#endif

#endif /* LIBSSA_SSA_H */
