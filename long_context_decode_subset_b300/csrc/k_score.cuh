// k_score.cuh -- K0 (per-step initialisation) and K1 (approximate scores on
// the tensor cores).
//
// Sources (page title, section):
//  * "FASA: Frequency-Aware Sparse Attention", section 3 (Method), Stage 1
//    "Token Importance Prediction": every token is scored online from a
//    fixed, pre-calibrated subset of dominant RoPE chunks only -- here the
//    key summary Ks[b][h][i][0..d_sel), stored contiguously at append time.
//  * The GQA group's query heads are combined by max:
//        s_i = fl32(scale * max_g sum_j q_g[S_ch[j]] * Ks[i][j]).
//  * Philox4x32-10 (Salmon et al., SC'11) draws each token's uniform; K1
//    keeps the top 16 bits of word 0, a lower bound of u to 2^-16, so that
//    the bucket pass lists only the tokens that can be drawn and the
//    attention kernel recomputes the full word for those few.
//
// K1 is persistent (one CTA per SM; three quarters of every unit's
// 512-token stages split evenly over the CTAs, the rest a shared queue that
// CTAs drain as they finish, since SMs stream at different rates) and
// warp-specialised:
//   warp 0   takes the stages, publishes each one's (unit, j) and issues its
//            TMA copies: two 256-token boxes of the summary (swizzled to the
//            64- or 32-byte row width so that the tensor cores read them as
//            K-major operands), into a ring; with a paged cache one box per
//            page piece (min(page_size, 256) tokens, a lane each), placed
//            where the 256-token box would put those rows;
//   warp 3   writes each stage's 1 KB query operand (the unit's G query
//            heads on the summary channels, same swizzle) beside it;
//   warp 1   issues tcgen05.mma (M = 128 tokens, N = 16 query-head slots,
//            K = d_sel; bf16 in, fp32 accumulators in tensor memory), four
//            tiles per stage, and commits to the "stage free" and
//            "accumulators ready" barriers;
//   warp 2   allocates and frees the tensor memory;
//   warps 4-19 (four warpgroups, one per 128-token tile) read the
//            accumulators back (tcgen05.ld), take the max over the G heads,
//            write the scores, count the top 12 order-key bits per unit, and
//            draw the 16-bit Philox prefixes;
//   warps 20-23 (decode chain only) add the shared histogram buffers the
//            epilogue hands over to the units' global histograms.
#pragma once
#include "common.cuh"

namespace ssa {

struct Params {
    CUtensorMap ks_map;        // key summary [Bt][Hkv][N][d_sel] as a 4-D tensor (K1)
    Plan pl;
    int32_t Bt, Hq, Hkv, d, d_sel;
    int32_t dense;             // every token selected with p = 1 (top_k >= N or budget = +inf)
    int32_t attend;            // K2 computes attention (else it only writes the compact list)
    int32_t src_mode;          // K2 rows: 0 the selection, 1 all tokens, 2 the caller's compact list
    int32_t strata;            // 0 top-k + p proportional to exp(s), 1 top-k + uniform, 2 top-p + p proportional to exp(s)
    float top_p;               // strata 2: the stratum's share of the softmax of the scores
    int32_t q_staged;          // q is copied from q_host into the workspace by K0: read it after the wait
    const uint16_t* q_host;    // the step's query in pinned host memory (q_staged), [Bt][Hq][d]
    const uint16_t* q;         // [Bt][Hq][d]
    const uint16_t* K;         // [Bt][Hkv][N][d] with the strides below
    const uint16_t* V;
    const int32_t* sel_ch;     // [Hkv][d_sel]
    int64_t kv_sb, kv_sh;
    float scale;
    float budget;
    int64_t top_k;
    uint64_t seed;
    char* ws;                  // workspace base
    float* s_dst;              // K1 writes the scores here ([U][N])
    const float* s_src;        // K2 reads the scores here ([U][N])
    const int32_t* idx_in;     // K2 source 2: [U][cap] / count [U]
    const float* p_in;
    const int32_t* count_in;
    int32_t* idx_out;          // compact list out (may be null): [U][cap] / count [U]
    float* p_out;
    int32_t* count_out;
    int64_t cap;
    float* out;                // [Bt][Hq][d]
    float* lse;                // [Bt][Hq]
    // append step (K0 or append_kernel), active when k_new is set: the new
    // token's rows [Bt][Hkv][d] go to position app_pos of K, V and Ks
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint16_t* app_K;
    uint16_t* app_V;
    uint16_t* app_Ks;
    int64_t app_pos;
    int64_t ks_sb, ks_sh;
    // paged, variable-length cache: K, V and Ks are page pools
    // [num_pages][Hkv][page_size][d or d_sel]; token t of sequence b sits in
    // page block_table[b][t >> log_ps] at slot t & (page_size - 1), and
    // sequence b holds seq_lens[b] <= pl.N tokens (the append, when given,
    // writes position seq_lens[b] - 1)
    int32_t paged;
    int32_t log_ps;
    int32_t max_pages;         // block-table entries per sequence
    int32_t log_box;           // log2 of the summary's TMA box height, min(page_size, 256)
    int64_t num_pages;
    const int32_t* block_table;
    const int32_t* seq_lens;
    // early stop (the unit kernel's early-stop variant): the list of each
    // unit is in descending score order; the attention keeps the blocks of
    // 128 rows up to the first whose share of the softmax denominator is
    // below tau for every head, and writes their number to blocks_out [U]
    float tau;
    int32_t* blocks_out;
};

__device__ __forceinline__ uint32_t* ws_status(const Params& p) { return reinterpret_cast<uint32_t*>(p.ws + p.pl.o_status); }
__device__ __forceinline__ UnitCtrl* ws_ctrl(const Params& p) { return reinterpret_cast<UnitCtrl*>(p.ws + p.pl.o_ctrl); }
__device__ __forceinline__ uint32_t* ws_hist1(const Params& p) { return reinterpret_cast<uint32_t*>(p.ws + p.pl.o_hist1); }
// level-2 histogram (the next 12 key bits of the threshold bucket's members), [U][kBins]
__device__ __forceinline__ uint32_t* ws_hist2(const Params& p) { return ws_hist1(p) + (size_t)p.pl.U * kBins; }
__device__ __forceinline__ float2* ws_zpart(const Params& p) { return reinterpret_cast<float2*>(p.ws + p.pl.o_zpart); }
__device__ __forceinline__ uint32_t* ws_kcnt(const Params& p) { return reinterpret_cast<uint32_t*>(p.ws + p.pl.o_kcnt); }
__device__ __forceinline__ float* ws_part(const Params& p) { return reinterpret_cast<float*>(p.ws + p.pl.o_part); }
__device__ __forceinline__ unsigned long long* ws_topp(const Params& p) { return reinterpret_cast<unsigned long long*>(p.ws + p.pl.o_topp); }
__device__ __forceinline__ uint2* ws_cand(const Params& p) { return reinterpret_cast<uint2*>(p.ws + p.pl.o_cand); }
__device__ __forceinline__ int32_t* ws_sel_idx(const Params& p) { return reinterpret_cast<int32_t*>(p.ws + p.pl.o_sel_idx); }
__device__ __forceinline__ float* ws_sel_p(const Params& p) { return reinterpret_cast<float*>(p.ws + p.pl.o_sel_p); }
__device__ __forceinline__ uint16_t* ws_ubuf(const Params& p) { return reinterpret_cast<uint16_t*>(p.ws + p.pl.o_ubuf); }
__device__ __forceinline__ int32_t* ws_es_count(const Params& p) { return reinterpret_cast<int32_t*>(p.ws + p.pl.o_es); }
__device__ __forceinline__ float* ws_es_part(const Params& p) { return reinterpret_cast<float*>(p.ws + p.pl.o_esp); }
__device__ __forceinline__ uint2* ws_es_sort(const Params& p) { return reinterpret_cast<uint2*>(p.ws + p.pl.o_ess); }

// Strata 1 (top-k + uniform): the remainder's size n - min(k, n) in fp32,
// the normaliser Z of p = min(1, B / Z) for a unit of n tokens.
__device__ __forceinline__ float uniform_z(const Params& p, int64_t n)
{
    return (float)(n - min(p.top_k, n));
}

// Tokens of sequence b: pl.N, or (PAGED) seq_lens[b]; a length outside
// [0, pl.N] is flagged and clamped.  The kernels that read a paged cache are
// separate instantiations (PAGED), so that the contiguous ones carry none of
// its code.
template <bool PAGED>
__device__ __forceinline__ int64_t unit_len(const Params& p, int b)
{
    if constexpr (!PAGED) return p.pl.N;
    const int32_t n = __ldg(p.seq_lens + b);
    if (n < 0 || (int64_t)n > p.pl.N) {
        flag(ws_status(p), DEV_BAD_INDEX);
        return n < 0 ? 0 : p.pl.N;
    }
    return n;
}

// The pool page holding token t of sequence b (t < pl.N); a page id outside
// [0, num_pages) is flagged and replaced by page 0, so that no access leaves
// the pools.
__device__ __forceinline__ int32_t page_of(const Params& p, int b, int64_t t)
{
    const int32_t pg = __ldg(p.block_table + (int64_t)b * p.max_pages + (t >> p.log_ps));
    if ((uint64_t)(uint32_t)pg >= (uint64_t)p.num_pages) {
        flag(ws_status(p), DEV_BAD_INDEX);
        return 0;
    }
    return pg;
}

// Token t of sequence b as a pool token: page * page_size + slot (below 2^31).
__device__ __forceinline__ int32_t pool_token(const Params& p, int b, int64_t t)
{
    return (page_of(p, b, t) << p.log_ps) | (int32_t)(t & ((1 << p.log_ps) - 1));
}

// The row (in head_dim or d_sel units) of pool token pt of KV head h in a pool.
__device__ __forceinline__ int64_t pool_row(const Params& p, int h, int32_t pt)
{
    return ((((int64_t)(pt >> p.log_ps)) * p.Hkv + h) << p.log_ps) + (pt & ((1 << p.log_ps) - 1));
}

// ---------------------------------------------------------------------------
// K0: zero the unit's control block and histograms.  One CTA per unit.  It
// lets the next kernel launch at once: K1 streams the summary meanwhile and
// waits for K0 only before its first histogram flush.
// ---------------------------------------------------------------------------
// The append step for unit u = (b, h_kv), the step just before the decode path
// ("FASA: Frequency-Aware Sparse Attention", section 3, Stage 1: a token's
// dominant channels are stored contiguously when it is appended):
//   K[b][h][pos] = k_new[b][h],  V[b][h][pos] = v_new[b][h],
//   Ks[b][h][pos][j] = k_new[b][h][S_ch[h][j]],
// pos = app_pos, or (paged) the sequence's last position seq_lens[b] - 1 in
// its page (nothing for an empty sequence).  An out-of-range channel is
// flagged and clamped.
__device__ __forceinline__ void append_unit(const Params& p, int u, int tid, int nthreads)
{
    const int b = u / p.Hkv, h = u % p.Hkv;
    const int d = p.d;
    const int64_t src = ((int64_t)b * p.Hkv + h) * d;
    int64_t dst, ks_dst;
    if (p.paged) {   // the last of the sequence's tokens, in its page
        const int64_t pos = unit_len<true>(p, b) - 1;
        if (pos < 0) return;
        const int64_t row = pool_row(p, h, pool_token(p, b, pos));
        dst = row * d;
        ks_dst = row * p.d_sel;
    } else {
        dst = (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh + p.app_pos * d;
        ks_dst = (int64_t)b * p.ks_sb + (int64_t)h * p.ks_sh + p.app_pos * p.d_sel;
    }
    const int nq = d / 8;   // 16-byte pieces of a row
    for (int i = tid; i < 2 * nq; i += nthreads) {
        if (i < nq)
            reinterpret_cast<uint4*>(p.app_K + dst)[i] = reinterpret_cast<const uint4*>(p.k_new + src)[i];
        else
            reinterpret_cast<uint4*>(p.app_V + dst)[i - nq] = reinterpret_cast<const uint4*>(p.v_new + src)[i - nq];
    }
    for (int j = tid; j < p.d_sel; j += nthreads) {
        int ch = p.sel_ch[h * p.d_sel + j];
        if ((unsigned)ch >= (unsigned)d) {
            flag(ws_status(p), DEV_BAD_INDEX);
            ch = ch < 0 ? 0 : d - 1;
        }
        p.app_Ks[ks_dst + j] = p.k_new[src + ch];
    }
}

__global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ Params p)
{
    append_unit(p, blockIdx.x, threadIdx.x, 128);
}

__global__ void __launch_bounds__(256) init_kernel(const __grid_constant__ Params p)
{
    grid_dep_launch();
    const int u = blockIdx.x;
    const int tid = threadIdx.x;
    if (p.k_new != nullptr) append_unit(p, u, tid, 256);   // read by K1 only after its wait for this grid
    if (p.q_staged) {
        // the unit's G query rows from pinned host memory into the workspace
        // copy every later kernel reads (after its wait for this grid)
        const int G = p.Hq / p.Hkv, b = u / p.Hkv, h = u % p.Hkv;
        const int64_t off = ((int64_t)b * p.Hq + (int64_t)h * G) * p.d;
        for (int i = tid; i < G * p.d / 8; i += 256)
            reinterpret_cast<uint4*>(const_cast<uint16_t*>(p.q) + off)[i] = reinterpret_cast<const uint4*>(p.q_host + off)[i];
    }
    uint4* z = reinterpret_cast<uint4*>(ws_ctrl(p) + u);
    if (tid < (int)(sizeof(UnitCtrl) / 16)) z[tid] = make_uint4(0, 0, 0, 0);
    if (p.src_mode != 0) return;   // no selection: no histograms
    uint4* h1 = reinterpret_cast<uint4*>(ws_hist1(p) + (size_t)u * kBins);
    uint4* h2 = reinterpret_cast<uint4*>(ws_hist2(p) + (size_t)u * kBins);
    for (int i = tid; i < kBins / 4; i += 256) {
        h1[i] = make_uint4(0, 0, 0, 0);
        h2[i] = make_uint4(0, 0, 0, 0);
    }
    if (p.strata == 2) {   // the top-p stratum's mass histograms
        uint4* t = reinterpret_cast<uint4*>(ws_topp(p) + (size_t)u * kTopPBins * 3);
        for (int i = tid; i < (int)(kTopPUnitBytes / 16); i += 256) t[i] = make_uint4(0, 0, 0, 0);
    }
}

// ---------------------------------------------------------------------------
// K1: scores
// ---------------------------------------------------------------------------

// warp 0: copies; 1: MMA; 2: tensor memory; 3: query operand; 4-19: epilogue;
// with the histogram, 20-23: add the histogram buffers the epilogue hands over
// to global memory
constexpr int k1EpiThreads = 512;
constexpr int kHistWarps = 4;
__host__ __device__ constexpr int k1_threads(bool hist) { return hist ? 640 + 32 * kHistWarps : 640; }
constexpr int kGrab = 2;         // stages a CTA takes from the shared queue at a time
constexpr int kPreIssue = 1;     // stages issued before the set-up barrier
constexpr int kInfo = 32;        // stage descriptors in flight (> ring stages + accumulator buffers)

// HIST: the histogram is kept in two shared buffers of 16-bit counts, two
// bins to a word (the one being filled and the one warps 20-23 are adding to the
// unit's global histogram); a buffer is handed over at every change of unit
// and after kHistRun stages of one unit, so that no count passes 65535.
constexpr int kHistRun = 127;    // 127 stages x 512 tokens = 65024 counts at most (Plan::hist_run <= this)
template <int DSEL, bool HIST>
struct K1Cfg {
    static constexpr uint32_t ROW = DSEL * 2;                        // bytes per token row
    static constexpr uint32_t BOX = 256u * ROW;                      // one TMA box
    static constexpr uint32_t STAGE = (uint32_t)kStageTok * ROW;     // 32 KB or 16 KB
    static constexpr int S = (int)((192u * 1024u) / STAGE);          // 6 or 12 stages
    static constexpr int NB = 4;                                     // accumulator buffers
    static constexpr uint32_t TCOLS = 256;                           // NB x 4 tiles x 16 columns
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, 16);
    static constexpr uint32_t HWORDS = kBins / 2;                    // words per histogram buffer
    static constexpr uint32_t OFF_BOP = (uint32_t)S * STAGE;
    static constexpr uint32_t OFF_HIST = OFF_BOP + (uint32_t)S * kQselBytes;
    static constexpr uint32_t OFF_QROWS = OFF_HIST + (HIST ? 2u * HWORDS * 4u : 0u);   // G query rows (<= 2 KB)
    static constexpr uint32_t OFF_INFO = OFF_QROWS + 2048u;                     // kInfo stage descriptors
    static constexpr uint32_t OFF_HCTL = OFF_INFO + kInfo * 8u;                 // histogram hand-over words
    static constexpr uint32_t OFF_BAR = OFF_HCTL + 16u;
    static constexpr uint32_t SMEM = OFF_BAR + (3u * S + 2u * NB + 4u) * 8u + 16u + 1024u;   // + alignment slack
    static_assert(STAGE % 1024 == 0, "stages keep the swizzle atoms aligned");
    static_assert(kInfo > S + NB, "a descriptor outlives its stage's epilogue");
};

template <int DSEL, bool HIST>
constexpr uint32_t k1_smem_bytes() { return K1Cfg<DSEL, HIST>::SMEM; }

// K1's work: every unit's stages j < sf are split evenly and contiguously over
// the CTAs in (unit, j) order; the stages j >= sf of all units form a queue, in
// (unit, j) order, that the CTAs drain kGrab at a time (its last `grid` stages
// one at a time) once their own share is
// done (a counter in unit 0's control block, zeroed by K0), so that CTAs that
// stream faster take more of it.  A unit of n tokens has ceil(n / 512) stages,
// sf = 3/4 of them (rounded down) static: the same for every unit of a
// contiguous cache, per sequence for a paged one, whose stages are then
// located through a cursor over the sequences.
__host__ __device__ constexpr int32_t stages_of(int64_t n) { return (int32_t)((n + kStageTok - 1) / kStageTok); }
__host__ __device__ constexpr int32_t static_of(int32_t nst) { return (int32_t)((int64_t)nst * 3 / 4); }

// The sequence whose units hold index g of one part (static or queue) of a
// paged schedule: its first index, stages per unit in the part, first stage
// and length.
struct K1Cursor {
    int b;
    int64_t base;
    int32_t per, off, len;
};

// PAGED: every method is warp-collective (warp 0, all lanes, same results);
// else thread 0 of the CTA runs them.
template <bool PAGED>
struct K1Sched {
    int64_t s_cur, s_end;      // this CTA's static stages [s_cur, s_end)
    int64_t d_cur, d_end;      // the current queue chunk
    int64_t pending;           // the next chunk's start (a grab in flight), or -1
    int64_t dtotal;            // queued stages in all
    uint32_t* counter;
    bool waited;
    K1Cursor sc, dc;           // paged: the static and the queue cursor

    __device__ void init(const Params& p, uint32_t* ctr)
    {
        const Plan& pl = p.pl;
        int64_t st;
        if constexpr (!PAGED) {
            st = (int64_t)pl.U * pl.sf;
            dtotal = (int64_t)pl.U * (pl.nst - pl.sf);
        } else {
            long long a = 0, d = 0;
            for (int b = (int)(threadIdx.x & 31); b < p.Bt; b += 32) {
                const int32_t nst = stages_of(unit_len<true>(p, b)), sf = static_of(nst);
                a += sf;
                d += nst - sf;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, o);
                d += __shfl_xor_sync(0xffffffffu, d, o);
            }
            st = (int64_t)a * p.Hkv;
            dtotal = (int64_t)d * p.Hkv;
        }
        s_cur = st * blockIdx.x / gridDim.x;
        s_end = st * (blockIdx.x + 1) / gridDim.x;
        d_cur = d_end = 0;
        pending = -1;
        counter = ctr;
        waited = false;
        sc = K1Cursor{-1, 0, 0, 0, 0};
        dc = sc;
    }
    __device__ int64_t grab()
    {
        if (!waited) {
            grid_dep_wait();   // K0 has zeroed the counter
            waited = true;
        }
        if constexpr (!PAGED) return (int64_t)atomicAdd(counter, 1u);
        uint32_t v = 0;
        if ((threadIdx.x & 31) == 0) v = atomicAdd(counter, 1u);
        return (int64_t)__shfl_sync(0xffffffffu, v, 0);
    }
    // paged: move cursor c forward to the sequence holding index g of its
    // part, 32 sequences at a time; false if no sequence does
    __device__ bool seek(const Params& p, K1Cursor& c, int64_t g, bool queue)
    {
        const int lane = (int)(threadIdx.x & 31);
#pragma unroll 1
        while (g >= c.base + (int64_t)p.Hkv * c.per) {
            if (c.b + 1 >= p.Bt) return false;
            const int bb = c.b + 1 + lane;
            int32_t len = 0, per = 0, off = 0;
            if (bb < p.Bt) {
                len = (int32_t)unit_len<true>(p, bb);
                const int32_t nst = stages_of(len), sf = static_of(nst);
                per = queue ? nst - sf : sf;
                off = queue ? sf : 0;
            }
            const long long w = (long long)p.Hkv * per;
            long long incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int64_t start = c.base + (int64_t)p.Hkv * c.per;   // sequence c.b + 1's first index
            const uint32_t hit = __ballot_sync(0xffffffffu, bb < p.Bt && g < start + incl);
            const int l = hit ? __ffs(hit) - 1 : min(31, p.Bt - 1 - (c.b + 1));
            c.b = c.b + 1 + l;
            c.base = start + __shfl_sync(0xffffffffu, incl - w, l);
            c.per = __shfl_sync(0xffffffffu, per, l);
            c.off = __shfl_sync(0xffffffffu, off, l);
            c.len = __shfl_sync(0xffffffffu, len, l);
        }
        return true;
    }
    // index g of a part as (unit, j) and the unit's length
    __device__ bool locate(const Params& p, int64_t g, bool queue, int& u, int& j, int64_t& len)
    {
        const Plan& pl = p.pl;
        if constexpr (!PAGED) {
            const int32_t per = queue ? pl.nst - pl.sf : pl.sf;
            u = (int)(g / per);
            j = (queue ? pl.sf : 0) + (int)(g % per);
            len = pl.N;
            return true;
        } else {
            K1Cursor& c = queue ? dc : sc;
            if (!seek(p, c, g, queue)) return false;
            const int64_t r = g - c.base;
            u = c.b * p.Hkv + (int)(r / c.per);
            j = c.off + (int)(r % c.per);
            len = c.len;
            return true;
        }
    }
    // the next stage (unit, j) and its unit's length; false at the end of the work
    __device__ bool next(const Params& p, int& u, int& j, int64_t& len)
    {
        if (s_cur < s_end) {
            const int64_t g = s_cur++;
            if (s_cur + 1 >= s_end && pending < 0 && dtotal > 0) pending = grab();   // one stage ahead
            return locate(p, g, false, u, j, len);
        }
        if (d_cur == d_end) {
            if (dtotal == 0) return false;
            if (pending < 0) pending = grab();
            // ticket t: stages [kGrab t, kGrab t + kGrab) while the queue is long, then single stages for its
            // last `grid` stages, so that the CTAs run out of work within a stage of one another
            const int64_t tail = min(dtotal, (int64_t)gridDim.x);
            const int64_t pairs = (dtotal - tail) / kGrab;
            const int64_t d0 = pending < pairs ? pending * kGrab : pairs * kGrab + (pending - pairs);
            if (d0 >= dtotal) return false;
            d_cur = d0;
            d_end = pending < pairs ? d0 + kGrab : d0 + 1;
            pending = grab();   // the next chunk's grab goes out now
        }
        return locate(p, d_cur++, true, u, j, len);
    }
};

template <int G, int DSEL, bool HIST, bool UBUF, bool PAGED>
__global__ void __launch_bounds__(k1_threads(HIST), 1) score_kernel(const __grid_constant__ Params p)
{
    using CF = K1Cfg<DSEL, HIST>;
    constexpr int S = CF::S, NB = CF::NB;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    unsigned char* ring = smem;
    unsigned char* bop = smem + CF::OFF_BOP;
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + CF::OFF_HIST);
    uint16_t* qrows = reinterpret_cast<uint16_t*>(smem + CF::OFF_QROWS);
    int2* info = reinterpret_cast<int2*>(smem + CF::OFF_INFO);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + CF::OFF_BAR);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + NB;
    uint64_t* ready = tempty + NB;   // a stage's (unit, j) is published
    uint64_t* hdone = ready + S;     // [2] the epilogue has left histogram buffer b
    uint64_t* hfree = hdone + 2;     // [2] warps 20-23 have added buffer b to global memory and zeroed it
    uint32_t* tslot = reinterpret_cast<uint32_t*>(hfree + 2);
    int* hctl = reinterpret_cast<int*>(smem + CF::OFF_HCTL);   // unit of buffer 0, of buffer 1, hand-overs + 1

    const Plan& pl = p.pl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* status = ws_status(p);

    // the producer (thread 0, or with a paged cache warp 0): takes stage c,
    // publishes its (unit, j) and issues its TMA copies: two 256-token boxes
    // of a contiguous summary, or one box per page (at most 256 tokens, a
    // lane each) of a paged one, skipping the boxes past the sequence's end;
    // false at the end marker
    K1Sched<PAGED> sch;
    int c_issued = 0;
    bool ended = false;
    auto produce = [&](int c) -> bool {
        const int st = c % S;
        if (c >= S) {
            if (lane == 0 && !mbar_wait_bounded(&empty[st], (uint32_t)((c / S) - 1) & 1u)) flag(status, DEV_TIMEOUT);
            if constexpr (PAGED) __syncwarp();
        }
        int u = -1, j = 0;
        int64_t len = 0;
        if (!sch.next(p, u, j, len)) u = -1;
        if (lane == 0) {
            info[c % kInfo] = make_int2(u, j);
            mbar_arrive(&ready[st]);
        }
        if (u < 0) {
            if (lane == 0) mbar_arrive(&full[st]);   // the end marker carries no copies
            return false;
        }
        const int b = u / p.Hkv, h = u % p.Hkv;
        unsigned char* dst = ring + (size_t)st * CF::STAGE;
        const uint64_t pol = l2_policy_evict_first();
        if constexpr (!PAGED) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[st], CF::STAGE);
                tma_load_4d(dst, &p.ks_map, 0, j * kStageTok, h, b, &full[st], pol);
                tma_load_4d(dst + CF::BOX, &p.ks_map, 0, j * kStageTok + 256, h, b, &full[st], pol);
            }
        } else {
            const int64_t t0 = (int64_t)j * kStageTok;
            const int nbox = (int)((min((int64_t)kStageTok, len - t0) + (1 << p.log_box) - 1) >> p.log_box);
            const uint32_t box_bytes = (CF::ROW << p.log_box);
            if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)nbox * box_bytes);
            __syncwarp();
            for (int i = lane; i < nbox; i += 32) {
                const int64_t t = t0 + ((int64_t)i << p.log_box);
                tma_load_4d(dst + (size_t)i * box_bytes, &p.ks_map, 0, (int)(t & ((1 << p.log_ps) - 1)), h,
                            page_of(p, b, t), &full[st], pol);
            }
        }
        return true;
    };
    if (PAGED ? warp == 0 : tid == 0) {
        if (lane == 0) {
            for (int i = 0; i < S; ++i) {
                mbar_init(&full[i], 2);    // the summary copies (with their bytes) + the query operand
                mbar_init(&empty[i], 1);
                mbar_init(&ready[i], 1);
            }
            for (int i = 0; i < NB; ++i) {
                mbar_init(&tfull[i], 1);
                mbar_init(&tempty[i], k1EpiThreads / 32);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&hdone[i], k1EpiThreads / 32);
                mbar_init(&hfree[i], kHistWarps);
            }
            hctl[2] = 0;
            fence_mbar_init();
            tma_prefetch_desc(&p.ks_map);
        }
        if constexpr (PAGED) __syncwarp();
        // the first stage's copies go out before the block-wide set-up ends;
        // the rest of the ring follows it (each issue takes a few hundred
        // cycles, and the query operand waits for the set-up barrier)
        sch.init(p, &ws_ctrl(p)[0].k1_next);
        for (; c_issued < kPreIssue && !ended; ++c_issued) ended = !produce(c_issued);
    }
    if constexpr (HIST) {
        for (int i = tid; i < 2 * (int)CF::HWORDS; i += k1_threads(HIST)) hist[i] = 0u;
    }
    if (warp == 2) tmem_alloc(tslot, CF::TCOLS);
    // the query operand's inputs: the G query rows and the channel list of a
    // unit (the first unit's fetched before the summary copies start, so that
    // they do not queue behind them)
    constexpr int QPL = G >= 2 ? G / 2 : 1;   // 16-byte pieces of the G rows per lane (d <= 128)
    const int nch = G * p.d / 8;
    uint4 nq[QPL];
    int nsel = 0;
    auto fetch_q = [&](int uu) {
        const int bb = uu / p.Hkv, hh = uu % p.Hkv;
        const uint4* qsrc = reinterpret_cast<const uint4*>(p.q + ((int64_t)bb * p.Hq + (int64_t)hh * G) * p.d);
#pragma unroll
        for (int i = 0; i < QPL; ++i) {
            const int ci = lane + 32 * i;
            nq[i] = (ci < nch) ? __ldg(qsrc + ci) : make_uint4(0u, 0u, 0u, 0u);
        }
        nsel = (lane < DSEL) ? __ldg(p.sel_ch + (int64_t)hh * DSEL + lane) : 0;
    };
    int first_u = -1;
    if (warp == 3) {
        if constexpr (!PAGED) {
            const int64_t st = (int64_t)pl.U * pl.sf;
            const int64_t g0 = st * blockIdx.x / gridDim.x;
            if (g0 < st * (blockIdx.x + 1) / gridDim.x) first_u = (int)(g0 / pl.sf);
        } else {   // the first static stage's unit, found as the producer finds it
            K1Sched<true> s3;
            s3.init(p, nullptr);
            int uu, jj;
            int64_t ll;
            if (s3.s_cur < s3.s_end && s3.locate(p, s3.s_cur, false, uu, jj, ll)) first_u = uu;
        }
        if (first_u >= 0) {
            if (p.q_staged) grid_dep_wait();   // K0 copies the query into the workspace
            fetch_q(first_u);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    // the next kernel may be scheduled now: its CTAs take SMs as this grid's
    // CTAs leave and wait for this grid to complete
    grid_dep_launch();
    SSA_MARK(0);

    if (warp == 0) {
        // the producer carries on from where the set-up left it
        if (PAGED || lane == 0) {
#pragma unroll 1
            for (int c = c_issued; !ended; ++c) ended = !produce(c);
        }
        SSA_MARKW(22);
    } else if (warp == 3) {
        // the stage's query operand: row g < G = q_g[S_ch[j]] over j, rows
        // G..15 zero, K-major in the 64/32-byte swizzled layout the TMA writes
        // for the summary (lane l builds half of row l / 2)
        constexpr int HALF = DSEL / 2;   // channels per lane: 16 or 8 (two or one 16-byte chunks)
        const int r = lane >> 1, hf = lane & 1;
        uint4 vals[HALF / 8];
        int cur_u = -1;
#pragma unroll 1
        for (int c = 0;; ++c) {
            const int st = c % S;
            if (lane == 0 && !mbar_wait_bounded(&ready[st], (uint32_t)(c / S) & 1u)) flag(status, DEV_TIMEOUT);
            __syncwarp();
            const int u = info[c % kInfo].x;
            if (u < 0) {
                if (lane == 0) mbar_arrive(&full[st]);
                break;
            }
            if (u != cur_u) {
                if (u != first_u || cur_u >= 0) fetch_q(u);
                cur_u = u;
                // stage the unit's rows, then gather the channels
#pragma unroll
                for (int i = 0; i < QPL; ++i) {
                    const int ci = lane + 32 * i;
                    if (ci < nch) reinterpret_cast<uint4*>(qrows)[ci] = nq[i];
                }
                int sel = nsel;
                if ((unsigned)sel >= (unsigned)p.d) {
                    if (lane < DSEL) flag(status, DEV_BAD_INDEX);
                    sel = 0;
                }
                __syncwarp();
                uint16_t v[HALF];
#pragma unroll
                for (int k = 0; k < HALF; ++k) {
                    const int ch = __shfl_sync(0xffffffffu, sel, hf * HALF + k);
                    v[k] = (r < G) ? qrows[r * p.d + ch] : (uint16_t)0;
                }
#pragma unroll
                for (int q8 = 0; q8 < HALF / 8; ++q8)
                    vals[q8] = make_uint4((uint32_t)v[q8 * 8 + 0] | ((uint32_t)v[q8 * 8 + 1] << 16),
                                          (uint32_t)v[q8 * 8 + 2] | ((uint32_t)v[q8 * 8 + 3] << 16),
                                          (uint32_t)v[q8 * 8 + 4] | ((uint32_t)v[q8 * 8 + 5] << 16),
                                          (uint32_t)v[q8 * 8 + 6] | ((uint32_t)v[q8 * 8 + 7] << 16));
                __syncwarp();
            }
            unsigned char* row = bop + (size_t)st * kQselBytes + (size_t)r * CF::ROW;
#pragma unroll
            for (int q8 = 0; q8 < HALF / 8; ++q8) {
                const int chunk = hf * (HALF / 8) + q8;
                const int phys = (DSEL == 32) ? (chunk ^ ((r >> 1) & 3)) : (chunk ^ ((r >> 2) & 1));
                *reinterpret_cast<uint4*>(row + phys * 16) = vals[q8];
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[st]);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t ring_a = smem_addr(ring), bop_a = smem_addr(bop);
#pragma unroll 1
            for (int c = 0;; ++c) {
                const int st = c % S, nb = c % NB;
                if (!mbar_wait_bounded(&full[st], (uint32_t)(c / S) & 1u)) flag(status, DEV_TIMEOUT);
                if (c >= NB && !mbar_wait_bounded(&tempty[nb], (uint32_t)((c / NB) - 1) & 1u)) flag(status, DEV_TIMEOUT);
                if (info[c % kInfo].x < 0) {   // end of the work: pass the marker on
                    mbar_arrive(&tfull[nb]);
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = ring_a + (uint32_t)st * CF::STAGE;
                const uint32_t b0 = bop_a + (uint32_t)st * kQselBytes;
                const uint32_t dcol = tbase + (uint32_t)nb * 64u;
#pragma unroll
                for (int tile = 0; tile < 4; ++tile) {
#pragma unroll
                    for (int ks = 0; ks < DSEL / 16; ++ks) {
                        const uint64_t ad = smem_desc_kmajor_swz(a0 + (uint32_t)tile * 128u * CF::ROW + ks * 32u, CF::ROW);
                        const uint64_t bd = smem_desc_kmajor_swz(b0 + ks * 32u, CF::ROW);
                        tc_mma_bf16(dcol + (uint32_t)tile * 16u, ad, bd, CF::IDESC, ks > 0 ? 1u : 0u);
                    }
                }
                tc_commit(&empty[st]);
                tc_commit(&tfull[nb]);
            }
        }
    } else if (warp >= 20) {
        if constexpr (HIST) {
            // warps 20-23 add each histogram buffer the epilogue hands over to
            // its unit's global histogram and zero it (a quarter each), so that
            // the epilogue never stops for a change of unit
            constexpr int QW = (int)CF::HWORDS / kHistWarps;
            const int w0 = (warp - 20) * QW;
            volatile int* hc = hctl;
            uint32_t* hist1 = ws_hist1(p);
            grid_dep_wait();   // K0 has zeroed the global histograms
#pragma unroll 1
            for (int f = 0;; ++f) {
                const int b = f & 1;
                if (!mbar_wait_bounded_sleep(&hdone[b], (uint32_t)(f >> 1) & 1u, 256u)) {
                    flag(status, DEV_TIMEOUT);
                    break;
                }
                const int total = hc[2];   // hand-overs + 1 once the epilogue has finished, else 0
                if (total != 0 && f >= total - 1) break;
                uint32_t* hb = hist + (size_t)b * CF::HWORDS;
                uint32_t* g = hist1 + (size_t)hc[b] * kBins;
#pragma unroll 4
                for (int i = w0 + lane; i < w0 + QW; i += 32) {
                    const uint32_t v = hb[i];
                    if (v) {
                        if (v & 0xffffu) atomicAdd(g + 2 * i, v & 0xffffu);
                        if (v >> 16) atomicAdd(g + 2 * i + 1, v >> 16);
                        hb[i] = 0u;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&hfree[b]);
            }
        }
    } else if (warp >= 4) {
        const int tile = (warp - 4) >> 2, quarter = warp & 3, etid = tid - 128;
        const uint32_t k0 = (uint32_t)(p.seed & 0xffffffffu), k1 = (uint32_t)(p.seed >> 32);
        volatile int* hc = hctl;
        int cur_u = -1;
        int hb = 0, nuse = 0, run = 0;     // histogram buffer in use, uses so far, stages in this use
        uint32_t* hcur = hist;
        uint32_t ub = 0u, uh = 0u;          // the unit's batch and KV head
        float* srow = nullptr;
        uint16_t* urow = nullptr;
        int64_t nu = 0;                     // the unit's tokens
        const uint32_t tl = ((uint32_t)(quarter * 32) << 16) + (uint32_t)tile * 16u;   // lane quarter, tile columns
#pragma unroll 1
        for (int c = 0;; ++c) {
            const int nb = c % NB;
            if (!mbar_wait_bounded(&tfull[nb], (uint32_t)(c / NB) & 1u)) flag(status, DEV_TIMEOUT);
            const int2 in = info[c % kInfo];
            if (in.x < 0) break;
            const int u = in.x, j = in.y;
            if (c == 0 && warp == 4) SSA_MARKW(21);
            if (u != cur_u || (HIST && run == pl.hist_run)) {
                if constexpr (HIST) {
                    if (cur_u >= 0) {
                        // hand the filled buffer to warps 20-23 and take the other one
                        if (warp == 4 && lane == 0) hc[hb] = cur_u;
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&hdone[hb]);
                        hb ^= 1;
                        ++nuse;
                        if (nuse >= 2 && !mbar_wait_bounded(&hfree[hb], (uint32_t)((nuse - 2) >> 1) & 1u))
                            flag(status, DEV_TIMEOUT);
                        hcur = hist + (size_t)hb * CF::HWORDS;
                    }
                    run = 0;
                }
                cur_u = u;
                ub = (uint32_t)(u / p.Hkv);
                uh = (uint32_t)(u % p.Hkv);
                srow = p.s_dst + (int64_t)u * pl.N;
                nu = unit_len<PAGED>(p, (int)ub);
                if constexpr (UBUF) urow = ws_ubuf(p) + (int64_t)u * pl.np;
            }
            if constexpr (HIST) ++run;
            tc_fence_after();
            const int t = j * kStageTok + tile * 128 + quarter * 32 + lane;
            const uint32_t taddr = tbase + tl + (uint32_t)nb * 64u;
            uint32_t rr[G];
            if constexpr (G == 1) tmem_ld_x1(taddr, rr);
            else if constexpr (G == 2) tmem_ld_x2(taddr, rr);
            else if constexpr (G == 4) tmem_ld_x4(taddr, rr);
            else tmem_ld_x8(taddr, rr);
            // the token's Philox word does not depend on the accumulator: it is
            // computed while the load is in flight
            uint32_t x0 = 0u;
            if constexpr (UBUF) x0 = philox_word0((uint32_t)t, uh, ub, 0u, k0, k1);
            tmem_ld_wait_after(x0);
            tmem_regs_ready(rr);
            float best = __uint_as_float(rr[0]);
#pragma unroll
            for (int g = 1; g < G; ++g) best = fmaxf(best, __uint_as_float(rr[g]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[nb]);
            if (t < nu) {
                const float s = best * p.scale;
                if (!isfinite(s)) flag(status, DEV_NONFINITE);
                srow[t] = s;
                if constexpr (HIST) {
                    const uint32_t key = okey(s) >> 20;
                    atomicAdd(&hcur[key >> 1], 1u << ((key & 1u) * 16u));
                }
                if constexpr (UBUF) urow[t] = (uint16_t)(x0 >> 16);
            }
        }
        if (warp == 4) SSA_MARKW(23);
        if constexpr (HIST) {
            // warps 20-23 stop at the hand-over they wait for; the buffer in use is
            // added to global memory here, by all the epilogue warps
            if (warp == 4 && lane == 0) hc[2] = nuse + 1;
            __syncwarp();
            if (lane == 0) mbar_arrive(&hdone[hb]);
            if (cur_u >= 0) {
                grid_dep_wait();   // K0 has zeroed the global histograms
                named_bar_sync(1, k1EpiThreads);
                uint32_t* g = ws_hist1(p) + (size_t)cur_u * kBins;
#pragma unroll 1
                for (int i = etid; i < (int)CF::HWORDS; i += k1EpiThreads) {
                    const uint32_t v = hcur[i];
                    if (v & 0xffffu) atomicAdd(g + 2 * i, v & 0xffffu);
                    if (v >> 16) atomicAdd(g + 2 * i + 1, v >> 16);
                }
            }
        }
        if (warp == 4) SSA_MARKW(24);
    }
    SSA_MARK(1);
    SSA_GT(0);
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tbase, CF::TCOLS);
    }
}

// K1 for ssa_select (scores given): per-unit histogram of the top 12 key bits
// and the 16-bit Philox prefixes.  One CTA per (unit, tile).
__global__ void __launch_bounds__(kInThreads) score_input_kernel(const __grid_constant__ Params p)
{
    __shared__ uint32_t hist[kBins];
    const Plan& pl = p.pl;
    const int u = blockIdx.x / pl.ntile, tile = blockIdx.x % pl.ntile;
    const int tid = threadIdx.x;
    const int64_t t0 = (int64_t)tile * pl.tt;
    const int n = (int)min((int64_t)pl.tt, pl.N - t0);
    const int b = u / p.Hkv, h = u % p.Hkv;
    const uint32_t k0 = (uint32_t)(p.seed & 0xffffffffu), k1 = (uint32_t)(p.seed >> 32);
    uint32_t* status = ws_status(p);
    for (int i = tid; i < kBins; i += kInThreads) hist[i] = 0u;
    __syncthreads();
    grid_dep_wait();
    for (int i = tid; i < n; i += kInThreads) {
        const int64_t t = t0 + i;
        const float s = p.s_src[(int64_t)u * pl.N + t];
        if (!isfinite(s)) flag(status, DEV_NONFINITE);
        atomicAdd(&hist[okey(s) >> 20], 1u);
        const uint32_t x0 = philox_word0((uint32_t)t, (uint32_t)h, (uint32_t)b, 0u, k0, k1);
        ws_ubuf(p)[(int64_t)u * pl.np + t] = (uint16_t)(x0 >> 16);
    }
    __syncthreads();
    uint32_t* hist1 = ws_hist1(p) + (size_t)u * kBins;
    for (int i = tid; i < kBins; i += kInThreads)
        if (hist[i]) atomicAdd(hist1 + i, hist[i]);
    grid_dep_launch();
}

}  // namespace ssa
