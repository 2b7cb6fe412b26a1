// k_attend.cuh -- K2, the unit kernel: the stratified selection's decisions
// and the exact softmax attention over the selected rows with the inclusion
// correction, a group of CTAs per (batch, KV head) unit.
//
// Sources (page title, section):
//  * "FASA: Frequency-Aware Sparse Attention", section 3, Stage 2 "Focused
//    Attention Computation": full-precision attention over the selected
//    tokens only, at their original positions.
//  * "Stratified Sparse Attention speeds up decoding 2.96x on a 1M context",
//    section "How SSA splits the cache into strata": each selected token is
//    corrected by its inclusion probability; here the weight 1/p_i enters the
//    logit as -log p_i, so numerator and denominator are both corrected:
//        l_i = scale * q_g . K_i - log p_i,   o_g = sum_i softmax(l)_i V_i.
//  * "S2O" (online permutation and early stopping), technical summary,
//    Method section 1: rows are gathered by index arrays, the physical layout
//    in HBM is kept; section 3: the online-softmax state (m, l, acc), merged
//    across splits.
//
// The C CTAs of a unit each own one tile of its tokens.  With the selection
// (source 0) every CTA runs the tile pass (k_select.cuh) and arrives on the
// unit's counter; once all C have arrived every CTA resolves the k-th token
// and Z (the same deterministic computation in each), decides its own
// tile's listed tokens (top-k stratum, or the draw u < p with the exact p)
// and keeps the chosen rows in index order.  With
// every token kept (source 1) a CTA takes its tile's tokens with p = 1; with
// the caller's lists (source 2) an even share of the unit's list.  The kept
// rows go through the tensor cores 128 at a time -- S = K Q^T and
// O^T = V^T P with tcgen05.mma, fp32 accumulators in tensor memory, P split
// into two bf16 terms (hi + lo) so that the products keep fp32-level
// accuracy -- and the last CTA of the unit to finish merges the CTAs'
// (m, l, acc) partials in rank order.  Every wait on another CTA is bounded
// in time (a timeout sets SSA_DEV_TIMEOUT); the grid is one wave, so every
// CTA of a unit is resident together.
#pragma once
#include "k_select.cuh"

namespace ssa {

// What the decisions need from the selection (source 0 only): the resolve's
// results.
struct UnitSel {
    uint32_t theta;
    int64_t cut;
    float m, Z;
    bool sampling;
};

// A paged cache's tile of pages: the block-table entries [p0, p0 + n) of
// sequence b in shared memory (n = 0 when they do not fit: then the table
// is read from global memory).
struct PageCache {
    const int32_t* ent;
    int64_t p0;
    int32_t n;
};

// Token t of sequence b as a pool token (page * page_size + slot), its page
// id from the cache when there; an id outside [0, num_pages) is flagged and
// replaced by page 0.
__device__ __forceinline__ int32_t pool_token_c(const Params& p, const PageCache& pc, int b, int64_t t)
{
    const int64_t pi = t >> p.log_ps;
    int32_t pg;
    if (pi - pc.p0 >= 0 && pi - pc.p0 < pc.n) {
        pg = pc.ent[pi - pc.p0];
        if ((uint64_t)(uint32_t)pg >= (uint64_t)p.num_pages) {
            flag(ws_status(p), DEV_BAD_INDEX);
            pg = 0;
        }
    } else {
        pg = page_of(p, b, t);
    }
    return (pg << p.log_ps) | (int32_t)(t & ((1 << p.log_ps) - 1));
}

// Entries [c0, c0 + n) of this CTA's list (n <= LIST) from source `mode`
// (0 the selection, 1 all tokens, 2 the caller's list): staged through
// ridx / rval (cp.async, one wave), decided, and the kept ones written in
// list order to cidx (the token, or with a paged cache its pool token) /
// clp (log p) [0, nk).  Returns nk (every thread).
// Source 0: the list is the concatenation of the tile's warp slices, pre[]
// their exclusive prefix (pre[kSelWarps] = length).  With a compact list
// requested, the kept (index, p) pairs also go to the unit's staging area at
// stage_at.  NT threads; ends with a block barrier.
// Copies entries [c0, c0 + n) of the tile's list (the concatenation of its
// warp slices, pre[] their exclusive prefix) to ridx / rval with cp.async,
// one commit group; the caller waits for it.  NT threads.
template <int NT>
__device__ void stage_list(const Params& p, int u, int tile, int64_t c0, int n, const uint32_t* pre,
                           int32_t* ridx, float* rval)
{
    const Plan& pl = p.pl;
    const int W2 = pl.tt / kSelWarps;
    const int32_t* sidx = ws_sel_idx(p) + (size_t)u * pl.np;
    const float* sp = ws_sel_p(p) + (size_t)u * pl.np;
#pragma unroll 1
    for (int i = threadIdx.x; i < n; i += NT) {
        const int64_t pos = c0 + i;
        int lo_l = 0, hi_l = kSelWarps;   // pre[lo_l] <= pos < pre[hi_l]
        while (hi_l - lo_l > 1) {
            const int mid = (lo_l + hi_l) >> 1;
            if ((int64_t)pre[mid] <= pos) lo_l = mid; else hi_l = mid;
        }
        const size_t at = (size_t)tile * pl.tt + (size_t)lo_l * W2 + (size_t)(pos - pre[lo_l]);
        cp_async_4(ridx + i, sidx + at);
        cp_async_4(rval + i, sp + at);
    }
    cp_async_commit();
}

template <int LIST, int NT, bool PAGED>
__device__ int stage_decide(const Params& p, int mode, int u, int b, int h, int tile, int64_t c0, int n,
                            int64_t stage_at, const uint32_t* pre, const UnitSel& us, int32_t* ridx, float* rval,
                            int32_t* cidx, float* clp, uint32_t* scan, const PageCache& pc, bool prestaged)
{
    constexpr int PER = (LIST + NT - 1) / NT;   // entries per thread at most
    static_assert(PER <= 32, "one keep bit per entry in a word");
    const Plan& pl = p.pl;
    const int tid = threadIdx.x;
    uint32_t* status = ws_status(p);
    if (mode == 0) {
        if (!prestaged) stage_list<NT>(p, u, tile, c0, n, pre, ridx, rval);   // else already in flight
    } else if (mode == 2) {
#pragma unroll 1
        for (int i = tid; i < n; i += NT) {
            cp_async_4(ridx + i, p.idx_in + (int64_t)u * p.cap + c0 + i);
            cp_async_4(rval + i, p.p_in + (int64_t)u * p.cap + c0 + i);
        }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    SSA_MARK(28);
    // the decisions for this thread's consecutive entries [e0, e1) (at most
    // PER of them, spread evenly over the threads); one bit each
    const int e0 = (int)((int64_t)n * tid / NT), e1 = (int)((int64_t)n * (tid + 1) / NT);
    uint32_t kbits = 0, kcount = 0;
#pragma unroll 1
    for (int e = 0; e < e1 - e0; ++e) {
        const int i = e0 + e;
        int32_t j;
        float pv;
        bool keep;
        if (mode == 1) {
            j = (int32_t)(c0 + i);
            pv = 1.0f;
            keep = true;
        } else {
            j = ridx[i];
            pv = rval[i];
            if (mode == 0) {
                const bool is_cand = ((uint32_t)j & kCandFlag) != 0u;
                j = (int32_t)((uint32_t)j & ~kCandFlag);
                keep = false;
                if (pv == INFINITY) {                     // above the threshold bucket
                    keep = true;
                    pv = 1.0f;
                } else {
                    float ev = pv;                        // a remainder term ...
                    if (is_cand) {                        // ... or a candidate's score
                        const uint32_t k = okey(pv);
                        if (k > us.theta || (k == us.theta && (int64_t)j <= us.cut)) {
                            keep = true;
                            pv = 1.0f;
                        }
                        ev = (p.strata == 1) ? 1.0f : expf(__fsub_rn(pv, us.m));
                    }
                    if (!keep) {
                        pv = us.sampling ? prob_from_term(ev, p.budget, us.Z) : 0.0f;
                        keep = pv > 0.0f && token_uniform(p.seed, j, h, b) < pv;
                    }
                }
            } else {
                keep = j >= 0 && (int64_t)j < pl.N && pv > 0.0f && pv <= 1.0f;
                if (!keep) flag(status, DEV_BAD_INDEX);
            }
            ridx[i] = j;
            rval[i] = pv;
        }
        if (keep) {
            kbits |= 1u << e;
            ++kcount;
        }
    }
    // the kept entries in list order (a paged cache's block-table reads for
    // them all go out first, together)
    uint32_t nk;
    uint32_t at = block_excl_scan<NT>(kcount, scan, nk);
    int32_t pt[PER];
    if constexpr (PAGED) {
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            pt[e] = 0;
            if (e < e1 - e0 && ((kbits >> e) & 1u))
                pt[e] = pool_token_c(p, pc, b, (mode == 1) ? c0 + e0 + e : (int64_t)ridx[e0 + e]);
        }
    }
#pragma unroll 1
    for (int e = 0; e < e1 - e0; ++e) {
        if (!((kbits >> e) & 1u)) continue;
        const int i = e0 + e;
        const int32_t j = (mode == 1) ? (int32_t)(c0 + i) : ridx[i];
        const float pv = (mode == 1) ? 1.0f : rval[i];
        if constexpr (PAGED) {
            int32_t ptv = 0;   // pt[e], picked without indexing the array by a variable
#pragma unroll
            for (int x = 0; x < PER; ++x) ptv = (x == e) ? pt[x] : ptv;
            cidx[at] = ptv;
        } else {
            cidx[at] = j;
        }
        clp[at] = logf(pv);
        if (p.idx_out) {
            if (stage_at + at < pl.N)
                ws_cand(p)[(size_t)u * pl.N + (size_t)(stage_at + at)] = make_uint2((uint32_t)j, __float_as_uint(pv));
            else
                flag(status, DEV_OVERFLOW);
        }
        ++at;
    }
    __syncthreads();
    SSA_MARK(29);
    return (int)nk;
}

// ---------------------------------------------------------------------------
// the unit kernel
// ---------------------------------------------------------------------------

constexpr int kUGatherWarps = 11;   // warps 5 .. 15 gather the K and V rows
static_assert((5 + kUGatherWarps) * 32 == kSelThreads, "the attention roles fill the block");

// A chunk is one 128-row MMA operand of K (and one of V) rows in the
// 128-byte swizzled layout: row i's 16-byte piece c at piece c ^ (i & 7) of
// the row's 64-dim plane.  At head_dim 64 only the first plane is gathered:
// S reads only it, and O's rows for dims 64..127 (from the second plane,
// whatever it holds) are never read back.
constexpr int kPageCache = 2048;   // block-table entries of its tile a CTA keeps in shared memory (paged)

template <int G, int D, int LIST, bool PAGED = false>   // LIST: list entries staged at a time
struct UCfg {
    static constexpr int CH = 128;                                 // listed rows per chunk
    static constexpr uint32_t PLANE = CH * 128u;                   // 64 dims x 128 rows, 128-byte swizzle
    static constexpr uint32_t KV = 2u * PLANE;                     // one K or V chunk (32 KB)
    static constexpr uint32_t QPLANE = 16u * 128u;                 // 64 elements x 16 rows
    static constexpr uint32_t OFF_K = 0;                           // 2 chunks
    static constexpr uint32_t OFF_V = OFF_K + 2u * KV;             // 2 chunks
    static constexpr uint32_t OFF_Q = OFF_V + 2u * KV;             // query operand: 16 x 128, 4 KB
    // before the attention, [0, OFF_Q) holds the selection pass's staging
    // (and the resolve's) and its shared state
    static constexpr uint32_t OFF_SEL = kSelStageBytes;
    static constexpr uint32_t OFF_P = OFF_Q + 2u * QPLANE;         // 2 x P operand: 16 columns x 128 rows
    static constexpr uint32_t OFF_LIST = OFF_P + 2u * 2u * QPLANE; // cidx, clp
    static constexpr uint32_t OFF_RAW = OFF_LIST + (uint32_t)LIST * 8u;       // raw list staging
    static constexpr uint32_t OFF_RED = OFF_RAW + (uint32_t)LIST * 8u;        // [2][2][4][G] floats
    static constexpr uint32_t OFF_BAR = (OFF_RED + 2u * 2u * 4u * G * 4u + 7u) & ~7u;
    static constexpr uint32_t NBAR = 14;                           // k/v_full, k/v_free, s_full, p_ready, o_full (x2)
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;      // tensor-memory slot, counts
    static constexpr uint32_t OFF_PRE = OFF_MISC + 64u;            // the tile list's slice prefix
    static constexpr uint32_t OFF_PCACHE = (OFF_PRE + (uint32_t)(kSelWarps + 1) * 4u + 15u) & ~15u;   // paged
    static constexpr uint32_t OFF_ROFF = OFF_PCACHE + (PAGED ? kPageCache * 4u : 0u);   // paged: 2 x CH row offsets
    static constexpr uint32_t SMEM = OFF_ROFF + (PAGED ? 2u * CH * 8u : 0u) + 1024u;     // + alignment slack
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 16);       // S = K Q^T
    static constexpr uint32_t IDESC_O = idesc_bf16_f32_amn(128, 16);   // O^T = V^T P
    static constexpr uint32_t TCOLS = 64;                          // S x2 (cols 0-31), O x2 (cols 32-63)
    static_assert(2 * G <= 16, "P's hi and lo columns fit in N = 16");
    static_assert(OFF_SEL % 16 == 0 && OFF_SEL + sizeof(SelShared) <= OFF_Q, "selection state fits the K/V chunks");
    static_assert(D == 64 || D == 128, "head_dim");
};

template <int G, int D, int LIST, bool PAGED = false>
constexpr uint32_t unit_smem_bytes() { return UCfg<G, D, LIST, PAGED>::SMEM; }


// Early stop: the number of leading blocks the unit keeps ("S2O ...",
// technical summary, Method section 2).  parts holds nb block partials
// (acc [G][D], m [G], l [G]); with M_g the largest m of head g and
// w_g(b) = l_g(b) exp(m_g(b) - M_g), block b's gain ratio is
// w_g(b) / sum_{b' <= b} w_g(b'), and the unit stops after the first block
// whose ratio is below tau for every head (block 0 included always).
// Block-wide (kSelThreads); uses nb * G * 2 floats of `sm` and misc[6].
// Every thread returns the count.
template <int G, int D>
__device__ __noinline__ int es_keep_blocks(const Params& p, const float* parts, int nb, float* sm, uint32_t* misc)
{
    constexpr int PS = G * D + 2 * G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float* w = sm;            // [nb][G]
    float* mx = sm + nb * G;  // [G]
    for (int i = tid; i < nb * G; i += kSelThreads) w[i] = __ldcg(parts + (size_t)(i / G) * PS + G * D + (i % G));
    if (tid == 0) misc[6] = (uint32_t)nb;
    __syncthreads();
    // per head (one warp each): the largest m, then the inclusive prefix of w and the test
    if (warp < G) {
        float m = -INFINITY;
        for (int b = lane; b < nb; b += 32) m = fmaxf(m, w[b * G + warp]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) mx[warp] = m;
    }
    __syncthreads();
    if (warp < G) {
        const float M = mx[warp];
        float run = 0.0f;
#pragma unroll 1
        for (int b0 = 0; b0 < nb; b0 += 32) {
            const int b = b0 + lane;
            float wb = 0.0f;
            if (b < nb) {
                const float mb = w[b * G + warp];
                const float lb = __ldcg(parts + (size_t)b * PS + G * D + G + warp);
                wb = (mb == -INFINITY) ? 0.0f : lb * expf(mb - M);
            }
            float incl = wb;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const float pref = run + incl;
            run += __shfl_sync(0xffffffffu, incl, 31);
            // a block of this head is "below" when its share is under tau; kept in the sign of w
            if (b < nb) w[b * G + warp] = (wb < p.tau * pref) ? 1.0f : 0.0f;
        }
    }
    __syncthreads();
    for (int b = tid; b < nb; b += kSelThreads) {
        bool all = true;
#pragma unroll
        for (int g = 0; g < G; ++g) all = all && w[b * G + g] != 0.0f;
        if (all) atomicMin(&misc[6], (uint32_t)b);
    }
    __syncthreads();
    const int stop = (int)misc[6];
    __syncthreads();
    return stop < nb ? stop + 1 : nb;
}

// Thread roles in the attention (kSelThreads): warps 0-3 epilogue
// (tensor-memory lanes = chunk rows for S, = head dims for O), warp 4 issues
// the MMAs (and owns the tensor memory), warps 5 .. 15 gather the K and V
// rows.  Chunk g uses buffers g & 1; barrier phases count chunks over the
// whole CTA.  Grid: U * C CTAs, C = pl.ntile per unit, one wave.
// The unit kernel's variants: a contiguous cache, a paged one, and the
// early-stop attention (a contiguous cache, the caller's lists in descending
// score order, one CTA per unit).
constexpr int kVarContig = 0, kVarPaged = 1, kVarEarlyStop = 2;

template <int G, int D, int LIST, int VAR>
__global__ void __launch_bounds__(kSelThreads, 1) unit_kernel(const __grid_constant__ Params p)
{
    constexpr bool PAGED = VAR == kVarPaged;
    constexpr bool ES = VAR == kVarEarlyStop;
    using CF = UCfg<G, D, LIST, PAGED>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    __shared__ uint32_t scan[kSelWarps];
    int32_t* cidx = reinterpret_cast<int32_t*>(smem + CF::OFF_LIST);
    float* clp = reinterpret_cast<float*>(smem + CF::OFF_LIST + LIST * 4);
    float* red = reinterpret_cast<float*>(smem + CF::OFF_RED);   // [parity][max | sum][warp][G]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CF::OFF_BAR);
    uint64_t* k_full = bars;
    uint64_t* v_full = bars + 2;
    uint64_t* k_free = bars + 4;
    uint64_t* v_free = bars + 6;
    uint64_t* s_full = bars + 8;
    uint64_t* p_ready = bars + 10;
    uint64_t* o_full = bars + 12;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + CF::OFF_MISC);   // [0] tensor memory, [2] last, [4..5] offsets
    uint32_t* pre = reinterpret_cast<uint32_t*>(smem + CF::OFF_PRE);

    const Plan& pl = p.pl;
    const int C = pl.ntile;
    const int u = blockIdx.x / C, r = blockIdx.x % C;   // r: the CTA's rank (tile) in its unit
    const int b = u / p.Hkv, h = u % p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* status = ws_status(p);

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 32 * kUGatherWarps);   // every gather thread's copies
            mbar_init(&v_full[i], 32 * kUGatherWarps);
            mbar_init(&k_free[i], 1);
            mbar_init(&v_free[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 4);   // one arrive per epilogue warp
            mbar_init(&o_full[i], 1);
        }
        fence_mbar_init();
    }
    if (warp == 4 && p.attend) tmem_alloc(&misc[0], CF::TCOLS);
    // the query operand: head slot n < G = q_n (the scale is applied to S),
    // slots G..15 zero; K-major, 128-byte swizzle, two 64-dim planes (a query
    // the chain's first kernel stages is read after the wait for it)
    if (p.q_staged) grid_dep_wait();
    if (tid < 256) {
        const int n = tid >> 4, pc = tid & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < G && p.attend && pc < D / 8)
            v = *reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + (int64_t)h * G + n) * D + pc * 8);
        *reinterpret_cast<uint4*>(smem + CF::OFF_Q + (pc >> 3) * CF::QPLANE + n * 128 + (((pc & 7) ^ (n & 7)) << 4)) = v;
        fence_proxy_async_smem();
    }
    // a paged cache: the sequence's length and the block-table entries of this
    // CTA's tile go to shared memory before the wait (the chain's kernels do
    // not write them)
    PageCache pc{nullptr, 0, 0};
    int64_t nu = pl.N;   // the unit's tokens
    if constexpr (PAGED) {
        nu = unit_len<true>(p, b);
        int32_t* ent = reinterpret_cast<int32_t*>(smem + CF::OFF_PCACHE);
        const int64_t t0 = (int64_t)r * pl.tt, t1 = min(nu, t0 + pl.tt);
        pc.ent = ent;
        pc.p0 = t0 >> p.log_ps;
        const int64_t np = t1 > t0 ? ((t1 - 1) >> p.log_ps) - pc.p0 + 1 : 0;
        pc.n = np <= kPageCache ? (int32_t)np : 0;
        for (int i = tid; i < pc.n; i += kSelThreads) ent[i] = __ldg(p.block_table + (int64_t)b * p.max_pages + pc.p0 + i);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = misc[0];
    SSA_GT(4);
    grid_dep_wait();
    SSA_MARK(7);
    SSA_GT(5);

    // this CTA's list: [lo, hi)
    UnitCtrl* ctrl = ws_ctrl(p) + u;
    UnitSel us{0u, -1, 0.0f, 0.0f, false};
    int64_t lo = 0, hi = 0;
    int32_t es_nb = 0, es_b0 = 0;   // early stop: the unit's blocks, this CTA's first block
    int mode = p.src_mode;
    SelShared& sh = *reinterpret_cast<SelShared*>(smem + CF::OFF_SEL);
    // the stratum's size: k, or (top-p) found from the unit's score masses;
    // a paged cache's unit whose stratum holds all its tokens keeps every one
    // with p = 1 (a sequence shorter than k)
    uint32_t k_unit = 0;
    bool prestaged = false;   // the first list chunk's copies are in flight
    if (mode == 0) {
        k_unit = (p.strata == 2) ? topp_size(p, u, r, nu, sh, smem) : (uint32_t)min(p.top_k, (int64_t)0xffffffff);
        if (PAGED && (int64_t)k_unit >= nu) mode = 1;
    }
    if (mode == 0) {
        const TileSel ts = tile_pass(p, u, r, nu, k_unit, sh, smem);
        if (tid == 0) {
            uint32_t run = 0;
            for (int w = 0; w < kSelWarps; ++w) {
                pre[w] = run;
                run += sh.wcnt[w];
            }
            pre[kSelWarps] = run;
            // the tile's lists, candidates, level-2 counts and share of Z are written
            __threadfence();
            atomicAdd(&ctrl->arrive, 1u);
        }
        SSA_MARK(3);
        // the first list chunk is this CTA's own: its copies to shared memory
        // go out now and land while the unit's other tiles finish and the
        // resolve runs (the resolve stages in other bytes)
        __syncthreads();
        stage_list<kSelThreads>(p, u, r, 0, (int)min((int64_t)LIST, (int64_t)pre[kSelWarps]), pre,
                                reinterpret_cast<int32_t*>(smem + CF::OFF_RAW),
                                reinterpret_cast<float*>(smem + CF::OFF_RAW + LIST * 4));
        prestaged = true;
        // every tile of the unit has arrived: resolve the k-th token and Z
        // (every CTA computes the same result)
        if (tid == 0 && !wait_geq_bounded(&ctrl->arrive, (uint32_t)C)) flag(status, DEV_TIMEOUT);
        __syncthreads();
        resolve_unit(p, u, nu, ts.f1, ts.above1, ts.target, ts.m, sh, reinterpret_cast<uint2*>(smem));
        __syncthreads();
        us.theta = sh.r_theta;
        us.cut = sh.r_cut;
        us.m = sh.r_m;
        us.Z = sh.r_Z;
        SSA_MARK(4);
        hi = pre[kSelWarps];
    } else if (mode == 1) {
        lo = min(nu, (int64_t)r * pl.tt);
        hi = min(nu, lo + pl.tt);
    } else {
        const int64_t c = p.count_in[u];
        const int64_t total = c < 0 ? 0 : (c > p.cap ? p.cap : c);
        if constexpr (ES) {   // whole 128-row blocks of the ordered list
            es_nb = (int32_t)((total + CF::CH - 1) / CF::CH);
            es_b0 = (int32_t)((int64_t)es_nb * r / C);
            lo = (int64_t)es_b0 * CF::CH;
            hi = min(total, (int64_t)es_nb * (r + 1) / C * CF::CH);
        } else {
            lo = total * r / C;
            hi = total * (r + 1) / C;
        }
    }
    SSA_MARK(11);
    us.sampling = p.budget > 0.0f && us.Z > 0.0f;
    const int64_t stage_base = (mode == 0) ? (int64_t)r * pl.tt : lo;   // the compact list's staging
    // row j of the unit: Kb + j * D (a paged cache: the pool row of pool token j)
    const uint16_t* Kb = PAGED ? p.K : p.K + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;
    const uint16_t* Vb = PAGED ? p.V : p.V + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;

    // epilogue state: running (m, l) per head (the same in every epilogue
    // thread) and this thread's head dim of the accumulator
    float m_run[G], l_run[G], acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.0f;
        acc[g] = 0.0f;
    }
    int gbase = 0;        // chunks done before this list chunk
    int64_t kept = 0;
    const uint32_t k_a = smem_addr(smem + CF::OFF_K), v_a = smem_addr(smem + CF::OFF_V);
    const uint32_t q_a = smem_addr(smem + CF::OFF_Q), p_a = smem_addr(smem + CF::OFF_P);
#pragma unroll 1
    for (int64_t c0 = lo; c0 < hi; c0 += LIST) {
        const int n = (int)min((int64_t)LIST, hi - c0);
        int32_t* ridx = reinterpret_cast<int32_t*>(smem + CF::OFF_RAW);
        float* rval = reinterpret_cast<float*>(smem + CF::OFF_RAW + LIST * 4);
        const int nk = stage_decide<LIST, kSelThreads, PAGED>(p, mode, u, b, h, r, c0, n, stage_base + kept, pre, us,
                                                              ridx, rval, cidx, clp, scan, pc,
                                                              prestaged && c0 == lo);
        kept += nk;
        const int nc = p.attend ? (nk + CF::CH - 1) / CF::CH : 0;
        if (warp >= 5) {
            // gather: the chunk's K rows, then its V rows, into the 128-byte
            // swizzled planes (rows past the list read as zeros).  An item is
            // one row and one 16-byte piece of each of its 64-dim planes:
            // eight consecutive threads cover a row's 128-byte plane
            // segments, and one address computation serves both planes.  K
            // and V buffers are released separately: a chunk's K copies go
            // out once S of the chunk two back has read its buffer, its V
            // copies once that chunk's O has.  Each thread's copies arrive on
            // k_full / v_full when they land (cp.async.mbarrier.arrive), so
            // publishing never waits on a later chunk's buffer.
            const int gt = tid - 160;   // 0 .. 32 * kUGatherWarps - 1
#pragma unroll 1
            for (int c = 0; c < nc; ++c) {
                const int g = gbase + c, bf = g & 1;
                const uint32_t ph = (uint32_t)((g - 2) >> 1) & 1u;   // the release of chunk g - 2
                if (g >= 2) {
                    if (lane == 0 && !mbar_wait_bounded(&k_free[bf], ph)) flag(status, DEV_TIMEOUT);
                    __syncwarp();
                }
                int64_t* roff = reinterpret_cast<int64_t*>(smem + CF::OFF_ROFF) + bf * CF::CH;
                if constexpr (PAGED) {
                    // the chunk's pool rows, once per row (double-buffered: a buffer is rewritten only after
                    // every gather thread has passed the next chunk's barrier)
                    if (gt < CF::CH) {
                        const int row = c * CF::CH + gt;
                        roff[gt] = row < nk ? pool_row(p, h, cidx[row]) : 0;
                    }
                    named_bar_sync(2, 32 * kUGatherWarps);
                }
                auto copy_rows = [&](unsigned char* dst, const uint16_t* src) {
#pragma unroll 1
                    for (int it = gt; it < CF::CH * 8; it += 32 * kUGatherWarps) {
                        const int i = it >> 3, pc = it & 7;
                        const int row = c * CF::CH + i;
                        const bool valid = row < nk;
                        int64_t j;
                        if constexpr (PAGED) j = roff[i];
                        else j = valid ? (int64_t)cidx[row] : 0;
                        const uint32_t off = (uint32_t)i * 128u + ((uint32_t)(pc ^ (i & 7)) << 4);
                        const uint16_t* sp = src + j * D + pc * 8;
                        cp_async_16_zfill(dst + off, sp, valid);
                        if constexpr (D == 128) cp_async_16_zfill(dst + CF::PLANE + off, sp + 64, valid);
                    }
                };
                copy_rows(smem + CF::OFF_K + bf * CF::KV, Kb);
                cp_async_mbar_arrive(&k_full[bf]);
                if (warp == 5 && c < 3) SSA_MARKW(30 + c);
                if (g >= 2) {
                    if (lane == 0 && !mbar_wait_bounded(&v_free[bf], ph)) flag(status, DEV_TIMEOUT);
                    __syncwarp();
                }
                copy_rows(smem + CF::OFF_V + bf * CF::KV, Vb);
                cp_async_mbar_arrive(&v_full[bf]);
            }
            cp_async_wait<0>();
        } else if (warp == 4) {
            if (lane == 0) {
                auto mma_s = [&](int g) {   // S[g & 1] = K_g Q^T; releases K_g's buffer
                    const int bf = g & 1;
                    fence_proxy_async_smem();   // the copies (generic proxy) before the MMA's reads
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t a = k_a + bf * CF::KV + (ks >> 2) * CF::PLANE + (ks & 3) * 32u;
                        const uint32_t bq = q_a + (ks >> 2) * CF::QPLANE + (ks & 3) * 32u;
                        tc_mma_bf16(tbase + bf * 16u, smem_desc_kmajor_swz(a, 128), smem_desc_kmajor_swz(bq, 128),
                                    CF::IDESC_S, ks > 0 ? 1u : 0u);
                    }
                    tc_commit(&s_full[bf]);
                    tc_commit(&k_free[bf]);
                };
                auto mma_o = [&](int g) {   // O^T[g & 1] = V_g^T P_g; releases V_g's buffer
                    const int bf = g & 1;
                    fence_proxy_async_smem();
                    tc_fence_after();
                    // A = the V rows read MN-major (64-dim atoms PLANE apart,
                    // 8-row groups 1 KB apart), 16 rows a step
#pragma unroll
                    for (int ks = 0; ks < CF::CH / 16; ++ks) {
                        const uint32_t a = v_a + bf * CF::KV + ks * 2048u;
                        const uint32_t bp = p_a + bf * 2u * CF::QPLANE + (ks >> 2) * CF::QPLANE + (ks & 3) * 32u;
                        tc_mma_bf16(tbase + 32u + bf * 16u, smem_desc_mn_sw128(a, CF::PLANE, 1024u),
                                    smem_desc_kmajor_swz(bp, 128), CF::IDESC_O, ks > 0 ? 1u : 0u);
                    }
                    tc_commit(&o_full[bf]);
                    tc_commit(&v_free[bf]);
                };
                // Whichever product can go out next does: S of chunk cs once
                // its K rows have landed (at most one chunk ahead of O: two S
                // buffers), O of chunk co once P is written and its V rows
                // have landed.  S of chunk g + 1 thus runs while the
                // epilogue turns S of chunk g into P, and O of chunk g while
                // it works on chunk g + 1.
                int cs = 0, co = 0;
                uint64_t t0 = 0;
                bool idle = false;
#pragma unroll 1
                while (co < nc) {
                    const int gs = gbase + cs, go = gbase + co;
                    const bool s_next = cs < nc && cs <= co + 1;
                    if (s_next && mbar_test_wait(&k_full[gs & 1], (uint32_t)(gs >> 1) & 1u)) {
                        if (cs < 3) SSA_MARKW(33 + cs);
                        mma_s(gs);
                        ++cs;
                        idle = false;
                    } else if (co < cs && mbar_test_wait(&p_ready[go & 1], (uint32_t)(go >> 1) & 1u) &&
                               mbar_test_wait(&v_full[go & 1], (uint32_t)(go >> 1) & 1u)) {
                        if (co < 3) SSA_MARKW(36 + co);
                        mma_o(go);
                        ++co;
                        idle = false;
                    } else if (!idle) {
                        t0 = global_timer_ns();
                        idle = true;
                    } else if (global_timer_ns() - t0 > 2000000000ull) {
                        // a wait ran out: record it and go on in order
                        flag(status, DEV_TIMEOUT);
                        if (s_next) {
                            mma_s(gs);
                            ++cs;
                        } else {
                            mma_o(go);
                            ++co;
                        }
                        idle = false;
                    } else {
                        __nanosleep(32);
                    }
                }
            }
        } else {
            // epilogue (tid = tensor-memory lane).  Iteration c turns S of
            // chunk c into P (softmax) and then folds O of chunk c - 1, so
            // that the O product of a chunk runs while the next chunk's
            // softmax does; (mc, lc) of the chunk waiting for its fold are
            // kept in mcP, lcP.
            const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
            float mcP[G], lcP[G];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                mcP[gg] = -INFINITY;
                lcP[gg] = 0.0f;
            }
#pragma unroll 1
            for (int c = 0; c <= nc; ++c) {
                float mc[G], lc[G];
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    mc[gg] = -INFINITY;
                    lc[gg] = 0.0f;
                }
                if (c < nc) {
                    const int g = gbase + c, bf = g & 1;
                    if (lane == 0 && !mbar_wait_bounded(&s_full[bf], (uint32_t)(g >> 1) & 1u)) flag(status, DEV_TIMEOUT);
                    __syncwarp();
                    tc_fence_after();
                    float s[G];
                    {
                        uint32_t rr[8];
                        tmem_ld_x8(lane_base + bf * 16u, rr);
                        tmem_ld_wait();
                        tmem_regs_ready(rr);
#pragma unroll
                        for (int gg = 0; gg < G; ++gg) s[gg] = __uint_as_float(rr[gg]);
                    }
                    const int row = c * CF::CH + tid;
                    const bool valid = row < nk;
                    const float lp = valid ? clp[row] : 0.0f;
                    float x[G];
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) {
                        x[gg] = valid ? s[gg] * p.scale - lp : -INFINITY;
                        float mx = x[gg];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                        if (lane == 0) red[((bf * 2 + 0) * 4 + warp) * G + gg] = mx;
                    }
                    named_bar_sync(1, 128);
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) {
                        float mx = red[((bf * 2 + 0) * 4 + 0) * G + gg];
#pragma unroll
                        for (int w = 1; w < 4; ++w) mx = fmaxf(mx, red[((bf * 2 + 0) * 4 + w) * G + gg]);
                        mc[gg] = mx;
                    }
                    // P = exp(x - m_chunk) as bf16 hi + lo, columns gg and G + gg of
                    // the K-major B operand (128-byte swizzle, two 64-row planes)
                    unsigned char* pb = smem + CF::OFF_P + bf * 2u * CF::QPLANE + (tid >> 6) * CF::QPLANE;
                    const int r64 = tid & 63;
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) {
                        const float w = (valid && mc[gg] != -INFINITY) ? expf(x[gg] - mc[gg]) : 0.0f;
                        const __nv_bfloat16 whi = __float2bfloat16_rn(w);
                        const __nv_bfloat16 wlo = __float2bfloat16_rn(w - __bfloat162float(whi));
                        const int nh = gg, nl = G + gg;
                        *reinterpret_cast<__nv_bfloat16*>(pb + nh * 128 + (((r64 >> 3) ^ (nh & 7)) << 4) + (r64 & 7) * 2) = whi;
                        *reinterpret_cast<__nv_bfloat16*>(pb + nl * 128 + (((r64 >> 3) ^ (nl & 7)) << 4) + (r64 & 7) * 2) = wlo;
                        float sm = w;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
                        if (lane == 0) red[((bf * 2 + 1) * 4 + warp) * G + gg] = sm;
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    named_bar_sync(1, 128);
                    if (lane == 0) mbar_arrive(&p_ready[bf]);
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) {
                        float sm = 0.0f;
#pragma unroll
                        for (int w = 0; w < 4; ++w) sm += red[((bf * 2 + 1) * 4 + w) * G + gg];
                        lc[gg] = sm;
                    }
                }
                if (c > 0) {
                    // fold O of chunk c - 1 (this thread's head dim, hi + lo columns) into acc
                    const int g = gbase + c - 1, bf = g & 1;
                    if (lane == 0 && !mbar_wait_bounded(&o_full[bf], (uint32_t)(g >> 1) & 1u)) flag(status, DEV_TIMEOUT);
                    __syncwarp();
                    tc_fence_after();
                    float o[2 * G];
                    if constexpr (G == 8) {
                        uint32_t rr[16];
                        tmem_ld_x16(lane_base + 32u + bf * 16u, rr);
                        tmem_ld_wait();
                        tmem_regs_ready(rr);
#pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = __uint_as_float(rr[k]);
                    } else {
                        uint32_t rr[8];
                        tmem_ld_x8(lane_base + 32u + bf * 16u, rr);
                        tmem_ld_wait();
                        tmem_regs_ready(rr);
#pragma unroll
                        for (int k = 0; k < 2 * G; ++k) o[k] = __uint_as_float(rr[k]);
                    }
                    tc_fence_before();
                    if constexpr (ES) {
                        // early stop: every block's own (m, l, acc) partial; the merge applies the gain test
                        constexpr int PS = G * D + 2 * G;
                        float* bp = ws_es_part(p) + ((size_t)u * pl.esb + (size_t)(es_b0 + g)) * PS;
                        if (tid < D) {
#pragma unroll
                            for (int gg = 0; gg < G; ++gg) bp[gg * D + tid] = o[gg] + o[G + gg];
                        }
                        if (tid == 0) {
#pragma unroll
                            for (int gg = 0; gg < G; ++gg) {
                                bp[G * D + gg] = mcP[gg];
                                bp[G * D + G + gg] = lcP[gg];
                            }
                        }
                    } else {
#pragma unroll
                        for (int gg = 0; gg < G; ++gg) {
                            const float mn = fmaxf(m_run[gg], mcP[gg]);
                            const float ar = (m_run[gg] == -INFINITY) ? 0.0f : expf(m_run[gg] - mn);
                            const float ac = (mcP[gg] == -INFINITY) ? 0.0f : expf(mcP[gg] - mn);
                            acc[gg] = acc[gg] * ar + (o[gg] + o[G + gg]) * ac;
                            l_run[gg] = l_run[gg] * ar + lcP[gg] * ac;
                            m_run[gg] = mn;
                        }
                    }
                    if (c <= 3) SSA_MARK(59 + c);
                }
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    mcP[gg] = mc[gg];
                    lcP[gg] = lc[gg];
                }
            }
        }
        gbase += nc;
        __syncthreads();   // every role is done with this list chunk
    }
    SSA_MARK(8);

    // this CTA's partial (acc per head dim, then (m, l) per head) in the
    // unit's partials array
    constexpr int PS = G * D + 2 * G;
    float* gpart = ws_part(p) + ((size_t)u * pl.tcap + r) * PS;
    if (warp < 4 && p.attend) {
        if (tid < D) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg) gpart[gg * D + tid] = acc[gg];
        }
        if (tid == 0) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                gpart[G * D + gg] = m_run[gg];
                gpart[G * D + G + gg] = l_run[gg];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4 && p.attend) {
        tc_fence_after();
        tmem_dealloc(tbase, CF::TCOLS);
    }

    // the compact list: every CTA's kept entries are in index order and the
    // CTAs' tiles (or list shares) are in rank order, so CTA r's entries go
    // after those of ranks < r
    if (p.count_out || p.idx_out) {
        uint32_t* kcnt = ws_kcnt(p) + (size_t)u * pl.tcap;
        if (tid == 0) {
            kcnt[r] = (uint32_t)kept;
            __threadfence();
            atomicAdd(&ctrl->karrive, 1u);
            if (!wait_geq_bounded(&ctrl->karrive, (uint32_t)C)) flag(status, DEV_TIMEOUT);
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t before = 0, all = 0;
#pragma unroll 1
            for (int k = lane; k < C; k += 32) {
                const uint32_t v = __ldcg(kcnt + k);
                all += v;
                before += (k < r) ? v : 0u;
            }
            before = warp_sum_u32(before);
            all = warp_sum_u32(all);
            if (lane == 0) {
                misc[4] = before;
                misc[5] = all;
            }
        }
        __syncthreads();
        const uint32_t before = misc[4];
        if (r == 0 && tid == 0 && p.count_out) p.count_out[u] = (int32_t)misc[5];
        if (p.idx_out) {
            const uint2* stage = ws_cand(p) + (size_t)u * pl.N + (size_t)stage_base;
#pragma unroll 1
            for (int64_t o = tid; o < kept; o += kSelThreads) {
                const int64_t dst = (int64_t)before + o;
                if (stage_base + o >= pl.N) break;   // flagged when staged
                const uint2 v = __ldcg(stage + o);
                if (dst < p.cap) {
                    p.idx_out[(int64_t)u * p.cap + dst] = (int32_t)v.x;
                    p.p_out[(int64_t)u * p.cap + dst] = __uint_as_float(v.y);
                } else {
                    flag(status, DEV_OVERFLOW);
                }
            }
        }
    }
    SSA_MARK(12);
    SSA_GT(6);
    if (!p.attend) return;
    // the last CTA of the unit to finish merges the partials in rank order
    // and writes the unit's output rows and log-sum-exp
    if (tid == 0) {
        __threadfence();
        misc[2] = (atomicAdd(&ctrl->done, 1u) == (uint32_t)(C - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!misc[2]) return;
    __threadfence();
    // the partials are staged in shared memory (the K/V chunk buffers) a
    // group at a time with one wave of copies, then merged in rank order
    const float* parts = ws_part(p) + (size_t)u * pl.tcap * PS;
    int nparts = C;
    if constexpr (ES) {
        // the blocks' partials, the first es_keep of them: the gain test on the blocks' (m, l)
        parts = ws_es_part(p) + (size_t)u * pl.esb * PS;
        nparts = es_keep_blocks<G, D>(p, parts, es_nb, reinterpret_cast<float*>(smem), misc);
        if (tid == 0 && p.blocks_out) p.blocks_out[u] = nparts;
    }
    float* sp = reinterpret_cast<float*>(smem);
    constexpr int KB = (int)(CF::OFF_Q / (PS * 4u));   // partials per group
    static_assert(KB >= 1, "a partial fits the staging");
    constexpr int EPT = (G * D + kSelThreads - 1) / kSelThreads;   // elements per thread (one head)
    const int e0 = tid * EPT;
    const bool mine = e0 < G * D;
    const int gg = mine ? e0 / D : 0;
    float M = -INFINITY, Ls = 0.0f, A[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) A[e] = 0.0f;
#pragma unroll 1
    for (int k0 = 0; k0 < nparts; k0 += KB) {
        const int nk = min(KB, nparts - k0);
        if (k0 > 0) __syncthreads();   // the previous group is consumed
#pragma unroll 1
        for (int i = tid; i < nk * PS; i += kSelThreads) cp_async_4(sp + i, parts + (size_t)k0 * PS + i);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        if (mine) {
            float Mg = -INFINITY;
#pragma unroll 1
            for (int k = 0; k < nk; ++k) Mg = fmaxf(Mg, sp[k * PS + G * D + gg]);
            if (Mg != -INFINITY) {
                const float Mn = fmaxf(M, Mg);
                const float a = (M == -INFINITY) ? 0.0f : expf(M - Mn);
                Ls *= a;
#pragma unroll
                for (int e = 0; e < EPT; ++e) A[e] *= a;
#pragma unroll 1
                for (int k = 0; k < nk; ++k) {
                    const float mk = sp[k * PS + G * D + gg];
                    const float wgt = (mk == -INFINITY) ? 0.0f : expf(mk - Mn);
                    Ls = fmaf(sp[k * PS + G * D + G + gg], wgt, Ls);
#pragma unroll
                    for (int e = 0; e < EPT; ++e) A[e] = fmaf(sp[k * PS + e0 + e], wgt, A[e]);
                }
                M = Mn;
            }
        }
    }
    if (mine) {
        const int64_t head = (int64_t)b * p.Hq + (int64_t)h * G + gg;
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            const int c = (e0 + e) % D;
            p.out[head * D + c] = (Ls > 0.0f) ? A[e] / Ls : 0.0f;
            if (c == 0) p.lse[head] = (Ls > 0.0f) ? M + logf(Ls) : -INFINITY;
        }
    }
    SSA_MARK(9);
    SSA_GT(7);
}

// ---------------------------------------------------------------------------
// the early-stop order
// ---------------------------------------------------------------------------
// ("S2O: early stopping for sparse attention via online permutation",
// technical summary, Method section 2: blocks are processed in descending
// estimated importance.)  One CTA of kOrderThreads per unit sorts the unit's
// list (idx_in / p_in, count_in entries, row stride cap) by its rows'
// scores s_src[u][idx] descending, ties by list position, and writes the
// ordered list to the workspace's selection rows (stride pl.np) and its
// length to the early-stop counts.
//
// The sort is a least-significant-digit radix sort of the 32-bit keys
// (~order key, so ascending is descending score), four passes of 8 bits,
// each stable: warp w owns a contiguous run of the elements and walks it 32
// at a time, an element's rank among the batch's equal digits comes from
// eight ballots (one per digit bit), and the digits' offsets are an exclusive scan over
// (digit, warp) -- so equal keys keep their list order.  The elements (key,
// position) ping-pong between two arrays, in shared memory for lists of up to
// kOrderSmemRows rows and in the workspace for longer ones (the CTA's own
// writes, read back after a block barrier).  Lists longer than
// kOrderCap (or than a row) keep their first entries and set
// SSA_DEV_OVERFLOW; an index outside [0, N) sets SSA_DEV_BAD_INDEX and sorts
// last.  The input may be the output rows: every read of the input ends
// before the first write.
constexpr int kOrderThreads = 1024;
constexpr int kOrderCap = kEsMaxRows;
constexpr int kOrderWarps = kOrderThreads / 32;
constexpr uint32_t kOrderCounters = (uint32_t)kOrderWarps * 256u * 4u;   // per-warp digit counters
constexpr int kOrderSmemRows = 12288;   // lists up to this long sort in shared memory, longer ones in the workspace
constexpr uint32_t kOrderSmem = kOrderCounters + (uint32_t)kOrderWarps * 4u +   // + the scan's scratch
                                2u * kOrderSmemRows * 8u;                       // + the two element arrays

// The lanes of the warp whose 8-bit digit equals this lane's, among the
// lanes with `ok` set (eight ballots, one per bit).
__device__ __forceinline__ uint32_t digit_peers(uint32_t d, bool ok)
{
    uint32_t peers = __ballot_sync(0xffffffffu, ok);
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const bool bit = (d >> b) & 1u;
        const uint32_t m = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? m : ~m;
    }
    return peers;
}

__global__ void __launch_bounds__(kOrderThreads, 1) order_kernel(const __grid_constant__ Params p)
{
    extern __shared__ __align__(16) unsigned char osm[];
    // [warp][digit] (a warp's digits in different banks): counts, then running offsets
    uint32_t* cnt = reinterpret_cast<uint32_t*>(osm);
    const Plan& pl = p.pl;
    const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* status = ws_status(p);
    SSA_MARK(30);
    grid_dep_wait();   // the lists may come from the previous kernel
    SSA_MARK(31);
    int64_t n64 = p.count_in[u];
    n64 = n64 < 0 ? 0 : (n64 > p.cap ? p.cap : n64);
    const int64_t room = min((int64_t)kOrderCap, pl.np);
    if (n64 > room) {
        if (tid == 0) flag(status, DEV_OVERFLOW);
        n64 = room;
    }
    const int n = (int)n64;
    const int32_t* idx = p.idx_in + (int64_t)u * p.cap;
    const float* pin = p.p_in + (int64_t)u * p.cap;
    const float* srow = p.s_src + (int64_t)u * pl.N;
    // the element arrays: in shared memory when the list fits, else in the workspace (generic pointers)
    uint2* bufA;
    uint2* bufB;
    if (n <= kOrderSmemRows) {
        bufA = reinterpret_cast<uint2*>(osm + kOrderCounters + kOrderWarps * 4);
        bufB = bufA + kOrderSmemRows;
    } else {
        bufA = ws_es_sort(p) + (size_t)u * 2 * pl.esr;
        bufB = bufA + pl.esr;
    }
    for (int i = tid; i < n; i += kOrderThreads) {
        uint32_t k = 0xffffffffu;
        const int32_t j = idx[i];
        if (j >= 0 && (int64_t)j < pl.N) k = ~okey(srow[j]);
        else flag(status, DEV_BAD_INDEX);
        bufA[i] = make_uint2(k, (uint32_t)i);
    }
    __syncthreads();
    SSA_MARK(32);
    const int per = (n + kOrderWarps - 1) / kOrderWarps;   // elements of each warp's run
    const int w0 = min(n, warp * per), w1 = min(n, w0 + per);
#pragma unroll 1
    for (int shift = 0; shift < 32; shift += 8) {
        for (int i = tid; i < 256 * kOrderWarps; i += kOrderThreads) cnt[i] = 0u;
        __syncthreads();
        // this warp's count of each digit
#pragma unroll 1
        for (int b = w0; b < w1; b += 32) {
            const int i = b + lane;
            const bool ok = i < w1;
            const uint32_t d = ok ? (bufA[i].x >> shift) & 0xffu : 0u;
            const uint32_t peers = digit_peers(d, ok);
            if (ok && lane == __ffs(peers) - 1) cnt[warp * 256 + d] += (uint32_t)__popc(peers);
        }
        __syncthreads();
        // exclusive scan over (digit, warp) in that order: thread t holds entries [8t, 8t + 8), entry
        // d * warps + w stored at cnt[w * 256 + d]
        {
            constexpr int E = 256 * kOrderWarps / kOrderThreads;
            uint32_t v[E], local = 0;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int x = tid * E + e;
                v[e] = cnt[(x % kOrderWarps) * 256 + x / kOrderWarps];
                local += v[e];
            }
            uint32_t total;
            uint32_t run = block_excl_scan<kOrderThreads>(local, reinterpret_cast<uint32_t*>(osm + kOrderCounters),
                                                          total);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int x = tid * E + e;
                cnt[(x % kOrderWarps) * 256 + x / kOrderWarps] = run;
                run += v[e];
            }
        }
        __syncthreads();
        // the stable scatter: this warp's elements in order, each after the earlier equal digits
#pragma unroll 1
        for (int b = w0; b < w1; b += 32) {
            const int i = b + lane;
            const bool ok = i < w1;
            const uint2 e = ok ? bufA[i] : make_uint2(0u, 0u);
            const uint32_t d = ok ? (e.x >> shift) & 0xffu : 0u;
            const uint32_t peers = digit_peers(d, ok);
            const uint32_t rank = (uint32_t)__popc(peers & lanemask_lt());
            uint32_t base = 0;
            if (ok) base = cnt[warp * 256 + d];
            __syncwarp();
            if (ok) {
                bufB[base + rank] = e;
                if (lane == __ffs(peers) - 1) cnt[warp * 256 + d] = base + (uint32_t)__popc(peers);
            }
            __syncwarp();
        }
        __syncthreads();
        uint2* t = bufA;
        bufA = bufB;
        bufB = t;
        SSA_MARK(33 + shift / 8);
    }
    // the ordered list: every read of the input rows, then the writes (the input may be those rows)
    int32_t* oidx = ws_sel_idx(p) + (size_t)u * pl.np;
    float* op = ws_sel_p(p) + (size_t)u * pl.np;
    for (int i = tid; i < n; i += kOrderThreads) {
        const uint32_t ps = bufA[i].y;
        bufB[i] = make_uint2((uint32_t)idx[ps], __float_as_uint(pin[ps]));
    }
    __syncthreads();
    for (int i = tid; i < n; i += kOrderThreads) {
        const uint2 v = bufB[i];
        oidx[i] = (int32_t)v.x;
        op[i] = __uint_as_float(v.y);
    }
    if (tid == 0) ws_es_count(p)[u] = n;
    SSA_MARK(37);
    grid_dep_launch();
}

// Append-time summary: Ks[b][h][i][j] = K[b][h][i][sel_ch[h][j]].
__global__ void pack_summary_kernel(const uint16_t* __restrict__ K, const int32_t* __restrict__ sel_ch,
                                    uint16_t* __restrict__ Ks, int32_t Hkv, int32_t d, int32_t d_sel,
                                    int64_t N, int64_t kv_sb, int64_t kv_sh, int64_t ks_sb, int64_t ks_sh,
                                    int64_t total, uint32_t* status)
{
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(e % d_sel);
        const int64_t i = (e / d_sel) % N;
        const int64_t bh = e / ((int64_t)d_sel * N);
        const int h = (int)(bh % Hkv);
        const int64_t b = bh / Hkv;
        int ch = sel_ch[h * d_sel + j];
        if ((unsigned)ch >= (unsigned)d) {
            flag(status, DEV_BAD_INDEX);
            ch = ch < 0 ? 0 : d - 1;
        }
        Ks[b * ks_sb + h * ks_sh + i * d_sel + j] = K[b * kv_sb + h * kv_sh + i * d + ch];
    }
}

}  // namespace ssa
