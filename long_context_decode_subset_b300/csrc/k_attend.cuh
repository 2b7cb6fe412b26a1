// k_attend.cuh -- K3: exact softmax attention over the selected rows with
// the inclusion correction.
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
// P CTAs per unit each take an even share of the unit's selected list
// (positions [r * R / P, (r + 1) * R / P)), staged in shared memory in
// chunks; every CTA first takes the final keep decisions for its entries
// (top-k stratum, or the draw u < p with the exact p) and keeps the chosen
// rows in list order.  Two kernels then do the attention:
//  * attend_tc_kernel (head_dim 128): the rows go through the tensor cores
//    128 at a time -- S = K Q^T and O^T = V^T P with tcgen05.mma, fp32
//    accumulators in tensor memory, P split into two bf16 terms (hi + lo) so
//    that the products keep fp32-level accuracy -- and the P CTAs of a unit,
//    in clusters of 4, merge their (m, l, acc) through distributed shared
//    memory (then the clusters' partials through global memory);
//  * attend_kernel (head_dim 64): CUDA cores, every warp streaming its rows
//    with cp.async; the last CTA of a unit merges the P partials.
#pragma once
#include "k_select.cuh"

namespace ssa {


// ---------------------------------------------------------------------------
// shared pieces: the unit's list, the final decisions, the compact list
// ---------------------------------------------------------------------------

// What the decisions need from the selection (per-tile lists only).
struct UnitSel {
    uint32_t theta;
    int64_t cut;
    float m, Z;
    bool sampling;
};

__device__ __forceinline__ UnitSel load_unit_sel(const Params& p, int u)
{
    UnitSel s{0u, -1, 0.0f, 0.0f, false};
    if (p.src_mode == 0) {
        const UnitCtrl* ctrl = ws_ctrl(p) + u;
        s.theta = __ldcg(&ctrl->theta);
        s.cut = __ldcg(&ctrl->idx_cut);
        s.m = __ldcg(&ctrl->m);
        s.Z = __ldcg(&ctrl->Z);
    }
    s.sampling = p.budget > 0.0f && s.Z > 0.0f;
    return s;
}

// The unit's list length.  For per-tile lists (source 0) also the exclusive
// prefix of the per-slice counts, pre[0..nlists] in shared memory (counts
// staged with cp.async).  NT threads; ends with a block barrier.
template <int NT>
__device__ int64_t list_total(const Params& p, int u, int nlists, uint32_t* pre, uint32_t* scan)
{
    const int tid = threadIdx.x;
    int64_t total = 0;
    if (p.src_mode == 0) {
        const uint32_t* sc = ws_scount(p) + (size_t)u * nlists;
#pragma unroll 1
        for (int l = tid; l < nlists; l += NT) cp_async_4(pre + l, sc + l);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        const int l0 = nlists * tid / NT, l1 = nlists * (tid + 1) / NT;
        uint32_t mine = 0;
#pragma unroll 1
        for (int l = l0; l < l1; ++l) {
            const uint32_t c = pre[l];
            pre[l] = mine;
            mine += c;
        }
        uint32_t tot;
        const uint32_t before = block_excl_scan<NT>(mine, scan, tot);
#pragma unroll 1
        for (int l = l0; l < l1; ++l) pre[l] += before;
        if (tid == 0) pre[nlists] = tot;
        total = tot;
    } else if (p.src_mode == 1) {
        total = p.pl.N;
    } else {
        const int64_t c = p.count_in[u];
        total = c < 0 ? 0 : (c > p.cap ? p.cap : c);
    }
    __syncthreads();
    return total;
}

// Entries [c0, c0 + n) of the unit's list (n <= LIST): staged through
// ridx / rval (cp.async, one wave), decided, and the kept ones written in
// list order to cidx / clp (log p) [0, nk).  Returns nk (every thread).
// With a compact list requested, the kept (index, p) pairs also go to the
// unit's staging area at stage_at.  NT threads; ends with a block barrier.
template <int LIST, int NT>
__device__ int stage_decide(const Params& p, int u, int b, int h, int64_t c0, int n, int64_t stage_at,
                            const uint32_t* pre, int nlists, const UnitSel& us, int32_t* ridx, float* rval,
                            int32_t* cidx, float* clp, uint32_t* scan)
{
    constexpr int PER = (LIST + NT - 1) / NT;   // entries per thread at most
    static_assert(PER <= 32, "one keep bit per entry in a word");
    const Plan& pl = p.pl;
    const int tid = threadIdx.x;
    const int W2 = pl.tt / kSelWarps;
    uint32_t* status = ws_status(p);
    const int32_t* sidx = ws_sel_idx(p) + (size_t)u * pl.np;
    const float* sp = ws_sel_p(p) + (size_t)u * pl.np;
    if (p.src_mode == 0) {
#pragma unroll 1
        for (int i = tid; i < n; i += NT) {
            const int64_t pos = c0 + i;
            int lo_l = 0, hi_l = nlists;   // pre[lo_l] <= pos < pre[hi_l]
            while (hi_l - lo_l > 1) {
                const int mid = (lo_l + hi_l) >> 1;
                if ((int64_t)pre[mid] <= pos) lo_l = mid; else hi_l = mid;
            }
            const size_t at = (size_t)(lo_l / kSelWarps) * pl.tt + (size_t)(lo_l % kSelWarps) * W2 + (pos - pre[lo_l]);
            cp_async_4(ridx + i, sidx + at);
            cp_async_4(rval + i, sp + at);
        }
    } else if (p.src_mode == 2) {
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
        if (p.src_mode == 1) {
            j = (int32_t)(c0 + i);
            pv = 1.0f;
            keep = true;
        } else {
            j = ridx[i];
            pv = rval[i];
            if (p.src_mode == 0) {
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
                        ev = expf(__fsub_rn(pv, us.m));
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
    // the kept entries in list order
    uint32_t nk;
    uint32_t at = block_excl_scan<NT>(kcount, scan, nk);
#pragma unroll 1
    for (int e = 0; e < e1 - e0; ++e) {
        if (!((kbits >> e) & 1u)) continue;
        const int i = e0 + e;
        const int32_t j = (p.src_mode == 1) ? (int32_t)(c0 + i) : ridx[i];
        const float pv = (p.src_mode == 1) ? 1.0f : rval[i];
        cidx[at] = j;
        clp[at] = logf(pv);
        if (p.idx_out)
            ws_cand(p)[(size_t)u * pl.N + (size_t)(stage_at + at)] = make_uint2((uint32_t)j, __float_as_uint(pv));
        ++at;
    }
    __syncthreads();
    SSA_MARK(29);
    return (int)nk;
}

// Records this CTA's kept count; the last CTA of the unit (returned true)
// writes the count and, if asked, the compact list in list order (copied
// from the per-CTA staging).  `koff` is shared scratch of at least
// kMaxSplit + 1 words.  NT threads.
template <int NT>
__device__ bool finish_lists(const Params& p, int u, int P, int r, int64_t kept, int64_t total, uint32_t* koff,
                             uint32_t* flag_smem)
{
    const Plan& pl = p.pl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* kept_all = ws_kept(p) + (size_t)u * kMaxSplit;
    __syncthreads();   // the CTA's writes, then one fence and the count (cumulative)
    if (tid == 0) {
        kept_all[r] = (uint32_t)kept;
        __threadfence();
        *flag_smem = (atomicAdd(&ws_ctrl(p)[u].k3_done, 1u) == (uint32_t)(P - 1)) ? 1u : 0u;
    }
    __syncthreads();
    const bool last = *flag_smem != 0u;
    if (!last) return false;
    __threadfence();
    if (p.count_out || p.idx_out) {
        if (warp == 0) {
            uint32_t run = 0;
#pragma unroll 1
            for (int r0 = 0; r0 < P; r0 += 32) {
                const uint32_t v = (r0 + lane < P) ? __ldcg(kept_all + r0 + lane) : 0u;
                const uint32_t x = warp_incl_scan(v);
                if (r0 + lane < P) koff[r0 + lane] = run + x - v;
                run += __shfl_sync(0xffffffffu, x, 31);
            }
            if (lane == 0) koff[P] = run;
        }
        __syncthreads();
        const uint32_t kept_total = koff[P];
        if (p.count_out && tid == 0) p.count_out[u] = (int32_t)kept_total;
        if (p.idx_out) {
            const uint2* stage = ws_cand(p) + (size_t)u * pl.N;
#pragma unroll 1
            for (uint32_t o = tid; o < kept_total; o += NT) {
                int lo_r = 0, hi_r = P;   // koff[lo_r] <= o < koff[hi_r]
                while (hi_r - lo_r > 1) {
                    const int mid = (lo_r + hi_r) >> 1;
                    if (koff[mid] <= o) lo_r = mid; else hi_r = mid;
                }
                const int64_t src = total * lo_r / P + (int64_t)(o - koff[lo_r]);
                const uint2 v = __ldcg(stage + src);
                if ((int64_t)o < p.cap) {
                    p.idx_out[(int64_t)u * p.cap + o] = (int32_t)v.x;
                    p.p_out[(int64_t)u * p.cap + o] = __uint_as_float(v.y);
                } else {
                    flag(ws_status(p), DEV_OVERFLOW);
                }
            }
        }
        __syncthreads();
    }
    return true;
}

// Merge NP partials [NP][G * D + 2G] (acc, then m, then l) in a fixed order
// (index ascending) and write the unit's output rows and log-sum-exp.  One
// wave of loads per thread: each of the first 256 threads owns
// G * D / 256 elements of one head and reads that head's (m, l) of all
// partials itself.
template <int G, int D>
__device__ void merge_partials(const Params& p, int b, int h, const float* parts, int NP)
{
    constexpr int MT = 256;   // merging threads
    constexpr int PS = G * D + 2 * G;   // floats per partial
    constexpr int EPT = (G * D + MT - 1) / MT;   // elements per thread (same head)
    static_assert((G * D) % MT == 0 || G * D < MT, "elements split evenly");
    if (threadIdx.x >= MT) return;
    const int e0 = threadIdx.x * EPT;
    if (e0 >= G * D) return;
    const int g = e0 / D;
    float M = -INFINITY;
#pragma unroll 1
    for (int r0 = 0; r0 < NP; r0 += 16) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (r0 + j < NP) M = fmaxf(M, __ldcg(parts + (size_t)(r0 + j) * PS + G * D + g));
    }
    float Ls = 0.0f, A[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) A[e] = 0.0f;
    if (M != -INFINITY) {
#pragma unroll 1
        for (int r0 = 0; r0 < NP; r0 += 8) {
            float mr[8], lr[8], ar[8][EPT];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float* pr = parts + (size_t)(r0 + j) * PS;
                const bool ok = r0 + j < NP;
                mr[j] = ok ? __ldcg(pr + G * D + g) : -INFINITY;
                lr[j] = ok ? __ldcg(pr + G * D + G + g) : 0.0f;
#pragma unroll
                for (int e = 0; e < EPT; ++e) ar[j][e] = ok ? __ldcg(pr + e0 + e) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float wgt = (mr[j] == -INFINITY) ? 0.0f : expf(mr[j] - M);
                Ls = fmaf(lr[j], wgt, Ls);
#pragma unroll
                for (int e = 0; e < EPT; ++e) A[e] = fmaf(ar[j][e], wgt, A[e]);
            }
        }
    }
    const int64_t head = (int64_t)b * p.Hq + (int64_t)h * G + g;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const int c = (e0 + e) % D;
        p.out[head * D + c] = (Ls > 0.0f) ? A[e] / Ls : 0.0f;
        if (c == 0) p.lse[head] = (Ls > 0.0f) ? M + logf(Ls) : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// attend_tc_kernel: head_dim 128, tensor cores, clusters of kClusterCtas CTAs
// ---------------------------------------------------------------------------

constexpr int kClusterCtas = 4;   // attend_tc_kernel: the CTAs of a unit merged on chip
constexpr int kTcGatherWarps = 7;                       // warps 5 .. 11
constexpr int kTcThreads = (5 + kTcGatherWarps) * 32;   // 384

// A chunk is one 128-row MMA operand of K (and one of V) rows in the
// 128-byte swizzled layout: row i's 16-byte piece c at piece c ^ (i & 7) of
// the row's 64-dim plane.
template <int G, int LIST>   // LIST: list entries staged at a time (1024 or 4096)
struct KTCfg {
    static constexpr int D = 128;
    static constexpr int CH = 128;                                 // listed rows per chunk
    static constexpr uint32_t PLANE = CH * 128u;                   // 64 dims x 128 rows, 128-byte swizzle
    static constexpr uint32_t KV = 2u * PLANE;                     // one K or V chunk (32 KB)
    static constexpr uint32_t QPLANE = 16u * 128u;                 // 64 elements x 16 rows
    static constexpr uint32_t OFF_K = 0;                           // 2 chunks
    static constexpr uint32_t OFF_V = OFF_K + 2u * KV;             // 2 chunks
    static constexpr uint32_t OFF_Q = OFF_V + 2u * KV;             // query operand: 16 x 128, 4 KB
    static constexpr uint32_t OFF_P = OFF_Q + 2u * QPLANE;         // 2 x P operand: 16 columns x 128 rows
    static constexpr uint32_t OFF_LIST = OFF_P + 2u * 2u * QPLANE; // cidx, clp
    static constexpr uint32_t OFF_RAW = OFF_LIST + (uint32_t)LIST * 8u;       // raw list staging
    static constexpr uint32_t OFF_PART = OFF_RAW + (uint32_t)LIST * 8u;       // (acc, m, l): G * D + 2G floats
    static constexpr uint32_t OFF_RED = OFF_PART + (uint32_t)(G * D + 2 * G) * 4u;   // [2][2][4][G] floats
    static constexpr uint32_t OFF_BAR = (OFF_RED + 2u * 2u * 4u * G * 4u + 7u) & ~7u;
    static constexpr uint32_t NBAR = 10;                           // kv_full, kv_free, s_full, p_ready, o_full (x2)
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;      // tensor-memory slot, flags
    static constexpr uint32_t OFF_PRE = OFF_MISC + 64u;
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 16);       // S = K Q^T
    static constexpr uint32_t IDESC_O = idesc_bf16_f32_amn(128, 16);   // O^T = V^T P
    static constexpr uint32_t TCOLS = 64;                          // S x2 (cols 0-31), O x2 (cols 32-63)
    static_assert(2 * G <= 16, "P's hi and lo columns fit in N = 16");
};

template <int G, int LIST>
constexpr uint32_t ktc_smem_bytes(int nlists)
{
    return KTCfg<G, LIST>::OFF_PRE + (uint32_t)(nlists + 1) * 4u + 1024u;   // + alignment slack
}

// Thread roles (kTcThreads): warps 0-3 epilogue (tensor-memory lanes =
// chunk rows for S, = head dims for O), warp 4 issues the MMAs (and owns the
// tensor memory), warps 5 .. 11 gather the K and V rows.  Chunk g uses buffers
// g & 1; barrier phases count chunks over the whole CTA.
template <int G, int LIST>
__global__ void __launch_bounds__(kTcThreads, 1) attend_tc_kernel(const __grid_constant__ Params p)
{
    using CF = KTCfg<G, LIST>;
    constexpr int CL = kClusterCtas;
    constexpr int D = CF::D;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    __shared__ uint32_t scan[kTcThreads / 32];
    int32_t* cidx = reinterpret_cast<int32_t*>(smem + CF::OFF_LIST);
    float* clp = reinterpret_cast<float*>(smem + CF::OFF_LIST + LIST * 4);
    float* part = reinterpret_cast<float*>(smem + CF::OFF_PART);
    float* red = reinterpret_cast<float*>(smem + CF::OFF_RED);   // [parity][max | sum][warp][G]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CF::OFF_BAR);
    uint64_t* kv_full = bars;
    uint64_t* kv_free = bars + 2;
    uint64_t* s_full = bars + 4;
    uint64_t* p_ready = bars + 6;
    uint64_t* o_full = bars + 8;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + CF::OFF_MISC);   // [0] tensor memory, [1], [2] flags
    uint32_t* pre = reinterpret_cast<uint32_t*>(smem + CF::OFF_PRE);

    const Plan& pl = p.pl;
    const int P = pl.P;
    const int u = blockIdx.x / P, r = blockIdx.x % P;
    const int b = u / p.Hkv, h = u % p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nlists = pl.ntile * kSelWarps;
    uint32_t* status = ws_status(p);

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kv_full[i], 32 * kTcGatherWarps);   // every gather thread's copies
            mbar_init(&kv_free[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 4);   // one arrive per epilogue warp
            mbar_init(&o_full[i], 1);
        }
        fence_mbar_init();
    }
    if (warp == 4) tmem_alloc(&misc[0], CF::TCOLS);
    // the query operand: head slot n < G = q_n (the scale is applied to S),
    // slots G..15 zero; K-major, 128-byte swizzle, two 64-dim planes
    if (tid < 256) {
        const int n = tid >> 4, pc = tid & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < G && p.attend)
            v = *reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + (int64_t)h * G + n) * D + pc * 8);
        *reinterpret_cast<uint4*>(smem + CF::OFF_Q + (pc >> 3) * CF::QPLANE + n * 128 + (((pc & 7) ^ (n & 7)) << 4)) = v;
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = misc[0];
    SSA_GT(4);
    grid_dep_wait();
    SSA_MARK(7);
    SSA_GT(5);

    const int64_t total = list_total<kTcThreads>(p, u, nlists, pre, scan);
    SSA_MARK(11);
    const int64_t lo = total * r / P, hi = total * (r + 1) / P;
    const UnitSel us = load_unit_sel(p, u);
    const uint16_t* Kb = p.K + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;
    const uint16_t* Vb = p.V + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;

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
        const int nk = stage_decide<LIST, kTcThreads>(p, u, b, h, c0, n, lo + kept, pre, nlists, us, ridx, rval, cidx,
                                                         clp, scan);
        kept += nk;
        const int nc = p.attend ? (nk + CF::CH - 1) / CF::CH : 0;
        if (warp >= 5) {
            // gather: 16-byte pieces of the chunk's K and V rows into the
            // 128-byte swizzled planes (rows past the list read as zeros)
            const int gt = tid - 160;   // 0 .. 32 * kTcGatherWarps - 1
            // each thread's copies of chunk c arrive on kv_full when they land
            // (cp.async.mbarrier.arrive), so publishing never waits on a later
            // chunk's buffer
#pragma unroll 1
            for (int c = 0; c < nc; ++c) {
                const int g = gbase + c, bf = g & 1;
                if (g >= 2) {
                    if (lane == 0 && !mbar_wait_bounded(&kv_free[bf], (uint32_t)((g - 2) >> 1) & 1u)) flag(status, DEV_TIMEOUT);
                    __syncwarp();
                }
                unsigned char* kd = smem + CF::OFF_K + bf * CF::KV;
                unsigned char* vd = smem + CF::OFF_V + bf * CF::KV;
#pragma unroll 1
                for (int q = gt; q < CF::CH * 16; q += 32 * kTcGatherWarps) {
                    const int i = q >> 4, pc = q & 15;
                    const int row = c * CF::CH + i;
                    const bool valid = row < nk;
                    const int64_t j = valid ? (int64_t)cidx[row] : 0;
                    const uint32_t off = (uint32_t)(pc >> 3) * CF::PLANE + (uint32_t)i * 128u + ((uint32_t)((pc & 7) ^ (i & 7)) << 4);
                    cp_async_16_zfill(kd + off, Kb + j * D + pc * 8, valid);
                    cp_async_16_zfill(vd + off, Vb + j * D + pc * 8, valid);
                }
                cp_async_mbar_arrive(&kv_full[bf]);
            }
            cp_async_wait<0>();
        } else if (warp == 4) {
            if (lane == 0) {
                auto mma_s = [&](int g) {   // S[g & 1] = K_g Q^T
                    const int bf = g & 1;
                    if (!mbar_wait_bounded(&kv_full[bf], (uint32_t)(g >> 1) & 1u)) flag(status, DEV_TIMEOUT);
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
                };
                // S of chunk g, then (once P_g is written) O of chunk g: the MMA
                // that frees a K/V buffer never waits on a later chunk's copies
#pragma unroll 1
                for (int c = 0; c < nc; ++c) {
                    const int g = gbase + c, bf = g & 1;
                    mma_s(g);
                    if (!mbar_wait_bounded(&p_ready[bf], (uint32_t)(g >> 1) & 1u)) flag(status, DEV_TIMEOUT);
                    tc_fence_after();
                    // O^T[g & 1] = V_g^T P_g: A = the V rows read MN-major (64-dim
                    // atoms PLANE apart, 8-row groups 1 KB apart), 16 rows a step
#pragma unroll
                    for (int ks = 0; ks < CF::CH / 16; ++ks) {
                        const uint32_t a = v_a + bf * CF::KV + ks * 2048u;
                        const uint32_t bp = p_a + bf * 2u * CF::QPLANE + (ks >> 2) * CF::QPLANE + (ks & 3) * 32u;
                        tc_mma_bf16(tbase + 32u + bf * 16u, smem_desc_mn_sw128(a, CF::PLANE, 1024u),
                                    smem_desc_kmajor_swz(bp, 128), CF::IDESC_O, ks > 0 ? 1u : 0u);
                    }
                    tc_commit(&o_full[bf]);
                    tc_commit(&kv_free[bf]);
                }
            }
        } else {
            // epilogue (tid = tensor-memory lane)
            const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < nc; ++c) {
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
                float x[G], mc[G], lc[G];
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
                // fold O_g (this thread's head dim, hi + lo columns) into acc
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
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    const float mn = fmaxf(m_run[gg], mc[gg]);
                    const float ar = (m_run[gg] == -INFINITY) ? 0.0f : expf(m_run[gg] - mn);
                    const float ac = (mc[gg] == -INFINITY) ? 0.0f : expf(mc[gg] - mn);
                    acc[gg] = acc[gg] * ar + (o[gg] + o[G + gg]) * ac;
                    l_run[gg] = l_run[gg] * ar + lc[gg] * ac;
                    m_run[gg] = mn;
                }
            }
        }
        gbase += nc;
        __syncthreads();   // every role is done with this list chunk
    }
    SSA_MARK(8);

    // this CTA's partial: acc per head dim, then (m, l) per head
    if (warp < 4) {
#pragma unroll
        for (int gg = 0; gg < G; ++gg) part[gg * D + tid] = acc[gg];
        if (tid == 0) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                part[G * D + gg] = m_run[gg];
                part[G * D + G + gg] = l_run[gg];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tbase, CF::TCOLS);
    }
    if (p.count_out || p.idx_out)   // the merge below needs no "last CTA"
        finish_lists<kTcThreads>(p, u, P, r, kept, total, reinterpret_cast<uint32_t*>(smem + CF::OFF_K), &misc[1]);
    SSA_MARK(12);
    SSA_GT(6);
    // merge the cluster's partials on chip (rank order); with one cluster
    // per unit it writes the output, with several each writes a cluster
    // partial and the last cluster to finish merges them in cluster order
    cluster_sync();
    if (p.attend && cluster_rank() == 0) {
        const int ncl = P / CL, cl = r / CL;
        constexpr int PS = G * D + 2 * G;
        float* cpart = ws_part(p) + ((size_t)u * kMaxSplit + cl) * PS;
        constexpr int EPT = (G * D + 255) / 256;
        const int e0 = tid * EPT;
        if (tid < 256 && e0 < G * D) {
            const int gg = e0 / D;
            float mr[CL], M = -INFINITY;
#pragma unroll
            for (int k = 0; k < CL; ++k) {
                mr[k] = ld_dsmem_f32(part + G * D + gg, (uint32_t)k);
                M = fmaxf(M, mr[k]);
            }
            float Ls = 0.0f, A[EPT];
#pragma unroll
            for (int e = 0; e < EPT; ++e) A[e] = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
                for (int k = 0; k < CL; ++k) {
                    const float wgt = (mr[k] == -INFINITY) ? 0.0f : expf(mr[k] - M);
                    Ls = fmaf(ld_dsmem_f32(part + G * D + G + gg, (uint32_t)k), wgt, Ls);
#pragma unroll
                    for (int e = 0; e < EPT; ++e) A[e] = fmaf(ld_dsmem_f32(part + e0 + e, (uint32_t)k), wgt, A[e]);
                }
            }
            if (ncl == 1) {
                const int64_t head = (int64_t)b * p.Hq + (int64_t)h * G + gg;
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    const int c = (e0 + e) % D;
                    p.out[head * D + c] = (Ls > 0.0f) ? A[e] / Ls : 0.0f;
                    if (c == 0) p.lse[head] = (Ls > 0.0f) ? M + logf(Ls) : -INFINITY;
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPT; ++e) cpart[e0 + e] = A[e];
                if (e0 % D == 0) {
                    cpart[G * D + gg] = M;
                    cpart[G * D + G + gg] = Ls;
                }
            }
        }
        if (ncl > 1) {
            __syncthreads();   // the cluster partial's writes, then one fence and the count
            if (tid == 0) {
                __threadfence();
                misc[2] = (atomicAdd(&ws_ctrl(p)[u].k3_cdone, 1u) == (uint32_t)(ncl - 1)) ? 1u : 0u;
            }
            __syncthreads();
            if (misc[2]) {
                __threadfence();
                merge_partials<G, D>(p, b, h, ws_part(p) + (size_t)u * kMaxSplit * PS, ncl);
            }
        }
    }
    cluster_sync();   // the cluster's shared memory stays until rank 0 has read it
    SSA_MARK(9);
    SSA_GT(7);
}

// ---------------------------------------------------------------------------
// attend_kernel: CUDA cores (head_dim 64)
// ---------------------------------------------------------------------------

template <int G, int D>
struct K3Cfg {
    static constexpr int DPL = (G <= 4) ? 8 : 4;              // dims per lane (16 or 8 bytes)
    static constexpr int LPR = D / DPL;                       // lanes per row
    static constexpr int RPW = 32 / LPR;                      // rows per warp per step
    static constexpr int RPS = k3Warps * RPW;                 // rows per CTA step
    static constexpr int NS = 8;                              // steps in flight per warp
    static constexpr uint32_t ROWB = D * 2u;
    static constexpr uint32_t STAGE_W = (uint32_t)RPW * 2u * ROWB;    // K and V rows of one warp step
    static constexpr uint32_t RING = (uint32_t)k3Warps * NS * STAGE_W;
    static constexpr uint32_t MERGE = (uint32_t)k3Warps * G * D * 4u;
    static constexpr uint32_t OFF_CHUNK = RING > MERGE ? RING : MERGE;
    static constexpr int CHUNK = 1024;                        // list entries staged at a time
    static constexpr uint32_t OFF_PRE = OFF_CHUNK + (uint32_t)CHUNK * 8u;
    static_assert(OFF_CHUNK >= (uint32_t)CHUNK * 8u, "the raw chunk staging fits in front of the kept lists");
};

// Dynamic shared memory of attend_kernel for nlists per-tile lists.
template <int G, int D>
constexpr uint32_t k3_smem_bytes(int nlists)
{
    return K3Cfg<G, D>::OFF_PRE + (uint32_t)(nlists + 1) * 4u + 128u;
}

struct K3Shared {
    uint32_t scan[k3Warps];
    float wm[k3Warps][8], wl[k3Warps][8];
    uint32_t is_last;
};

template <int G, int D>
__global__ void __launch_bounds__(k3Threads) attend_kernel(const __grid_constant__ Params p)
{
    using CF = K3Cfg<G, D>;
    constexpr int DPL = CF::DPL;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                           ~static_cast<uintptr_t>(127));
    __shared__ K3Shared ks;
    int32_t* cidx = reinterpret_cast<int32_t*>(smem + CF::OFF_CHUNK);
    float* clp = reinterpret_cast<float*>(smem + CF::OFF_CHUNK + CF::CHUNK * 4);
    uint32_t* pre = reinterpret_cast<uint32_t*>(smem + CF::OFF_PRE);

    const Plan& pl = p.pl;
    const int P = pl.P;
    const int u = blockIdx.x / P, r = blockIdx.x % P;
    const int b = u / p.Hkv, h = u % p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nlists = pl.ntile * kSelWarps;   // K2 writes one list per warp slice of a tile
    SSA_GT(4);
    grid_dep_wait();
    SSA_MARK(7);
    SSA_GT(5);

    const int64_t total = list_total<k3Threads>(p, u, nlists, pre, ks.scan);
    SSA_MARK(11);
    const int64_t lo = total * r / P, hi = total * (r + 1) / P;
    const uint16_t* Kb = p.K + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;
    const uint16_t* Vb = p.V + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;
    const UnitSel us = load_unit_sel(p, u);

    const int sub = lane / CF::LPR, li = lane % CF::LPR;
    float qv[G][DPL];
    float mrun[G], lrun[G], acc[G][DPL];
    if (p.attend) {
        const uint16_t* qb = p.q + ((int64_t)b * p.Hq + (int64_t)h * G) * D + li * DPL;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < DPL; ++c) qv[g][c] = bf16_at(qb + (int64_t)g * D + c);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        mrun[g] = -INFINITY;
        lrun[g] = 0.0f;
#pragma unroll
        for (int c = 0; c < DPL; ++c) acc[g][c] = 0.0f;
    }
    unsigned char* wring = smem + (size_t)warp * CF::NS * CF::STAGE_W + (size_t)sub * 2u * CF::ROWB + li * DPL * 2;
    int64_t kept = 0;   // entries this CTA keeps

#pragma unroll 1
    for (int64_t c0 = lo; c0 < hi; c0 += CF::CHUNK) {
        const int n = (int)min((int64_t)CF::CHUNK, hi - c0);
        __syncthreads();   // the previous chunk is consumed
        int32_t* ridx = reinterpret_cast<int32_t*>(smem);
        float* rval = reinterpret_cast<float*>(smem + CF::CHUNK * 4);
        const int nk = stage_decide<CF::CHUNK, k3Threads>(p, u, b, h, c0, n, lo + kept, pre, nlists, us, ridx, rval,
                                                          cidx, clp, ks.scan);
        kept += nk;
        if (!p.attend) continue;
        const int nsteps = (nk + CF::RPS - 1) / CF::RPS;
        auto issue = [&](int step) {
            const int row = step * CF::RPS + warp * CF::RPW + sub;
            if (step < nsteps && row < nk) {
                const int32_t j = cidx[row];
                if (j >= 0) {
                    unsigned char* dst = wring + (size_t)(step % CF::NS) * CF::STAGE_W;
                    if constexpr (DPL == 8) {
                        cp_async_16(dst, Kb + (int64_t)j * D + li * DPL);
                        cp_async_16(dst + CF::ROWB, Vb + (int64_t)j * D + li * DPL);
                    } else {
                        cp_async_8(dst, Kb + (int64_t)j * D + li * DPL);
                        cp_async_8(dst + CF::ROWB, Vb + (int64_t)j * D + li * DPL);
                    }
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int s = 0; s < CF::NS - 1; ++s) issue(s);
#pragma unroll 1
        for (int step = 0; step < nsteps; ++step) {
            issue(step + CF::NS - 1);
            cp_async_wait<CF::NS - 1>();
            const int row = step * CF::RPS + warp * CF::RPW + sub;
            const bool valid = row < nk;
            const float lp = valid ? clp[row] : 0.0f;
            const unsigned char* src = wring + (size_t)(step % CF::NS) * CF::STAGE_W;
            float kf[DPL], vf[DPL];
            if constexpr (DPL == 8) {
                const uint4 kw = *reinterpret_cast<const uint4*>(src);
                const uint4 vw = *reinterpret_cast<const uint4*>(src + CF::ROWB);
                const uint32_t ka[4] = {kw.x, kw.y, kw.z, kw.w}, va[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    kf[2 * i] = bf16_lo(ka[i]);
                    kf[2 * i + 1] = bf16_hi(ka[i]);
                    vf[2 * i] = bf16_lo(va[i]);
                    vf[2 * i + 1] = bf16_hi(va[i]);
                }
            } else {
                const uint2 kw = *reinterpret_cast<const uint2*>(src);
                const uint2 vw = *reinterpret_cast<const uint2*>(src + CF::ROWB);
                kf[0] = bf16_lo(kw.x); kf[1] = bf16_hi(kw.x); kf[2] = bf16_lo(kw.y); kf[3] = bf16_hi(kw.y);
                vf[0] = bf16_lo(vw.x); vf[1] = bf16_hi(vw.x); vf[2] = bf16_lo(vw.y); vf[3] = bf16_hi(vw.y);
            }
            float dot[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float sacc = 0.0f;
#pragma unroll
                for (int c = 0; c < DPL; ++c) sacc = fmaf(qv[g][c], kf[c], sacc);
                dot[g] = sacc;
            }
#pragma unroll
            for (int o = CF::LPR / 2; o > 0; o >>= 1)
#pragma unroll
                for (int g = 0; g < G; ++g) dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], o);
            if (valid) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float x = dot[g] * p.scale - lp;
                    if (x > mrun[g]) {
                        const float a = expf(mrun[g] - x);
                        lrun[g] *= a;
#pragma unroll
                        for (int c = 0; c < DPL; ++c) acc[g][c] *= a;
                        mrun[g] = x;
                    }
                    const float w = expf(x - mrun[g]);
                    lrun[g] += w;
#pragma unroll
                    for (int c = 0; c < DPL; ++c) acc[g][c] = fmaf(w, vf[c], acc[g][c]);
                }
            }
        }
        cp_async_wait<0>();
    }
    SSA_MARK(8);

    float* part = ws_part(p) + ((size_t)u * P + r) * (size_t)(G * D + 2 * G);
    if (p.attend) {
        // merge the row streams of a warp (lanes li, li + LPR, ...)
#pragma unroll
        for (int o = CF::LPR; o < 32; o <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mo = __shfl_xor_sync(0xffffffffu, mrun[g], o);
                const float lo_ = __shfl_xor_sync(0xffffffffu, lrun[g], o);
                const float M = fmaxf(mrun[g], mo);
                const float a = (mrun[g] == -INFINITY) ? 0.0f : expf(mrun[g] - M);
                const float ao = (mo == -INFINITY) ? 0.0f : expf(mo - M);
                lrun[g] = lrun[g] * a + lo_ * ao;
#pragma unroll
                for (int c = 0; c < DPL; ++c) {
                    const float xo = __shfl_xor_sync(0xffffffffu, acc[g][c], o);
                    acc[g][c] = acc[g][c] * a + xo * ao;
                }
                mrun[g] = M;
            }
        }
        __syncthreads();   // the ring is reused for the warp partials
        float* wpart = reinterpret_cast<float*>(smem);   // [k3Warps][G][D]
        if (lane < CF::LPR) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int c = 0; c < DPL; ++c) wpart[((size_t)warp * G + g) * D + li * DPL + c] = acc[g][c];
        }
        if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                ks.wm[warp][g] = mrun[g];
                ks.wl[warp][g] = lrun[g];
            }
        }
        __syncthreads();
#pragma unroll 1
        for (int i = tid; i < G * D; i += k3Threads) {
            const int g = i / D, c = i % D;
            float M = -INFINITY;
            for (int w = 0; w < k3Warps; ++w) M = fmaxf(M, ks.wm[w][g]);
            float A = 0.0f, Ls = 0.0f;
            if (M != -INFINITY) {
                for (int w = 0; w < k3Warps; ++w) {
                    const float mw = ks.wm[w][g];
                    if (mw == -INFINITY) continue;
                    const float e = expf(mw - M);
                    A = fmaf(wpart[((size_t)w * G + g) * D + c], e, A);
                    Ls = fmaf(ks.wl[w][g], e, Ls);
                }
            }
            part[i] = A;
            if (c == 0) {
                part[G * D + g] = M;
                part[G * D + G + g] = Ls;
            }
        }
    }
    __syncthreads();
    const bool last = finish_lists<k3Threads>(p, u, P, r, kept, total, reinterpret_cast<uint32_t*>(smem), &ks.is_last);
    SSA_MARK(12);
    SSA_GT(6);
    if (!last || !p.attend) return;
    SSA_MARK(14);
    merge_partials<G, D>(p, b, h, ws_part(p) + (size_t)u * P * (size_t)(G * D + 2 * G), P);
    SSA_MARK(9);
    SSA_GT(7);
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
