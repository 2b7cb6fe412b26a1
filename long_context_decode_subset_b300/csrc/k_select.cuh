// k_select.cuh -- K2: the threshold bucket pass of the stratified selection
// ("Stratified Sparse Attention speeds up decoding 2.96x on a 1M context",
// section "How SSA splits the cache into strata"):
//
//   T  = the k tokens with the highest scores under the order (order key
//        desc, index asc), read deterministically;
//   R  = every other token j, kept independently with probability
//        p_j = min(1, fl32(fl32(B * e_j) / Z)),  e_j = fl32(expf(fl32(s_j - m))),
//        Z = sum over R of e_j (rounded once to fp32),
//        decided by u_j < p_j with u_j = (x0 >> 8) * 2^-24, x0 = word 0 of
//        Philox4x32-10(key = seed, counter = (j, h_kv, b, 0)).
//   p is independent of m; m is the lower edge of the 12-bit order-key
//   bucket f that holds the k-th score (the largest when k = 0).
//
// Selection pass of the unit kernel (K2): one CTA of 512 threads per (unit,
// tile); each of its 16
// warps owns a contiguous slice of the tile (tile / 16 tokens), staged
// through shared memory, and walks it in index order:
//   * a token above bucket f is in T: it joins the slice's list (p = 1);
//   * a token of bucket f is a candidate: it joins the slice's list (with
//     its score) and the unit's candidate array (for the exact k-th);
//   * a token below bucket f is in R: its term e joins the tile's share of
//     Z (compensated sum, fixed order), and it joins the slice's list only
//     if it could be drawn at all: p <= B e / Z_lb for a lower bound Z_lb
//     of Z read off the histogram (every term of bucket c is at least
//     exp(floor_c - m)), and u is at least its 16-bit prefix (drawn by the
//     score kernel), so prefix >= B e / Z_lb rules it out for good.
// Once every tile of the unit has arrived, each CTA resolves the exact k-th
// token among the candidates (the same computation in every CTA of the unit,
// so no CTA waits for another's result) -- in shared memory: a 12-bit histogram, then the few members
// sharing 24 key bits ranked exactly (key desc, index asc) -- and completes
// Z: the tiles' shares in tile order plus the remainder candidates' terms,
// summed exactly as 128-bit integers (every such term is an fp32 value of at
// least one; terms of 2^81 and more, i.e. scores more than 450 apart from m,
// are flagged as out of range).  Every CTA then makes the final decision for
// its own listed tokens (k_attend.cuh).
#pragma once
#include "k_score.cuh"

namespace ssa {

constexpr uint32_t kCandFlag = 0x80000000u;   // list entry: a candidate (its value is the score)

struct SelShared {
    uint32_t scan[kSelWarps];
    uint32_t bcast[8];
    float zw[kSelWarps][2];
    float zlb[kSelWarps];
    uint32_t is_last;
    uint32_t ncand_cta;
    // resolve
    uint32_t hist[2048];   // the tie path's histograms
    uint32_t nbound;
    uint2 bound[256];
    unsigned long long zi[kSelWarps][2];
    uint32_t coff[kMaxTiles + 1];   // per-tile candidate offsets
    uint32_t wcnt[kSelWarps];       // the tile pass: list length of each warp slice
    double dscan[kSelWarps];        // the top-p select: the warps' mass sums
    double pick_m[2];               // ... the crossing bin's mass above and its own
    uint32_t pick_u[3];             // ... the crossing bin, the tokens above, its own
    // the resolve's results: order key of the k-th score, the tie cut, m and Z
    uint32_t r_theta;
    int32_t r_cut;
    float r_m, r_Z;
};

// What each (unit, tile) CTA leaves for the resolve: its share of Z
// (compensated pair) and its candidate count (its candidates sit in the
// tile's own segment of the unit's candidate array).
struct TilePart {
    float zh, zl;
    uint32_t ncand, pad;
};

constexpr int kSlice = 512;           // tokens a warp stages at a time (two chunks in flight)
constexpr int kResStage = kSelWarps * kSlice * 2 * 6 / 8;   // candidates the resolve stages at a time (same memory)
static_assert(kResStage * 8 <= kSelWarps * kSlice * 2 * 6, "the resolve's staging fits the pass's");


__device__ __forceinline__ void zacc(float& zh, float& zl, float v)
{
    float sh, er;
    two_sum(zh, v, sh, er);
    zh = sh;
    zl = __fadd_rn(zl, er);
}

// Exact 128-bit fixed-point accumulation (LSB 2^-23) of an fp32 value
// 1 <= e < 2^81: e = mant * 2^(ex - 23) with a 24-bit mant, so e is the
// integer mant << ex in units of 2^-23 and no bit is lost.  Returns false
// (and adds nothing) for a larger e.
__device__ __forceinline__ bool iacc(unsigned long long& lo, unsigned long long& hi, float e)
{
    const uint32_t u = __float_as_uint(e);
    const int ex = (int)(u >> 23) - 127;
    if (ex < 0 || ex > 80) return ex < 0 && e == 0.0f;
    const unsigned long long mant = (unsigned long long)((u & 0x7fffffu) | 0x800000u);
    unsigned long long add_lo, add_hi;
    if (ex == 0) {
        add_lo = mant;
        add_hi = 0ull;
    } else if (ex < 64) {
        add_lo = mant << ex;
        add_hi = mant >> (64 - ex);
    } else {
        add_lo = 0ull;
        add_hi = mant << (ex - 64);
    }
    const unsigned long long nlo = lo + add_lo;
    hi += add_hi + (nlo < lo ? 1ull : 0ull);
    lo = nlo;
    return true;
}

// The 128-bit count (hi, lo) of 2^-23 units as an unevaluated pair of floats
// (c_hi + c_lo equals it to a relative 2^-47): its leading 63 bits `top`
// (value = top * 2^(sh - 23) up to the dropped low bits), top rounded to a
// float, and the rest of top, both scaled by the power of two.
__device__ __forceinline__ void u128_to_float2(unsigned long long hi, unsigned long long lo, float& c_hi, float& c_lo)
{
    int sh;
    unsigned long long top;
    if (hi == 0ull) {
        sh = (lo >> 63) ? 1 : 0;
        top = lo >> sh;
    } else {
        const int L = 127 - __clzll((long long)hi);   // leading bit, 64..127
        sh = L - 62;                                  // 2..65: the leading bit lands on bit 62
        top = (sh >= 64) ? (hi >> (sh - 64)) : ((hi << (64 - sh)) | (lo >> sh));
    }
    const float th = __ull2float_rn(top);                                    // <= 2^63, exact as an integer
    const long long rest = (long long)(top - (unsigned long long)th);        // |rest| < 2^39
    const float scale = __int_as_float((sh - 23 + 127) << 23);               // 2^(sh - 23), normal
    c_hi = __fmul_rn(th, scale);
    c_lo = __fmul_rn(__ll2float_rn(rest), scale);
}

// Many members share the top 24 key bits (ties, near-constant scores): the
// last 8 key bits by histogram, then the tie by index (radix levels on the
// index bits [20, 31), [9, 20), [0, 9) over the members equal to theta; bins
// are counted in reverse so that the largest-first search finds the smallest
// index); then the members outside the stratum add their terms.  Every level
// walks the unit's candidates again (rare: a slow path).
template <class Fetch>
__device__ __noinline__ void resolve_ties(const Params& p, int u, uint32_t pre24, uint32_t t3, uint32_t E, float m,
                                          SelShared& sh, Fetch& fetch, unsigned long long& ilo,
                                          unsigned long long& ihi, bool& bad, uint32_t& theta, int64_t& idx_cut)
{
    const int tid = threadIdx.x;
    uint32_t* status = ws_status(p);
    __syncthreads();
#pragma unroll 1
    for (int i = tid; i < 256; i += kSelThreads) sh.hist[i] = 0u;
    __syncthreads();
#pragma unroll 1
    for (uint32_t i = tid; i < E; i += kSelThreads) {
        const uint2 e = fetch(i);
        if ((e.x >> 8) == pre24) atomicAdd(&sh.hist[e.x & 0xffu], 1u);
    }
    __syncthreads();
    const Found f3 = find_rank_desc<kSelThreads, 256, false>(sh.hist, t3, sh.scan, sh.bcast, status);
    theta = (pre24 << 8) | f3.bin;
    uint32_t rt = t3 - f3.above;   // the rt-th smallest index among the ties at theta
    uint32_t prefix = 0;
    const int shifts[3] = {20, 9, 0};
    const uint32_t masks[3] = {0u, 0xfff00000u, 0xfffffe00u};
#pragma unroll 1
    for (int level = 0; level < 3; ++level) {
        const int shift = shifts[level];
        __syncthreads();
#pragma unroll 1
        for (int i = tid; i < 2048; i += kSelThreads) sh.hist[i] = 0u;
        __syncthreads();
#pragma unroll 1
        for (uint32_t i = tid; i < E; i += kSelThreads) {
            const uint2 e = fetch(i);
            if (e.x == theta && (e.y & masks[level]) == prefix)
                atomicAdd(&sh.hist[2047u - ((e.y >> shift) & 0x7ffu)], 1u);
        }
        __syncthreads();
        const Found fi = find_rank_desc<kSelThreads, 2048, false>(sh.hist, rt, sh.scan, sh.bcast, status);
        prefix |= (2047u - fi.bin) << shift;
        rt -= fi.above;
    }
    idx_cut = (p.top_k == 0) ? -1 : (int64_t)prefix;
    if (p.budget > 0.0f) {
#pragma unroll 1
        for (uint32_t i = tid; i < E; i += kSelThreads) {
            const uint2 e = fetch(i);
            const bool inT = e.x > theta || (e.x == theta && (int64_t)e.y <= idx_cut);
            if ((e.x >> 8) == pre24 && !inT) bad |= !iacc(ilo, ihi, expf(__fsub_rn(okey_value(e.x), m)));
        }
    }
    __syncthreads();
}

__device__ __noinline__ void resolve_unit(const Params& p, int u, int64_t nu, uint32_t f1, uint32_t above1,
                                         uint32_t target, float m, SelShared& sh, uint2* cs)
{
    const Plan& pl = p.pl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* status = ws_status(p);
    const bool want_z = p.budget > 0.0f && p.strata != 1;   // the uniform sampler's Z is n - k
    const TilePart* tp = reinterpret_cast<const TilePart*>(ws_zpart(p)) + (size_t)u * pl.tcap;
    // one wave of loads: the tiles' candidate counts and shares of Z (two
    // tiles per thread: at most kMaxTiles tiles) and the candidates' level-2
    // histogram (the next 12 key bits, counted by the tiles; 8 bins per
    // thread, top bin first)
    uint32_t cnt2[2];
    float tzh[2], tzl[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int t = 2 * tid + j;
        const bool ok = t < pl.ntile;
        cnt2[j] = ok ? __ldcg(&tp[t].ncand) : 0u;
        tzh[j] = ok ? __ldcg(&tp[t].zh) : 0.0f;
        tzl[j] = ok ? __ldcg(&tp[t].zl) : 0.0f;
    }
    const uint32_t* hist2 = ws_hist2(p) + (size_t)u * kBins;
    constexpr int CH = kBins / kSelThreads;
    uint32_t c[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) c[j] = __ldcg(hist2 + (kBins - 1 - (tid * CH + j)));
    if (tid == 0) sh.nbound = 0;
    uint32_t E;
    const uint32_t before = block_excl_scan<kSelThreads>(cnt2[0] + cnt2[1], sh.scan, E);
    if (2 * tid < pl.ntile) sh.coff[2 * tid] = before;
    if (2 * tid + 1 < pl.ntile) sh.coff[2 * tid + 1] = before + cnt2[0];
    if (tid == 0) sh.coff[pl.ntile] = E;
    // f2: the level-2 bin holding the k-th score
    const uint32_t t2 = target - above1;
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < CH; ++j) local += c[j];
    if (tid == 0) {
        sh.bcast[0] = 0;
        sh.bcast[1] = 0xffffffffu;
    }
    uint32_t tot2;
    const uint32_t excl = block_excl_scan<kSelThreads>(local, sh.scan, tot2);
    if (local > 0 && excl < t2 && t2 <= excl + local) {
        uint32_t cum = excl;
        bool done = false;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (!done && cum + c[j] >= t2) {
                sh.bcast[0] = (uint32_t)(kBins - 1 - (tid * CH + j));
                sh.bcast[1] = cum;
                done = true;
            }
            cum += c[j];
        }
    }
    __syncthreads();
    Found f2{sh.bcast[0], sh.bcast[1]};
    if (f2.above == 0xffffffffu || tot2 != E) {   // counts disagree: cannot happen
        if (tid == 0) flag(status, DEV_BAD_INDEX);
        f2.bin = 0;
        f2.above = 0;
    }
    const uint32_t pre24 = (f1 << 12) | f2.bin;
    const uint32_t t3 = t2 - f2.above;   // rank among the pre24 members (1-based)
    SSA_MARK(5);

    // one pass over the candidates: above pre24 -> in T; below -> in R, its
    // term summed exactly; equal -> the member list in shared memory.  The
    // candidates are staged in shared memory kResStage at a time, each warp
    // copying whole tile segments (cp.async).
    const uint2* cand = ws_cand(p) + (size_t)u * pl.N;
    auto fetch = [&](uint32_t i) -> uint2 {   // the i-th candidate in tile order (slow path)
        int lo_t = 0, hi_t = pl.ntile;          // coff[lo_t] <= i < coff[hi_t]
        while (hi_t - lo_t > 1) {
            const int mid = (lo_t + hi_t) >> 1;
            if (sh.coff[mid] <= i) lo_t = mid; else hi_t = mid;
        }
        return __ldcg(cand + (size_t)lo_t * pl.tt + (i - sh.coff[lo_t]));
    };
    unsigned long long ilo = 0ull, ihi = 0ull;
    bool bad = false;
#pragma unroll 1
    for (uint32_t r0 = 0; r0 < E; r0 += kResStage) {
        const uint32_t r1 = min(E, r0 + (uint32_t)kResStage);
        __syncthreads();   // the previous round is consumed
#pragma unroll 1
        for (int t = warp; t < pl.ntile; t += kSelWarps) {
            const uint32_t a = max(sh.coff[t], r0), e = min(sh.coff[t + 1], r1);
            const uint2* src = cand + (size_t)t * pl.tt + (a - sh.coff[t]);
#pragma unroll 1
            for (uint32_t i = lane; a + i < e; i += 32) cp_async_8(cs + (a - r0) + i, src + i);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
#pragma unroll 1
        for (uint32_t i = tid; i < r1 - r0; i += kSelThreads) {
            const uint2 v = cs[i];
            const uint32_t p24 = v.x >> 8;
            if (p24 < pre24) {
                if (want_z) bad |= !iacc(ilo, ihi, expf(__fsub_rn(okey_value(v.x), m)));
            } else if (p24 == pre24) {
                const uint32_t slot = atomicAdd(&sh.nbound, 1u);
                if (slot < 256u) sh.bound[slot] = v;
            }
        }
    }
    __syncthreads();
    SSA_MARK(6);
    const uint32_t nb = sh.nbound;
    uint32_t theta = 0;
    int64_t idx_cut = -1;
    if (nb <= 256u) {
        // rank every pre24 member exactly (key desc, index asc)
        if (tid == 0) {
            sh.bcast[4] = 0xffffffffu;
            sh.bcast[5] = 0;
        }
        __syncthreads();
        if ((uint32_t)tid < nb) {
            const uint2 me = sh.bound[tid];
            uint32_t ahead = 0;
#pragma unroll 1
            for (uint32_t i = 0; i < nb; ++i) {
                const uint2 o = sh.bound[i];
                ahead += (o.x > me.x || (o.x == me.x && o.y < me.y)) ? 1u : 0u;
            }
            if (ahead + 1 == t3) {
                sh.bcast[4] = me.x;
                sh.bcast[5] = me.y;
            }
        }
        __syncthreads();
        if (sh.bcast[4] == 0xffffffffu) {   // inconsistent counts: cannot happen
            if (tid == 0) flag(status, DEV_BAD_INDEX);
            sh.bcast[4] = pre24 << 8;
            sh.bcast[5] = 0;
        }
        theta = sh.bcast[4];
        idx_cut = (int64_t)sh.bcast[5];
        if (p.top_k == 0) idx_cut = -1;   // k = 0: empty stratum, the k-th score only fixes m
        // the members outside the stratum add their terms
        if (want_z && (uint32_t)tid < nb) {
            const uint2 me = sh.bound[tid];
            const bool inT = me.x > theta || (me.x == theta && (int64_t)me.y <= idx_cut);
            if (!inT) bad |= !iacc(ilo, ihi, expf(__fsub_rn(okey_value(me.x), m)));
        }
        __syncthreads();
    } else {
        resolve_ties(p, u, pre24, t3, E, m, sh, fetch, ilo, ihi, bad, theta, idx_cut);
    }
    if (bad) flag(status, DEV_NONFINITE);
    SSA_MARK(13);

    // normaliser: tile shares (compensated, fixed tree) + the exact sum of the
    // remainder candidates' terms
    float zh = 0.0f, zl = 0.0f;
    comp_add(zh, zl, tzh[0], tzl[0]);
    comp_add(zh, zl, tzh[1], tzl[1]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long l2 = __shfl_xor_sync(0xffffffffu, ilo, o);
        const unsigned long long h2 = __shfl_xor_sync(0xffffffffu, ihi, o);
        const unsigned long long nlo = ilo + l2;
        ihi += h2 + (nlo < ilo ? 1ull : 0ull);
        ilo = nlo;
        const float fh = __shfl_xor_sync(0xffffffffu, zh, o);
        const float fl = __shfl_xor_sync(0xffffffffu, zl, o);
        comp_add(zh, zl, fh, fl);
    }
    if (lane == 0) {
        sh.zw[warp][0] = zh;
        sh.zw[warp][1] = zl;
        sh.zi[warp][0] = ilo;
        sh.zi[warp][1] = ihi;
    }
    __syncthreads();
    if (warp == 0) {   // the warps' sums, a fixed tree over 16 lanes
        float hh = lane < kSelWarps ? sh.zw[lane][0] : 0.0f, ll = lane < kSelWarps ? sh.zw[lane][1] : 0.0f;
        unsigned long long slo = lane < kSelWarps ? sh.zi[lane][0] : 0ull, shi = lane < kSelWarps ? sh.zi[lane][1] : 0ull;
#pragma unroll
        for (int o = kSelWarps / 2; o > 0; o >>= 1) {
            const unsigned long long l2 = __shfl_xor_sync(0xffffffffu, slo, o);
            const unsigned long long h2 = __shfl_xor_sync(0xffffffffu, shi, o);
            const unsigned long long nlo = slo + l2;
            shi += h2 + (nlo < slo ? 1ull : 0ull);
            slo = nlo;
            const float fh = __shfl_xor_sync(0xffffffffu, hh, o);
            const float fl = __shfl_xor_sync(0xffffffffu, ll, o);
            comp_add(hh, ll, fh, fl);
        }
        if (lane != 0) return;
        float c_hi, c_lo;
        u128_to_float2(shi, slo, c_hi, c_lo);
        comp_add(hh, ll, c_hi, c_lo);
        sh.r_theta = theta;
        sh.r_cut = (int32_t)idx_cut;
        sh.r_m = m;
        sh.r_Z = (p.strata == 1) ? uniform_z(p, nu) : __fadd_rn(hh, ll);
    }
}

// ---------------------------------------------------------------------------
// The top-p stratum's size
// ---------------------------------------------------------------------------
// ("Stratified Sparse Attention speeds up decoding 2.96x on a 1M context",
// section "How SSA splits the cache into strata": top-p is a special case of
// the deterministic stratum.)  The stratum is the fewest tokens, taken in the
// top-k order (order key desc, index asc), whose share of sum_j exp(s_j) over
// all N tokens reaches top_p.  Its size is found by a mass-weighted radix
// select across the unit's tiles: every tile adds, per bin of the current
// radix level, its tokens' count and their terms w = expf(s - M) (M above
// every score, so w <= 1) as exact fixed point -- w * 2^63 truncated to an
// integer, split into two 32-bit halves summed in 64-bit words, so the sums
// are exact and independent of order -- to the unit's histogram; once every
// tile has arrived, each CTA finds the first bin from the top whose
// cumulative mass reaches the remaining target.  Three levels (12, 12 and 8
// key bits) leave the key of the crossing token; its ties have equal terms,
// so the number of them the stratum needs is a division.

struct MassPick {
    uint32_t bin;          // the crossing bin
    uint32_t count_above;  // tokens in higher bins
    uint32_t count_bin;    // tokens in the crossing bin
    double mass_above;     // mass of the higher bins
    double mass_bin;       // mass of the crossing bin
    double total;          // mass of every bin
};

// The bin, from the top of the unit's NB-bin mass histogram h ([3][NB]
// words: high part, low part, count), whose cumulative mass first reaches
// the target: `target` times the histogram's total when `frac` is set, else
// `target` itself (if rounding leaves it unreached, the lowest non-empty
// bin).  Block-wide (kSelThreads); every thread returns it.
template <int NB>
__device__ MassPick mass_pick(const unsigned long long* h, double target, bool frac, SelShared& sh)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int CH = NB >= kSelThreads ? NB / kSelThreads : 1;
    constexpr double kHiUnit = 1.0 / 2147483648.0;            // 2^-31: one unit of the high part
    constexpr double kLoUnit = kHiUnit / 4294967296.0;       // 2^-63
    double wm[CH];
    uint32_t wc[CH];
    double lm = 0.0;
    uint32_t lc = 0, deepest = 0;   // deepest: 1 + the lowest non-empty position of this thread (0: none)
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        const int pos = tid * CH + j;   // pos-th bin from the top
        wm[j] = 0.0;
        wc[j] = 0u;
        if (pos < NB) {
            const int bin = NB - 1 - pos;
            wm[j] = (double)__ldcg(h + bin) * kHiUnit + (double)__ldcg(h + NB + bin) * kLoUnit;
            wc[j] = (uint32_t)__ldcg(h + 2 * NB + bin);
            if (wc[j]) deepest = (uint32_t)pos + 1u;
        }
        lm += wm[j];
        lc += wc[j];
    }
    double xm = lm;
    uint32_t xc = lc, dmax = deepest;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double ym = __shfl_up_sync(0xffffffffu, xm, o);
        const uint32_t yc = __shfl_up_sync(0xffffffffu, xc, o);
        if (lane >= o) {
            xm += ym;
            xc += yc;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dmax = max(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
    if (lane == 31) {
        sh.dscan[warp] = xm;
        sh.scan[warp] = xc;
    }
    if (lane == 0) sh.wcnt[warp] = dmax;
    if (tid == 0) sh.pick_u[0] = 0xffffffffu;
    __syncthreads();
    double em = 0.0, total = 0.0;
    uint32_t ec = 0;
    dmax = 0;
    for (int w = 0; w < kSelWarps; ++w) {
        if (w < warp) {
            em += sh.dscan[w];
            ec += sh.scan[w];
        }
        total += sh.dscan[w];
        dmax = max(dmax, sh.wcnt[w]);
    }
    em += xm - lm;   // exclusive prefix of this thread's bins
    ec += xc - lc;
    const double tgt = frac ? target * total : target;
    if (lc > 0 && em < tgt && tgt <= em + lm) {
        double cum = em;
        uint32_t cc = ec;
        bool done = false;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (!done && wc[j] > 0 && cum + wm[j] >= tgt) {
                sh.pick_u[0] = (uint32_t)(NB - 1 - (tid * CH + j));
                sh.pick_u[1] = cc;
                sh.pick_u[2] = wc[j];
                sh.pick_m[0] = cum;
                sh.pick_m[1] = wm[j];
                done = true;
            }
            cum += wm[j];
            cc += wc[j];
        }
    }
    __syncthreads();
    if (sh.pick_u[0] == 0xffffffffu && dmax > 0 && (int)(dmax - 1) / CH == tid) {
        // unreached: the lowest non-empty bin (this thread holds it)
        const int pos = (int)dmax - 1, jl = pos % CH;
        double cum = em;
        uint32_t cc = ec;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (j == jl) {
                sh.pick_u[0] = (uint32_t)(NB - 1 - pos);
                sh.pick_u[1] = cc;
                sh.pick_u[2] = wc[j];
                sh.pick_m[0] = cum;
                sh.pick_m[1] = wm[j];
            }
            cum += wm[j];
            cc += wc[j];
        }
    }
    __syncthreads();
    MassPick r{sh.pick_u[0], sh.pick_u[1], sh.pick_u[2], sh.pick_m[0], sh.pick_m[1], total};
    if (r.bin == 0xffffffffu) r = MassPick{0u, 0u, 0u, 0.0, 0.0, total};   // no token at all
    __syncthreads();
    return r;
}

// One radix level of the top-p select over this tile: every token whose
// order key matches `prefix` in its bits from `hi_shift` up (every token when
// hi_shift is 32) adds its count and term to bin (key >> lo_shift) & (NB - 1)
// of the CTA's histogram in shared memory, which is then added to the unit's
// histogram h.  Shared memory: NB * 20 bytes of histogram, then 16 warps'
// 256-score staging (16 KB).
template <int NB>
__device__ void mass_level(const Params& p, int u, int tile, int64_t nu, float M, uint32_t prefix, int hi_shift,
                           int lo_shift, unsigned long long* h, unsigned char* smem)
{
    const Plan& pl = p.pl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long* sA = reinterpret_cast<unsigned long long*>(smem);
    unsigned long long* sB = sA + NB;
    uint32_t* sC = reinterpret_cast<uint32_t*>(sB + NB);
    float* stg = reinterpret_cast<float*>(smem + 80 * 1024) + warp * 256;
    for (int i = tid; i < NB; i += kSelThreads) {
        sA[i] = 0ull;
        sB[i] = 0ull;
        sC[i] = 0u;
    }
    __syncthreads();
    const int W2 = pl.tt / kSelWarps;
    const int64_t base = (int64_t)tile * pl.tt + (int64_t)warp * W2;
    const float* S = p.s_src + (int64_t)u * pl.N;
#pragma unroll 1
    for (int c0 = 0; c0 < W2; c0 += 256) {
        const int n = min(256, W2 - c0);
        __syncwarp();
#pragma unroll 1
        for (int i = lane; i < n; i += 32) cp_async_4(stg + i, S + min(base + c0 + i, pl.N - 1));
        cp_async_commit();
        cp_async_wait<0>();
        __syncwarp();
#pragma unroll 1
        for (int i = lane; i < n; i += 32) {
            if (base + c0 + i >= nu) continue;
            const float sv = stg[i];
            const uint32_t k = okey(sv);
            if (hi_shift < 32 && (k >> hi_shift) != prefix) continue;
            const uint32_t bin = (k >> lo_shift) & (uint32_t)(NB - 1);
            const float w = expf(__fsub_rn(sv, M));
            const unsigned long long v = __float2ull_rz(w * 9223372036854775808.0f);   // w * 2^63, w <= 1
            atomicAdd(&sA[bin], v >> 32);
            atomicAdd(&sB[bin], v & 0xffffffffull);
            atomicAdd(&sC[bin], 1u);
        }
    }
    __syncthreads();
    for (int i = tid; i < NB; i += kSelThreads) {
        if (sC[i]) {
            atomicAdd(h + i, sA[i]);
            atomicAdd(h + NB + i, sB[i]);
            atomicAdd(h + 2 * NB + i, (unsigned long long)sC[i]);
        }
    }
}

// All tiles of unit u have added their level to the unit's histogram.
__device__ __forceinline__ void mass_level_arrive(const Params& p, int u, int level)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        UnitCtrl* ctrl = ws_ctrl(p) + u;
        __threadfence();
        atomicAdd(&ctrl->tp_arrive[level], 1u);
        if (!wait_geq_bounded(&ctrl->tp_arrive[level], (uint32_t)p.pl.ntile)) flag(ws_status(p), DEV_TIMEOUT);
    }
    __syncthreads();
}

// The size of unit u's top-p stratum over its nu tokens (every CTA of the
// unit returns the same value, at least 1).  Block-wide; uses the first 96 KB
// of `smem`.
__device__ __noinline__ uint32_t topp_size(const Params& p, int u, int tile, int64_t nu, SelShared& sh,
                                           unsigned char* smem)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long* h0 = ws_topp(p) + (size_t)u * kTopPBins * 3;
    unsigned long long* h1 = h0 + (size_t)4096 * 3;
    unsigned long long* h2 = h1 + (size_t)4096 * 3;
    // M: the lower edge of the bucket above the highest non-empty bucket of
    // the unit's count histogram (above every score, so every term is <= 1)
    const uint32_t* hist1 = ws_hist1(p) + (size_t)u * kBins;
    uint32_t top = 0;
    for (int i = tid; i < kBins; i += kSelThreads)
        if (__ldcg(hist1 + i)) top = max(top, (uint32_t)i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) top = max(top, __shfl_xor_sync(0xffffffffu, top, o));
    if (lane == 0) sh.scan[warp] = top;
    __syncthreads();
    for (int w = 0; w < kSelWarps; ++w) top = max(top, sh.scan[w]);
    __syncthreads();
    float M = okey_value(min(top + 1u, (uint32_t)(kBins - 1)) << 20);
    if (!isfinite(M)) {   // scores at the top of the binary32 range: no margin above them
        if (tid == 0) flag(ws_status(p), DEV_NONFINITE);
        M = 3.4028234663852886e38f;
    }
    // level 0: the 12-bit order-key buckets
    mass_level<4096>(p, u, tile, nu, M, 0u, 32, 20, h0, smem);
    mass_level_arrive(p, u, 0);
    const MassPick a = mass_pick<4096>(h0, (double)p.top_p, true, sh);
    const double t1 = (double)p.top_p * a.total - a.mass_above;   // the target left inside bucket a
    // level 1: the next 12 bits of bucket a's members
    mass_level<4096>(p, u, tile, nu, M, a.bin, 20, 8, h1, smem);
    mass_level_arrive(p, u, 1);
    const MassPick b = mass_pick<4096>(h1, t1, false, sh);
    const double t2 = t1 - b.mass_above;
    // level 2: the last 8 bits of the members sharing those 24 bits
    mass_level<256>(p, u, tile, nu, M, (a.bin << 12) | b.bin, 8, 0, h2, smem);
    mass_level_arrive(p, u, 2);
    const MassPick c = mass_pick<256>(h2, t2, false, sh);
    // the crossing key's ties have equal terms: the stratum takes the fewest
    // of them (in index order) whose mass reaches what is left
    uint32_t r = 1;
    if (c.count_bin > 0 && c.mass_bin > 0.0) {
        const double w = c.mass_bin / (double)c.count_bin, rem = t2 - c.mass_above;
        double need = floor(rem / w);
        if (need * w < rem) need += 1.0;   // the fewest ties whose mass reaches what is left
        r = (uint32_t)fmin(fmax(need, 1.0), (double)c.count_bin);
    }
    return a.count_above + b.count_above + c.count_above + r;
}

// ---------------------------------------------------------------------------
// The selection pass of one (unit, tile): block-wide, kSelThreads threads.
// ---------------------------------------------------------------------------

// What the pass leaves for the resolve (rank 0): the bucket of the k-th
// score, the number of tokens above it, the rank sought and the reference
// point m.
struct TileSel {
    uint32_t f1, above1, target;
    float m;
};

// Dynamic shared memory the pass stages its warps' chunks in (scores and
// Philox prefixes); the resolve stages candidates in the same bytes.
constexpr uint32_t kSelStageBytes = (uint32_t)kSelWarps * kSlice * 2u * 6u;

__device__ __noinline__ TileSel tile_pass(const Params& p, int u, int tile, int64_t nu, uint32_t k_unit,
                                          SelShared& sh, unsigned char* k2dyn)
{
    const Plan& pl = p.pl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W2 = pl.tt / kSelWarps;
    uint32_t* status = ws_status(p);
    SSA_MARK(2);

    const int64_t base = (int64_t)tile * pl.tt + (int64_t)warp * W2;   // this warp's first token
    // the part of the slice inside the unit's nu tokens (chunks past it are not walked)
    const int Wv = (int)max((int64_t)0, min((int64_t)W2, nu - base));
    const float* S = p.s_src + (int64_t)u * pl.N;
    const uint16_t* ub = ws_ubuf(p) + (size_t)u * pl.np + base;
    const float B = p.budget;
    const bool sampling = B > 0.0f;
    const bool uniform = p.strata == 1;   // every remainder token has the same p: e = 1, Z = n - k
    // Each warp stages its slice kSlice tokens at a time (scores and Philox
    // prefixes, cp.async) into two buffers: the next chunk's copies are in
    // flight while the current one is walked.  The first chunk's copies go
    // out before the histogram search.  Loops are kept rolled: the code runs
    // once per launch, so its size, not its instruction count, sets its time.
    float* ssc = reinterpret_cast<float*>(k2dyn) + warp * 2 * kSlice;
    uint16_t* su = reinterpret_cast<uint16_t*>(k2dyn + kSelWarps * kSlice * 2 * 4) + warp * 2 * kSlice;
    // whole 16-byte score copies when the unit's row and the warp's slice allow
    const bool s16 = ((uint64_t)u * (uint64_t)pl.N) % 4 == 0 && base + W2 <= pl.N;
    auto stage = [&](int c0) {
        const int n = min(kSlice, W2 - c0);
        float* dsc = ssc + ((c0 / kSlice) & 1) * kSlice;
        uint16_t* dsu = su + ((c0 / kSlice) & 1) * kSlice;
        if (s16) {
#pragma unroll 1
            for (int i = lane * 4; i < n; i += 128) cp_async_16(dsc + i, S + base + c0 + i);
        } else {
#pragma unroll 1
            for (int i = lane; i < n; i += 32) cp_async_4(dsc + i, S + min(base + c0 + i, pl.N - 1));
        }
        if (sampling) {
#pragma unroll 1
            for (int i = lane * 8; i < n; i += 256) cp_async_16(dsu + i, ub + c0 + i);
        }
        cp_async_commit();
    };
    if (Wv > 0) stage(0);

    // bucket f1 of the k-th score (the largest when k = 0): each thread reads
    // 8 bins of the unit's histogram, top bin first
    const uint32_t target = k_unit > 0 ? k_unit : 1u;
    const uint32_t* hist1 = ws_hist1(p) + (size_t)u * kBins;
    constexpr int CH = kBins / kSelThreads;
    uint32_t c[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) c[j] = __ldcg(hist1 + (kBins - 1 - (tid * CH + j)));
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < CH; ++j) local += c[j];
    if (tid == 0) {
        sh.bcast[0] = 0;
        sh.bcast[1] = 0xffffffffu;
        sh.ncand_cta = 0;
    }
    uint32_t total;
    const uint32_t excl = block_excl_scan<kSelThreads>(local, sh.scan, total);
    if (local > 0 && excl < target && target <= excl + local) {
        uint32_t cum = excl;
        bool done = false;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (!done && cum + c[j] >= target) {
                sh.bcast[0] = (uint32_t)(kBins - 1 - (tid * CH + j));
                sh.bcast[1] = cum;
                done = true;
            }
            cum += c[j];
        }
    }
    __syncthreads();
    Found f1{sh.bcast[0], sh.bcast[1]};
    if (f1.above == 0xffffffffu) {   // fewer than k tokens counted: inconsistent inputs
        if (tid == 0) flag(status, DEV_BAD_INDEX);
        f1.bin = 0;
        f1.above = 0;
    }
    const float m = okey_value(f1.bin << 20);
    SSA_MARK(16);

    // Z_lb from the same bins: every term of bucket c < f1 is at least
    // expf(fl32(floor_c - m)); 0.999 covers the rounding
    float zlb = 0.0f;
    if (sampling) {
        float part = 0.0f;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const uint32_t cb = (uint32_t)(kBins - 1 - (tid * CH + j));
            const float fl = okey_value(cb << 20);
            if (cb < f1.bin && c[j] && isfinite(fl)) part = fmaf((float)c[j], expf(__fsub_rn(fl, m)), part);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) sh.zlb[warp] = part;
        __syncthreads();
        for (int w = 0; w < kSelWarps; ++w) zlb += sh.zlb[w];
        zlb *= 0.999f;
    }
    if (uniform) zlb = uniform_z(p, nu);   // the exact normaliser
    // u >= prefix * 2^-16 >= B e / Z_lb >= p (any Z >= Z_lb): the token cannot be drawn
    const float bound_scale = (zlb > 0.0f) ? __fdiv_ru(B, zlb) : INFINITY;
    SSA_MARK(17);

    int32_t* sidx = ws_sel_idx(p) + (size_t)u * pl.np + base;
    float* sval = ws_sel_p(p) + (size_t)u * pl.np + base;
    // the tile's candidates go to its own segment of the unit's candidate
    // array (their order is free: the resolve ranks and sums exactly)
    uint2* cseg = ws_cand(p) + (size_t)u * pl.N + (size_t)tile * pl.tt;
    uint32_t* hist2 = ws_hist2(p) + (size_t)u * kBins;   // level-2 histogram of the unit's candidates
    uint32_t cnt = 0;
    float zh4[4] = {0.0f, 0.0f, 0.0f, 0.0f}, zl4[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // four (hi, lo) Z accumulators
    // the prefix test in units of 2^-16: prefix < B e / Z_lb * 2^16 (a power-of-two scale, exact)
    const float bound16 = __fmul_rn(bound_scale, 65536.0f);
#pragma unroll 1
    for (int c0 = 0; c0 < Wv; c0 += kSlice) {
        // the next chunk's copies go out before this one is walked
        if (c0 / kSlice < 4) SSA_MARKG(16 + c0 / kSlice);
        if (c0 + kSlice < Wv) {
            __syncwarp();
            stage(c0 + kSlice);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        const float* csc = ssc + ((c0 / kSlice) & 1) * kSlice;
        const uint16_t* csu = su + ((c0 / kSlice) & 1) * kSlice;
        const int n = min(kSlice, W2 - c0);   // a multiple of 32
        // tokens [0, nvalid) of the chunk are in the cache (the unit's tail past nu is not)
        const int nvalid = (int)min((int64_t)n, nu - (base + c0));
        const uint32_t t0 = (uint32_t)(base + c0);   // token indices fit 31 bits
        // each lane takes four consecutive tokens of a 128-token group; the
        // group's kept tokens are listed in index order at the warp's
        // running count plus the lane's exclusive prefix
#pragma unroll 1
        for (int g0 = 0; g0 < n; g0 += 128) {
            if ((c0 + g0) / 128 < 16) SSA_MARKG((c0 + g0) / 128);
            const int i0 = g0 + 4 * lane;
            float sv[4];
            uint32_t pr[4] = {0u, 0u, 0u, 0u};
            if (i0 < n) {
                const float4 v = *reinterpret_cast<const float4*>(csc + i0);
                sv[0] = v.x; sv[1] = v.y; sv[2] = v.z; sv[3] = v.w;
                if (sampling) {
                    const uint2 w = *reinterpret_cast<const uint2*>(csu + i0);
                    pr[0] = w.x & 0xffffu; pr[1] = w.x >> 16; pr[2] = w.y & 0xffffu; pr[3] = w.y >> 16;
                }
            } else {
                sv[0] = sv[1] = sv[2] = sv[3] = 0.0f;
            }
            // the four tokens are classified without branches (their chains
            // interleave); the rare candidates are written after the loop
            uint32_t kbits = 0;
            float val[4];
            uint32_t kq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool valid = i0 + q < nvalid;
                const uint32_t k = okey(sv[q]);
                const uint32_t b1 = k >> 20;
                const bool above = valid && b1 > f1.bin;
                const bool is_cand = valid && b1 == f1.bin;
                const bool below = sampling && valid && b1 < f1.bin;
                const float e = uniform ? 1.0f : expf(__fsub_rn(sv[q], m));
                if (!uniform) zacc(zh4[q], zl4[q], below ? e : 0.0f);
                const bool drawn = below && __fmul_ru(e, bound16) > __uint2float_rn(pr[q]);
                val[q] = above ? INFINITY : (below ? e : sv[q]);
                kbits |= ((uint32_t)(above || is_cand || drawn) << q) | ((uint32_t)is_cand << (4 + q));
                kq[q] = k;
            }
            if (kbits & 0xf0u) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (kbits & (0x10u << q)) {   // a candidate: flagged in the list
                        cseg[atomicAdd(&sh.ncand_cta, 1u)] = make_uint2(kq[q], t0 + (uint32_t)(i0 + q));
                        atomicAdd(hist2 + ((kq[q] >> 8) & 0xfffu), 1u);
                    }
                }
            }
            // the lane's first list slot: the warp's count so far plus the kept
            // tokens of the lower lanes, from one ballot per token position
            const uint32_t lt = lanemask_lt();
            uint32_t o = cnt, nkw = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t bq = __ballot_sync(0xffffffffu, (kbits >> q) & 1u);
                o += (uint32_t)__popc(bq & lt);
                nkw += (uint32_t)__popc(bq);
            }
            if (kbits & 0xfu) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (kbits & (1u << q)) {
                        const uint32_t t = t0 + (uint32_t)(i0 + q);
                        sidx[o] = (int32_t)(t | ((kbits & (0x10u << q)) ? kCandFlag : 0u));
                        sval[o] = val[q];
                        ++o;
                    }
                }
            }
            cnt += nkw;
        }
    }
    SSA_MARK(18);
    float zh = zh4[0], zl = zl4[0];
    comp_add(zh, zl, zh4[1], zl4[1]);
    comp_add(zh, zl, zh4[2], zl4[2]);
    comp_add(zh, zl, zh4[3], zl4[3]);
    if (lane == 0) sh.wcnt[warp] = cnt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, zh, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, zl, o);
        comp_add(zh, zl, h2, l2);
    }
    if (lane == 0) {
        sh.zw[warp][0] = zh;
        sh.zw[warp][1] = zl;
    }
    __syncthreads();   // the CTA's list and candidate writes; the caller's fence covers them (cumulative)
    SSA_MARK(19);
    if (warp == 0) {   // the warps' shares, a fixed tree over 16 lanes
        float hh = lane < kSelWarps ? sh.zw[lane][0] : 0.0f, ll = lane < kSelWarps ? sh.zw[lane][1] : 0.0f;
#pragma unroll
        for (int o = kSelWarps / 2; o > 0; o >>= 1) {
            const float fh = __shfl_xor_sync(0xffffffffu, hh, o);
            const float fl = __shfl_xor_sync(0xffffffffu, ll, o);
            comp_add(hh, ll, fh, fl);
        }
        if (lane == 0) {
            TilePart tpo;
            tpo.zh = hh;
            tpo.zl = ll;
            tpo.ncand = sh.ncand_cta;
            tpo.pad = 0;
            reinterpret_cast<TilePart*>(ws_zpart(p))[(size_t)u * pl.tcap + tile] = tpo;
        }
    }
    return TileSel{f1.bin, f1.above, target, m};
}

}  // namespace ssa
