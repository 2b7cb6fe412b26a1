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
// One CTA of 512 threads per (unit, tile); each warp owns a 512-token slice
// of the tile and walks it in index order:
//   * a token above bucket f is in T: it joins the slice's list (p = 1);
//   * a token of bucket f is a candidate: it joins the slice's list (with
//     its score) and the unit's candidate array (for the exact k-th);
//   * a token below bucket f is in R: its term e joins the tile's share of
//     Z (compensated sum, fixed order), and it joins the slice's list only
//     if it could be drawn at all: p <= B e / Z_lb for a lower bound Z_lb
//     of Z read off the histogram (every term of bucket c is at least
//     exp(floor_c - m)), so u >= B e / Z_lb rules it out for good.
// The last tile of a unit to finish (a counter in the unit's control block)
// resolves the exact k-th token among the candidates -- in shared memory:
// a 12-bit histogram, then the few members sharing 24 key bits ranked
// exactly (key desc, index asc) -- and completes Z: the tiles' shares in
// tile order plus the remainder candidates' terms, summed exactly as 128-bit
// integers (every such term is an fp32 value of at least one; terms of
// 2^81 and more, i.e. scores more than 450 apart from m, are flagged as
// out of range).  The
// attention kernel makes the final decision for every listed token.
#pragma once
#include "k_score.cuh"

namespace ssa {

constexpr int kBatch = 16;            // strips loaded per thread before use
constexpr int kCandSmem = 8192;       // candidates the resolve stages in shared memory
constexpr uint32_t kCandFlag = 0x80000000u;   // list entry: a candidate (its value is the score)

struct SelShared {
    uint32_t scan[kSelWarps];
    uint32_t bcast[8];
    float zw[kSelWarps][2];
    float zlb[kSelWarps];
    uint32_t is_last;
    uint32_t ncand_cta, cand_base;
    // resolve
    uint32_t hist[kBins];
    uint32_t nbound;
    uint2 bound[256];
    unsigned long long zi[kSelWarps][2];
};

// Dynamic shared memory of K2: the resolve's candidate staging.
inline uint32_t k2_smem_bytes() { return (uint32_t)kCandSmem * 8u; }

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

__device__ void resolve_unit(const Params& p, int u, uint32_t f1, uint32_t above1, uint32_t target, float m,
                             SelShared& sh, uint2* cs)
{
    const Plan& pl = p.pl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* status = ws_status(p);
    const bool want_z = p.budget > 0.0f;
    UnitCtrl* ctrl = ws_ctrl(p) + u;
    const uint32_t E = __ldcg(&ctrl->ncand);
    const uint2* cand = ws_cand(p) + (size_t)u * pl.N;
    const bool staged = E <= (uint32_t)kCandSmem;
    auto entry = [&](uint32_t i) -> uint2 { return staged ? cs[i] : __ldcg(cand + i); };
    if (staged) {
        for (uint32_t i0 = 0; i0 < E; i0 += kSelThreads * 4) {
            uint2 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t i = i0 + j * kSelThreads + tid;
                v[j] = (i < E) ? __ldcg(cand + i) : make_uint2(0u, 0u);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t i = i0 + j * kSelThreads + tid;
                if (i < E) cs[i] = v[j];
            }
        }
    }
    for (int i = tid; i < kBins; i += kSelThreads) sh.hist[i] = 0u;
    if (tid == 0) sh.nbound = 0;
    __syncthreads();
    // level 2: the next 12 key bits of the bucket's members
    for (uint32_t i = tid; i < E; i += kSelThreads) atomicAdd(&sh.hist[(entry(i).x >> 8) & 0xfffu], 1u);
    __syncthreads();
    const Found f2 = find_rank_desc<kSelThreads, kBins, false>(sh.hist, target - above1, sh.scan, sh.bcast, status);
    const uint32_t pre24 = (f1 << 12) | f2.bin;
    const uint32_t t3 = target - above1 - f2.above;   // rank among the pre24 members (1-based)
    for (uint32_t i = tid; i < E; i += kSelThreads) {
        const uint2 e = entry(i);
        if ((e.x >> 8) == pre24) {
            const uint32_t slot = atomicAdd(&sh.nbound, 1u);
            if (slot < 256u) sh.bound[slot] = e;
        }
    }
    __syncthreads();
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
        __syncthreads();
    } else {
        // many members share the top 24 bits (ties, near-constant scores): the
        // last 8 key bits by histogram, then the tie by index (radix levels on
        // the index bits [20, 31), [9, 20), [0, 9) over the members equal to
        // theta; bins are counted in reverse so that the largest-first search
        // finds the smallest index)
        __syncthreads();
        for (int i = tid; i < 256; i += kSelThreads) sh.hist[i] = 0u;
        __syncthreads();
        for (uint32_t i = tid; i < E; i += kSelThreads) {
            const uint2 e = entry(i);
            if ((e.x >> 8) == pre24) atomicAdd(&sh.hist[e.x & 0xffu], 1u);
        }
        __syncthreads();
        const Found f3 = find_rank_desc<kSelThreads, 256, false>(sh.hist, t3, sh.scan, sh.bcast, status);
        theta = (pre24 << 8) | f3.bin;
        uint32_t rt = t3 - f3.above;   // the rt-th smallest index among the ties at theta
        uint32_t prefix = 0;
        const int shifts[3] = {20, 9, 0};
        const uint32_t masks[3] = {0u, 0xfff00000u, 0xfffffe00u};
#pragma unroll
        for (int level = 0; level < 3; ++level) {
            const int shift = shifts[level];
            __syncthreads();
            for (int i = tid; i < 2048; i += kSelThreads) sh.hist[i] = 0u;
            __syncthreads();
            for (uint32_t i = tid; i < E; i += kSelThreads) {
                const uint2 e = entry(i);
                if (e.x == theta && (e.y & masks[level]) == prefix)
                    atomicAdd(&sh.hist[2047u - ((e.y >> shift) & 0x7ffu)], 1u);
            }
            __syncthreads();
            const Found fi = find_rank_desc<kSelThreads, 2048, false>(sh.hist, rt, sh.scan, sh.bcast, status);
            prefix |= (2047u - fi.bin) << shift;
            rt -= fi.above;
        }
        idx_cut = (int64_t)prefix;
    }
    if (p.top_k == 0) idx_cut = -1;   // k = 0: empty stratum, the k-th score only fixes m

    // normaliser: tile shares (tile order, compensated) + remainder candidates (exact)
    float zh = 0.0f, zl = 0.0f;
    {
        const float2* zp = ws_zpart(p) + (size_t)u * pl.ntile;
        for (int t0 = 0; t0 < pl.ntile; t0 += kSelThreads * 4) {
            float2 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = t0 + j * kSelThreads + tid;
                v[j] = (t < pl.ntile) ? __ldcg(zp + t) : make_float2(0.0f, 0.0f);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) comp_add(zh, zl, v[j].x, v[j].y);
        }
    }
    unsigned long long ilo = 0ull, ihi = 0ull;
    if (want_z) {
        for (uint32_t i = tid; i < E; i += kSelThreads) {
            const uint2 e = entry(i);
            const bool inT = e.x > theta || (e.x == theta && (int64_t)e.y <= idx_cut);
            if (!inT && !iacc(ilo, ihi, expf(__fsub_rn(okey_value(e.x), m)))) flag(status, DEV_NONFINITE);
        }
    }
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
    if (tid == 0) {
        float hh = 0.0f, ll = 0.0f;
        unsigned long long slo = 0ull, shi = 0ull;
        for (int w = 0; w < kSelWarps; ++w) {
            comp_add(hh, ll, sh.zw[w][0], sh.zw[w][1]);
            const unsigned long long nlo = slo + sh.zi[w][0];
            shi += sh.zi[w][1] + (nlo < slo ? 1ull : 0ull);
            slo = nlo;
        }
        // the integer sum (units of 2^-23) as a double, then as two floats
        const double d = __ull2double_rn(shi) * 2199023255552.0 + __ull2double_rn(slo) * 1.1920928955078125e-07;
        const float c_hi = __double2float_rn(d);
        const float c_lo = __double2float_rn(d - (double)c_hi);
        comp_add(hh, ll, c_hi, c_lo);
        ctrl->theta = theta;
        ctrl->idx_cut = (int32_t)idx_cut;
        ctrl->m = m;
        ctrl->Z = __fadd_rn(hh, ll);
    }
}

// ---------------------------------------------------------------------------
// K2: per (unit, tile)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads, 2) bucket_kernel(const __grid_constant__ Params p)
{
    extern __shared__ uint2 cstage[];
    __shared__ SelShared sh;
    const Plan& pl = p.pl;
    const int u = blockIdx.x / pl.ntile, tile = blockIdx.x % pl.ntile;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W2 = pl.tt / kSelWarps;
    const int b = u / p.Hkv, h = u % p.Hkv;
    uint32_t* status = ws_status(p);
    grid_dep_wait();
    SSA_MARK(2);

    const uint32_t target = (uint32_t)(p.top_k > 0 ? p.top_k : 1);
    const uint32_t* hist1 = ws_hist1(p) + (size_t)u * kBins;
    const Found f1 = find_rank_desc<kSelThreads, kBins, true>(hist1, target, sh.scan, sh.bcast, status);
    const float m = okey_value(f1.bin << 20);
    const float B = p.budget;
    const bool sampling = B > 0.0f;

    // Z_lb: every term of bucket c < f1 is at least expf(fl32(floor_c - m)); 0.999 covers rounding
    float zlb = 0.0f;
    if (sampling) {
        constexpr int CH = kBins / kSelThreads;
        float part = 0.0f;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const uint32_t c = (uint32_t)(tid * CH + j);
            if (c < f1.bin) {
                const uint32_t n = __ldcg(hist1 + c);
                const float fl = okey_value(c << 20);
                if (n && isfinite(fl)) part = fmaf((float)n, expf(__fsub_rn(fl, m)), part);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) sh.zlb[warp] = part;
        __syncthreads();
        for (int w = 0; w < kSelWarps; ++w) zlb += sh.zlb[w];
        zlb *= 0.999f;
    }
    // u >= B e / Z_lb implies u >= p for any Z >= Z_lb: the token cannot be drawn
    const float bound_scale = (zlb > 0.0f) ? __fdiv_ru(B, zlb) : INFINITY;

    const int64_t base = (int64_t)tile * pl.tt + (int64_t)warp * W2;   // this warp's first token
    const float* S = p.s_src + (int64_t)u * pl.N;
    const uint8_t* ub = ws_ubuf(p) + (size_t)u * pl.np;
    int32_t* sidx = ws_sel_idx(p) + (size_t)u * pl.np + base;
    float* sval = ws_sel_p(p) + (size_t)u * pl.np + base;
    uint2* cand = ws_cand(p) + (size_t)u * pl.N;
    UnitCtrl* ctrl = ws_ctrl(p) + u;
    if (tid == 0) sh.ncand_cta = 0;
    __syncthreads();
    uint32_t cnt = 0;
    float zh = 0.0f, zl = 0.0f;
    for (int st0 = 0; st0 < W2; st0 += 32 * kBatch) {
        float sv[kBatch];
        uint32_t u8v[kBatch / 4];   // four Philox bytes per word
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int64_t t = base + st0 + j * 32 + lane;
            sv[j] = (st0 + j * 32 < W2 && t < pl.N) ? __ldcg(S + t) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kBatch / 4; ++j) u8v[j] = 0u;
        if (sampling) {
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int64_t t = base + st0 + j * 32 + lane;
                if (st0 + j * 32 < W2 && t < pl.N) u8v[j >> 2] |= (uint32_t)__ldcg(ub + t) << (8 * (j & 3));
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (st0 + j * 32 >= W2) break;   // uniform across the warp
            const int64_t t = base + st0 + j * 32 + lane;
            const bool valid = t < pl.N;
            const uint32_t k = okey(sv[j]);
            const uint32_t b1 = k >> 20;
            const bool above = valid && b1 > f1.bin;
            const bool is_cand = valid && b1 == f1.bin;
            bool keep = above || is_cand;
            float val = above ? INFINITY : sv[j];
            if (valid && b1 < f1.bin && sampling) {
                const float e = expf(__fsub_rn(sv[j], m));
                zacc(zh, zl, e);
                const float pmax = __fmul_ru(e, bound_scale);
                const uint32_t v8 = (u8v[j >> 2] >> (8 * (j & 3))) & 0xffu;
                if (pmax > (float)v8 * 0.00390625f) keep = token_uniform(p.seed, t, h, b) < pmax;
                val = e;
            }
            const uint32_t km = __ballot_sync(0xffffffffu, keep);
            if (keep) {
                const uint32_t o = cnt + __popc(km & lanemask_lt());
                sidx[o] = (int32_t)((uint32_t)t | (is_cand ? kCandFlag : 0u));
                sval[o] = val;
            }
            cnt += __popc(km);
            const uint32_t cm = __ballot_sync(0xffffffffu, is_cand);
            if (cm) {   // candidates gather in shared memory first (one global reservation per CTA)
                uint32_t slot0 = 0;
                if (lane == __ffs(cm) - 1) slot0 = atomicAdd(&sh.ncand_cta, (uint32_t)__popc(cm));
                slot0 = __shfl_sync(0xffffffffu, slot0, __ffs(cm) - 1);
                const uint32_t slot = slot0 + __popc(cm & lanemask_lt());
                if (is_cand && slot < (uint32_t)kCandSmem) cstage[slot] = make_uint2(k, (uint32_t)t);
            }
        }
    }
    if (lane == 0) ws_scount(p)[((size_t)u * pl.ntile + tile) * kSelWarps + warp] = cnt;
    __syncthreads();
    {
        // reserve the tile's share of the unit's candidate array and copy it out
        // (the array's order is free: the resolve ranks exactly and sums exactly)
        const uint32_t nc = sh.ncand_cta;
        if (tid == 0) sh.cand_base = nc ? atomicAdd(&ctrl->ncand, nc) : 0u;
        __syncthreads();
        const uint32_t cb = sh.cand_base;
        if (nc <= (uint32_t)kCandSmem) {
            for (uint32_t i = tid; i < nc; i += kSelThreads) cand[cb + i] = cstage[i];
        } else {   // too many for the staging: walk the tile again and write them all
            if (tid == 0) sh.ncand_cta = 0;
            __syncthreads();
            for (int st0 = 0; st0 < W2; st0 += 32) {
                const int64_t t = base + st0 + lane;
                const bool valid = t < pl.N;
                const uint32_t k = valid ? okey(__ldcg(S + t)) : 0u;
                const bool is_cand = valid && (k >> 20) == f1.bin;
                const uint32_t cm = __ballot_sync(0xffffffffu, is_cand);
                if (cm) {
                    uint32_t slot0 = 0;
                    if (lane == __ffs(cm) - 1) slot0 = atomicAdd(&sh.ncand_cta, (uint32_t)__popc(cm));
                    slot0 = __shfl_sync(0xffffffffu, slot0, __ffs(cm) - 1);
                    const uint32_t slot = slot0 + __popc(cm & lanemask_lt());
                    if (is_cand) cand[cb + slot] = make_uint2(k, (uint32_t)t);
                }
            }
        }
        __syncthreads();
    }
    SSA_MARK(10);
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
    __syncthreads();
    if (tid == 0) {
        float hh = 0.0f, ll = 0.0f;
        for (int w = 0; w < kSelWarps; ++w) comp_add(hh, ll, sh.zw[w][0], sh.zw[w][1]);
        ws_zpart(p)[(size_t)u * pl.ntile + tile] = make_float2(hh, ll);
        __threadfence();
        const uint32_t prev = atomicAdd(&ctrl->k2a_done, 1u);
        sh.is_last = (prev == (uint32_t)(pl.ntile - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (sh.is_last) {
        __threadfence();
        SSA_MARK(3);
        resolve_unit(p, u, f1.bin, f1.above, target, m, sh, cstage);
        SSA_MARK(4);
    }
    grid_dep_launch();
}

}  // namespace ssa
