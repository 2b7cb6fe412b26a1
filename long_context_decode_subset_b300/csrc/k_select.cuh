// k_select.cuh -- K2a (threshold bucket, candidates, normaliser) and K2c
// (decisions): the stratified selection of "Stratified Sparse Attention
// speeds up decoding 2.96x on a 1M context", section "How SSA splits the
// cache into strata".
//
//   T  = the k tokens with the highest scores under the order (order key
//        desc, index asc), read deterministically;
//   R  = every other token j, kept independently with probability
//        p_j = min(1, fl32(fl32(B * e_j) / Z)),  e_j = fl32(expf(fl32(s_j - m))),
//        Z = sum over R of e_j (rounded once to fp32),
//        decided by u_j < p_j with u_j = (x0 >> 8) * 2^-24, x0 = word 0 of
//        Philox4x32-10(key = seed, counter = (j, h_kv, b, 0)).
//   p is independent of m; m is the lower edge of the 12-bit order-key
//   bucket that holds the k-th score (the largest when k = 0), so every
//   term is at most exp(|s_(k)| / 8) and Z can be summed in the same pass
//   that finds that bucket's members.
//
// Both kernels run one CTA of 512 threads per (unit, tile); each warp owns a
// contiguous slice of the tile and writes its candidates / selected tokens
// in index order into its own slots, so every list and every floating-point
// reduction has a fixed order (the results do not depend on scheduling).
// Loads are issued in batches (16 per thread) before any is used: these
// kernels move little data and are bound by memory latency.
#pragma once
#include "k_score.cuh"

namespace ssa {

constexpr int kBatch = 16;   // strips (or list entries) loaded per thread before use
constexpr int kDecBatch = 8;  // the same in the decision kernel (it keeps more live per strip)

struct SelShared {
    uint32_t scan[kSelWarps];
    uint32_t bcast[8];
    float zw[kSelWarps][2];
};

// Exact position of the k-th token among the members of the threshold
// bucket, and the normaliser.  Run by the last K2a CTA of unit u.
struct ResolveShared {
    uint32_t scan[kSelWarps];
    uint32_t bcast[8];
    uint32_t hist3[256];
    uint32_t nbound;
    uint2 bound[256];        // members sharing the top 24 key bits with the k-th score
    float bterm[256];        // their remainder terms, by rank
    float zw[kSelWarps][2];
};

// Dynamic shared memory of K2a: the per-list offsets of the candidate lists.
inline uint32_t k2a_smem_bytes(int nlists) { return (uint32_t)(nlists + 1) * 4u; }

__device__ __forceinline__ void zacc(float& zh, float& zl, float v)
{
    float sh, er;
    two_sum(zh, v, sh, er);
    zh = sh;
    zl = __fadd_rn(zl, er);
}

// The candidate lists of unit u, flattened in index order: entry q lies in
// list l with coff[l] <= q < coff[l + 1].
struct CandLists {
    const uint2* cand;       // the unit's slots
    const uint32_t* coff;    // shared memory, nlists + 1 offsets
    int nlists, tt, W2;
    __device__ __forceinline__ const uint2* at(uint32_t q) const
    {
        int lo = 0, hi = nlists;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (coff[mid] <= q) lo = mid; else hi = mid;
        }
        return cand + (size_t)(lo / kSelWarps) * tt + (size_t)(lo % kSelWarps) * W2 + (q - coff[lo]);
    }
};

__device__ void resolve_unit(const Params& p, int u, uint32_t f1, uint32_t above1, uint32_t target, float m,
                             ResolveShared& rs, uint32_t* coff)
{
    const Plan& pl = p.pl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* status = ws_status(p);
    const bool want_z = p.budget > 0.0f;
    const uint32_t* ccount = ws_ccount(p) + (size_t)u * pl.ntile * kSelWarps;
    const int nlists = pl.ntile * kSelWarps;
    const CandLists cl{ws_cand(p) + (size_t)u * pl.np, coff, nlists, pl.tt, pl.tt / kSelWarps};

    // list offsets (each thread a contiguous range of lists, loaded at once)
    {
        const int l0 = nlists * tid / kSelThreads, l1 = nlists * (tid + 1) / kSelThreads;
        uint32_t mine = 0;
        for (int l = l0; l < l1; l += 32) {
            uint32_t c[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) c[j] = (l + j < l1) ? __ldcg(ccount + l + j) : 0u;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (l + j < l1) coff[l + j] = mine;
                mine += c[j];
            }
        }
        uint32_t tot;
        const uint32_t before = block_excl_scan<kSelThreads>(mine, rs.scan, tot);
        for (int l = l0; l < l1; ++l) coff[l] += before;
        if (tid == 0) coff[nlists] = tot;
        __syncthreads();
    }
    const uint32_t E = coff[nlists];

    // level 2: the next 12 key bits of the bucket's members
    const Found f2 = find_rank_desc<kSelThreads, kBins, true>(ws_hist2(p) + (size_t)u * kBins, target - above1,
                                                            rs.scan, rs.bcast, status);
    const uint32_t pre24 = (f1 << 12) | f2.bin;
    const uint32_t t3 = target - above1 - f2.above;   // rank among the pre24 members (1-based)

    // walk the members: below pre24 -> remainder terms; pre24 -> ranked exactly
    if (tid == 0) rs.nbound = 0;
    __syncthreads();
    float zh = 0.0f, zl = 0.0f;
    for (uint32_t q0 = 0; q0 < E; q0 += kSelThreads * kBatch) {
        uint2 e[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const uint32_t q = q0 + (uint32_t)(j * kSelThreads + tid);
            e[j] = (q < E) ? __ldcg(cl.at(q)) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const uint32_t q = q0 + (uint32_t)(j * kSelThreads + tid);
            if (q >= E) continue;
            const uint32_t k24 = e[j].x >> 8;
            if (k24 < pre24) {
                if (want_z) zacc(zh, zl, expf(__fsub_rn(okey_value(e[j].x), m)));
            } else if (k24 == pre24) {
                const uint32_t slot = atomicAdd(&rs.nbound, 1u);
                if (slot < 256u) rs.bound[slot] = e[j];
            }
        }
    }
    __syncthreads();
    const uint32_t nb = rs.nbound;
    uint32_t theta;
    int64_t idx_cut;
    if (nb <= 256u) {
        // rank every pre24 member exactly (key desc, index asc)
        if (tid == 0) {
            rs.bcast[4] = 0xffffffffu;
            rs.bcast[5] = 0;
        }
        __syncthreads();
        uint32_t my_rank = 0xffffffffu;
        uint2 me = make_uint2(0, 0);
        if ((uint32_t)tid < nb) {
            me = rs.bound[tid];
            uint32_t ahead = 0;
            for (uint32_t i = 0; i < nb; ++i) {
                const uint2 o = rs.bound[i];
                ahead += (o.x > me.x || (o.x == me.x && o.y < me.y)) ? 1u : 0u;
            }
            my_rank = ahead + 1;
            if (my_rank == t3) {
                rs.bcast[4] = me.x;
                rs.bcast[5] = me.y;
            }
        }
        __syncthreads();
        if (rs.bcast[4] == 0xffffffffu) {   // inconsistent counts: cannot happen
            if (tid == 0) flag(status, DEV_BAD_INDEX);
            rs.bcast[4] = pre24 << 8;
            rs.bcast[5] = 0;
        }
        theta = rs.bcast[4];
        idx_cut = (int64_t)rs.bcast[5];
        if (p.top_k == 0) idx_cut = -1;   // k = 0: empty stratum, the k-th score only fixes m
        // remainder terms of these members, summed in rank order
        if ((uint32_t)tid < nb) {
            const bool inT = me.x > theta || (me.x == theta && (int64_t)me.y <= idx_cut);
            rs.bterm[my_rank - 1] = (!inT && want_z) ? expf(__fsub_rn(okey_value(me.x), m)) : 0.0f;
        }
        __syncthreads();
        if (tid == 0) {
            float bh = 0.0f, bl = 0.0f;
            for (uint32_t r = 0; r < nb; ++r) zacc(bh, bl, rs.bterm[r]);
            comp_add(zh, zl, bh, bl);
        }
    } else {
        // many members share the top 24 bits (ties, near-constant scores):
        // last 8 bits by histogram, then the tie by index order (the
        // flattened lists are in index order), in rounds of one entry per thread
        for (int i = tid; i < 256; i += kSelThreads) rs.hist3[i] = 0u;
        __syncthreads();
        for (uint32_t q = tid; q < E; q += kSelThreads) {
            const uint2 e = __ldcg(cl.at(q));
            if ((e.x >> 8) == pre24) atomicAdd(&rs.hist3[e.x & 0xffu], 1u);
        }
        __syncthreads();
        const Found f3 = find_rank_desc<kSelThreads, 256, false>(rs.hist3, t3, rs.scan, rs.bcast, status);
        theta = (pre24 << 8) | f3.bin;
        const uint32_t rt = t3 - f3.above;   // rank among the ties at theta, in index order
        uint32_t seen = 0;
        if (tid == 0) rs.bcast[6] = 0;
        __syncthreads();
        for (uint32_t q0 = 0; q0 < E && seen < rt; q0 += kSelThreads) {
            const uint32_t q = q0 + tid;
            const uint2 e = (q < E) ? __ldcg(cl.at(q)) : make_uint2(0u, 0u);
            const bool tie = q < E && e.x == theta;
            uint32_t n;
            const uint32_t before = block_excl_scan<kSelThreads>(tie ? 1u : 0u, rs.scan, n);
            if (tie && seen + before + 1 == rt) rs.bcast[6] = e.y;
            seen += n;
        }
        __syncthreads();
        idx_cut = (int64_t)rs.bcast[6];
        if (p.top_k == 0) idx_cut = -1;
        // remainder terms of the pre24 members
        if (want_z) {
            for (uint32_t q = tid; q < E; q += kSelThreads) {
                const uint2 e = __ldcg(cl.at(q));
                if ((e.x >> 8) != pre24) continue;
                const bool inT = e.x > theta || (e.x == theta && (int64_t)e.y <= idx_cut);
                if (!inT) zacc(zh, zl, expf(__fsub_rn(okey_value(e.x), m)));
            }
        }
    }

    // normaliser: tile partials + candidate terms, fixed assignment and tree
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, zh, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, zl, o);
        comp_add(zh, zl, h2, l2);
    }
    if (lane == 0) {
        rs.zw[warp][0] = zh;
        rs.zw[warp][1] = zl;
    }
    __syncthreads();
    if (tid == 0) {
        float hh = 0.0f, ll = 0.0f;
        for (int w = 0; w < kSelWarps; ++w) comp_add(hh, ll, rs.zw[w][0], rs.zw[w][1]);
        UnitCtrl* ctrl = ws_ctrl(p) + u;
        ctrl->theta = theta;
        ctrl->idx_cut = (int32_t)idx_cut;
        ctrl->m = m;
        ctrl->Z = __fadd_rn(hh, ll);
    }
}

// ---------------------------------------------------------------------------
// K2a: per (unit, tile)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads, 2) bucket_kernel(const __grid_constant__ Params p)
{
    extern __shared__ uint32_t coff[];
    __shared__ SelShared sh;
    __shared__ ResolveShared rs;
    __shared__ uint32_t is_last;
    const Plan& pl = p.pl;
    const int u = blockIdx.x / pl.ntile, tile = blockIdx.x % pl.ntile;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W2 = pl.tt / kSelWarps;
    uint32_t* status = ws_status(p);
    grid_dep_wait();
    SSA_MARK(2);

    const uint32_t target = (uint32_t)(p.top_k > 0 ? p.top_k : 1);
    const Found f1 = find_rank_desc<kSelThreads, kBins, true>(ws_hist1(p) + (size_t)u * kBins, target, sh.scan,
                                                            sh.bcast, status);
    const float m = okey_value(f1.bin << 20);
    const bool want_z = p.budget > 0.0f;

    const int64_t base = (int64_t)tile * pl.tt + (int64_t)warp * W2;   // this warp's first token
    const float* S = p.s_src + (int64_t)u * pl.N;
    uint2* cand = ws_cand(p) + (size_t)u * pl.np + base;
    uint32_t* hist2 = ws_hist2(p) + (size_t)u * kBins;
    uint32_t cnt = 0;
    float zh = 0.0f, zl = 0.0f;
    for (int st0 = 0; st0 < W2; st0 += 32 * kBatch) {
        float sv[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int64_t t = base + st0 + j * 32 + lane;
            sv[j] = (st0 + j * 32 < W2 && t < pl.N) ? __ldcg(S + t) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (st0 + j * 32 >= W2) break;   // uniform across the warp
            const int64_t t = base + st0 + j * 32 + lane;
            const bool valid = t < pl.N;
            const uint32_t k = okey(sv[j]);
            const uint32_t b1 = k >> 20;
            const bool is_cand = valid && b1 == f1.bin;
            if (is_cand) atomicAdd(hist2 + ((k >> 8) & 0xfffu), 1u);
            const uint32_t mask = __ballot_sync(0xffffffffu, is_cand);
            if (is_cand) cand[cnt + __popc(mask & lanemask_lt())] = make_uint2(k, (uint32_t)t);
            cnt += __popc(mask);
            if (valid && want_z && b1 < f1.bin) zacc(zh, zl, expf(__fsub_rn(sv[j], m)));
        }
    }
    if (lane == 0) ws_ccount(p)[((size_t)u * pl.ntile + tile) * kSelWarps + warp] = cnt;
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
        const uint32_t prev = atomicAdd(&ws_ctrl(p)[u].k2a_done, 1u);
        is_last = (prev == (uint32_t)(pl.ntile - 1)) ? 1u : 0u;
    }
    __syncthreads();
    grid_dep_launch();
    if (is_last) {
        __threadfence();
        SSA_MARK(3);
        resolve_unit(p, u, f1.bin, f1.above, target, m, rs, coff);
        SSA_MARK(4);
    }
}

// ---------------------------------------------------------------------------
// K2c: decisions, per (unit, tile); selected tokens in index order per warp
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads, 2) decide_kernel(const __grid_constant__ Params p)
{
    // xrej[v] / xacc[v]: thresholds on x = fl32(s - m) for a token whose uniform
    // has top 8 bits v, u in [v / 256, (v + 1) / 256): x < xrej[v] implies
    // p <= v / 256 <= u (reject); x > xacc[v] implies p >= (v + 1) / 256 > u
    // (accept).  The margin (1e-4 + 1e-5 |threshold| in x) exceeds the error
    // of the fp32 logarithms that place the thresholds plus the rounding of
    // expf (2 ulp) and of the product and quotient that form p, so either
    // shortcut agrees with the exact rule; tokens in between take the exact
    // rule.
    __shared__ float xrej[256], xacc[256];
    const Plan& pl = p.pl;
    const int u = blockIdx.x / pl.ntile, tile = blockIdx.x % pl.ntile;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W2 = pl.tt / kSelWarps;
    const int b = u / p.Hkv, h = u % p.Hkv;
    const int64_t base = (int64_t)tile * pl.tt + (int64_t)warp * W2;
    const float* S = p.s_src + (int64_t)u * pl.N;
    const uint8_t* ub = ws_ubuf(p) + (size_t)u * pl.np;
    int32_t* sidx = ws_sel_idx(p) + (size_t)u * pl.np + base;
    float* sp = ws_sel_p(p) + (size_t)u * pl.np + base;
    grid_dep_wait();
    SSA_MARK(5);
    const UnitCtrl* ctrl = ws_ctrl(p) + u;
    const uint32_t theta = __ldcg(&ctrl->theta);
    const int64_t idx_cut = __ldcg(&ctrl->idx_cut);
    const float m = __ldcg(&ctrl->m);
    const float Z = __ldcg(&ctrl->Z);
    const float B = p.budget;
    const bool sampling = B > 0.0f && Z > 0.0f;
    if (sampling && tid < 256) {
        const float lzb = logf(Z) - logf(B) - 5.545177444479562f;   // log(Z / (256 B))
        const float lo = lzb + logf((float)tid);                      // log(v Z / (256 B)); -inf at v = 0
        const float hi = lzb + logf((float)(tid + 1));
        xrej[tid] = (tid == 0) ? -INFINITY : lo - 1e-4f - 1e-5f * fabsf(lo);
        xacc[tid] = hi + 1e-4f + 1e-5f * fabsf(hi);
    }
    __syncthreads();

    uint32_t cnt = 0;
    for (int st0 = 0; st0 < W2; st0 += 32 * kDecBatch) {
        float sv[kDecBatch];
        uint32_t u8[kDecBatch];
#pragma unroll
        for (int j = 0; j < kDecBatch; ++j) {
            const int64_t t = base + st0 + j * 32 + lane;
            const bool ok = st0 + j * 32 < W2 && t < pl.N;
            sv[j] = ok ? __ldcg(S + t) : 0.0f;
            u8[j] = ok ? (uint32_t)__ldcg(ub + t) : 0u;
        }
#pragma unroll
        for (int j = 0; j < kDecBatch; ++j) {
            if (st0 + j * 32 >= W2) break;   // uniform across the warp
            const int64_t t = base + st0 + j * 32 + lane;
            bool sel = false;
            float pr = 1.0f;
            if (t < pl.N) {
                const uint32_t k = okey(sv[j]);
                if (k > theta || (k == theta && t <= idx_cut)) {
                    sel = true;
                } else if (sampling) {
                    const float x = __fsub_rn(sv[j], m);
                    if (!(x < xrej[u8[j]])) {
                        pr = prob_from_term(expf(x), B, Z);
                        if (pr > 0.0f) {
                            const float lo8 = (float)u8[j] * 0.00390625f;   // u lies in [lo8, lo8 + 2^-8)
                            if (x > xacc[u8[j]] || pr >= lo8 + 0.00390625f) sel = true;
                            else if (pr > lo8) sel = token_uniform(p.seed, t, h, b) < pr;
                        }
                    }
                }
            }
            const uint32_t mask = __ballot_sync(0xffffffffu, sel);
            if (sel) {
                const uint32_t o = cnt + __popc(mask & lanemask_lt());
                sidx[o] = (int32_t)t;
                sp[o] = pr;
            }
            cnt += __popc(mask);
        }
    }
    if (lane == 0) ws_scount(p)[((size_t)u * pl.ntile + tile) * kSelWarps + warp] = cnt;
    SSA_MARK(6);
    grid_dep_launch();
}

}  // namespace ssa
