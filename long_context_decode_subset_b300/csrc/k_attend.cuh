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
// (positions [r * R / P, (r + 1) * R / P)); the list is staged in shared
// memory in chunks.  Every warp streams its rows' K and V straight from HBM
// with cp.async (each lane copies, and later reads, its own 16- or 8-byte
// piece of a row; NS steps in flight per warp), so the gather needs no block
// barrier.  The CTA's (m, l, acc) partial goes to the workspace; the last CTA
// of a unit to finish merges the P partials in a fixed order.
#pragma once
#include "k_select.cuh"

namespace ssa {

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

// Dynamic shared memory of K3 for nlists per-tile lists.
template <int G, int D>
constexpr uint32_t k3_smem_bytes(int nlists)
{
    return K3Cfg<G, D>::OFF_PRE + (uint32_t)(nlists + 1) * 4u + 128u;
}

struct K3Shared {
    uint32_t scan[k3Warps];
    uint32_t bcast[4];
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
    const int nlists = pl.ntile * kSelWarps;   // K2c writes one list per warp slice of a tile
    const int W2 = pl.tt / kSelWarps;
    uint32_t* status = ws_status(p);
    SSA_GT(4);
    grid_dep_wait();
    SSA_MARK(7);
    SSA_GT(5);

    // the unit's list length and (per-tile lists) its prefix over the lists
    int64_t total = 0;
    if (p.src_mode == 0) {
        const uint32_t* sc = ws_scount(p) + (size_t)u * nlists;
#pragma unroll 1
        for (int l = tid; l < nlists; l += k3Threads) cp_async_4(pre + l, sc + l);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        const int l0 = nlists * tid / k3Threads, l1 = nlists * (tid + 1) / k3Threads;
        uint32_t mine = 0;
#pragma unroll 1
        for (int l = l0; l < l1; ++l) {
            const uint32_t c = pre[l];
            pre[l] = mine;
            mine += c;
        }
        uint32_t tot;
        const uint32_t before = block_excl_scan<k3Threads>(mine, ks.scan, tot);
        for (int l = l0; l < l1; ++l) pre[l] += before;
        if (tid == 0) pre[nlists] = tot;
        total = tot;
    } else if (p.src_mode == 1) {
        total = pl.N;
    } else {
        const int64_t c = p.count_in[u];
        total = c < 0 ? 0 : (c > p.cap ? p.cap : c);
    }
    __syncthreads();
    SSA_MARK(11);
    const int64_t lo = total * r / P, hi = total * (r + 1) / P;
    const uint16_t* Kb = p.K + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;
    const uint16_t* Vb = p.V + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;
    const int32_t* sidx = ws_sel_idx(p) + (size_t)u * pl.np;
    const float* sp = ws_sel_p(p) + (size_t)u * pl.np;

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
    // the unit's threshold and normaliser (per-tile lists only)
    uint32_t d_theta = 0;
    int64_t d_cut = -1;
    float d_m = 0.0f, d_Z = 0.0f;
    if (p.src_mode == 0) {
        const UnitCtrl* ctrl = ws_ctrl(p) + u;
        d_theta = __ldcg(&ctrl->theta);
        d_cut = __ldcg(&ctrl->idx_cut);
        d_m = __ldcg(&ctrl->m);
        d_Z = __ldcg(&ctrl->Z);
    }
    const bool d_sampling = p.budget > 0.0f && d_Z > 0.0f;
    int64_t kept = 0;   // entries this CTA keeps

    for (int64_t c0 = lo; c0 < hi; c0 += CF::CHUNK) {
        const int n = (int)min((int64_t)CF::CHUNK, hi - c0);
        __syncthreads();   // the previous chunk is consumed
        constexpr int PER = CF::CHUNK / k3Threads;   // consecutive entries per thread
        // the chunk's raw entries into shared memory (cp.async, one wave)
        int32_t* ridx = reinterpret_cast<int32_t*>(smem);
        float* rval = reinterpret_cast<float*>(smem + CF::CHUNK * 4);
        if (p.src_mode == 0) {
#pragma unroll 1
            for (int i = tid; i < n; i += k3Threads) {
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
            for (int i = tid; i < n; i += k3Threads) {
                cp_async_4(ridx + i, p.idx_in + (int64_t)u * p.cap + c0 + i);
                cp_async_4(rval + i, p.p_in + (int64_t)u * p.cap + c0 + i);
            }
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        SSA_MARK(28);
        // final decisions for this thread's PER consecutive entries (per-tile
        // lists: the top-k stratum, then the draw u < p); one bit each
        uint32_t kbits = 0, kcount = 0;
#pragma unroll 1
        for (int e = 0; e < PER; ++e) {
            const int i = tid * PER + e;
            if (i >= n) break;
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
                            if (k > d_theta || (k == d_theta && (int64_t)j <= d_cut)) {
                                keep = true;
                                pv = 1.0f;
                            }
                            ev = expf(__fsub_rn(pv, d_m));
                        }
                        if (!keep) {
                            pv = d_sampling ? prob_from_term(ev, p.budget, d_Z) : 0.0f;
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
        // keep the chosen entries in list order: cidx / clp[0, nk)
        uint32_t nk_u;
        uint32_t at = block_excl_scan<k3Threads>(kcount, ks.scan, nk_u);
        const int nk = (int)nk_u;
#pragma unroll 1
        for (int e = 0; e < PER; ++e) {
            if (!((kbits >> e) & 1u)) continue;
            const int i = tid * PER + e;
            const int32_t j = (p.src_mode == 1) ? (int32_t)(c0 + i) : ridx[i];
            const float pv = (p.src_mode == 1) ? 1.0f : rval[i];
            cidx[at] = j;
            clp[at] = logf(pv);
            if (p.idx_out) {   // staged for the unit's compact list
                uint2* stage = ws_cand(p) + (size_t)u * pl.N + (size_t)(lo + kept);
                stage[at] = make_uint2((uint32_t)j, __float_as_uint(pv));
            }
            ++at;
        }
        SSA_MARK(29);
        kept += nk;
        __syncthreads();
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
    uint32_t* kept_all = ws_kept(p) + (size_t)u * kMaxSplit;
    if (tid == 0) kept_all[r] = (uint32_t)kept;
    __threadfence();
    __syncthreads();
    if (tid == 0) ks.is_last = (atomicAdd(&ws_ctrl(p)[u].k3_done, 1u) == (uint32_t)(P - 1)) ? 1u : 0u;
    __syncthreads();
    SSA_MARK(12);
    SSA_GT(6);
    if (!ks.is_last) return;
    __threadfence();
    if (p.count_out || p.idx_out) {
        // the unit's kept entries: prefix over the P CTAs, then (if asked) the
        // compact list in list order, copied from the per-CTA staging
        uint32_t* koff = reinterpret_cast<uint32_t*>(smem);   // [P + 1]
        if (warp == 0) {
            uint32_t run = 0;
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
            for (uint32_t o = tid; o < kept_total; o += k3Threads) {
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
                    flag(status, DEV_OVERFLOW);
                }
            }
        }
        __syncthreads();
    }
    SSA_MARK(14);
    if (!p.attend) return;
    // merge the P partials in a fixed order (r ascending).  Every thread owns
    // G * D / k3Threads accumulator elements of one head g and reads that
    // head's (m, l) of all P partials itself, so the merge is one wave of
    // loads and no block barrier.
    const float* parts = ws_part(p) + (size_t)u * P * (size_t)(G * D + 2 * G);
    constexpr int PS = G * D + 2 * G;   // floats per partial
    constexpr int EPT = (G * D + k3Threads - 1) / k3Threads;   // elements per thread (same head)
    static_assert((G * D) % k3Threads == 0 || G * D < k3Threads, "elements split evenly");
    const int e0 = tid * EPT;
    if (e0 < G * D) {
        const int g = e0 / D;
        float M = -INFINITY;
        for (int r0 = 0; r0 < P; r0 += 16) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (r0 + j < P) M = fmaxf(M, __ldcg(parts + (size_t)(r0 + j) * PS + G * D + g));
        }
        float Ls = 0.0f, A[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) A[e] = 0.0f;
        if (M != -INFINITY) {
            for (int r0 = 0; r0 < P; r0 += 8) {
                float mr[8], lr[8], ar[8][EPT];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float* pr = parts + (size_t)(r0 + j) * PS;
                    const bool ok = r0 + j < P;
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
