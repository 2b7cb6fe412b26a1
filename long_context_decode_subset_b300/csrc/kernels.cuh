// kernels.cuh -- the libssa device code: one thread-block cluster per
// (batch, KV head) unit runs the whole Stratified Sparse Attention decode
// step for that unit.
//
// Sources (page title, section):
//  * "FASA: Frequency-Aware Sparse Attention", section 3 (Method), Stage 1
//    "Token Importance Prediction": every token is scored from a fixed,
//    pre-calibrated subset of dominant RoPE chunks only; Stage 2 "Focused
//    Attention Computation": full-precision attention over the selected
//    tokens only, at their original positions.
//  * "Stratified Sparse Attention speeds up decoding 2.96x on a 1M context",
//    section "How SSA splits the cache into strata": high-estimate tokens are
//    read deterministically; the rest are sampled with probability
//    proportional to the approximate attention; each sampled token is
//    corrected by its inclusion probability.
//  * "S2O" (online permutation and early stopping), technical summary,
//    Method section 1 (rows are gathered by index arrays, the physical layout
//    in HBM is kept) and section 3 (the online-softmax state (m, l, acc)).
//  * Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
//    Easy as 1, 2, 3", SC'11.
//
// Work split.  A unit's N tokens are cut into C contiguous segments, one per
// CTA of the unit's cluster (C in {1, 2, 4, 8, 16}).  Each CTA:
//   1. streams its segment of the key summary through a ring of bulk
//      asynchronous copies into shared memory and scores every token (fp32
//      FMA; the G query heads of the group reduced by max), keeping the
//      scores in shared memory (or global scratch when the segment is too
//      long) and building a 4096-bin histogram of the top 12 bits of the
//      order-preserving score key;
//   2. finds the exact k-th largest key with three radix levels (12, 12 and
//      8 bits), merging the per-CTA histograms through distributed shared
//      memory (a slice of bins per CTA);
//   3. resolves ties at the threshold by index (lowest indices first);
//   4. sums exp(s - m) over the remainder EXACTLY as a 160-bit fixed-point
//      integer (every fp32 value is an integer multiple of 2^-149), merges
//      the per-CTA sums and rounds once to fp32;
//   5. decides every token (top-k, or a Philox uniform against p), records
//      the decisions as ballot bit masks, and writes the selected indices and
//      probabilities in ascending token order at offsets from a cluster-wide
//      prefix sum;
//   6. takes an even share of the unit's selected list, gathers those K and V
//      rows into shared memory with bulk asynchronous copies (one copy per
//      row, physical layout untouched), runs the corrected online softmax on
//      CUDA cores, and
//   7. merges the per-warp and then per-CTA (m, l, acc) states (the latter
//      through distributed shared memory) into the unit's outputs.
// Every wait is bounded in time; every CTA reaches every cluster barrier.
#pragma once
#include <cooperative_groups.h>
#include <cstdint>

#include "ptx.cuh"

namespace ssa {
namespace cg = cooperative_groups;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;                      // radix levels 1 and 2 (12 bits)
constexpr int kBins3 = 256;                      // radix level 3 (8 bits)
constexpr uint32_t kRingBytes = 96u * 1024u;     // summary ring / attend ring / merge scratch
constexpr int kSegAlign = 512;                   // segments are multiples of 16 warps x 32 lanes
constexpr int kAttendStages = 4;
constexpr int kMaxScoreStages = 12;
constexpr uint32_t kSmemLimit = 227u * 1024u;

constexpr int MODE_SCORE = 1;
constexpr int MODE_SELECT = 2;
constexpr int MODE_ATTEND = 4;

constexpr uint32_t DEV_NONFINITE = 0x1u;
constexpr uint32_t DEV_OVERFLOW = 0x2u;
constexpr uint32_t DEV_TIMEOUT = 0x4u;
constexpr uint32_t DEV_BAD_INDEX = 0x8u;

struct Params {
    int32_t Bt, Hq, Hkv, d, d_sel;
    int64_t N;
    int64_t kv_sb, kv_sh, ks_sb, ks_sh;
    const uint16_t* q;
    const uint16_t* K;
    const uint16_t* V;
    const uint16_t* Ks;
    const int32_t* sel_ch;
    float scale;
    int64_t top_k;
    float budget;
    uint64_t seed;
    const float* s_in;      // select-only: the scores to select from
    float* s_out;           // scores written to global memory (may be null in decode)
    int32_t* idx;           // selected lists [units][cap]
    float* p;
    int32_t* count;         // [units]
    int64_t cap;
    float* out;             // [Bt][Hq][d]
    float* lse;             // [Bt][Hq]
    uint32_t* status;       // device status word
    int32_t C;              // CTAs per unit
    int64_t seg_len;        // tokens per CTA
};

// Shared-memory scalars and small arrays.
struct Misc {
    uint64_t score_full[kMaxScoreStages];
    uint64_t att_full[kAttendStages];
    float att_logp[kAttendStages][64];
    uint32_t warp_u32[kWarps];
    uint32_t bcast[16];
    unsigned long long zwarp[kWarps][5];
    unsigned long long zpart[5];     // this CTA's exact normaliser limbs (read by peers)
    uint32_t slice_tot;              // this CTA's merged-slice total (read by peers)
    uint32_t cta_count;              // this CTA's selected count (read by peers)
    float fbcast[4];
    float wm[kWarps][8], wl[kWarps][8];
    float cm[8], cl[8];              // this CTA's softmax partial (read by peers)
};

struct Layout {
    uint32_t ring, sbuf, histA, histB, merged, bits, misc, total;
};

__host__ __device__ inline uint32_t align_up_u32(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int mode, bool resident, int64_t seg_len, int C)
{
    Layout L{};
    uint32_t o = 0;
    L.ring = o;
    o += kRingBytes;
    if (mode & MODE_SELECT) {
        L.sbuf = o;
        if (resident) o += align_up_u32((uint32_t)(seg_len * 4), 128);
        L.histA = o;
        o += kBins * 4;
        L.histB = o;
        o += kBins * 4;
        L.merged = o;
        if (C > 1) o += align_up_u32(2u * (uint32_t)(kBins / C) * 4u, 128);
        L.bits = o;
        o += align_up_u32((uint32_t)(seg_len / 32) * 4u, 128);
    } else if (mode & MODE_ATTEND) {
        L.histB = o;  // the CTA's (acc) partial
        o += kBins * 4;
    }
    L.misc = o;
    o += align_up_u32((uint32_t)sizeof(Misc), 128);
    L.total = o;
    return L;
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------

// Order-preserving key of an fp32 value (-0 sorts below +0).
__device__ __forceinline__ uint32_t okey(float x)
{
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float okey_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_at(const uint16_t* p) { return __uint_as_float(((uint32_t)*p) << 16); }

__device__ __forceinline__ void flag(uint32_t* status, uint32_t bits)
{
    if (status) atomicOr(status, bits);
}

// Philox4x32-10 (SC'11): ten rounds of two 32x32->64-bit products of the
// even words by the round multipliers, high halves xored into the odd words
// with the round key, key bumped by the Weyl constants.  Only word 0 of the
// output is used.
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a_hi = __umulhi(0xD2511F53u, c0);
        const uint32_t a_lo = 0xD2511F53u * c0;
        const uint32_t b_hi = __umulhi(0xCD9E8D57u, c2);
        const uint32_t b_lo = 0xCD9E8D57u * c2;
        c0 = b_hi ^ c1 ^ k0;
        c1 = b_lo;
        c2 = a_hi ^ c3 ^ k1;
        c3 = a_lo;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

// u = (x0 >> 8) * 2^-24 for token j of unit (b, h_kv).
__device__ __forceinline__ float token_uniform(uint64_t seed, int64_t j, int h_kv, int b)
{
    const uint32_t x0 = philox_word0((uint32_t)j, (uint32_t)h_kv, (uint32_t)b, 0u,
                                     (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32));
    return __uint2float_rn(x0 >> 8) * 5.9604644775390625e-08f;
}

// p = min(1, fl32(fl32(B * e) / Z)) with e = expf(fl32(s - m)).
__device__ __forceinline__ float inclusion_prob(float s, float m, float budget, float Z)
{
    const float e = expf(__fsub_rn(s, m));
    const float t = __fmul_rn(budget, e);
    return fminf(__fdiv_rn(t, Z), 1.0f);
}

// Exact accumulation of a non-negative fp32 e <= 1 into five 64-bit limb
// sums: e * 2^149 = M << sh (M < 2^24, sh <= 126) spans 32-bit digits
// sh/32 and sh/32 + 1; each limb collects 32-bit digits without carry
// propagation (fewer than 2^31 terms per limb cannot overflow 64 bits).
__device__ __forceinline__ void exact_add(unsigned long long (&z)[5], float e, uint32_t* status)
{
    const uint32_t u = __float_as_uint(e);
    const uint32_t ex = u >> 23;            // sign is 0
    if (ex >= 255u) { flag(status, DEV_NONFINITE); return; }
    uint32_t mant = u & 0x7fffffu;
    uint32_t sh = 0;
    if (ex) { mant |= 0x800000u; sh = ex - 1; }
    if (sh > 126u) { flag(status, DEV_NONFINITE); return; }   // e > 1 cannot happen on R
    const uint32_t digit = sh >> 5;
    const unsigned long long v = (unsigned long long)mant << (sh & 31u);
    const unsigned long long lo = v & 0xffffffffull, hi = v >> 32;
#pragma unroll
    for (int i = 0; i < 5; ++i)
        z[i] += (digit == (uint32_t)i) ? lo : ((digit + 1u == (uint32_t)i) ? hi : 0ull);
}

// Round sum(z[i] * 2^(32 i)) * 2^-149 to the nearest fp32, ties to even.
__device__ inline float exact_to_float(const unsigned long long (&z)[5])
{
    uint32_t dig[6];
    unsigned long long carry = 0;
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        const unsigned long long v = z[i] + carry;
        dig[i] = (uint32_t)v;
        carry = v >> 32;
    }
    dig[5] = (uint32_t)carry;
    int top = -1;
    for (int i = 5; i >= 0; --i)
        if (dig[i]) { top = 32 * i + 31 - __clz(dig[i]); break; }
    if (top < 0) return 0.0f;
    if (top < 24) return __uint_as_float(dig[0]);   // M * 2^-149 with M < 2^24: the bits are M itself
    // 64-bit window holding bits [top-63, top] (lower bits only matter for the sticky bit)
    auto bits_from = [&](int lo_bit) -> unsigned long long {  // 64 bits starting at lo_bit (may be < 0)
        unsigned long long w = 0;
        for (int k = 63; k >= 0; --k) {
            const int bpos = lo_bit + k;
            const uint32_t bit = (bpos >= 0 && bpos < 192) ? ((dig[bpos >> 5] >> (bpos & 31)) & 1u) : 0u;
            w = (w << 1) | bit;
        }
        return w;
    };
    const unsigned long long win = bits_from(top - 63);       // bit 63 = top
    uint32_t mant = (uint32_t)(win >> 40);                     // 24 bits [top-23, top]
    const uint32_t guard = (uint32_t)(win >> 39) & 1u;
    bool sticky = (win & ((1ull << 39) - 1)) != 0;
    for (int bpos = top - 64; bpos >= 0 && !sticky; --bpos)
        sticky = (dig[bpos >> 5] >> (bpos & 31)) & 1u;
    if (guard && (sticky || (mant & 1u))) {
        ++mant;
        if (mant == (1u << 24)) { mant >>= 1; ++top; }
    }
    const uint32_t biased = (uint32_t)(top - 22);               // value = mant * 2^(top - 172)
    return __uint_as_float((biased << 23) | (mant & 0x7fffffu));
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exclusive prefix over the block of one value per thread; also the total.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, Misc& ms, uint32_t& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ms.warp_u32[warp] = x;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = ms.warp_u32[w];
        before += (w < warp) ? t : 0u;
        tot += t;
    }
    __syncthreads();
    total = tot;
    return before + x - v;
}

struct Found {
    uint32_t bin, above, in;
};

// counts[0..n) are histogram bins in ascending key order.  Find the bin
// holding the t-th largest element (t >= 1): above = elements in higher
// bins, in = elements in that bin.
__device__ Found find_rank_desc(const uint32_t* counts, int n, uint32_t t, Misc& ms, uint32_t* status)
{
    const int tid = threadIdx.x;
    const int chunk = (n + kThreads - 1) / kThreads;
    uint32_t local = 0;
    for (int j = 0; j < chunk; ++j) {
        const int pos = tid * chunk + j;
        if (pos < n) local += counts[n - 1 - pos];
    }
    uint32_t total;
    const uint32_t excl = block_excl_scan(local, ms, total);
    if (local > 0 && excl < t && t <= excl + local) {
        uint32_t cum = excl;
        for (int j = 0; j < chunk; ++j) {
            const int pos = tid * chunk + j;
            if (pos >= n) break;
            const uint32_t c = counts[n - 1 - pos];
            if (cum + c >= t) {
                ms.bcast[0] = (uint32_t)(n - 1 - pos);
                ms.bcast[1] = cum;
                ms.bcast[2] = c;
                break;
            }
            cum += c;
        }
    }
    if (tid == 0 && total < t) {  // cannot happen for consistent inputs
        ms.bcast[0] = 0;
        ms.bcast[1] = 0;
        ms.bcast[2] = 0;
        flag(status, DEV_BAD_INDEX);
    }
    __syncthreads();
    const Found f{ms.bcast[0], ms.bcast[1], ms.bcast[2]};
    __syncthreads();
    return f;
}

// One radix level across the cluster: every CTA's local histogram `hloc`
// (nb bins) is complete on entry.  CTA r sums bins [r*nb/C, (r+1)*nb/C)
// over all peers; the slice holding rank t is located from the slice totals
// and scanned.  Every CTA returns the same answer.
__device__ Found level_find(cg::cluster_group& cluster, uint32_t* hloc, int nb, uint32_t t, int C,
                            int rank, uint32_t* merged, Misc& ms, uint32_t* status)
{
    if (C == 1) {
        __syncthreads();
        return find_rank_desc(hloc, nb, t, ms, status);
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    cluster.sync();
    const int per = nb / C;
    const int lo = rank * per;
    uint32_t tot = 0;
    for (int i = tid; i < per; i += kThreads) {
        uint32_t s = 0;
        for (int r = 0; r < C; ++r) s += cluster.map_shared_rank(hloc, r)[lo + i];
        merged[i] = s;
        tot += s;
    }
    uint32_t total;
    block_excl_scan(tot, ms, total);
    if (tid == 0) ms.slice_tot = total;
    cluster.sync();
    if (warp == 0) {
        // lane r looks at slice C-1-r (highest bins first)
        const uint32_t v = (lane < C) ? *cluster.map_shared_rank(&ms.slice_tot, C - 1 - lane) : 0u;
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        const uint32_t excl = x - v;
        const bool hit = lane < C && v > 0 && excl < t && t <= x;
        const uint32_t m = __ballot_sync(0xffffffffu, hit);
        if (m) {
            if (lane == __ffs(m) - 1) {
                ms.bcast[4] = (uint32_t)(C - 1 - lane);
                ms.bcast[5] = excl;
            }
        } else if (lane == 0) {
            ms.bcast[4] = 0;
            ms.bcast[5] = 0;
            flag(status, DEV_BAD_INDEX);
        }
    }
    __syncthreads();
    const int sstar = (int)ms.bcast[4];
    const uint32_t above_s = ms.bcast[5];
    uint32_t* fetched = merged + per;
    const uint32_t* remote = cluster.map_shared_rank(merged, sstar);
    for (int i = tid; i < per; i += kThreads) fetched[i] = remote[i];
    __syncthreads();
    Found f = find_rank_desc(fetched, per, t - above_s, ms, status);
    f.bin += (uint32_t)(sstar * per);
    f.above += above_s;
    return f;
}

// Segment position of the nth (1-based) token whose key equals theta, in
// index order, within this CTA's segment.
__device__ int find_nth_tie(const float* S, int len, uint32_t theta, uint32_t nth, int W, Misc& ms)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int base = warp * W;
    uint32_t cnt = 0;
    for (int t0 = 0; t0 < W; t0 += 32) {
        const int pos = base + t0 + lane;
        const bool tie = pos < len && okey(S[pos]) == theta;
        cnt += __popc(__ballot_sync(0xffffffffu, tie));
    }
    if (lane == 0) ms.warp_u32[warp] = cnt;
    __syncthreads();
    uint32_t excl = 0;
    for (int w = 0; w < warp; ++w) excl += ms.warp_u32[w];
    __syncthreads();
    if (excl < nth && nth <= excl + cnt) {
        uint32_t run = excl;
        for (int t0 = 0; t0 < W; t0 += 32) {
            const int pos = base + t0 + lane;
            const bool tie = pos < len && okey(S[pos]) == theta;
            uint32_t mask = __ballot_sync(0xffffffffu, tie);
            const uint32_t c = __popc(mask);
            if (run + c >= nth) {
                for (uint32_t k = 1; k < nth - run; ++k) mask &= mask - 1;
                if (lane == 0) ms.bcast[7] = (uint32_t)(base + t0 + __ffs(mask) - 1);
                break;
            }
            run += c;
        }
    }
    __syncthreads();
    const int r = (int)ms.bcast[7];
    __syncthreads();
    return r;
}

// ---------------------------------------------------------------------------
// phase 1: approximate scores from the key summary
// ---------------------------------------------------------------------------

template <int G, int DSEL>
struct ScoreCfg {
    static constexpr int CPT = (G <= 4) ? 16 : 8;            // summary channels per thread
    static constexpr int TPT = DSEL / CPT;                   // threads per token
    static constexpr int TOK = kThreads / TPT;               // tokens per ring stage
    static constexpr uint32_t STAGE_BYTES = (uint32_t)TOK * DSEL * 2u;
    static constexpr int STAGES = (int)(kRingBytes / STAGE_BYTES) < kMaxScoreStages
                                      ? (int)(kRingBytes / STAGE_BYTES) : kMaxScoreStages;
    static_assert(DSEL % CPT == 0, "d_sel must be a multiple of the per-thread channel count");
    static_assert(STAGES >= 2, "ring too small");
};

// Scores of segment tokens [s0, s0 + len) of unit (b, h).  sdst (shared or
// global) receives them at segment-relative positions; gdst (may be null)
// gets a second, global copy; hist (may be null) counts the top 12 key bits.
template <int G, int DSEL>
__device__ void phase_score(const Params& p, unsigned char* ring, Misc& ms, int b, int h, int64_t s0,
                            int len, float* sdst, float* gdst, uint32_t* hist)
{
    using SC = ScoreCfg<G, DSEL>;
    const int tid = threadIdx.x;
    const int part = tid % SC::TPT;
    const int tok = tid / SC::TPT;

    float qr[G][SC::CPT];
    {
        const int32_t* sel = p.sel_ch + (int64_t)h * DSEL + part * SC::CPT;
        const uint16_t* qb = p.q + ((int64_t)b * p.Hq + (int64_t)h * G) * p.d;
#pragma unroll
        for (int c = 0; c < SC::CPT; ++c) {
            int ch = sel[c];
            if ((unsigned)ch >= (unsigned)p.d) {
                flag(p.status, DEV_BAD_INDEX);
                ch = 0;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) qr[g][c] = bf16_at(qb + (int64_t)g * p.d + ch);
        }
    }

    const uint16_t* src = p.Ks + (int64_t)b * p.ks_sb + (int64_t)h * p.ks_sh + s0 * DSEL;
    const int nchunks = (len + SC::TOK - 1) / SC::TOK;
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int c) {
        const int st = c % SC::STAGES;
        const int ntok = min(SC::TOK, len - c * SC::TOK);
        const uint32_t bytes = (uint32_t)ntok * DSEL * 2u;
        mbar_arrive_expect_tx(&ms.score_full[st], bytes);
        bulk_copy_g2s_hint(ring + (size_t)st * SC::STAGE_BYTES, src + (int64_t)c * SC::TOK * DSEL, bytes,
                           &ms.score_full[st], pol);
    };
    if (tid == 0)
        for (int c = 0; c < min(nchunks, SC::STAGES); ++c) issue(c);

    for (int c = 0; c < nchunks; ++c) {
        const int st = c % SC::STAGES;
        if (!mbar_wait_bounded(&ms.score_full[st], (uint32_t)(c / SC::STAGES) & 1u))
            flag(p.status, DEV_TIMEOUT);
        const int t = c * SC::TOK + tok;
        float acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = 0.0f;
        if (t < len) {
            const uint4* kp = reinterpret_cast<const uint4*>(ring + (size_t)st * SC::STAGE_BYTES +
                                                             (size_t)tid * SC::CPT * 2);
            constexpr int NV = SC::CPT / 8;
            uint4 piece[NV];
            if constexpr (NV == 2) {
                // odd lane quads load their second 16-byte piece first: conflict-free shared loads
                const bool rot = (tid >> 2) & 1;
                const uint4 a = kp[rot ? 1 : 0];
                const uint4 c2 = kp[rot ? 0 : 1];
                piece[0] = rot ? c2 : a;
                piece[1] = rot ? a : c2;
            } else {
                piece[0] = kp[0];
            }
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const uint4 w = piece[v];
                const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float k0 = bf16_lo(wd[i]), k1 = bf16_hi(wd[i]);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        acc[g] = fmaf(qr[g][v * 8 + 2 * i], k0, acc[g]);
                        acc[g] = fmaf(qr[g][v * 8 + 2 * i + 1], k1, acc[g]);
                    }
                }
            }
        }
#pragma unroll
        for (int o = 1; o < SC::TPT; o <<= 1)
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], o);
        if (t < len && part == 0) {
            float best = acc[0];
#pragma unroll
            for (int g = 1; g < G; ++g) best = fmaxf(best, acc[g]);
            const float s = best * p.scale;
            if (!isfinite(s)) flag(p.status, DEV_NONFINITE);
            sdst[t] = s;
            if (gdst) gdst[t] = s;
            if (hist) atomicAdd(&hist[okey(s) >> 20], 1u);
        }
        __syncthreads();
        if (tid == 0 && c + SC::STAGES < nchunks) issue(c + SC::STAGES);
    }
}

// ---------------------------------------------------------------------------
// phase 6: corrected attention over a share of the selected list
// ---------------------------------------------------------------------------

template <int G, int D>
struct AttCfg {
    static constexpr int DPL = (G <= 4) ? 8 : 4;             // dims per lane
    static constexpr int LPR = D / DPL;                      // lanes per row
    static constexpr int RPW = 32 / LPR;                     // rows per warp per batch
    static constexpr int RB = kWarps * RPW;                  // rows per batch
    static constexpr uint32_t ROW_BYTES = D * 2u;
    static constexpr uint32_t BATCH_BYTES = (uint32_t)RB * 2u * ROW_BYTES;
    static_assert(RB <= 64, "att_logp holds 64 rows per stage");
    static_assert(kAttendStages * BATCH_BYTES <= kRingBytes, "attend ring too large");
    static_assert((size_t)kWarps * G * D * 4 <= kRingBytes, "warp partials do not fit");
};

template <int G, int D>
__device__ void phase_attend(const Params& p, cg::cluster_group& cluster, unsigned char* ring, float* cpart,
                             Misc& ms, int b, int h, int rank, int C, int64_t count_u,
                             const int32_t* idx_list, const float* p_list)
{
    using AC = AttCfg<G, D>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t lo = count_u * rank / C, hi = count_u * (rank + 1) / C;
    const int rows = (int)(hi - lo);
    const int nbatch = (rows + AC::RB - 1) / AC::RB;
    const uint16_t* Kb = p.K + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;
    const uint16_t* Vb = p.V + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh;

    fence_proxy_async_smem();
    __syncthreads();

    auto issue = [&](int j) {  // warp 0
        const int st = j % kAttendStages;
        unsigned char* kdst = ring + (size_t)st * AC::BATCH_BYTES;
        unsigned char* vdst = kdst + (size_t)AC::RB * AC::ROW_BYTES;
        int64_t tok[2] = {0, 0};
        bool ok[2] = {false, false};
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            const int r = lane + 32 * k2;
            if (r < AC::RB) {
                const int64_t gr = lo + (int64_t)j * AC::RB + r;
                float lp = __int_as_float(0x7f800000);  // +inf marks an empty slot
                if (gr < hi) {
                    const int32_t i = __ldcg(idx_list + gr);
                    const float pv = __ldcg(p_list + gr);
                    if (i < 0 || (int64_t)i >= p.N || !(pv > 0.0f) || !(pv <= 1.0f)) {
                        flag(p.status, DEV_BAD_INDEX);
                    } else {
                        lp = logf(pv);
                        tok[k2] = i;
                        ok[k2] = true;
                    }
                }
                ms.att_logp[st][r] = lp;
            }
        }
        const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, ok[0])) + __popc(__ballot_sync(0xffffffffu, ok[1]));
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&ms.att_full[st], nvalid * 2u * AC::ROW_BYTES);
        __syncwarp();
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            if (ok[k2]) {
                const int r = lane + 32 * k2;
                bulk_copy_g2s(kdst + (size_t)r * AC::ROW_BYTES, Kb + tok[k2] * D, AC::ROW_BYTES, &ms.att_full[st]);
                bulk_copy_g2s(vdst + (size_t)r * AC::ROW_BYTES, Vb + tok[k2] * D, AC::ROW_BYTES, &ms.att_full[st]);
            }
        }
    };

    const int sub = lane / AC::LPR, li = lane % AC::LPR;
    float qv[G][AC::DPL];
    {
        const uint16_t* qb = p.q + ((int64_t)b * p.Hq + (int64_t)h * G) * D + li * AC::DPL;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < AC::DPL; ++c) qv[g][c] = bf16_at(qb + (int64_t)g * D + c);
    }
    float mrun[G], lrun[G], acc[G][AC::DPL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        mrun[g] = -INFINITY;
        lrun[g] = 0.0f;
#pragma unroll
        for (int c = 0; c < AC::DPL; ++c) acc[g][c] = 0.0f;
    }

    if (warp == 0)
        for (int j = 0; j < min(nbatch, kAttendStages); ++j) issue(j);

    for (int j = 0; j < nbatch; ++j) {
        const int st = j % kAttendStages;
        if (!mbar_wait_bounded(&ms.att_full[st], (uint32_t)(j / kAttendStages) & 1u))
            flag(p.status, DEV_TIMEOUT);
        const int r = warp * AC::RPW + sub;
        const float lp = ms.att_logp[st][r];
        const bool valid = lp != __int_as_float(0x7f800000);
        const unsigned char* krow = ring + (size_t)st * AC::BATCH_BYTES + (size_t)r * AC::ROW_BYTES + li * AC::DPL * 2;
        const unsigned char* vrow = krow + (size_t)AC::RB * AC::ROW_BYTES;
        float kf[AC::DPL], vf[AC::DPL];
        if constexpr (AC::DPL == 8) {
            const uint4 kw = *reinterpret_cast<const uint4*>(krow);
            const uint4 vw = *reinterpret_cast<const uint4*>(vrow);
            const uint32_t ka[4] = {kw.x, kw.y, kw.z, kw.w}, va[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                kf[2 * i] = bf16_lo(ka[i]);
                kf[2 * i + 1] = bf16_hi(ka[i]);
                vf[2 * i] = bf16_lo(va[i]);
                vf[2 * i + 1] = bf16_hi(va[i]);
            }
        } else {
            const uint2 kw = *reinterpret_cast<const uint2*>(krow);
            const uint2 vw = *reinterpret_cast<const uint2*>(vrow);
            kf[0] = bf16_lo(kw.x); kf[1] = bf16_hi(kw.x); kf[2] = bf16_lo(kw.y); kf[3] = bf16_hi(kw.y);
            vf[0] = bf16_lo(vw.x); vf[1] = bf16_hi(vw.x); vf[2] = bf16_lo(vw.y); vf[3] = bf16_hi(vw.y);
        }
        float dot[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float s = 0.0f;
#pragma unroll
            for (int c = 0; c < AC::DPL; ++c) s = fmaf(qv[g][c], kf[c], s);
            dot[g] = s;
        }
#pragma unroll
        for (int o = AC::LPR / 2; o > 0; o >>= 1)
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
                    for (int c = 0; c < AC::DPL; ++c) acc[g][c] *= a;
                    mrun[g] = x;
                }
                const float w = expf(x - mrun[g]);
                lrun[g] += w;
#pragma unroll
                for (int c = 0; c < AC::DPL; ++c) acc[g][c] = fmaf(w, vf[c], acc[g][c]);
            }
        }
        __syncthreads();
        if (warp == 0 && j + kAttendStages < nbatch) issue(j + kAttendStages);
    }

    // merge the row streams of one warp (lanes li, li + LPR, ...)
#pragma unroll
    for (int o = AC::LPR; o < 32; o <<= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float mo = __shfl_xor_sync(0xffffffffu, mrun[g], o);
            const float lo_ = __shfl_xor_sync(0xffffffffu, lrun[g], o);
            const float M = fmaxf(mrun[g], mo);
            const float a = (mrun[g] == -INFINITY) ? 0.0f : expf(mrun[g] - M);
            const float ao = (mo == -INFINITY) ? 0.0f : expf(mo - M);
            lrun[g] = lrun[g] * a + lo_ * ao;
#pragma unroll
            for (int c = 0; c < AC::DPL; ++c) {
                const float xo = __shfl_xor_sync(0xffffffffu, acc[g][c], o);
                acc[g][c] = acc[g][c] * a + xo * ao;
            }
            mrun[g] = M;
        }
    }
    float* wpart = reinterpret_cast<float*>(ring);   // [kWarps][G][D]
    if (lane < AC::LPR) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < AC::DPL; ++c) wpart[((size_t)warp * G + g) * D + li * AC::DPL + c] = acc[g][c];
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            ms.wm[warp][g] = mrun[g];
            ms.wl[warp][g] = lrun[g];
        }
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += kThreads) {
        const int g = i / D, c = i % D;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ms.wm[w][g]);
        float A = 0.0f, Ls = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < kWarps; ++w) {
                const float mw = ms.wm[w][g];
                if (mw == -INFINITY) continue;
                const float e = expf(mw - M);
                A = fmaf(wpart[((size_t)w * G + g) * D + c], e, A);
                Ls = fmaf(ms.wl[w][g], e, Ls);
            }
        }
        cpart[i] = A;
        if (c == 0) {
            ms.cm[g] = M;
            ms.cl[g] = Ls;
        }
    }
    if (C > 1) cluster.sync(); else __syncthreads();
    const int per = (G * D) / C;
    for (int i = rank * per + tid; i < (rank + 1) * per; i += kThreads) {
        const int g = i / D, c = i % D;
        float M = -INFINITY;
        for (int r = 0; r < C; ++r) M = fmaxf(M, *cluster.map_shared_rank(&ms.cm[g], r));
        float A = 0.0f, Ls = 0.0f;
        if (M != -INFINITY) {
            for (int r = 0; r < C; ++r) {
                const float mr = *cluster.map_shared_rank(&ms.cm[g], r);
                if (mr == -INFINITY) continue;
                const float e = expf(mr - M);
                A = fmaf(*cluster.map_shared_rank(&cpart[i], r), e, A);
                Ls = fmaf(*cluster.map_shared_rank(&ms.cl[g], r), e, Ls);
            }
        }
        const int64_t head = (int64_t)b * p.Hq + (int64_t)h * G + g;
        p.out[head * D + c] = (Ls > 0.0f) ? A / Ls : 0.0f;
        if (c == 0) p.lse[head] = (Ls > 0.0f) ? M + logf(Ls) : -INFINITY;
    }
    if (C > 1) cluster.sync();
}

// ---------------------------------------------------------------------------
// the unit kernel
// ---------------------------------------------------------------------------

template <int G, int DSEL, int D, int MODE, bool RES>
__global__ void __launch_bounds__(kThreads, 1) unit_kernel(const __grid_constant__ Params p)
{
    constexpr bool SCORE = (MODE & MODE_SCORE) != 0;
    constexpr bool SELECT = (MODE & MODE_SELECT) != 0;
    constexpr bool ATTEND = (MODE & MODE_ATTEND) != 0;
    extern __shared__ __align__(1024) unsigned char smem[];

    const Layout L = make_layout(MODE, RES, p.seg_len, p.C);
    Misc& ms = *reinterpret_cast<Misc*>(smem + L.misc);
    cg::cluster_group cluster = cg::this_cluster();
    const int C = p.C;
    const int rank = (int)(blockIdx.x % (unsigned)C);
    const int unit = (int)(blockIdx.x / (unsigned)C);
    const int b = unit / p.Hkv, h = unit % p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t N = p.N;
    const int64_t s0 = min(N, (int64_t)rank * p.seg_len);
    const int len = (int)(min(N, s0 + p.seg_len) - s0);
    unsigned char* ring = smem + L.ring;
    uint32_t* histA = reinterpret_cast<uint32_t*>(smem + L.histA);
    uint32_t* histB = reinterpret_cast<uint32_t*>(smem + L.histB);
    float* sbuf = reinterpret_cast<float*>(smem + L.sbuf);

    if (tid == 0) {
        for (int i = 0; i < kMaxScoreStages; ++i) mbar_init(&ms.score_full[i], 1);
        for (int i = 0; i < kAttendStages; ++i) mbar_init(&ms.att_full[i], 1);
        fence_mbar_init();
    }
    if constexpr (SELECT) {
        for (int i = tid; i < kBins; i += kThreads) {
            histA[i] = 0u;
            histB[i] = 0u;
        }
    }
    __syncthreads();

    // --- scores of this CTA's segment -------------------------------------
    const float* S = nullptr;  // segment-relative scores
    if constexpr (SCORE) {
        float* gseg = p.s_out ? p.s_out + (int64_t)unit * N + s0 : nullptr;
        if constexpr (SELECT && RES) {
            phase_score<G, DSEL>(p, ring, ms, b, h, s0, len, sbuf, gseg, histA);
            S = sbuf;
        } else {
            phase_score<G, DSEL>(p, ring, ms, b, h, s0, len, gseg, nullptr, SELECT ? histA : nullptr);
            S = gseg;
        }
        if constexpr (!SELECT && !ATTEND) return;
    } else if constexpr (SELECT) {
        const float* gin = p.s_in + (int64_t)unit * N + s0;
        for (int t = tid; t < len; t += kThreads) {
            const float s = gin[t];
            if (!isfinite(s)) flag(p.status, DEV_NONFINITE);
            if constexpr (RES) sbuf[t] = s;
            atomicAdd(&histA[okey(s) >> 20], 1u);
        }
        S = RES ? sbuf : gin;
    }

    int64_t count_u = 0;
    if constexpr (SELECT) {
        const bool everything = (p.top_k >= N) || isinf(p.budget);
        uint32_t theta = 0u;
        int idx_cut = -1;
        float m = 0.0f, Zf = 0.0f;
        if (!everything && N > 0) {
            uint32_t* merged = reinterpret_cast<uint32_t*>(smem + L.merged);
            const uint32_t target = (uint32_t)(p.top_k > 0 ? p.top_k : 1);
            const Found f1 = level_find(cluster, histA, kBins, target, C, rank, merged, ms, p.status);
            for (int i = tid; i < kBins3; i += kThreads) histA[i] = 0u;   // level-3 histogram
            for (int t = tid; t < len; t += kThreads) {
                const uint32_t k = okey(S[t]);
                if ((k >> 20) == f1.bin) atomicAdd(&histB[(k >> 8) & 0xfffu], 1u);
            }
            const Found f2 = level_find(cluster, histB, kBins, target - f1.above, C, rank, merged, ms, p.status);
            const uint32_t pre24 = (f1.bin << 12) | f2.bin;
            for (int t = tid; t < len; t += kThreads) {
                const uint32_t k = okey(S[t]);
                if ((k >> 8) == pre24) atomicAdd(&histA[k & 0xffu], 1u);
            }
            const Found f3 = level_find(cluster, histA, kBins3, target - f1.above - f2.above, C, rank, merged,
                                        ms, p.status);
            theta = (pre24 << 8) | f3.bin;
            m = okey_value(theta);
            const int64_t c_gt = (int64_t)f1.above + f2.above + f3.above;

            // ties at theta: the lowest indices go to the top-k stratum
            const uint32_t eq_local = histA[f3.bin];
            uint32_t tie_off = 0;
            if (C > 1) {
                if (warp == 0) {
                    uint32_t v = (lane < rank) ? cluster.map_shared_rank(histA, lane)[f3.bin] : 0u;
                    v = warp_sum_u32(v);
                    if (lane == 0) ms.bcast[6] = v;
                }
                __syncthreads();
                tie_off = ms.bcast[6];
            }
            const int64_t need = (p.top_k > 0) ? p.top_k - c_gt : 0;
            int64_t ln = need - (int64_t)tie_off;
            ln = ln < 0 ? 0 : (ln > (int64_t)eq_local ? (int64_t)eq_local : ln);
            if (ln == 0) idx_cut = -1;
            else if (ln == (int64_t)eq_local) idx_cut = 0x7fffffff;
            else idx_cut = find_nth_tie(S, len, theta, (uint32_t)ln, (int)(p.seg_len / kWarps), ms);

            // exact normaliser over the remainder
            if (p.budget > 0.0f) {
                unsigned long long z[5] = {0ull, 0ull, 0ull, 0ull, 0ull};
                for (int t = tid; t < len; t += kThreads) {
                    const float s = S[t];
                    const uint32_t k = okey(s);
                    const bool inT = k > theta || (k == theta && t <= idx_cut);
                    if (!inT) exact_add(z, expf(__fsub_rn(s, m)), p.status);
                }
#pragma unroll
                for (int i = 0; i < 5; ++i) {
                    unsigned long long v = z[i];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) ms.zwarp[warp][i] = v;
                }
                __syncthreads();
                if (tid < 5) {
                    unsigned long long v = 0;
                    for (int w = 0; w < kWarps; ++w) v += ms.zwarp[w][tid];
                    ms.zpart[tid] = v;
                }
                if (C > 1) cluster.sync(); else __syncthreads();
                if (warp == 0) {
                    unsigned long long zz[5];
#pragma unroll
                    for (int i = 0; i < 5; ++i) {
                        unsigned long long v = (lane < C) ? cluster.map_shared_rank(&ms.zpart[0], lane)[i] : 0ull;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                        zz[i] = v;
                    }
                    if (lane == 0) ms.fbcast[0] = exact_to_float(zz);
                }
                __syncthreads();
                Zf = ms.fbcast[0];
            }
        }

        // decisions: one ballot mask per 32-token strip
        uint32_t* bits = reinterpret_cast<uint32_t*>(smem + L.bits);
        const int W = (int)(p.seg_len / kWarps);
        const int nstrip = W / 32;
        const int base = warp * W;
        const bool sampling = !everything && p.budget > 0.0f && Zf > 0.0f;
        uint32_t cnt = 0;
        for (int st = 0; st < nstrip; ++st) {
            const int pos = base + st * 32 + lane;
            bool sel = false;
            if (pos < len) {
                if (everything) {
                    sel = true;
                } else {
                    const float s = S[pos];
                    const uint32_t k = okey(s);
                    if (k > theta || (k == theta && pos <= idx_cut)) {
                        sel = true;
                    } else if (sampling) {
                        const float pr = inclusion_prob(s, m, p.budget, Zf);
                        if (pr > 0.0f) sel = token_uniform(p.seed, s0 + pos, h, b) < pr;
                    }
                }
            }
            const uint32_t mask = __ballot_sync(0xffffffffu, sel);
            if (lane == 0) bits[warp * nstrip + st] = mask;
            cnt += __popc(mask);
        }
        if (lane == 0) ms.warp_u32[warp] = cnt;
        __syncthreads();
        uint32_t warp_off = 0, cta_total = 0;
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t t = ms.warp_u32[w];
            warp_off += (w < warp) ? t : 0u;
            cta_total += t;
        }
        __syncthreads();
        if (tid == 0) ms.cta_count = cta_total;
        if (C > 1) cluster.sync(); else __syncthreads();
        if (warp == 0) {
            const uint32_t v = (lane < C) ? *cluster.map_shared_rank(&ms.cta_count, lane) : 0u;
            const uint32_t before = warp_sum_u32(lane < rank ? v : 0u);
            const uint32_t total = warp_sum_u32(v);
            if (lane == 0) {
                ms.bcast[8] = before;
                ms.bcast[9] = total;
            }
        }
        __syncthreads();
        const int64_t my_off = ms.bcast[8];
        count_u = ms.bcast[9];
        int32_t* idx_u = p.idx + (int64_t)unit * p.cap;
        float* p_u = p.p + (int64_t)unit * p.cap;
        uint32_t run = 0;
        bool over = false;
        for (int st = 0; st < nstrip; ++st) {
            const uint32_t mask = bits[warp * nstrip + st];
            if ((mask >> lane) & 1u) {
                const int pos = base + st * 32 + lane;
                const int64_t o = my_off + warp_off + run + __popc(mask & lanemask_lt());
                float pr = 1.0f;
                if (!everything) {
                    const float s = S[pos];
                    const uint32_t k = okey(s);
                    if (!(k > theta || (k == theta && pos <= idx_cut))) pr = inclusion_prob(s, m, p.budget, Zf);
                }
                if (o < p.cap) {
                    idx_u[o] = (int32_t)(s0 + pos);
                    p_u[o] = pr;
                } else {
                    over = true;
                }
            }
            run += __popc(mask);
        }
        if (over) flag(p.status, DEV_OVERFLOW);
        if (rank == 0 && tid == 0 && p.count) p.count[unit] = (int32_t)count_u;
        if constexpr (ATTEND) {
            if (C > 1) cluster.sync(); else __syncthreads();
        }
    } else if constexpr (ATTEND) {
        int64_t c = p.count[unit];
        count_u = c < 0 ? 0 : (c > p.cap ? p.cap : c);
    }

    if constexpr (ATTEND) {
        if (count_u > p.cap) count_u = p.cap;
        phase_attend<G, D>(p, cluster, ring, reinterpret_cast<float*>(smem + L.histB), ms, b, h, rank, C,
                           count_u, p.idx + (int64_t)unit * p.cap, p.p + (int64_t)unit * p.cap);
    } else if constexpr (SELECT) {
        if (C > 1) cluster.sync();   // peers may still read this CTA's shared memory
    }
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
