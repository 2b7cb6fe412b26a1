// common.cuh -- shared definitions of the libssa kernels: the work plan, the
// workspace layout, the per-unit control block and small device helpers.
//
// A "unit" is one (batch b, KV head h_kv) pair; u = b * Hkv + h_kv.  One
// decode step runs three kernels on the caller's stream (programmatic
// dependent launch lets each start while the previous one drains):
//   K0 init     zero the per-unit counters and histograms (K1 starts at
//               once and waits for K0 only before its first histogram flush);
//   K1 score    every SM streams the key summary (TMA) and scores it on the
//               tensor cores; order-key histogram; 16-bit Philox prefixes;
//   K2 unit     a group of CTAs per unit, one per tile of the unit's tokens:
//               each CTA finds the bucket of the k-th score, lists every
//               token above it, its members (candidates) and the remainder
//               tokens that can still be drawn, and sums its share of the
//               normaliser; once every tile has arrived (a counter in the
//               unit's control block) every CTA resolves the exact k-th token
//               and Z (the same computation in each), decides its listed
//               tokens (top-k stratum, or the draw u < p), gathers the
//               kept K/V rows and runs the corrected attention on the tensor
//               cores; the last CTA of the unit merges the (m, l, acc)
//               partials.  The grid is one wave (every unit's CTAs resident
//               at once) and every wait has a time limit.
// K1 and K2 have separate instantiations for a paged cache (page pools and
// a block table), and K2 one for the early-stop attention, which follows an
// ordering kernel (one CTA per unit sorts its list by score).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

// Phase markers: no-ops unless a profiling build defines SSA_MARK(k) to
// record a timestamp for phase boundary k (SSA_MARKG(k) inside a loop, and
// SSA_NOTE(k, v) to record a value).
#ifndef SSA_MARK
#define SSA_MARK(k) ((void)0)
#endif
#ifndef SSA_GT
#define SSA_GT(k) ((void)0)
#endif
#ifndef SSA_MARKW
#define SSA_MARKW(k) ((void)0)
#endif
#ifndef SSA_NOTE
#define SSA_NOTE(k, v) ((void)0)
#endif
#ifndef SSA_MARKG
#define SSA_MARKG(k) ((void)0)
#endif

namespace ssa {

constexpr uint32_t DEV_NONFINITE = 0x1u;
constexpr uint32_t DEV_OVERFLOW = 0x2u;
constexpr uint32_t DEV_TIMEOUT = 0x4u;
constexpr uint32_t DEV_BAD_INDEX = 0x8u;

constexpr int kBins = 4096;            // 12-bit order-key buckets
constexpr int kStageTok = 512;         // K1: tokens per pipeline stage (4 MMA tiles of 128)
constexpr int kTileAlign = 512;        // K2: tiles are multiples of 512 tokens (32 per warp slice)
constexpr int kMaxTiles = 64;          // K2: tiles (CTAs) per unit at most
constexpr int kEsMaxRows = 32768;      // early stop: rows of a unit's list the ordering kernel sorts at most
constexpr int kSelThreads = 512;       // K2 block size; in the selection each warp owns a slice (a list) of the tile
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kInThreads = 256;        // score_input_kernel block size
constexpr int kQselBytes = 1024;       // B operand: 16 rows x d_sel bf16, swizzled
// top-p stratum: per unit, mass and count histograms of three radix levels
// (12, 12 and 8 key bits), each bin three 64-bit words (mass high part, mass
// low part, count)
constexpr int kTopPBins = 4096 + 4096 + 256;
constexpr size_t kTopPUnitBytes = (size_t)kTopPBins * 3 * 8;

// Per-unit control block (zeroed by K0).
struct UnitCtrl {
    uint32_t arrive;     // K2 tiles whose selection pass is done
    uint32_t k1_next;    // unit 0 only: K1's shared stage queue (stages taken)
    uint32_t karrive;    // K2 CTAs whose kept count is written
    uint32_t done;       // K2 CTAs whose attention partial is written
    uint32_t tp_arrive[3];   // top-p stratum: K2 tiles whose mass counts of level 0 / 1 / 2 are added
    uint32_t pad[9];
};
static_assert(sizeof(UnitCtrl) == 64, "control block is 64 bytes");

// Launch geometry and workspace offsets for one shape (computed on the host).
struct Plan {
    int32_t U;           // units
    int32_t G;           // query heads per KV head
    int64_t N;           // tokens per unit
    int32_t nst;         // K1 stages per unit
    int32_t sf;          // K1 stages per unit split statically over the CTAs (the rest are queued)
    int64_t stages;      // K1 stages in all
    int32_t k1_grid;     // K1 CTAs (persistent)
    int32_t tt;          // K2 tile tokens (multiple of kTileAlign)
    int32_t ntile;       // K2 tiles per unit = its CTAs (1..kMaxTiles)
    int64_t np;          // ntile * tt: padded tokens per unit
    int32_t hist_run;    // K1: stages of one unit per shared-histogram buffer (1..127)
    // workspace byte offsets
    int32_t tcap;        // tiles the per-tile arrays hold per unit (>= ntile)
    size_t o_status, o_ctrl, o_hist1, o_zpart, o_kcnt, o_part, o_cand, o_sel_idx, o_sel_p, o_scores, o_ubuf, o_hq,
        o_hout, o_hlse, o_topp, o_es, o_esp, o_ess, total;
    int32_t esb;         // early stop: 128-row blocks a unit's ordered list holds at most
    int32_t esr;         // early stop: rows a unit's ordered list holds at most (the sort's buffers)
};

// ---------------------------------------------------------------------------
// device helpers
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
        const uint64_t pa = (uint64_t)0xD2511F53u * c0;
        const uint64_t pb = (uint64_t)0xCD9E8D57u * c2;
        c0 = (uint32_t)(pb >> 32) ^ c1 ^ k0;
        c1 = (uint32_t)pb;
        c2 = (uint32_t)(pa >> 32) ^ c3 ^ k1;
        c3 = (uint32_t)pa;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

// u = (x0 >> 8) * 2^-24 for token j of unit (b, h_kv).
__device__ __forceinline__ float token_uniform(uint64_t seed, int64_t j, int h_kv, int b)
{
    const uint32_t x0 = philox_word0((uint32_t)j, (uint32_t)h_kv, (uint32_t)b, 0u, (uint32_t)(seed & 0xffffffffu),
                                     (uint32_t)(seed >> 32));
    return __uint2float_rn(x0 >> 8) * 5.9604644775390625e-08f;
}

// p = min(1, fl32(fl32(B * e) / Z)) for a remainder token with e = expf(fl32(s - m)).
__device__ __forceinline__ float prob_from_term(float e, float budget, float Z)
{
    return fminf(__fdiv_rn(__fmul_rn(budget, e), Z), 1.0f);
}

// Error-free sum: s + err == a + b exactly (Knuth's two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& err)
{
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    const float ap = __fsub_rn(s, bp);
    err = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// (hi, lo) += (h2, l2), compensated.
__device__ __forceinline__ void comp_add(float& hi, float& lo, float h2, float l2)
{
    float s, e;
    two_sum(hi, h2, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, l2));
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// Exclusive prefix over a block of NT threads of one value per thread; also
// the total.  `scratch` holds NT / 32 words.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch, uint32_t& total)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t x = warp_incl_scan(v);
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t t = scratch[w];
        before += (w < warp) ? t : 0u;
        tot += t;
    }
    __syncthreads();
    total = tot;
    return before + x - v;
}

struct Found {
    uint32_t bin, above;
};

// counts[0..NB) are histogram bins in ascending key order.  Find the bin
// holding the t-th largest element (t >= 1): `above` = elements in higher
// bins.  Block-wide (NT threads; NB a multiple or a divisor of NT); every thread returns
// the answer.  Each thread loads its NB / NT bins at once (a global
// histogram is read through L2: other CTAs wrote it).  bcast holds 2 words,
// scratch NT / 32 words.
template <int NT, int NB, bool GLOBAL>
__device__ Found find_rank_desc(const uint32_t* counts, uint32_t t, uint32_t* scratch, uint32_t* bcast,
                                uint32_t* status)
{
    constexpr int CH = NB >= NT ? NB / NT : 1;
    static_assert(NB % NT == 0 || NT % NB == 0, "bins must split evenly over the block");
    const int tid = threadIdx.x;
    uint32_t c[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        const int pos = tid * CH + j;   // pos-th bin from the top
        c[j] = (pos < NB) ? (GLOBAL ? __ldcg(counts + (NB - 1 - pos)) : counts[NB - 1 - pos]) : 0u;
    }
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < CH; ++j) local += c[j];
    if (tid == 0) {
        bcast[0] = 0;
        bcast[1] = 0xffffffffu;
    }
    uint32_t total;
    const uint32_t excl = block_excl_scan<NT>(local, scratch, total);
    if (local > 0 && excl < t && t <= excl + local) {
        uint32_t cum = excl;
        bool done = false;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (!done && cum + c[j] >= t) {
                bcast[0] = (uint32_t)(NB - 1 - (tid * CH + j));
                bcast[1] = cum;
                done = true;
            }
            cum += c[j];
        }
    }
    __syncthreads();
    Found f{bcast[0], bcast[1]};
    if (f.above == 0xffffffffu) {   // fewer than t elements: inconsistent inputs
        if (tid == 0) flag(status, DEV_BAD_INDEX);
        f.bin = 0;
        f.above = 0;
    }
    __syncthreads();
    return f;
}

}  // namespace ssa
