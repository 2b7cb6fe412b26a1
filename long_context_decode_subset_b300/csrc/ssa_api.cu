// ssa_api.cu -- host side of libssa: argument checks, the per-shape plan and
// workspace layout, launches, and the C entry points declared in
// include/ssa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>

#include "ssa.h"
#include "k_attend.cuh"

using namespace ssa;

namespace {

constexpr size_t kStatusBytes = 256;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }
bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

int env_int(const char* name, int dflt)
{
    const char* v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : dflt;
}

int device_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 148;
    }
    return n > 0 ? n : 148;
}

// Plan and workspace layout.  The layout does not depend on the device: the
// per-unit token arrays are sized for the largest tiling (at most kMaxTiles
// tiles of 512-token multiples pad a unit by less than kMaxTiles * 512
// tokens).  The tiling itself -- the unit kernel's CTAs per unit -- and the
// score kernel's grid do depend on the device; `tiles` > 0 gives the tile
// count (the tiles are then the fewest 512-token multiples that cover N in
// that many pieces) and `fit` the most tiles per unit one wave of the unit
// kernel holds.  SSA_FORCE_TILE (tokens per tile, if its tile count fits)
// and SSA_FORCE_SPLIT (tiles per unit) override the choice (the tests use
// them to cover many tilings on small inputs), and SSA_FORCE_HIST_RUN the
// score kernel's histogram hand-over period.
constexpr int64_t kPadTokens = (int64_t)kMaxTiles * kTileAlign;

// Tiles per unit the per-tile arrays are sized for: as many as two CTAs on
// every SM of a 148-SM device could give a unit, at most kMaxTiles.
int tile_cap(int64_t U) { return (int)std::max<int64_t>(1, std::min<int64_t>(kMaxTiles, (296 + U - 1) / std::max<int64_t>(U, 1))); }

ssa::Plan make_plan(const ssa_shape& s, int tiles, int fit = 1)
{
    ssa::Plan pl{};
    pl.U = s.batch * s.n_kv_heads;
    pl.G = s.n_q_heads / s.n_kv_heads;
    pl.N = s.ctx_len;
    const int64_t U = pl.U, N = s.ctx_len;
    pl.nst = (int32_t)((N + kStageTok - 1) / kStageTok);
    pl.stages = U * pl.nst;
    pl.sf = (int32_t)((int64_t)pl.nst * 3 / 4);   // the rest of each unit goes to K1's shared queue
    const int sms = tiles > 0 ? device_sms() : 148;
    pl.k1_grid = (int32_t)std::max<int64_t>(1, std::min<int64_t>(sms, pl.stages));
    const int64_t cmax = std::max<int64_t>(1, std::min<int64_t>(tile_cap(U), (N + kTileAlign - 1) / kTileAlign));
    int64_t c = std::max<int64_t>(1, std::min<int64_t>(tiles > 0 ? tiles : 1, cmax));
    int64_t tt = std::max<int64_t>(kTileAlign, ((N + c - 1) / c + kTileAlign - 1) / kTileAlign * kTileAlign);
    const int forced_tile = env_int("SSA_FORCE_TILE", 0);
    if (tiles > 0 && forced_tile >= kTileAlign && forced_tile % kTileAlign == 0 &&
        (N + forced_tile - 1) / forced_tile <= std::min<int64_t>(fit, tile_cap(U)) &&   // one wave
        (N + forced_tile - 1) / forced_tile * forced_tile < N + kPadTokens)   // within the sized padding
        tt = forced_tile;
    pl.tt = (int32_t)tt;
    pl.ntile = (int32_t)std::max<int64_t>(1, (N + tt - 1) / tt);
    pl.np = (int64_t)pl.ntile * tt;
    pl.tcap = tile_cap(U);
    // K1's histogram buffers are handed over after at most kHistRun stages of
    // one unit; SSA_FORCE_HIST_RUN lowers that (the tests use it to hand
    // buffers over at every stage or two)
    pl.hist_run = kHistRun;
    const int forced_run = env_int("SSA_FORCE_HIST_RUN", 0);
    if (forced_run >= 1 && forced_run <= kHistRun) pl.hist_run = forced_run;

    const int64_t D = s.head_dim, G = pl.G;
    const int64_t heads = (int64_t)s.batch * s.n_q_heads;
    const int64_t npmax = N + kPadTokens;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += align256(bytes);
        return at;
    };
    pl.o_status = take(kStatusBytes);
    pl.o_ctrl = take((size_t)U * sizeof(UnitCtrl));
    pl.o_hist1 = take((size_t)U * kBins * 4 * 2);   // level-1 then level-2 histograms
    pl.o_zpart = take((size_t)U * pl.tcap * 16);
    pl.o_kcnt = take((size_t)U * pl.tcap * 4);
    pl.o_part = take((size_t)U * pl.tcap * (size_t)(G * D + 2 * G) * 4);
    pl.o_cand = take((size_t)U * N * 8);
    pl.o_sel_idx = take((size_t)U * npmax * 4);
    pl.o_sel_p = take((size_t)U * npmax * 4);
    pl.o_scores = take((size_t)U * N * 4);
    pl.o_ubuf = take((size_t)U * npmax * 2);
    pl.o_hq = take((size_t)heads * D * 2);
    pl.o_hout = take((size_t)heads * D * 4);
    pl.o_hlse = take((size_t)heads * 4);
    pl.o_topp = take((size_t)U * kTopPUnitBytes);
    pl.o_es = take((size_t)U * 4);
    // early stop: every block's (acc, m, l) partial (sized, like the token
    // arrays, for the largest tiling: the layout does not depend on the plan)
    pl.esb = (int32_t)((std::min<int64_t>(kEsMaxRows, npmax) + 127) / 128);
    pl.o_esp = take((size_t)U * pl.esb * (size_t)(G * D + 2 * G) * 4);
    // early stop: the order kernel's two arrays of (key, position) per unit
    pl.esr = (int32_t)std::min<int64_t>(kEsMaxRows, npmax);
    pl.o_ess = take((size_t)U * 2 * pl.esr * 8);
    pl.total = o;
    return pl;
}

// Which stride fields a shape must carry: a contiguous cache's, all zero (a
// paged cache), or either (the calls that only size things).
enum StrideRule { kStridesContig, kStridesZero, kStridesAny };

bool zero_strides(const ssa_shape* s)
{
    return s->kv_stride_b == 0 && s->kv_stride_h == 0 && s->ks_stride_b == 0 && s->ks_stride_h == 0;
}

ssa_status check_shape(const ssa_shape* s, StrideRule rule = kStridesContig)
{
    if (!s) return SSA_ERR_INVALID_ARG;
    if (s->batch < 0 || s->n_kv_heads < 1 || s->n_q_heads < 1 || s->reserved != 0) return SSA_ERR_INVALID_ARG;
    if (s->n_q_heads % s->n_kv_heads != 0) return SSA_ERR_INVALID_ARG;
    const int G = s->n_q_heads / s->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SSA_ERR_UNSUPPORTED;
    if (s->head_dim != 64 && s->head_dim != 128) return SSA_ERR_UNSUPPORTED;
    if (s->d_sel != 16 && s->d_sel != 32) return SSA_ERR_UNSUPPORTED;
    if (s->ctx_len < 0 || s->ctx_len > (int64_t)INT32_MAX - 4096) return SSA_ERR_INVALID_ARG;
    if ((int64_t)s->batch * s->n_kv_heads > (int64_t)INT32_MAX / (kMaxTiles * 2)) return SSA_ERR_UNSUPPORTED;
    if (rule != kStridesContig && zero_strides(s)) return SSA_OK;
    if (rule == kStridesZero) return SSA_ERR_INVALID_ARG;
    const int64_t N = s->ctx_len;
    if (s->kv_stride_h < N * s->head_dim || s->ks_stride_h < N * s->d_sel) return SSA_ERR_INVALID_ARG;
    if (s->kv_stride_b < (int64_t)(s->n_kv_heads - 1) * s->kv_stride_h + N * s->head_dim) return SSA_ERR_INVALID_ARG;
    if (s->ks_stride_b < (int64_t)(s->n_kv_heads - 1) * s->ks_stride_h + N * s->d_sel) return SSA_ERR_INVALID_ARG;
    if (s->kv_stride_h % 8 || s->kv_stride_b % 8 || s->ks_stride_h % 8 || s->ks_stride_b % 8)
        return SSA_ERR_INVALID_ARG;
    return SSA_OK;
}

ssa_status check_ws(void* ws, size_t ws_bytes, const ssa::Plan& pl)
{
    if (!ws || !aligned(ws, 256)) return SSA_ERR_WORKSPACE;
    if (ws_bytes < pl.total) return SSA_ERR_WORKSPACE;
    return SSA_OK;
}

// Whether the device can read `ptr` directly: device (or managed) memory, or
// pinned host memory mapped into the device's address space at the same
// address (the K/V rows of the host-resident memory tier).  Pageable host
// memory is refused: a kernel reading it would fault.  `host_ok` false
// refuses host memory as well.
bool device_readable(const void* ptr, bool host_ok)
{
    if (!ptr) return true;   // null pointers are checked where they matter
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
    return host_ok && a.type == cudaMemoryTypeHost && a.devicePointer == ptr;
}

bool bad_scalars(int64_t top_k, float budget) { return top_k < 0 || !(budget >= 0.0f); }
bool bad_strata(int strata, float top_p)
{
    return strata < SSA_STRATA_SSA || strata > SSA_STRATA_TOP_P || !(top_p >= 0.0f) || std::isnan(top_p);
}

// The strata of a step.  Strata 1 keeps every remainder token with
// p = min(1, B / (N - min(k, N))), i.e. e = 1 and Z = N - min(k, N).  Top-p
// with top_p <= 0 is the SSA step with k = 0, with top_p >= 1 the step that
// keeps every token; otherwise the unit kernel finds each unit's stratum size
// (p.top_k is then only a nonzero placeholder).  Returns the k the host's
// dense test uses.
int64_t set_strata(ssa::Params& p, int strata, int64_t top_k, float top_p, int64_t N)
{
    p.strata = 0;
    if (strata == SSA_STRATA_UNIFORM) {
        p.strata = 1;
    } else if (strata == SSA_STRATA_TOP_P) {
        if (!(top_p > 0.0f)) top_k = 0;
        else if (top_p >= 1.0f) top_k = std::max<int64_t>(N, 1);
        else {
            p.strata = 2;
            p.top_p = top_p;
            top_k = 1;
        }
    }
    p.top_k = top_k;
    return top_k;
}
bool bad_scale(float scale) { return !(scale > 0.0f) || !std::isfinite(scale); }

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// The key summary [Bt][Hkv][N][d_sel] as a 4-D tensor for TMA: boxes of
// 256 tokens x d_sel channels, swizzled to the row width (64 or 32 bytes)
// so that the tensor cores read them as K-major operands.
ssa_status encode_summary_map(CUtensorMap* map, const ssa_bf16* Ks, const ssa_shape& s)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return SSA_ERR_CUDA;
    cuuint64_t dims[4] = {(cuuint64_t)s.d_sel, (cuuint64_t)s.ctx_len, (cuuint64_t)s.n_kv_heads, (cuuint64_t)s.batch};
    cuuint64_t strides[3] = {(cuuint64_t)s.d_sel * 2, (cuuint64_t)s.ks_stride_h * 2, (cuuint64_t)s.ks_stride_b * 2};
    cuuint32_t box[4] = {(cuuint32_t)s.d_sel, 256u, 1u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<ssa_bf16*>(Ks), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           s.d_sel == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SSA_OK : SSA_ERR_CUDA;
}

// A paged summary pool [num_pages][Hkv][page_size][d_sel] as a 4-D tensor:
// boxes of min(page_size, 256) tokens of one page and head, swizzled as above
// (a box lands where the 256-token box would put its rows).
ssa_status encode_paged_map(CUtensorMap* map, const ssa_bf16* Ks_pool, const ssa_paged_kv& pg, const ssa_shape& s)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return SSA_ERR_CUDA;
    const cuuint64_t row = (cuuint64_t)s.d_sel * 2;
    cuuint64_t dims[4] = {(cuuint64_t)s.d_sel, (cuuint64_t)pg.page_size, (cuuint64_t)s.n_kv_heads,
                          (cuuint64_t)pg.num_pages};
    cuuint64_t strides[3] = {row, row * (cuuint64_t)pg.page_size, row * (cuuint64_t)pg.page_size * s.n_kv_heads};
    cuuint32_t box[4] = {(cuuint32_t)s.d_sel, (cuuint32_t)std::min(pg.page_size, 256), 1u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<ssa_bf16*>(Ks_pool), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           s.d_sel == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SSA_OK : SSA_ERR_CUDA;
}

int log2_exact(int64_t v)
{
    int l = 0;
    while (((int64_t)1 << l) < v) ++l;
    return l;
}

// A paged cache's description, checked against the shape.
ssa_status check_paged(const ssa_paged_kv* pg, const ssa_shape& s)
{
    if (!pg || !pg->block_table || !pg->seq_lens) return SSA_ERR_INVALID_ARG;
    const int64_t ps = pg->page_size;
    if (ps < 16 || ps > (1 << 20) || (ps & (ps - 1)) != 0) return SSA_ERR_INVALID_ARG;
    if (pg->max_pages < 1 || pg->num_pages < 1) return SSA_ERR_INVALID_ARG;
    if (pg->num_pages > (int64_t)INT32_MAX / ps) return SSA_ERR_INVALID_ARG;   // pool tokens fit 31 bits
    if (s.ctx_len > (int64_t)pg->max_pages * ps) return SSA_ERR_INVALID_ARG;
    return SSA_OK;
}

typedef void (*kfn_t)(ssa::Params);

template <int G, int DSEL, bool PAGED>
kfn_t pick_score_hd(bool hist)
{
    return hist ? &score_kernel<G, DSEL, true, true, PAGED> : &score_kernel<G, DSEL, false, false, PAGED>;
}

template <bool PAGED>
kfn_t pick_score_p(int G, int dsel, bool hist)
{
    switch (G) {
        case 1: return dsel == 16 ? pick_score_hd<1, 16, PAGED>(hist) : pick_score_hd<1, 32, PAGED>(hist);
        case 2: return dsel == 16 ? pick_score_hd<2, 16, PAGED>(hist) : pick_score_hd<2, 32, PAGED>(hist);
        case 4: return dsel == 16 ? pick_score_hd<4, 16, PAGED>(hist) : pick_score_hd<4, 32, PAGED>(hist);
        default: return dsel == 16 ? pick_score_hd<8, 16, PAGED>(hist) : pick_score_hd<8, 32, PAGED>(hist);
    }
}

// The score kernel for this group size, summary width, histogram choice and cache layout.
kfn_t pick_score(int G, int dsel, bool hist, bool paged)
{
    return paged ? pick_score_p<true>(G, dsel, hist) : pick_score_p<false>(G, dsel, hist);
}

template <int G, int VAR>
kfn_t unit_fn(int d, uint32_t* smem)
{
    if (d == 128) {
        *smem = unit_smem_bytes<G, 128, 4096, VAR == kVarPaged>();
        return &unit_kernel<G, 128, 4096, VAR>;
    }
    *smem = unit_smem_bytes<G, 64, 4096, VAR == kVarPaged>();
    return &unit_kernel<G, 64, 4096, VAR>;
}

template <int VAR>
kfn_t pick_unit_v(int G, int d, uint32_t* smem)
{
    switch (G) {
        case 1: return unit_fn<1, VAR>(d, smem);
        case 2: return unit_fn<2, VAR>(d, smem);
        case 4: return unit_fn<4, VAR>(d, smem);
        default: return unit_fn<8, VAR>(d, smem);
    }
}

// The unit kernel for this group size, head_dim and variant (kVarContig,
// kVarPaged, kVarEarlyStop), and its dynamic shared memory.
kfn_t pick_unit(int G, int d, uint32_t* smem, int var = kVarContig)
{
    switch (var) {
        case kVarPaged: return pick_unit_v<kVarPaged>(G, d, smem);
        case kVarEarlyStop: return pick_unit_v<kVarEarlyStop>(G, d, smem);
        default: return pick_unit_v<kVarContig>(G, d, smem);
    }
}

// Raise `fn`'s dynamic shared-memory limit to `smem` (static plus dynamic
// above 48 KB needs it); remembered per kernel, per device.
bool allow_dynamic_smem(kfn_t fn, uint32_t smem)
{
    static std::mutex mu;
    static std::map<std::pair<void*, int>, uint32_t> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const auto key = std::make_pair((void*)fn, dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = done.find(key);
        if (it != done.end() && it->second >= smem) return true;
    }
    if (cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lk(mu);
    done[key] = std::max(done[key], smem);
    return true;
}

// Launch `fn` on `stream`.  Every kernel of a step after the first is a
// programmatic dependent launch: it may start while its predecessor drains
// and waits (griddepcontrol.wait) before reading its results.  The first
// kernel of a step is an ordinary launch: it starts after everything before
// it on the stream (the caller's writes of the query, say) has completed.
ssa_status launch(kfn_t fn, int64_t grid, int block, uint32_t smem, const ssa::Params& prm, cudaStream_t stream,
                  bool dependent)
{
    if (grid <= 0) return SSA_OK;
    if (grid > INT32_MAX) return SSA_ERR_UNSUPPORTED;
    if (smem > 0 && !allow_dynamic_smem(fn, smem)) return SSA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    unsigned na = 0;
    if (dependent) {
        at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? at : nullptr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, fn, prm) != cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    return SSA_OK;
}

ssa::Params base_params(const ssa_shape& s, const ssa::Plan& pl, void* ws)
{
    ssa::Params p;
    std::memset(&p, 0, sizeof p);
    p.pl = pl;
    p.Bt = s.batch;
    p.Hq = s.n_q_heads;
    p.Hkv = s.n_kv_heads;
    p.d = s.head_dim;
    p.d_sel = s.d_sel;
    p.kv_sb = s.kv_stride_b;
    p.kv_sh = s.kv_stride_h;
    p.ws = static_cast<char*>(ws);
    return p;
}

ssa_status launch_init(const ssa::Params& p, cudaStream_t stream)
{
    return launch(&init_kernel, p.pl.U, 256, 0, p, stream, false);
}

ssa_status launch_score(const ssa::Params& p, const ssa_shape& s, bool hist, cudaStream_t stream, bool dependent)
{
    const uint32_t smem = s.d_sel == 32 ? (hist ? k1_smem_bytes<32, true>() : k1_smem_bytes<32, false>())
                                        : (hist ? k1_smem_bytes<16, true>() : k1_smem_bytes<16, false>());
    return launch(pick_score(p.pl.G, s.d_sel, hist, p.paged != 0), p.pl.k1_grid, k1_threads(hist), smem, p, stream,
                  dependent);
}

// CTAs of `fn` resident per SM (cached per kernel, shared-memory size and device).
int blocks_per_sm(kfn_t fn, int block, uint32_t smem)
{
    static std::mutex mu;
    static std::map<std::tuple<void*, uint32_t, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    const auto key = std::make_tuple((void*)fn, smem, dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if ((smem > 0 && !allow_dynamic_smem(fn, smem)) ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, (const void*)fn, block, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    n = std::max(n, 1);
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = n;
    return n;
}

// The most tiles (CTAs) per unit the device holds at once with every unit
// getting the same number.  The CTAs of a unit wait on one another, so the
// unit kernel's grid must be one wave: U * tiles never exceeds this.
int unit_fit(const ssa_shape& s)
{
    const int64_t U = std::max<int64_t>(1, (int64_t)s.batch * s.n_kv_heads);
    uint32_t smem = 0;
    kfn_t fn = pick_unit(s.n_q_heads / s.n_kv_heads, s.head_dim, &smem);
    const int64_t slots = (int64_t)blocks_per_sm(fn, kSelThreads, smem) * device_sms();
    return (int)std::max<int64_t>(1, std::min<int64_t>(kMaxTiles, slots / U));
}

// The unit kernel's plan: as many tiles per unit as one wave holds, or
// SSA_FORCE_SPLIT of them (at most that many); the plan also caps the tiles
// at the 512-token pieces of the context and at the per-tile arrays.
ssa::Plan unit_plan(const ssa_shape& s)
{
    const int fit = unit_fit(s);
    const int forced = env_int("SSA_FORCE_SPLIT", 0);
    return make_plan(s, forced > 0 ? std::min(forced, fit) : fit, fit);
}

ssa_status launch_unit(const ssa::Params& p, const ssa_shape& s, cudaStream_t stream, bool dependent)
{
    uint32_t smem = 0;
    kfn_t fn = pick_unit(p.pl.G, s.head_dim, &smem, p.paged ? kVarPaged : kVarContig);
    if (smem > 227u * 1024u) return SSA_ERR_UNSUPPORTED;
    return launch(fn, (int64_t)p.pl.U * p.pl.ntile, kSelThreads, smem, p, stream, dependent);
}

// The early-stop attention after the lists are known (prm.idx_in / p_in /
// count_in / cap, scores prm.s_src): the order kernel sorts each unit's list
// into the workspace, then the unit kernel's early-stop variant attends over
// it, each CTA a run of whole 128-row blocks, and the last CTA of the unit
// applies the gain test to the blocks' partials and merges the kept ones.
// Both wait for the previous kernel.
ssa_status launch_early_stop(ssa::Params prm, const ssa_shape& s, float tau, int32_t* blocks, cudaStream_t stream)
{
    ssa_status st = launch(&order_kernel, prm.pl.U, kOrderThreads, kOrderSmem, prm, stream, true);
    if (st != SSA_OK) return st;
    char* w = prm.ws;
    prm.idx_in = reinterpret_cast<const int32_t*>(w + prm.pl.o_sel_idx);
    prm.p_in = reinterpret_cast<const float*>(w + prm.pl.o_sel_p);
    prm.count_in = reinterpret_cast<const int32_t*>(w + prm.pl.o_es);
    prm.cap = prm.pl.np;
    prm.src_mode = 2;
    prm.attend = 1;
    prm.idx_out = nullptr;
    prm.p_out = nullptr;
    prm.count_out = nullptr;
    prm.tau = tau;
    prm.blocks_out = blocks;
    uint32_t smem = 0;
    kfn_t fn = pick_unit(prm.pl.G, s.head_dim, &smem, kVarEarlyStop);
    return launch(fn, (int64_t)prm.pl.U * prm.pl.ntile, kSelThreads, smem, prm, stream, true);
}

bool bad_tau(float tau) { return !(tau >= 0.0f); }

}  // namespace

// Scratch for ssa_decode_static: one array per GPU that loads the library.
// Host code must not use its name as a device address; the address comes
// from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_static_scratch[SSA_STATIC_SCRATCH_BYTES];

namespace {

// The current CUDA context (driver entry point looked up once), or null.
CUcontext current_context()
{
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        else
            cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

// The array's device address in the current context, looked up once per
// context (a context created anew, e.g. after cudaDeviceReset, gets its own
// entry: the module and its array are loaded again there).
void* static_scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    CUcontext ctx = current_context();
    if (!ctx) {   // no context yet: the symbol lookup makes the device's primary context current
        void* tmp = nullptr;
        if (cudaGetSymbolAddress(&tmp, g_static_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        ctx = current_context();
        if (!ctx) return nullptr;
    }
    static std::mutex mu;
    static std::map<std::pair<CUcontext, int>, void*> addr;
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_pair(ctx, dev);
    auto it = addr.find(key);
    if (it != addr.end()) return it->second;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return nullptr;
    }
    addr[key] = ptr;
    return ptr;
}

}  // namespace

extern "C" {

const char* ssa_status_string(int status)
{
    switch (status) {
        case SSA_OK: return "ok";
        case SSA_ERR_INVALID_ARG: return "invalid argument";
        case SSA_ERR_UNSUPPORTED: return "unsupported shape";
        case SSA_ERR_WORKSPACE: return "workspace too small or misaligned";
        case SSA_ERR_CUDA: return "CUDA runtime error";
        case SSA_ERR_OVERFLOW: return "selection longer than list capacity";
        case SSA_ERR_NONFINITE: return "non-finite score";
        case SSA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case SSA_ERR_BAD_INDEX: return "index or channel out of range";
        default: return "unknown status";
    }
}

int ssa_version(void) { return 200; }

size_t ssa_workspace_bytes(const ssa_shape* shape, int64_t list_cap)
{
    (void)list_cap;
    if (check_shape(shape, kStridesAny) != SSA_OK) return 0;
    return make_plan(*shape, 0).total;
}

size_t ssa_select_capacity(const ssa_shape* shape)
{
    if (check_shape(shape, kStridesAny) != SSA_OK) return 0;
    return (size_t)shape->ctx_len;
}

ssa_status ssa_pack_summary(const ssa_bf16* K, const int32_t* sel_ch, ssa_bf16* Ks, void* ws, size_t ws_bytes,
                            const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!K || !sel_ch || !Ks) return SSA_ERR_INVALID_ARG;
    const ssa::Plan pl = make_plan(*shape, 0);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    const int64_t total = (int64_t)shape->batch * shape->n_kv_heads * shape->ctx_len * shape->d_sel;
    if (total == 0) return SSA_OK;
    const int threads = 256;
    const int64_t want = (total + threads - 1) / threads;
    const unsigned blocks = (unsigned)std::min<int64_t>(want, 148 * 32);
    uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + pl.o_status);
    pack_summary_kernel<<<blocks, threads, 0, stream>>>(K, sel_ch, Ks, shape->n_kv_heads, shape->head_dim,
                                                        shape->d_sel, shape->ctx_len, shape->kv_stride_b,
                                                        shape->kv_stride_h, shape->ks_stride_b,
                                                        shape->ks_stride_h, total, status);
    if (cudaGetLastError() != cudaSuccess) return SSA_ERR_CUDA;
    return SSA_OK;
}

ssa_status ssa_score(const ssa_bf16* q, const ssa_bf16* Ks, const int32_t* sel_ch, float scale, float* s_hat,
                     void* ws, size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!q || !Ks || !sel_ch || !s_hat) return SSA_ERR_INVALID_ARG;
    if (!aligned(Ks, 16) || !aligned(q, 16)) return SSA_ERR_INVALID_ARG;
    if (bad_scale(scale)) return SSA_ERR_INVALID_ARG;
    const ssa::Plan pl = make_plan(*shape, 1);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    if (shape->ctx_len == 0 || pl.U == 0) return SSA_OK;
    ssa::Params p = base_params(*shape, pl, ws);
    if ((st = encode_summary_map(&p.ks_map, Ks, *shape)) != SSA_OK) return st;
    p.q = q;
    p.sel_ch = sel_ch;
    p.scale = scale;
    p.s_dst = s_hat;
    p.src_mode = 1;   // no selection follows: K0 zeroes K1's stage queue only, no histograms
    if ((st = launch_init(p, stream)) != SSA_OK) return st;
    return launch_score(p, *shape, false, stream, true);
}

ssa_status ssa_select(const float* s_hat, int64_t top_k, float budget, uint64_t seed, int32_t* idx, float* p,
                      int32_t* count, int64_t list_cap, void* ws, size_t ws_bytes, const ssa_shape* shape,
                      cudaStream_t stream)
{
    return ssa_select_strata(s_hat, SSA_STRATA_SSA, top_k, 0.0f, budget, seed, idx, p, count, list_cap, ws, ws_bytes,
                             shape, stream);
}

ssa_status ssa_select_strata(const float* s_hat, int strata, int64_t top_k, float top_p, float budget, uint64_t seed,
                             int32_t* idx, float* p, int32_t* count, int64_t list_cap, void* ws, size_t ws_bytes,
                             const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!s_hat || !idx || !p || !count) return SSA_ERR_INVALID_ARG;
    if (bad_scalars(top_k, budget) || bad_strata(strata, top_p)) return SSA_ERR_INVALID_ARG;
    const ssa::Plan pl = unit_plan(*shape);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    if (pl.U == 0) return SSA_OK;
    ssa::Params prm = base_params(*shape, pl, ws);
    prm.s_src = s_hat;
    prm.budget = budget;
    prm.seed = seed;
    top_k = set_strata(prm, strata, top_k, top_p, shape->ctx_len);
    prm.idx_out = idx;
    prm.p_out = p;
    prm.count_out = count;
    prm.cap = list_cap > 0 ? list_cap : std::max<int64_t>(shape->ctx_len, 1);
    prm.dense = (top_k >= shape->ctx_len || std::isinf(budget)) ? 1 : 0;
    prm.src_mode = prm.dense ? 1 : 0;
    prm.attend = 0;
    // K0 zeroes the unit counters (and the histograms), the input kernel
    // counts the scores and draws the Philox prefixes, the unit kernel selects
    if ((st = launch_init(prm, stream)) != SSA_OK) return st;
    if (prm.dense) return launch_unit(prm, *shape, stream, true);   // every token, p = 1
    if ((st = launch(&score_input_kernel, (int64_t)pl.U * pl.ntile, kInThreads, 0, prm, stream, true)) != SSA_OK)
        return st;
    return launch_unit(prm, *shape, stream, true);
}

ssa_status ssa_attend(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const int32_t* idx, const float* p,
                      const int32_t* count, int64_t list_cap, float scale, float* out, float* lse, void* ws,
                      size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!q || !idx || !p || !count || !out || !lse || (shape->ctx_len > 0 && (!K || !V))) return SSA_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16) || !aligned(q, 16)) return SSA_ERR_INVALID_ARG;
    if (bad_scale(scale)) return SSA_ERR_INVALID_ARG;
    const ssa::Plan pl = unit_plan(*shape);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    if (!device_readable(K, true) || !device_readable(V, true) || !device_readable(q, false)) return SSA_ERR_INVALID_ARG;
    if (pl.U == 0) return SSA_OK;
    ssa::Params prm = base_params(*shape, pl, ws);
    prm.q = q;
    prm.K = K;
    prm.V = V;
    prm.scale = scale;
    prm.idx_in = idx;
    prm.p_in = p;
    prm.count_in = count;
    prm.cap = list_cap > 0 ? list_cap : std::max<int64_t>(shape->ctx_len, 1);
    prm.out = out;
    prm.lse = lse;
    prm.src_mode = 2;
    prm.attend = 1;
    // K0 zeroes the unit counters the CTAs of a unit meet on
    if ((st = launch_init(prm, stream)) != SSA_OK) return st;
    return launch_unit(prm, *shape, stream, true);
}

ssa_status ssa_attend_early_stop(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const int32_t* idx,
                                 const float* p, const int32_t* count, int64_t list_cap, const float* s_hat,
                                 float tau, float scale, float* out, float* lse, int32_t* blocks_opt, void* ws,
                                 size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!q || !idx || !p || !count || !s_hat || !out || !lse || (shape->ctx_len > 0 && (!K || !V)))
        return SSA_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16) || !aligned(q, 16)) return SSA_ERR_INVALID_ARG;
    if (bad_scale(scale) || bad_tau(tau)) return SSA_ERR_INVALID_ARG;
    const ssa::Plan pl = unit_plan(*shape);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    if (!device_readable(K, true) || !device_readable(V, true) || !device_readable(q, false)) return SSA_ERR_INVALID_ARG;
    if (pl.U == 0) return SSA_OK;
    ssa::Params prm = base_params(*shape, pl, ws);
    prm.q = q;
    prm.K = K;
    prm.V = V;
    prm.scale = scale;
    prm.s_src = s_hat;
    prm.idx_in = idx;
    prm.p_in = p;
    prm.count_in = count;
    prm.cap = list_cap > 0 ? list_cap : std::max<int64_t>(shape->ctx_len, 1);
    prm.out = out;
    prm.lse = lse;
    prm.src_mode = 2;
    if ((st = launch_init(prm, stream)) != SSA_OK) return st;   // zeroes the unit counters
    return launch_early_stop(prm, *shape, tau, blocks_opt, stream);
}

}  // extern "C"

namespace {

// The new token of a fused append (ssa_decode_append), or none.
struct AppendArgs {
    const ssa_bf16* k_new;
    const ssa_bf16* v_new;
    ssa_bf16* K;
    ssa_bf16* V;
    ssa_bf16* Ks;
};

void set_append(ssa::Params& p, const AppendArgs& a, int64_t pos, const ssa_shape& s)
{
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.app_K = a.K;
    p.app_V = a.V;
    p.app_Ks = a.Ks;
    p.app_pos = pos;
    p.ks_sb = s.ks_stride_b;
    p.ks_sh = s.ks_stride_h;
}

// The step.  `pg` (may be null) describes a paged cache: K, V and Ks are
// then its pools.
ssa_status decode_impl(const AppendArgs* app, const ssa_paged_kv* pg, int strata, float top_p, bool host_io,
                       const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const ssa_bf16* Ks,
                       const int32_t* sel_ch, int64_t top_k, float budget, uint64_t seed, float scale, float* out,
                       float* lse, float* s_hat_opt, int32_t* idx_opt, float* p_opt, int32_t* count_opt,
                       int64_t list_cap, void* ws, size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape, pg ? kStridesZero : kStridesContig);
    if (st != SSA_OK) return st;
    if (pg && (st = check_paged(pg, *shape)) != SSA_OK) return st;
    const bool empty = shape->ctx_len == 0;  // nothing is read from the cache
    if (!q || !sel_ch || !out || !lse || (!empty && (!K || !V || !Ks))) return SSA_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16) || !aligned(Ks, 16) || !aligned(q, 16)) return SSA_ERR_INVALID_ARG;
    if (bad_scalars(top_k, budget) || bad_scale(scale)) return SSA_ERR_INVALID_ARG;
    if ((idx_opt == nullptr) != (p_opt == nullptr)) return SSA_ERR_INVALID_ARG;
    const ssa::Plan pl = unit_plan(*shape);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    // K and V may sit in pinned host memory (the host-resident tier); the
    // summary the score kernel streams, and the query, live on the device
    if (!device_readable(K, true) || !device_readable(V, true) || !device_readable(Ks, false) ||
        !device_readable(q, host_io) || !device_readable(out, host_io) || !device_readable(lse, host_io))
        return SSA_ERR_INVALID_ARG;
    if (pg && (!device_readable(pg->block_table, false) || !device_readable(pg->seq_lens, false)))
        return SSA_ERR_INVALID_ARG;
    if (pl.U == 0) return SSA_OK;
    char* w = static_cast<char*>(ws);
    ssa::Params prm = base_params(*shape, pl, ws);
    if (pg) {
        prm.paged = 1;
        prm.log_ps = log2_exact(pg->page_size);
        prm.log_box = std::min(prm.log_ps, 8);
        prm.max_pages = pg->max_pages;
        prm.num_pages = pg->num_pages;
        prm.block_table = pg->block_table;
        prm.seq_lens = pg->seq_lens;
    }
    if (!empty && (st = pg ? encode_paged_map(&prm.ks_map, Ks, *pg, *shape) : encode_summary_map(&prm.ks_map, Ks, *shape)) !=
                      SSA_OK)
        return st;
    prm.q = q;
    if (host_io) {   // the first kernel stages the query from host memory into the workspace
        prm.q = reinterpret_cast<const ssa_bf16*>(w + pl.o_hq);
        prm.q_host = q;
        prm.q_staged = 1;
    }
    prm.K = K;
    prm.V = V;
    prm.sel_ch = sel_ch;
    prm.scale = scale;
    prm.budget = budget;
    prm.seed = seed;
    top_k = set_strata(prm, strata, top_k, top_p, shape->ctx_len);
    float* scores = s_hat_opt ? s_hat_opt : reinterpret_cast<float*>(w + pl.o_scores);
    prm.s_dst = scores;
    prm.s_src = scores;
    prm.idx_out = idx_opt;
    prm.p_out = p_opt;
    prm.count_out = count_opt;
    prm.cap = list_cap > 0 ? list_cap : std::max<int64_t>(shape->ctx_len, 1);
    prm.out = out;
    prm.lse = lse;
    prm.dense = (top_k >= shape->ctx_len || std::isinf(budget)) ? 1 : 0;
    prm.src_mode = prm.dense ? 1 : 0;
    prm.attend = 1;
    if (app) {
        // K0 writes the new token at ctx_len - 1 (paged: at each sequence's
        // last position).  The score kernel reads that summary row only from
        // its shared queue (the last stage of a unit is never in a CTA's
        // static share: sf < number of stages), i.e. after its wait for K0;
        // the attention reads rows after its own wait.
        if (pl.sf >= pl.nst) return SSA_ERR_UNSUPPORTED;
        set_append(prm, *app, shape->ctx_len - 1, *shape);
    }
    // K0 zeroes the unit counters, the score kernel's queue and the
    // histograms (and writes the appended token); a step that keeps every
    // token and wants no scores runs no score kernel
    const bool score = !empty && (!prm.dense || s_hat_opt);
    if ((st = launch_init(prm, stream)) != SSA_OK) return st;
    if (score && (st = launch_score(prm, *shape, !prm.dense, stream, true)) != SSA_OK) return st;
    return launch_unit(prm, *shape, stream, true);
}

}  // namespace

extern "C" {

ssa_status ssa_decode(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const ssa_bf16* Ks,
                      const int32_t* sel_ch, int64_t top_k, float budget, uint64_t seed, float scale, float* out,
                      float* lse, float* s_hat_opt, int32_t* idx_opt, float* p_opt, int32_t* count_opt,
                      int64_t list_cap, void* ws, size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream)
{
    return decode_impl(nullptr, nullptr, SSA_STRATA_SSA, 0.0f, false, q, K, V, Ks, sel_ch, top_k, budget, seed, scale, out,
                       lse, s_hat_opt, idx_opt, p_opt, count_opt, list_cap, ws, ws_bytes, shape, stream);
}

ssa_status ssa_decode_strata(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const ssa_bf16* Ks,
                             const int32_t* sel_ch, int strata, int64_t top_k, float top_p, float budget,
                             uint64_t seed, float scale, float* out, float* lse, float* s_hat_opt, int32_t* idx_opt,
                             float* p_opt, int32_t* count_opt, int64_t list_cap, void* ws, size_t ws_bytes,
                             const ssa_shape* shape, cudaStream_t stream)
{
    if (bad_strata(strata, top_p)) return SSA_ERR_INVALID_ARG;
    return decode_impl(nullptr, nullptr, strata, top_p, false, q, K, V, Ks, sel_ch, top_k, budget, seed, scale, out, lse,
                       s_hat_opt, idx_opt, p_opt, count_opt, list_cap, ws, ws_bytes, shape, stream);
}

ssa_status ssa_decode_early_stop(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const ssa_bf16* Ks,
                                 const int32_t* sel_ch, int64_t top_k, float budget, uint64_t seed, float scale,
                                 float tau, float* out, float* lse, int32_t* blocks_opt, void* ws, size_t ws_bytes,
                                 const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    const bool empty = shape->ctx_len == 0;
    if (!q || !sel_ch || !out || !lse || (!empty && (!K || !V || !Ks))) return SSA_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16) || !aligned(Ks, 16) || !aligned(q, 16)) return SSA_ERR_INVALID_ARG;
    if (bad_scalars(top_k, budget) || bad_scale(scale) || bad_tau(tau)) return SSA_ERR_INVALID_ARG;
    const ssa::Plan pl = unit_plan(*shape);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    if (!device_readable(K, true) || !device_readable(V, true) || !device_readable(Ks, false) ||
        !device_readable(q, false) || !device_readable(out, false) || !device_readable(lse, false))
        return SSA_ERR_INVALID_ARG;
    if (pl.U == 0) return SSA_OK;
    char* w = static_cast<char*>(ws);
    ssa::Params prm = base_params(*shape, pl, ws);
    if (!empty && (st = encode_summary_map(&prm.ks_map, Ks, *shape)) != SSA_OK) return st;
    prm.q = q;
    prm.K = K;
    prm.V = V;
    prm.sel_ch = sel_ch;
    prm.scale = scale;
    prm.budget = budget;
    prm.seed = seed;
    top_k = set_strata(prm, SSA_STRATA_SSA, top_k, 0.0f, shape->ctx_len);
    float* scores = reinterpret_cast<float*>(w + pl.o_scores);
    prm.s_dst = scores;
    prm.s_src = scores;
    prm.out = out;
    prm.lse = lse;
    prm.dense = (top_k >= shape->ctx_len || std::isinf(budget)) ? 1 : 0;
    prm.src_mode = prm.dense ? 1 : 0;
    // the selection writes each unit's list (ascending index) into the
    // workspace's selection rows; the early-stop launches order and attend it
    prm.attend = 0;
    prm.idx_out = reinterpret_cast<int32_t*>(w + pl.o_sel_idx);
    prm.p_out = reinterpret_cast<float*>(w + pl.o_sel_p);
    prm.count_out = reinterpret_cast<int32_t*>(w + pl.o_es);
    prm.cap = pl.np;
    if ((st = launch_init(prm, stream)) != SSA_OK) return st;
    if (!empty && (st = launch_score(prm, *shape, !prm.dense, stream, true)) != SSA_OK) return st;
    if ((st = launch_unit(prm, *shape, stream, true)) != SSA_OK) return st;
    prm.idx_in = prm.idx_out;
    prm.p_in = prm.p_out;
    prm.count_in = prm.count_out;
    return launch_early_stop(prm, *shape, tau, blocks_opt, stream);
}

ssa_status ssa_decode_append(const ssa_bf16* q, const ssa_bf16* k_new, const ssa_bf16* v_new, ssa_bf16* K,
                             ssa_bf16* V, ssa_bf16* Ks, const int32_t* sel_ch, int64_t top_k, float budget,
                             uint64_t seed, float scale, float* out, float* lse, void* ws, size_t ws_bytes,
                             const ssa_shape* shape, cudaStream_t stream)
{
    const ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (shape->ctx_len < 1 || !k_new || !v_new || !K || !V || !Ks) return SSA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return SSA_ERR_INVALID_ARG;
    const AppendArgs app{k_new, v_new, K, V, Ks};
    return decode_impl(&app, nullptr, SSA_STRATA_SSA, 0.0f, false, q, K, V, Ks, sel_ch, top_k, budget, seed, scale, out, lse,
                       nullptr, nullptr, nullptr, nullptr, 0, ws, ws_bytes, shape, stream);
}

ssa_status ssa_decode_paged(const ssa_bf16* q, const ssa_bf16* k_new, const ssa_bf16* v_new, ssa_bf16* K_pool,
                            ssa_bf16* V_pool, ssa_bf16* Ks_pool, const ssa_paged_kv* pages, const int32_t* sel_ch,
                            int64_t top_k, float budget, uint64_t seed, float scale, float* out, float* lse,
                            float* s_hat_opt, int32_t* idx_opt, float* p_opt, int32_t* count_opt, int64_t list_cap,
                            void* ws, size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream)
{
    if (!pages || (k_new == nullptr) != (v_new == nullptr)) return SSA_ERR_INVALID_ARG;
    if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))) return SSA_ERR_INVALID_ARG;
    if (k_new && shape && shape->ctx_len < 1) return SSA_ERR_INVALID_ARG;
    const AppendArgs app{k_new, v_new, K_pool, V_pool, Ks_pool};
    return decode_impl(k_new ? &app : nullptr, pages, SSA_STRATA_SSA, 0.0f, false, q, K_pool,
                       V_pool, Ks_pool, sel_ch, top_k, budget, seed, scale, out, lse, s_hat_opt, idx_opt, p_opt,
                       count_opt, list_cap, ws, ws_bytes, shape, stream);
}

ssa_status ssa_append(const ssa_bf16* k_new, const ssa_bf16* v_new, const int32_t* sel_ch, int64_t pos,
                      ssa_bf16* K, ssa_bf16* V, ssa_bf16* Ks, void* ws, size_t ws_bytes, const ssa_shape* shape,
                      cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!k_new || !v_new || !sel_ch || !K || !V || !Ks) return SSA_ERR_INVALID_ARG;
    if (pos < 0 || pos >= shape->ctx_len) return SSA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(K, 16) || !aligned(V, 16)) return SSA_ERR_INVALID_ARG;
    const ssa::Plan pl = make_plan(*shape, 0);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    if (pl.U == 0) return SSA_OK;
    ssa::Params prm = base_params(*shape, pl, ws);
    prm.sel_ch = sel_ch;
    set_append(prm, AppendArgs{k_new, v_new, K, V, Ks}, pos, *shape);
    return launch(&append_kernel, pl.U, 128, 0, prm, stream, false);
}

ssa_status ssa_decode_host(const ssa_bf16* q_host, const ssa_bf16* K, const ssa_bf16* V, const ssa_bf16* Ks,
                           const int32_t* sel_ch, int64_t top_k, float budget, uint64_t seed, float scale,
                           float* out_host, float* lse_host, void* ws, size_t ws_bytes, const ssa_shape* shape,
                           cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!q_host || !out_host || !lse_host) return SSA_ERR_INVALID_ARG;
    // pinned, mapped buffers: the kernels read q from host memory and write
    // out / lse into it (no copy is enqueued)
    if (device_readable(q_host, true) && device_readable(out_host, true) && device_readable(lse_host, true))
        return decode_impl(nullptr, nullptr, SSA_STRATA_SSA, 0.0f, true, q_host, K, V, Ks, sel_ch, top_k, budget, seed, scale,
                           out_host, lse_host, nullptr, nullptr, nullptr, nullptr, 0, ws, ws_bytes, shape, stream);
    // otherwise one staged copy in, the step, two staged copies out
    const ssa::Plan pl = make_plan(*shape, 0);
    if ((st = check_ws(ws, ws_bytes, pl)) != SSA_OK) return st;
    char* w = static_cast<char*>(ws);
    const size_t heads = (size_t)shape->batch * shape->n_q_heads;
    ssa_bf16* q_dev = reinterpret_cast<ssa_bf16*>(w + pl.o_hq);
    float* out_dev = reinterpret_cast<float*>(w + pl.o_hout);
    float* lse_dev = reinterpret_cast<float*>(w + pl.o_hlse);
    if (cudaMemcpyAsync(q_dev, q_host, heads * shape->head_dim * 2, cudaMemcpyHostToDevice, stream) != cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    st = ssa_decode(q_dev, K, V, Ks, sel_ch, top_k, budget, seed, scale, out_dev, lse_dev, nullptr, nullptr,
                    nullptr, nullptr, 0, ws, ws_bytes, shape, stream);
    if (st != SSA_OK) return st;
    if (cudaMemcpyAsync(out_host, out_dev, heads * shape->head_dim * 4, cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaMemcpyAsync(lse_host, lse_dev, heads * 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    return SSA_OK;
}

ssa_status ssa_decode_static(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const ssa_bf16* Ks,
                             const int32_t* sel_ch, int64_t top_k, float budget, uint64_t seed, float scale,
                             float* out, float* lse, uint32_t* device_flags, const ssa_shape* shape,
                             cudaStream_t stream)
{
    const ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    const ssa::Plan pl = make_plan(*shape, 0);
    if (pl.total > (size_t)SSA_STATIC_SCRATCH_BYTES) return SSA_ERR_WORKSPACE;
    void* ws = static_scratch_address();
    if (!ws) return SSA_ERR_CUDA;
    // the status word accumulates device flags: start this call from zero
    if (cudaMemsetAsync(ws, 0, kStatusBytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    const ssa_status rc = ssa_decode(q, K, V, Ks, sel_ch, top_k, budget, seed, scale, out, lse, nullptr, nullptr,
                                     nullptr, nullptr, 0, ws, (size_t)SSA_STATIC_SCRATCH_BYTES, shape, stream);
    if (rc != SSA_OK) return rc;
    if (device_flags &&
        cudaMemcpyAsync(device_flags, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    return SSA_OK;
}

ssa_status ssa_get_device_status(void* ws, cudaStream_t stream, uint32_t* flags_out)
{
    if (!ws || !aligned(ws, 256)) return SSA_ERR_WORKSPACE;
    uint32_t flags = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess ||
        cudaMemcpyAsync(&flags, ws, sizeof flags, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemsetAsync(ws, 0, sizeof flags, stream) != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    if (flags_out) *flags_out |= flags;
    if (flags & SSA_DEV_TIMEOUT) return SSA_ERR_DEVICE_TIMEOUT;
    if (flags & SSA_DEV_BAD_INDEX) return SSA_ERR_BAD_INDEX;
    if (flags & SSA_DEV_NONFINITE) return SSA_ERR_NONFINITE;
    if (flags & SSA_DEV_OVERFLOW) return SSA_ERR_OVERFLOW;
    return SSA_OK;
}

ssa_status ssa_query_plan(const ssa_shape* shape, int32_t* score_ctas, int32_t* tiles_per_unit,
                          int32_t* attend_ctas_per_unit)
{
    const ssa_status st = check_shape(shape, kStridesAny);
    if (st != SSA_OK) return st;
    const ssa::Plan pl = unit_plan(*shape);
    if (score_ctas) *score_ctas = pl.k1_grid;
    if (tiles_per_unit) *tiles_per_unit = pl.ntile;
    if (attend_ctas_per_unit) *attend_ctas_per_unit = pl.ntile;
    return SSA_OK;
}

}  // extern "C"
