// ssa_api.cu -- host side of libssa: argument checks, workspace layout,
// launch planning and the C entry points declared in include/ssa.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "ssa.h"
#include "kernels.cuh"

using namespace ssa;

namespace {

constexpr size_t kStatusBytes = 256;
constexpr int64_t kScoreTile = 8192;   // tokens per CTA for the standalone score launch

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
    size_t status, scores, idx, prob, count, hq, hout, hlse, total;
};

int64_t eff_cap(const ssa_shape& s, int64_t cap) { return cap > 0 ? cap : (s.ctx_len > 0 ? s.ctx_len : 1); }

WsLayout ws_layout(const ssa_shape& s, int64_t cap)
{
    const int64_t units = (int64_t)s.batch * s.n_kv_heads;
    const int64_t n = s.ctx_len > 0 ? s.ctx_len : 1;
    const int64_t c = eff_cap(s, cap);
    const int64_t heads = (int64_t)s.batch * s.n_q_heads;
    WsLayout L{};
    size_t o = 0;
    L.status = o;
    o += kStatusBytes;
    L.scores = o;
    o += align256((size_t)(units * n * 4));
    L.idx = o;
    o += align256((size_t)(units * c * 4));
    L.prob = o;
    o += align256((size_t)(units * c * 4));
    L.count = o;
    o += align256((size_t)(units * 4));
    L.hq = o;
    o += align256((size_t)(heads * s.head_dim * 2));
    L.hout = o;
    o += align256((size_t)(heads * s.head_dim * 4));
    L.hlse = o;
    o += align256((size_t)(heads * 4));
    L.total = o;
    return L;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

ssa_status check_shape(const ssa_shape* s)
{
    if (!s) return SSA_ERR_INVALID_ARG;
    if (s->batch < 0 || s->n_kv_heads < 1 || s->n_q_heads < 1 || s->reserved != 0) return SSA_ERR_INVALID_ARG;
    if (s->n_q_heads % s->n_kv_heads != 0) return SSA_ERR_INVALID_ARG;
    const int G = s->n_q_heads / s->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SSA_ERR_UNSUPPORTED;
    if (s->head_dim != 64 && s->head_dim != 128) return SSA_ERR_UNSUPPORTED;
    if (s->d_sel != 16 && s->d_sel != 32) return SSA_ERR_UNSUPPORTED;
    if (s->ctx_len < 0 || s->ctx_len >= (int64_t)INT32_MAX) return SSA_ERR_INVALID_ARG;
    const int64_t N = s->ctx_len;
    if (s->kv_stride_h < N * s->head_dim || s->ks_stride_h < N * s->d_sel) return SSA_ERR_INVALID_ARG;
    if (s->kv_stride_b < (int64_t)(s->n_kv_heads - 1) * s->kv_stride_h + N * s->head_dim) return SSA_ERR_INVALID_ARG;
    if (s->ks_stride_b < (int64_t)(s->n_kv_heads - 1) * s->ks_stride_h + N * s->d_sel) return SSA_ERR_INVALID_ARG;
    if (s->kv_stride_h % 8 || s->kv_stride_b % 8 || s->ks_stride_h % 8 || s->ks_stride_b % 8)
        return SSA_ERR_INVALID_ARG;
    return SSA_OK;
}

ssa_status check_ws(void* ws, size_t ws_bytes, const ssa_shape& s, int64_t cap)
{
    if (!ws || !aligned(ws, 256)) return SSA_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(s, cap).total) return SSA_ERR_WORKSPACE;
    return SSA_OK;
}

typedef void (*kfn_t)(Params);

template <int G, int MODE, bool RES>
kfn_t pick_dsel_d(int dsel, int d)
{
    if (dsel == 16) return d == 64 ? &unit_kernel<G, 16, 64, MODE, RES> : &unit_kernel<G, 16, 128, MODE, RES>;
    return d == 64 ? &unit_kernel<G, 32, 64, MODE, RES> : &unit_kernel<G, 32, 128, MODE, RES>;
}

template <int MODE, bool RES>
kfn_t pick_g(int G, int dsel, int d)
{
    switch (G) {
        case 1: return pick_dsel_d<1, MODE, RES>(dsel, d);
        case 2: return pick_dsel_d<2, MODE, RES>(dsel, d);
        case 4: return pick_dsel_d<4, MODE, RES>(dsel, d);
        default: return pick_dsel_d<8, MODE, RES>(dsel, d);
    }
}

template <int G>
kfn_t pick_score(int dsel)
{
    return dsel == 16 ? &unit_kernel<G, 16, 64, MODE_SCORE, false> : &unit_kernel<G, 32, 64, MODE_SCORE, false>;
}

template <int G>
kfn_t pick_attend(int d)
{
    return d == 64 ? &unit_kernel<G, 16, 64, MODE_ATTEND, false> : &unit_kernel<G, 16, 128, MODE_ATTEND, false>;
}

kfn_t pick_kernel(int mode, int G, int dsel, int d, bool res)
{
    switch (mode) {
        case MODE_SCORE:
            switch (G) {
                case 1: return pick_score<1>(dsel);
                case 2: return pick_score<2>(dsel);
                case 4: return pick_score<4>(dsel);
                default: return pick_score<8>(dsel);
            }
        case MODE_SELECT:
            return res ? &unit_kernel<1, 16, 64, MODE_SELECT, true> : &unit_kernel<1, 16, 64, MODE_SELECT, false>;
        case MODE_ATTEND:
            switch (G) {
                case 1: return pick_attend<1>(d);
                case 2: return pick_attend<2>(d);
                case 4: return pick_attend<4>(d);
                default: return pick_attend<8>(d);
            }
        default:
            return res ? pick_g<MODE_SCORE | MODE_SELECT | MODE_ATTEND, true>(G, dsel, d)
                       : pick_g<MODE_SCORE | MODE_SELECT | MODE_ATTEND, false>(G, dsel, d);
    }
}

int env_int(const char* name, int dflt)
{
    const char* v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : dflt;
}

std::mutex g_mu;

// Largest number of clusters of size C of this kernel that can be resident at once.
int max_active_clusters(kfn_t fn, int C, uint32_t smem)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    static std::map<std::tuple<void*, int, uint32_t, int>, int> cache;
    const auto key = std::make_tuple((void*)fn, C, smem, dev);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    bool ok = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
              cudaSuccess;
    if (ok && C > 8)
        ok = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(C * 64), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)C;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, (const void*)fn, &cfg) != cudaSuccess) n = 0;
    }
    if (!ok || n == 0) cudaGetLastError();
    std::lock_guard<std::mutex> lk(g_mu);
    cache[key] = n;
    return n;
}

struct Plan {
    int C = 1;
    bool res = false;
    int64_t seg = kSegAlign;
    uint32_t smem = 0;
    bool cluster = true;
};

int64_t round_seg(int64_t n, int C)
{
    const int64_t per = (n + C - 1) / C;
    return ((per + kSegAlign - 1) / kSegAlign) * kSegAlign;
}

// One cluster per unit: the largest C in {16, 8, 4, 2, 1} whose clusters
// all fit on the GPU at once (a single wave), without CTAs of fewer than
// 512 tokens.  SSA_FORCE_CLUSTER / SSA_FORCE_GLOBAL_SCORES override the
// choice (used by the tests to cover every path on small inputs).
Plan make_plan(int mode, const ssa_shape& s)
{
    const int G = s.n_q_heads / s.n_kv_heads;
    const int64_t units = (int64_t)s.batch * s.n_kv_heads;
    const int64_t n = s.ctx_len > 0 ? s.ctx_len : 1;
    Plan pl;
    if (mode == MODE_SCORE) {
        pl.seg = kScoreTile;
        pl.C = (int)((n + kScoreTile - 1) / kScoreTile);
        pl.cluster = false;
        pl.smem = make_layout(mode, false, pl.seg, 1).total;
        return pl;
    }
    const int forced = env_int("SSA_FORCE_CLUSTER", 0);
    const bool force_global = env_int("SSA_FORCE_GLOBAL_SCORES", 0) != 0;
    int maxC = 1;
    while (maxC < 16 && (int64_t)(maxC * 2) * kSegAlign <= n) maxC *= 2;
    Plan best;
    bool have_best = false;
    int64_t best_score = -1;
    for (int C = 16; C >= 1; C /= 2) {
        if (forced > 0 && C != forced) continue;
        if (forced <= 0 && C > maxC) continue;
        Plan cand;
        cand.C = C;
        cand.seg = (mode & MODE_SELECT) ? round_seg(n, C) : kSegAlign;
        cand.res = (mode & MODE_SELECT) && !force_global &&
                   make_layout(mode, true, cand.seg, C).total <= kSmemLimit;
        cand.smem = make_layout(mode, cand.res, cand.seg, C).total;
        if (cand.smem > kSmemLimit) continue;
        if (forced > 0) return cand;
        const int clusters = max_active_clusters(pick_kernel(mode, G, s.d_sel, s.head_dim, cand.res), C, cand.smem);
        if (clusters <= 0) continue;
        if (clusters >= units) return cand;
        // otherwise prefer the choice that keeps the most CTAs busy in one wave
        const int64_t busy = (int64_t)std::min<int64_t>(clusters, units) * C;
        if (busy > best_score) {
            best_score = busy;
            best = cand;
            have_best = true;
        }
    }
    if (have_best) return best;
    Plan fb;
    fb.C = 1;
    fb.seg = (mode & MODE_SELECT) ? round_seg(n, 1) : kSegAlign;
    fb.res = false;
    fb.smem = make_layout(mode, false, fb.seg, 1).total;
    return fb;
}

ssa_status launch(int mode, const ssa_shape& s, const Plan& pl, const Params& prm, cudaStream_t stream)
{
    const int G = s.n_q_heads / s.n_kv_heads;
    const int64_t units = (int64_t)s.batch * s.n_kv_heads;
    if (units == 0) return SSA_OK;
    if (pl.smem > kSmemLimit) return SSA_ERR_UNSUPPORTED;
    kfn_t fn = pick_kernel(mode, G, s.d_sel, s.head_dim, pl.res);
    if (cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    if (pl.cluster && pl.C > 8 &&
        cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    const int64_t blocks = units * pl.C;
    if (blocks > INT32_MAX) return SSA_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    if (pl.cluster) {
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)pl.C;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
    }
    Params p = prm;
    p.C = pl.C;
    p.seg_len = pl.seg;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, fn, p);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SSA_ERR_CUDA;
    }
    return SSA_OK;
}

Params base_params(const ssa_shape& s, void* ws)
{
    Params p = {};
    p.Bt = s.batch;
    p.Hq = s.n_q_heads;
    p.Hkv = s.n_kv_heads;
    p.d = s.head_dim;
    p.d_sel = s.d_sel;
    p.N = s.ctx_len;
    p.kv_sb = s.kv_stride_b;
    p.kv_sh = s.kv_stride_h;
    p.ks_sb = s.ks_stride_b;
    p.ks_sh = s.ks_stride_h;
    p.status = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_layout(s, 1).status);
    return p;
}

bool bad_scalars(int64_t top_k, float budget) { return top_k < 0 || !(budget >= 0.0f); }
bool bad_scale(float scale) { return !(scale > 0.0f) || !std::isfinite(scale); }

}  // namespace

// Scratch for ssa_decode_static: one array per GPU that loads the library.
// Host code must not use its name as a device address; the address comes
// from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_static_scratch[SSA_STATIC_SCRATCH_BYTES];

namespace {

void* static_scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    static std::mutex mu;
    static std::map<int, void*> addr;
    std::lock_guard<std::mutex> lk(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) return it->second;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return nullptr;
    }
    addr[dev] = ptr;
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

int ssa_version(void) { return 100; }

size_t ssa_workspace_bytes(const ssa_shape* shape, int64_t list_cap)
{
    if (check_shape(shape) != SSA_OK) return 0;
    return ws_layout(*shape, list_cap).total;
}

ssa_status ssa_pack_summary(const ssa_bf16* K, const int32_t* sel_ch, ssa_bf16* Ks, void* ws, size_t ws_bytes,
                            const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!K || !sel_ch || !Ks) return SSA_ERR_INVALID_ARG;
    if ((st = check_ws(ws, ws_bytes, *shape, 0)) != SSA_OK) return st;
    const int64_t total = (int64_t)shape->batch * shape->n_kv_heads * shape->ctx_len * shape->d_sel;
    if (total == 0) return SSA_OK;
    const Params bp = base_params(*shape, ws);
    const int threads = 256;
    const int64_t want = (total + threads - 1) / threads;
    const unsigned blocks = (unsigned)std::min<int64_t>(want, 148 * 32);
    pack_summary_kernel<<<blocks, threads, 0, stream>>>(K, sel_ch, Ks, shape->n_kv_heads, shape->head_dim,
                                                        shape->d_sel, shape->ctx_len, shape->kv_stride_b,
                                                        shape->kv_stride_h, shape->ks_stride_b,
                                                        shape->ks_stride_h, total, bp.status);
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
    if ((st = check_ws(ws, ws_bytes, *shape, 0)) != SSA_OK) return st;
    if (shape->ctx_len == 0) return SSA_OK;
    Params p = base_params(*shape, ws);
    p.q = q;
    p.Ks = Ks;
    p.sel_ch = sel_ch;
    p.scale = scale;
    p.s_out = s_hat;
    return launch(MODE_SCORE, *shape, make_plan(MODE_SCORE, *shape), p, stream);
}

ssa_status ssa_select(const float* s_hat, int64_t top_k, float budget, uint64_t seed, int32_t* idx, float* p,
                      int32_t* count, int64_t list_cap, void* ws, size_t ws_bytes, const ssa_shape* shape,
                      cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!s_hat || !idx || !p || !count) return SSA_ERR_INVALID_ARG;
    if (bad_scalars(top_k, budget)) return SSA_ERR_INVALID_ARG;
    if ((st = check_ws(ws, ws_bytes, *shape, list_cap)) != SSA_OK) return st;
    Params prm = base_params(*shape, ws);
    prm.s_in = s_hat;
    prm.top_k = top_k;
    prm.budget = budget;
    prm.seed = seed;
    prm.idx = idx;
    prm.p = p;
    prm.count = count;
    prm.cap = eff_cap(*shape, list_cap);
    return launch(MODE_SELECT, *shape, make_plan(MODE_SELECT, *shape), prm, stream);
}

ssa_status ssa_attend(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const int32_t* idx, const float* p,
                      const int32_t* count, int64_t list_cap, float scale, float* out, float* lse, void* ws,
                      size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!q || !idx || !p || !count || !out || !lse || (shape->ctx_len > 0 && (!K || !V))) return SSA_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16)) return SSA_ERR_INVALID_ARG;
    if (bad_scale(scale)) return SSA_ERR_INVALID_ARG;
    if ((st = check_ws(ws, ws_bytes, *shape, list_cap)) != SSA_OK) return st;
    Params prm = base_params(*shape, ws);
    prm.q = q;
    prm.K = K;
    prm.V = V;
    prm.scale = scale;
    prm.idx = const_cast<int32_t*>(idx);
    prm.p = const_cast<float*>(p);
    prm.count = const_cast<int32_t*>(count);
    prm.cap = eff_cap(*shape, list_cap);
    prm.out = out;
    prm.lse = lse;
    return launch(MODE_ATTEND, *shape, make_plan(MODE_ATTEND, *shape), prm, stream);
}

ssa_status ssa_decode(const ssa_bf16* q, const ssa_bf16* K, const ssa_bf16* V, const ssa_bf16* Ks,
                      const int32_t* sel_ch, int64_t top_k, float budget, uint64_t seed, float scale, float* out,
                      float* lse, float* s_hat_opt, int32_t* idx_opt, float* p_opt, int32_t* count_opt,
                      int64_t list_cap, void* ws, size_t ws_bytes, const ssa_shape* shape, cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    const bool empty = shape->ctx_len == 0;  // nothing is read from the cache
    if (!q || !sel_ch || !out || !lse || (!empty && (!K || !V || !Ks))) return SSA_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16) || !aligned(Ks, 16) || !aligned(q, 16)) return SSA_ERR_INVALID_ARG;
    if (bad_scalars(top_k, budget) || bad_scale(scale)) return SSA_ERR_INVALID_ARG;
    if ((st = check_ws(ws, ws_bytes, *shape, list_cap)) != SSA_OK) return st;
    const WsLayout wl = ws_layout(*shape, list_cap);
    char* w = static_cast<char*>(ws);
    const Plan pl = make_plan(MODE_SCORE | MODE_SELECT | MODE_ATTEND, *shape);
    Params prm = base_params(*shape, ws);
    prm.q = q;
    prm.K = K;
    prm.V = V;
    prm.Ks = Ks;
    prm.sel_ch = sel_ch;
    prm.scale = scale;
    prm.top_k = top_k;
    prm.budget = budget;
    prm.seed = seed;
    prm.s_out = s_hat_opt ? s_hat_opt : (pl.res ? nullptr : reinterpret_cast<float*>(w + wl.scores));
    prm.idx = idx_opt ? idx_opt : reinterpret_cast<int32_t*>(w + wl.idx);
    prm.p = p_opt ? p_opt : reinterpret_cast<float*>(w + wl.prob);
    prm.count = count_opt;
    prm.cap = eff_cap(*shape, list_cap);
    prm.out = out;
    prm.lse = lse;
    return launch(MODE_SCORE | MODE_SELECT | MODE_ATTEND, *shape, pl, prm, stream);
}

ssa_status ssa_decode_host(const ssa_bf16* q_host, const ssa_bf16* K, const ssa_bf16* V, const ssa_bf16* Ks,
                           const int32_t* sel_ch, int64_t top_k, float budget, uint64_t seed, float scale,
                           float* out_host, float* lse_host, void* ws, size_t ws_bytes, const ssa_shape* shape,
                           cudaStream_t stream)
{
    ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    if (!q_host || !out_host || !lse_host) return SSA_ERR_INVALID_ARG;
    if ((st = check_ws(ws, ws_bytes, *shape, 0)) != SSA_OK) return st;
    const WsLayout wl = ws_layout(*shape, 0);
    char* w = static_cast<char*>(ws);
    const size_t heads = (size_t)shape->batch * shape->n_q_heads;
    ssa_bf16* q_dev = reinterpret_cast<ssa_bf16*>(w + wl.hq);
    float* out_dev = reinterpret_cast<float*>(w + wl.hout);
    float* lse_dev = reinterpret_cast<float*>(w + wl.hlse);
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
    if (ws_layout(*shape, 0).total > (size_t)SSA_STATIC_SCRATCH_BYTES) return SSA_ERR_WORKSPACE;
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

ssa_status ssa_query_plan(const ssa_shape* shape, int32_t* cluster_size, int32_t* scores_resident,
                          int32_t* smem_bytes)
{
    const ssa_status st = check_shape(shape);
    if (st != SSA_OK) return st;
    const Plan pl = make_plan(MODE_SCORE | MODE_SELECT | MODE_ATTEND, *shape);
    if (cluster_size) *cluster_size = pl.C;
    if (scores_resident) *scores_resident = pl.res ? 1 : 0;
    if (smem_bytes) *smem_bytes = (int32_t)pl.smem;
    return SSA_OK;
}

}  // extern "C"
