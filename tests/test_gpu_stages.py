"""GPU parity, stage by stage, against the CPU oracle (small sizes that span
several tiles, ragged tails, several selection tile sizes and attention splits).

Tolerances:
  * pack: bit-exact.
  * score: |s_gpu - s_oracle| <= 1e-5 * scale * max_g sum_j |q_g[S_j] Ks_ij|
    (fp32 accumulation vs. the oracle's double; the plain relative form fails
    where s ~ 0).
  * select (given the oracle's scores): index sets identical except tokens
    with |u - p| <= 1e-6 (expf vs. a correctly rounded exp may move p by an
    ulp or two); p within 4 ulp.
  * attend (given the oracle's lists): out and lse within 2e-3 abs + 2e-3 rel.
"""
import contextlib
import math
import os

import numpy as np
import pytest
import torch

import long_context_decode_subset_b300 as ssa
import oracle
import workloads
from _util import compare_unit_lists, score_bound, u16

pytestmark = pytest.mark.gpu

DEV = "cuda"


@contextlib.contextmanager
def plan_env(tile=None, split=None):
    """Force the selection tile size (tokens) and the attention split (CTAs per unit)."""
    keys = ("SSA_FORCE_TILE", "SSA_FORCE_SPLIT")
    old = {k: os.environ.get(k) for k in keys}
    for k, v in zip(keys, (tile, split)):
        if v:
            os.environ[k] = str(v)
        else:
            os.environ.pop(k, None)
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


SMALL = {
    "tiny": workloads.CONFIGS["tiny"],
    "g4_d128": workloads.make_config("ministral8b_32k", batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=5000,
                                     top_k=50, budget=50.0, n_needles=8),
    "g8_d128": workloads.make_config("ministral8b_32k", batch=1, n_q_heads=16, n_kv_heads=2, ctx_len=3001,
                                     top_k=30, budget=31.0, n_needles=4),
    "g1_d64": workloads.make_config("ministral8b_32k", batch=2, n_q_heads=2, n_kv_heads=2, head_dim=64,
                                    ctx_len=1500, top_k=20, budget=20.0, n_needles=4),
    "g2_d128_s16": workloads.make_config("27b_128k_50x", batch=1, n_q_heads=4, n_kv_heads=2, ctx_len=4100,
                                         d_sel=16, top_k=41, budget=41.0, n_needles=4),
    "g8_d64_s16": workloads.make_config("ministral8b_32k", batch=1, n_q_heads=8, n_kv_heads=1, head_dim=64,
                                        d_sel=16, ctx_len=2600, top_k=26, budget=26.0, n_needles=4),
}

_cache = {}


def case(name, seed=0):
    key = (name, seed)
    if key not in _cache:
        cfg = SMALL[name]
        w = workloads.generate(cfg, seed, DEV)
        w["Ks"] = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
        torch.cuda.synchronize()
        _cache[key] = w
    return _cache[key]


def oracle_inputs(w):
    """Host copies for the oracle; its key summary is packed by the oracle, not taken from the GPU."""
    K, sel = u16(w["K"]), w["sel_ch"].cpu().numpy()
    return u16(w["q"]), K, u16(w["V"]), oracle.pack_summary(K, sel, w["cfg"].d_sel), sel


@pytest.mark.parametrize("name", list(SMALL))
def test_pack_summary_bit_exact(oracle_mod, name):
    w = case(name)
    cfg = w["cfg"]
    want = oracle_mod.pack_summary(u16(w["K"]), w["sel_ch"].cpu().numpy(), cfg.d_sel)
    assert np.array_equal(u16(w["Ks"]), want)


@pytest.mark.parametrize("name", list(SMALL))
def test_score_parity(oracle_mod, name):
    w = case(name)
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    s_gpu = ssa.ssa_score(w["q"], w["Ks"], w["sel_ch"], cfg.scale).cpu().numpy()
    s_ora = oracle_mod.score(q, Ks, sel, cfg.scale)
    tol = score_bound(q, Ks, sel, cfg.scale)
    assert np.all(np.abs(s_gpu - s_ora) <= tol), np.max(np.abs(s_gpu - s_ora) / tol)


def _select_and_compare(oracle_mod, s_np, k, B, seed, tile=None, split=None, cap=None):
    s = torch.from_numpy(s_np).to(DEV)
    Bt, Hkv, N = s_np.shape
    with plan_env(tile, split):
        idx, p, count = ssa.ssa_select(s, k, B, seed, list_cap=cap or 0)
        ws = None
    torch.cuda.synchronize()
    idx, p, count = idx.cpu().numpy(), p.cpu().numpy(), count.cpu().numpy()
    nb = 0
    for b in range(Bt):
        for h in range(Hkv):
            o_idx, o_p, m, Z, p_all = oracle_mod.select_unit(s_np[b, h], k, B, seed, b, h, want_p_all=True)
            n = int(count[b, h])
            nd, _ = compare_unit_lists(idx[b, h, :n], p[b, h, :n], o_idx, o_p, p_all,
                                       lambda j: oracle_mod.uniform(seed, j, h, b))
            nb += nd
            assert np.all(np.diff(idx[b, h, :n]) > 0), "selection not in ascending token order"
    return nb


@pytest.mark.parametrize("tile,split", [(None, None), (512, 1), (512, 7), (1024, 3), (2048, 64), (4096, 2)])
def test_select_parity_tiles_and_splits(oracle_mod, tile, split):
    w = case("g4_d128")
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    s_np = oracle_mod.score(q, Ks, sel, cfg.scale)
    nb = _select_and_compare(oracle_mod, s_np, cfg.top_k, cfg.budget, 7, tile, split)
    assert nb <= 2


@pytest.mark.parametrize("tile,split", [(None, None), (512, 5), (1024, 1)])
def test_select_edge_cases(oracle_mod, tile, split):
    rng = np.random.default_rng(11)
    Bt, Hkv = 1, 2
    for N, k, B, kind in [
        (3000, 40, 40.0, "ties"),            # heavy exact ties at the threshold
        (3000, 40, 40.0, "constant"),        # uniform hybrid: all scores equal
        (2500, 0, 30.0, "normal"),           # no top-k stratum: m = max
        (2500, 25, 0.0, "normal"),           # pure top-k
        (2500, 25, math.inf, "normal"),      # dense limit
        (700, 700, 10.0, "normal"),          # k >= N
        (700, 699, 10.0, "normal"),          # k = N - 1
        (1, 0, 5.0, "normal"),               # single token
        (513, 5, 5.0, "signed_zero"),        # -0 / +0 ordering
        (4097, 60, 1e6, "normal"),           # clipping: most p = 1
        (2000, 30, 30.0, "wide"),            # scores spanning many octaves
    ]:
        if kind == "ties":
            s = np.round(rng.standard_normal((Bt, Hkv, N)) * 2) / 4
        elif kind == "constant":
            s = np.full((Bt, Hkv, N), 0.375)
        elif kind == "signed_zero":
            s = np.where(rng.random((Bt, Hkv, N)) < 0.5, 0.0, -0.0) * np.ones((Bt, Hkv, N))
            s[..., ::7] = rng.standard_normal(s[..., ::7].shape)
        elif kind == "wide":
            s = rng.standard_normal((Bt, Hkv, N)) * np.exp2(rng.integers(-20, 6, (Bt, Hkv, N)))
        else:
            s = rng.standard_normal((Bt, Hkv, N)) * 1.5
        s = s.astype(np.float32)
        nb = _select_and_compare(oracle_mod, s, k, B, 3, tile, split)
        assert nb <= 2, (N, k, B, kind)


def test_select_overflow_flag(oracle_mod):
    s = torch.zeros((1, 1, 1000), device=DEV)
    idx, p, count = ssa.ssa_select(s, 100, math.inf, 0, list_cap=10)
    shape = ssa.make_shape(1, 1, 1, 64, 16, 1000)
    # the binding allocated its own workspace; re-run with one we can inspect
    ws = ssa.workspace(shape, 10)
    idx2, p2, c2 = ssa.ssa_select(s, 100, math.inf, 0, idx=idx, p=p, count=count, list_cap=10, ws=ws)
    st, flags = ssa.ssa_get_device_status(ws)
    assert flags & ssa.ssa.DEV_OVERFLOW and st == 5
    assert int(c2[0, 0]) == 1000 and idx2[0, 0].tolist() == list(range(10))


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("split", [None, 1, 13])
def test_attend_parity(oracle_mod, name, split):
    w = case(name)
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    r = oracle_mod.decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 5, cfg.scale)
    idx = torch.from_numpy(r["idx"]).to(DEV)
    p = torch.from_numpy(r["p"]).to(DEV)
    count = torch.from_numpy(r["count"].astype(np.int32)).to(DEV)
    with plan_env(None, split):
        out, lse = ssa.ssa_attend(w["q"], w["K"], w["V"], idx, p, count, cfg.scale)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    assert np.allclose(out, r["out"], atol=2e-3, rtol=2e-3), np.abs(out - r["out"]).max()
    assert np.allclose(lse, r["lse"], atol=2e-3, rtol=2e-3), np.abs(lse - r["lse"]).max()


def test_attend_empty_and_dense(oracle_mod):
    w = case("tiny")
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    N = cfg.ctx_len
    idx = torch.arange(N, dtype=torch.int32, device=DEV).view(1, 1, N)
    p = torch.ones((1, 1, N), device=DEV)
    count = torch.tensor([[N]], dtype=torch.int32, device=DEV)
    out, lse = ssa.ssa_attend(w["q"], w["K"], w["V"], idx, p, count, cfg.scale)
    d_out, d_lse = oracle_mod.dense_attention(q, K, V, cfg.scale)
    assert np.allclose(out.cpu().numpy(), d_out, atol=2e-3, rtol=2e-3)
    assert np.allclose(lse.cpu().numpy(), d_lse, atol=2e-3, rtol=2e-3)
    count.zero_()
    out, lse = ssa.ssa_attend(w["q"], w["K"], w["V"], idx, p, count, cfg.scale)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), float("-inf")])
def test_select_flags_nonfinite_scores(bad):
    """A non-finite score is an error the device reports (SSA_DEV_NONFINITE / SSA_ERR_NONFINITE); the
    selection's content is then unspecified, but the call completes and its lists stay in bounds."""
    s = torch.randn((1, 2, 1000), device=DEV)
    s[0, 1, 123] = bad
    shape = ssa.make_shape(1, 2, 2, 64, 16, 1000)
    ws = ssa.workspace(shape, 1000)
    idx, p, count = ssa.ssa_select(s, 10, 10.0, 0, list_cap=1000, ws=ws)
    st, flags = ssa.ssa_get_device_status(ws)
    assert flags & ssa.ssa.DEV_NONFINITE and st == 6, (st, hex(flags))
    c = count.cpu()
    assert torch.all((c >= 0) & (c <= 1000))
    for h in range(2):
        n = int(c[0, h])
        ids = idx[0, h, :n].cpu()
        assert torch.all((ids >= 0) & (ids < 1000))


def _uniform_p_all(oracle_mod, s_unit, k, B):
    """The uniform hybrid's inclusion probability of every token, from the oracle's own top-k stratum
    (1 on T, min(1, fl32(B / fl32(N - |T|))) on the remainder)."""
    N = s_unit.size
    t_idx = oracle_mod.select_unit(s_unit, k, 0.0, 0, 0, 0)[0]
    p_all = np.empty(N, np.float32)
    n_r = N - t_idx.size
    p_all[:] = 1.0 if (n_r == 0 or math.isinf(B)) else min(np.float32(1.0), np.float32(np.float32(B) / np.float32(n_r)))
    p_all[t_idx] = 1.0
    return p_all


def _select_uniform_and_compare(oracle_mod, s_np, k, B, seed, tile=None, split=None):
    s = torch.from_numpy(s_np).to(DEV)
    Bt, Hkv, N = s_np.shape
    with plan_env(tile, split):
        idx, p, count = ssa.ssa_select_strata(s, ssa.ssa.STRATA_UNIFORM, k, 0.0, B, seed)
    torch.cuda.synchronize()
    idx, p, count = idx.cpu().numpy(), p.cpu().numpy(), count.cpu().numpy()
    for b in range(Bt):
        for h in range(Hkv):
            o_idx, o_p = oracle_mod.select_unit_uniform(s_np[b, h], k, B, seed, b, h)
            n = int(count[b, h])
            # the same Philox uniforms against the same fp32 p: identical lists, p bit for bit
            assert np.array_equal(idx[b, h, :n], o_idx), (b, h, n, o_idx.size)
            assert np.array_equal(p[b, h, :n], o_p), (b, h)


@pytest.mark.parametrize("tile,split", [(None, None), (512, 1), (1024, 3), (4096, 2)])
def test_select_uniform_hybrid_parity(oracle_mod, tile, split):
    """The top-k + uniform hybrid (SSA_STRATA_UNIFORM) against the oracle's select_unit_uniform, given the
    oracle's scores, over several tilings."""
    w = case("g4_d128")
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    s_np = oracle_mod.score(q, Ks, sel, cfg.scale)
    _select_uniform_and_compare(oracle_mod, s_np, cfg.top_k, cfg.budget, 7, tile, split)


def test_select_uniform_hybrid_edge_cases(oracle_mod):
    rng = np.random.default_rng(21)
    for N, k, B, kind in [(3000, 40, 40.0, "ties"), (3000, 40, 40.0, "constant"), (2500, 0, 30.0, "normal"),
                          (2500, 25, 0.0, "normal"), (700, 699, 10.0, "normal"), (4097, 60, 1e6, "normal"),
                          (513, 5, 5.0, "signed_zero")]:
        if kind == "ties":
            s = np.round(rng.standard_normal((1, 2, N)) * 2) / 4
        elif kind == "constant":
            s = np.full((1, 2, N), 0.375)
        elif kind == "signed_zero":
            s = np.where(rng.random((1, 2, N)) < 0.5, 0.0, -0.0) * np.ones((1, 2, N))
        else:
            s = rng.standard_normal((1, 2, N)) * 1.5
        _select_uniform_and_compare(oracle_mod, s.astype(np.float32), k, B, 4)


def test_decode_uniform_hybrid_parity(oracle_mod):
    """The whole step with the uniform hybrid: the selection against the oracle's hybrid on the oracle's
    scores (boundary cases at the top-k edge excepted), the output against the oracle's attention over the
    oracle's lists."""
    w = case("g4_d128")
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    Bt, Hkv, N = cfg.batch, cfg.n_kv_heads, cfg.ctx_len
    G = cfg.group
    idx = torch.empty((Bt, Hkv, N), dtype=torch.int32, device=DEV)
    p = torch.empty((Bt, Hkv, N), dtype=torch.float32, device=DEV)
    count = torch.empty((Bt, Hkv), dtype=torch.int32, device=DEV)
    out, lse = ssa.ssa_decode_strata(w["q"], w["K"], w["V"], w["Ks"], w["sel_ch"], ssa.ssa.STRATA_UNIFORM,
                                     cfg.top_k, 0.0, cfg.budget, 9, cfg.scale, idx=idx, p=p, count=count)
    s_np = oracle_mod.score(q, Ks, sel, cfg.scale)
    for b in range(Bt):
        for h in range(Hkv):
            o_idx, o_p = oracle_mod.select_unit_uniform(s_np[b, h], cfg.top_k, cfg.budget, 9, b, h)
            n = int(count[b, h])
            g_idx = idx[b, h, :n].cpu().numpy()
            assert len(set(g_idx.tolist()) ^ set(o_idx.tolist())) <= 2
            out_o, lse_o = oracle_mod.attend_unit(q[b, h * G:(h + 1) * G], K[b, h], V[b, h], g_idx,
                                                  _uniform_p_all(oracle_mod, s_np[b, h], cfg.top_k, cfg.budget)[g_idx],
                                                  cfg.scale)
            assert np.allclose(out[b, h * G:(h + 1) * G].cpu().numpy(), out_o, atol=2e-3, rtol=2e-3)
            assert np.allclose(lse[b, h * G:(h + 1) * G].cpu().numpy(), lse_o, atol=2e-3, rtol=2e-3)


def _top_p_sizes(oracle_mod, s_unit, top_p, tol=2e-6):
    """The oracle's top-p stratum size and, where top_p falls within `tol` of a stratum edge (the GPU sums
    fp32 expf terms, the oracle double exp terms), the neighbouring size the GPU may find instead."""
    k, before, at = oracle_mod.top_p_shares(s_unit, top_p)
    sizes = [k]
    if k >= 1 and top_p - before <= tol * top_p:
        sizes.append(k - 1)
    if at - top_p <= tol * top_p and k < s_unit.size:
        sizes.append(k + 1)
    return sizes


def _select_top_p_and_compare(oracle_mod, s_np, top_p, B, seed, tile=None, split=None):
    s = torch.from_numpy(s_np).to(DEV)
    Bt, Hkv, N = s_np.shape
    with plan_env(tile, split):
        i0, p0, c0 = ssa.ssa_select_strata(s, ssa.STRATA_TOP_P, 0, top_p, 0.0, seed)   # the stratum alone
        idx, p, count = ssa.ssa_select_strata(s, ssa.STRATA_TOP_P, 0, top_p, B, seed)
    torch.cuda.synchronize()
    i0, c0 = i0.cpu().numpy(), c0.cpu().numpy()
    idx, p, count = idx.cpu().numpy(), p.cpu().numpy(), count.cpu().numpy()
    edges = 0
    for b in range(Bt):
        for h in range(Hkv):
            sizes = _top_p_sizes(oracle_mod, s_np[b, h], top_p)
            k = int(c0[b, h])
            assert k in sizes, (b, h, k, sizes)
            edges += k != sizes[0]
            t_idx = oracle_mod.select_unit(s_np[b, h], k, 0.0, seed, b, h)[0]
            assert np.array_equal(i0[b, h, :k], t_idx)
            o_idx, o_p, m, Z, p_all = oracle_mod.select_unit(s_np[b, h], k, B, seed, b, h, want_p_all=True)
            n = int(count[b, h])
            compare_unit_lists(idx[b, h, :n], p[b, h, :n], o_idx, o_p, p_all,
                               lambda j: oracle_mod.uniform(seed, j, h, b))
    return edges


@pytest.mark.parametrize("tile,split", [(None, None), (512, 1), (1024, 3), (4096, 2)])
def test_select_top_p_parity(oracle_mod, tile, split):
    """The top-p stratum (SSA_STRATA_TOP_P) against the oracle's top_p_count / select_unit_top_p, given the
    oracle's scores, over several tilings and stratum sizes."""
    w = case("g4_d128")
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    s_np = oracle_mod.score(q, Ks, sel, cfg.scale)
    for top_p in (0.01, 0.3, 0.9, 0.999):
        assert _select_top_p_and_compare(oracle_mod, s_np, top_p, cfg.budget, 7, tile, split) <= 1


def test_select_top_p_edge_cases(oracle_mod):
    rng = np.random.default_rng(31)
    for N, top_p, B, kind in [(3000, 0.5, 40.0, "constant"), (3000, 0.37, 40.0, "ties"), (2500, 0.8, 30.0, "wide"),
                              (513, 0.6, 5.0, "signed_zero"), (4097, 0.95, 1e6, "normal"), (1, 0.5, 5.0, "normal"),
                              (2000, 0.2, 0.0, "needles")]:
        if kind == "constant":
            s = np.full((1, 2, N), 0.375)
        elif kind == "ties":
            s = np.round(rng.standard_normal((1, 2, N)) * 2) / 4
        elif kind == "wide":
            s = rng.standard_normal((1, 2, N)) * np.exp2(rng.integers(-10, 4, (1, 2, N)))
        elif kind == "signed_zero":
            s = np.where(rng.random((1, 2, N)) < 0.5, 0.0, -0.0) * np.ones((1, 2, N))
            s[..., ::7] = rng.standard_normal(s[..., ::7].shape)
        elif kind == "needles":
            s = rng.standard_normal((1, 2, N)) * 1.5
            s[..., rng.choice(N, 12, replace=False)] += 9.0
        else:
            s = rng.standard_normal((1, 2, N)) * 1.5
        _select_top_p_and_compare(oracle_mod, s.astype(np.float32), top_p, B, 4)


def test_select_top_p_limits(oracle_mod):
    """top_p <= 0: no stratum (the SSA sampler with k = 0); top_p >= 1: every token."""
    s_np = (np.random.default_rng(2).standard_normal((1, 2, 3000)) * 1.5).astype(np.float32)
    s = torch.from_numpy(s_np).to(DEV)
    idx, p, count = ssa.ssa_select_strata(s, ssa.STRATA_TOP_P, 0, 0.0, 30.0, 3)
    for h in range(2):
        o_idx, o_p, m, Z, p_all = oracle_mod.select_unit(s_np[0, h], 0, 30.0, 3, 0, h, want_p_all=True)
        n = int(count[0, h])
        compare_unit_lists(idx[0, h, :n].cpu().numpy(), p[0, h, :n].cpu().numpy(), o_idx, o_p, p_all,
                           lambda j: oracle_mod.uniform(3, j, h, 0))
    idx, p, count = ssa.ssa_select_strata(s, ssa.STRATA_TOP_P, 0, 1.0, 30.0, 3)
    assert torch.all(count == 3000)


def test_decode_top_p_parity(oracle_mod):
    """The whole step with the top-p stratum: the lists against the oracle's on the oracle's scores (stratum
    and sampling boundaries excepted), the output against the oracle's attention over the GPU's index set with
    the oracle's inclusion probabilities."""
    w = case("g4_d128")
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    Bt, Hkv, N = cfg.batch, cfg.n_kv_heads, cfg.ctx_len
    G = cfg.group
    top_p = 0.9
    idx = torch.empty((Bt, Hkv, N), dtype=torch.int32, device=DEV)
    p = torch.empty((Bt, Hkv, N), dtype=torch.float32, device=DEV)
    count = torch.empty((Bt, Hkv), dtype=torch.int32, device=DEV)
    out, lse = ssa.ssa_decode_strata(w["q"], w["K"], w["V"], w["Ks"], w["sel_ch"], ssa.STRATA_TOP_P, 0, top_p,
                                     cfg.budget, 9, cfg.scale, idx=idx, p=p, count=count)
    s_np = oracle_mod.score(q, Ks, sel, cfg.scale)
    for b in range(Bt):
        for h in range(Hkv):
            o_idx, o_p, m, Z = oracle_mod.select_unit_top_p(s_np[b, h], top_p, cfg.budget, 9, b, h)
            _, _, _, _, p_all = oracle_mod.select_unit(s_np[b, h], oracle_mod.top_p_count(s_np[b, h], top_p),
                                                       cfg.budget, 9, b, h, want_p_all=True)
            n = int(count[b, h])
            g_idx = idx[b, h, :n].cpu().numpy()
            assert len(set(g_idx.tolist()) ^ set(o_idx.tolist())) <= 3
            out_o, lse_o = oracle_mod.attend_unit(q[b, h * G:(h + 1) * G], K[b, h], V[b, h], g_idx, p_all[g_idx],
                                                  cfg.scale)
            assert np.allclose(out[b, h * G:(h + 1) * G].cpu().numpy(), out_o, atol=2e-3, rtol=2e-3)
            assert np.allclose(lse[b, h * G:(h + 1) * G].cpu().numpy(), lse_o, atol=2e-3, rtol=2e-3)
