"""GPU end-to-end decode parity at small sizes, every plan, and the special
cases the pages name (dense limit, pure top-k, uniform hybrid)."""
import contextlib
import math
import os

import numpy as np
import pytest
import torch

import long_context_decode_subset_b300 as ssa
import workloads
from gpu_e2e import check_unit, gpu_decode
from test_gpu_stages import SMALL, case, oracle_inputs, plan_env
from _util import u16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("plan", [(None, None), (512, 1), (512, 9), (1024, 64), (2048, 3)])
def test_decode_parity(oracle_mod, name, plan):
    w = case(name)
    cfg = w["cfg"]
    with plan_env(*plan):
        g = gpu_decode(w, cfg.top_k, cfg.budget, 1)
    assert g["status"] == 0, hex(g["flags"])
    stats = {}
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            check_unit(oracle_mod, w, g, b, h, cfg.top_k, cfg.budget, 1, stats)
    assert stats.get("units_differing", 0) <= max(1, stats["units"] // 8), stats


@pytest.mark.parametrize("name", ["tiny", "g4_d128", "g8_d128"])
def test_dense_limit_equals_dense_attention(oracle_mod, name):
    w = case(name)
    cfg = w["cfg"]
    g = gpu_decode(w, cfg.top_k, math.inf, 0)
    q, K, V, Ks, sel = oracle_inputs(w)
    d_out, d_lse = oracle_mod.dense_attention(q, K, V, cfg.scale)
    assert np.all(g["count"].cpu().numpy() == cfg.ctx_len)
    assert np.allclose(g["out"].cpu().numpy(), d_out, atol=2e-3, rtol=2e-3)
    assert np.allclose(g["lse"].cpu().numpy(), d_lse, atol=2e-3, rtol=2e-3)


def test_budget_zero_is_pure_topk(oracle_mod):
    w = case("g4_d128")
    cfg = w["cfg"]
    g = gpu_decode(w, cfg.top_k, 0.0, 0)
    assert np.all(g["count"].cpu().numpy() == cfg.top_k)
    assert torch.all(g["p"][..., :cfg.top_k] == 1.0)
    stats = {}
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            check_unit(oracle_mod, w, g, b, h, cfg.top_k, 0.0, 0, stats)


def test_zero_query_on_summary_is_uniform_hybrid(oracle_mod):
    w = dict(case("g4_d128"))
    cfg = w["cfg"]
    q = w["q"].clone()
    G = cfg.group
    for h in range(cfg.n_kv_heads):
        q[:, h * G:(h + 1) * G, w["sel_ch"][h].long()] = 0
    w["q"] = q
    g = gpu_decode(w, cfg.top_k, cfg.budget, 2)
    assert torch.all(g["s_hat"] == 0)
    N, k = cfg.ctx_len, cfg.top_k
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            n = int(g["count"][b, h])
            idx = g["idx"][b, h, :n].cpu().numpy()
            p = g["p"][b, h, :n].cpu().numpy()
            assert set(range(k)) <= set(idx.tolist())
            assert np.all(p[idx >= k] == np.float32(cfg.budget) / np.float32(N - k))
    stats = {}
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            check_unit(oracle_mod, w, g, b, h, k, cfg.budget, 2, stats)


def test_k_at_least_n_and_empty_context(oracle_mod):
    w = case("tiny")
    cfg = w["cfg"]
    g = gpu_decode(w, cfg.ctx_len + 3, 5.0, 0)
    assert int(g["count"][0, 0]) == cfg.ctx_len
    q, K, V, Ks, sel = oracle_inputs(w)
    d_out, d_lse = oracle_mod.dense_attention(q, K, V, cfg.scale)
    assert np.allclose(g["out"].cpu().numpy(), d_out, atol=2e-3, rtol=2e-3)
    # N = 0: nothing to attend to
    K0 = w["K"][:, :, :0]
    Ks0 = w["Ks"][:, :, :0]
    out, lse = ssa.ssa_decode(w["q"], K0, K0, Ks0, w["sel_ch"], 3, 3.0, 0, cfg.scale)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_decode_is_deterministic_and_seed_dependent():
    w = case("g4_d128")
    cfg = w["cfg"]
    a = gpu_decode(w, cfg.top_k, cfg.budget, 42)
    b = gpu_decode(w, cfg.top_k, cfg.budget, 42)
    c = gpu_decode(w, cfg.top_k, cfg.budget, 43)
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["lse"], b["lse"])
    assert torch.equal(a["count"], b["count"])

    def lists(g):  # the first count entries of every unit (the rest of each row is unwritten)
        return [g["idx"][bb, h, :int(g["count"][bb, h])].tolist()
                for bb in range(cfg.batch) for h in range(cfg.n_kv_heads)]

    assert lists(a) == lists(b)
    assert lists(a) != lists(c)


def test_decode_host_matches_device_path():
    w = case("g8_d128")
    cfg = w["cfg"]
    g = gpu_decode(w, cfg.top_k, cfg.budget, 9)
    q_host = w["q"].cpu().pin_memory()
    out_h = torch.empty(g["out"].shape, dtype=torch.float32).pin_memory()
    lse_h = torch.empty(g["lse"].shape, dtype=torch.float32).pin_memory()
    shape = ssa.shape_of(w["q"], w["K"], w["Ks"])
    ws = ssa.workspace(shape)
    ssa.ssa_decode_host(q_host, w["K"], w["V"], w["Ks"], w["sel_ch"], cfg.top_k, cfg.budget, 9, cfg.scale,
                        out_h, lse_h, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h, g["out"].cpu()) and torch.equal(lse_h, g["lse"].cpu())
    # pageable host buffers take the staged-copy path: the same results
    q_p = w["q"].cpu()
    out_p = torch.full(g["out"].shape, float("nan"))
    lse_p = torch.full(g["lse"].shape, float("nan"))
    assert not q_p.is_pinned()
    ssa.ssa_decode_host(q_p, w["K"], w["V"], w["Ks"], w["sel_ch"], cfg.top_k, cfg.budget, 9, cfg.scale,
                        out_p, lse_p, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_p, g["out"].cpu()) and torch.equal(lse_p, g["lse"].cpu())


def test_strided_cache_layout(oracle_mod):
    # K / V / Ks inside larger caches (capacity > N): batch and head strides differ from the packed ones
    w = case("g1_d64")
    cfg = w["cfg"]
    cap_tokens = cfg.ctx_len + 77 * 8
    Bt, Hkv, N, d = w["K"].shape
    bigK = torch.zeros((Bt, Hkv, cap_tokens, d), dtype=torch.bfloat16, device=DEV)
    bigV = torch.zeros_like(bigK)
    bigK[:, :, :N] = w["K"]
    bigV[:, :, :N] = w["V"]
    K = bigK[:, :, :N]
    V = bigV[:, :, :N]
    bigKs = torch.zeros((Bt, Hkv, cap_tokens, cfg.d_sel), dtype=torch.bfloat16, device=DEV)
    Ks = bigKs[:, :, :N]
    ssa.ssa_pack_summary(K, w["sel_ch"], Ks=Ks)
    assert torch.equal(Ks, w["Ks"])
    ref = gpu_decode(w, cfg.top_k, cfg.budget, 4)
    out, lse = ssa.ssa_decode(w["q"], K, V, Ks, w["sel_ch"], cfg.top_k, cfg.budget, 4, cfg.scale)
    assert torch.equal(out, ref["out"]) and torch.equal(lse, ref["lse"])


@contextlib.contextmanager
def hist_run_env(run):
    old = os.environ.get("SSA_FORCE_HIST_RUN")
    os.environ["SSA_FORCE_HIST_RUN"] = str(run)
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("SSA_FORCE_HIST_RUN", None)
        else:
            os.environ["SSA_FORCE_HIST_RUN"] = old


_LONG = {}


def _long_case():
    """Two units of 160K tokens: ~4 score stages per CTA, runs of ~3 stages of one unit."""
    if not _LONG:
        cfg = workloads.make_config("ministral8b_32k", batch=1, n_q_heads=8, n_kv_heads=2, ctx_len=163840,
                                    top_k=1638, budget=1638.0, n_needles=8)
        w = workloads.generate(cfg, 0, DEV)
        w["Ks"] = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
        torch.cuda.synchronize()
        _LONG["w"] = w
    return _LONG["w"]


@pytest.mark.parametrize("name", ["g4_d128", "long"])
@pytest.mark.parametrize("run", [1, 2])
def test_decode_parity_with_frequent_histogram_handover(oracle_mod, name, run):
    """The score kernel hands its shared histogram buffer to the flush warps at a change of unit and
    after every `run` stages of one unit (at most 127 normally, which only contexts of millions of
    tokens with few units reach): forcing a hand-over every stage or two must not change the result."""
    w = _long_case() if name == "long" else case(name)
    cfg = w["cfg"]
    with hist_run_env(run):
        g = gpu_decode(w, cfg.top_k, cfg.budget, 3)
    assert g["status"] == 0, hex(g["flags"])
    stats = {}
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            check_unit(oracle_mod, w, g, b, h, cfg.top_k, cfg.budget, 3, stats)
    assert stats.get("units_differing", 0) <= max(1, stats["units"] // 8), stats
    ref = gpu_decode(w, cfg.top_k, cfg.budget, 3)
    assert torch.equal(g["out"], ref["out"]) and torch.equal(g["count"], ref["count"])


def test_workspace_reuse_and_junk():
    """A workspace full of junk (apart from a cleared status word), and one reused across calls of every kind,
    give the results of a fresh zeroed workspace bit for bit: each call resets the counters its kernels meet
    on, including the calls that keep every token or attend given lists."""
    w = case("g4_d128")
    cfg = w["cfg"]
    q, K, V, Ks, sel = w["q"], w["K"], w["V"], w["Ks"], w["sel_ch"]
    shape = ssa.shape_of(q, K, Ks)
    N = cfg.ctx_len

    def junk_ws(shp):
        ws = ssa.workspace(shp)
        ws.fill_(0xA5)
        ssa.ssa_get_device_status(ws)   # clears the status word
        return ws

    def dec(ws, k, B, seed, s_hat=None):
        out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), device=DEV)
        lse = torch.full((cfg.batch, cfg.n_q_heads), float("nan"), device=DEV)
        ssa.ssa_decode(q, K, V, Ks, sel, k, B, seed, cfg.scale, out=out, lse=lse, s_hat=s_hat, ws=ws)
        return out, lse

    calls = [(cfg.top_k, cfg.budget, 3), (cfg.top_k, math.inf, 0), (N + 5, cfg.budget, 0), (0, cfg.budget, 4)]
    ref = [dec(None, *c) for c in calls]
    ws = junk_ws(shape)
    for _ in range(2):   # the second round finds the first one's counters
        for c, r in zip(calls, ref):
            out, lse = dec(ws, *c)
            assert torch.equal(out, r[0]) and torch.equal(lse, r[1]), c
    assert ssa.ssa_get_device_status(ws)[0] == 0

    # the stage entry points: selection (sparse and every token) and attention over given lists
    s_hat = ssa.ssa_score(q, Ks, sel, cfg.scale, K_like=K)
    s_shape_ws = junk_ws(ssa.ssa.make_shape(cfg.batch, cfg.n_kv_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_sel, N))
    for k, B in ((cfg.top_k, cfg.budget), (N, cfg.budget)):
        r_idx, r_p, r_cnt = ssa.ssa_select(s_hat, k, B, 9)
        for _ in range(2):
            idx, p, cnt = ssa.ssa_select(s_hat, k, B, 9, ws=s_shape_ws)
            assert torch.equal(cnt, r_cnt)
            for b in range(cfg.batch):
                for h in range(cfg.n_kv_heads):
                    n = int(cnt[b, h])
                    assert torch.equal(idx[b, h, :n], r_idx[b, h, :n]) and torch.equal(p[b, h, :n], r_p[b, h, :n])
    r_out, r_lse = ssa.ssa_attend(q, K, V, r_idx, r_p, r_cnt, cfg.scale)
    ws = junk_ws(shape)
    for _ in range(2):
        out = torch.full_like(r_out, float("nan"))
        lse = torch.full_like(r_lse, float("nan"))
        ssa.ssa_attend(q, K, V, r_idx, r_p, r_cnt, cfg.scale, out=out, lse=lse, ws=ws)
        assert torch.equal(out, r_out) and torch.equal(lse, r_lse)
