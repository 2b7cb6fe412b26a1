"""GPU parity at the full synthetic workload sizes, in the launch
configuration the benchmark times (the automatic plan).

* End to end (ssa_decode): the oracle recomputes units one by one from scratch
  (its own key summary, score, selection, attention) from the same inputs
  (gpu_e2e.check_unit); the units it does not recompute are checked through
  properties that hold at any size (counts, ascending order, p in (0, 1],
  top-k stratum present, finite outputs).
* Stage by stage at full size: ssa_select fed the oracle's scores must give the
  oracle's index sets on every unit (apart from tokens with |u - p| <= 1e-6,
  counted and printed) with p within 4 ulp; ssa_attend fed the oracle's lists
  must give out / lse within 2e-3 on every unit.
"""
import math

import numpy as np
import pytest
import torch

import long_context_decode_subset_b300 as ssa
import workloads
from _util import compare_unit_lists, u16
from gpu_e2e import check_unit, gpu_decode

pytestmark = pytest.mark.gpu

# (workload, seed, units recomputed by the oracle: None = every unit)
FULL = [("ministral8b_32k", 0, None)]
FULL += [("ministral8b_128k", s, None) for s in range(10)]
FULL += [
    ("ministral8b_1m", 0, None),
    ("27b_128k_10x", 0, 8),
    ("27b_128k_20x", 0, 8),
    ("27b_128k_50x", 0, 8),
    ("27b_128k_100x", 0, 8),
    ("27b_128k_dense", 0, 4),
]


def _properties(g, cfg):
    count = g["count"].cpu().numpy()
    N, k, B = cfg.ctx_len, cfg.top_k, cfg.budget
    if math.isinf(B):
        assert np.all(count == N)
    else:
        assert np.all(count >= min(k, N))
        # E[count] = k + sum_R p <= k + B; a Poisson count stays far below +8 sigma
        assert np.all(count <= k + B + 8 * math.sqrt(B + 1) + 1)
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            n = int(count[b, h])
            idx = g["idx"][b, h, :n]
            p = g["p"][b, h, :n]
            assert bool(torch.all(idx[1:] > idx[:-1])), "not ascending"
            assert bool(torch.all((p > 0) & (p <= 1)))
            assert int((p == 1).sum()) >= min(k, n)
    assert torch.isfinite(g["out"]).all() and torch.isfinite(g["lse"]).all()


def _units(cfg, sample, seed):
    units = [(b, h) for b in range(cfg.batch) for h in range(cfg.n_kv_heads)]
    if sample is not None and sample < len(units):
        rng = np.random.default_rng(seed + 17)
        units = [units[i] for i in sorted(rng.choice(len(units), size=sample, replace=False))]
    return units


@pytest.mark.parametrize("name,seed,sample", FULL)
def test_full_size_parity(oracle_mod, name, seed, sample):
    cfg = workloads.CONFIGS[name]
    w = workloads.generate(cfg, seed, "cuda")
    w["Ks"] = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    g = gpu_decode(w, cfg.top_k, cfg.budget, seed)
    assert g["status"] == 0, hex(g["flags"])
    _properties(g, cfg)
    stats = {}
    for b, h in _units(cfg, sample, seed):
        check_unit(oracle_mod, w, g, b, h, cfg.top_k, cfg.budget, seed, stats)
    print(name, seed, stats)
    del w, g
    torch.cuda.empty_cache()


def _oracle_scores(oracle_mod, w, cfg):
    """The oracle's scores of every unit, from its own key summary."""
    K, sel = u16(w["K"]), w["sel_ch"].cpu().numpy()
    Ks = oracle_mod.pack_summary(K, sel, cfg.d_sel)
    return oracle_mod.score(u16(w["q"]), Ks, sel, cfg.scale)


@pytest.mark.parametrize("name", ["ministral8b_128k", "ministral8b_1m", "27b_128k_10x"])
def test_full_size_select_given_oracle_scores(oracle_mod, name):
    cfg = workloads.CONFIGS[name]
    seed = 4
    w = workloads.generate(cfg, 0, "cuda")
    s_np = _oracle_scores(oracle_mod, w, cfg)
    del w
    torch.cuda.empty_cache()
    s = torch.from_numpy(s_np).cuda()
    shape = ssa.make_shape(cfg.batch, cfg.n_kv_heads, cfg.n_kv_heads, 64, 16, cfg.ctx_len)
    ws = ssa.workspace(shape, cfg.ctx_len)
    idx, p, count = ssa.ssa_select(s, cfg.top_k, cfg.budget, seed, ws=ws)
    st, flags = ssa.ssa_get_device_status(ws)
    assert st == 0, hex(flags)
    idx, p, count = idx.cpu().numpy(), p.cpu().numpy(), count.cpu().numpy()
    boundary = 0
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            o_idx, o_p, m, Z, p_all = oracle_mod.select_unit(s_np[b, h], cfg.top_k, cfg.budget, seed, b, h,
                                                             want_p_all=True)
            n = int(count[b, h])
            nd, _ = compare_unit_lists(idx[b, h, :n], p[b, h, :n], o_idx, o_p, p_all,
                                       lambda j: oracle_mod.uniform(seed, j, h, b))
            boundary += nd
            assert np.all(np.diff(idx[b, h, :n]) > 0)
    print(f"{name}: {cfg.units} units, {boundary} boundary tokens (|u - p| <= 1e-6)")


@pytest.mark.parametrize("name", ["ministral8b_128k", "ministral8b_1m"])
def test_full_size_attend_given_oracle_lists(oracle_mod, name):
    cfg = workloads.CONFIGS[name]
    seed = 2
    w = workloads.generate(cfg, 0, "cuda")
    s_np = _oracle_scores(oracle_mod, w, cfg)
    G = cfg.group
    lists = {}
    cap = 1
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            o_idx, o_p, _, _ = oracle_mod.select_unit(s_np[b, h], cfg.top_k, cfg.budget, seed, b, h)
            lists[b, h] = (o_idx, o_p)
            cap = max(cap, o_idx.size)
    idx = np.zeros((cfg.batch, cfg.n_kv_heads, cap), np.int32)
    p = np.ones((cfg.batch, cfg.n_kv_heads, cap), np.float32)
    count = np.zeros((cfg.batch, cfg.n_kv_heads), np.int32)
    for (b, h), (o_idx, o_p) in lists.items():
        idx[b, h, :o_idx.size] = o_idx
        p[b, h, :o_p.size] = o_p
        count[b, h] = o_idx.size
    out, lse = ssa.ssa_attend(w["q"], w["K"], w["V"], torch.from_numpy(idx).cuda(), torch.from_numpy(p).cuda(),
                              torch.from_numpy(count).cuda(), cfg.scale)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    worst = 0.0
    for (b, h), (o_idx, o_p) in lists.items():
        qh = u16(w["q"][b, h * G:(h + 1) * G])
        out_o, lse_o = oracle_mod.attend_unit(qh, u16(w["K"][b, h]), u16(w["V"][b, h]), o_idx, o_p, cfg.scale)
        og, lg = out[b, h * G:(h + 1) * G], lse[b, h * G:(h + 1) * G]
        assert np.allclose(og, out_o, atol=2e-3, rtol=2e-3), (b, h, np.abs(og - out_o).max())
        assert np.allclose(lg, lse_o, atol=2e-3, rtol=2e-3), (b, h, np.abs(lg - lse_o).max())
        worst = max(worst, float(np.abs(og - out_o).max()))
    print(f"{name}: every unit within 2e-3, max |out - oracle| = {worst:.2e}")


def test_full_size_uniform_hybrid_given_oracle_scores(oracle_mod):
    """The top-k + uniform hybrid at the 128K workload in the automatic plan: identical lists, p bit for bit."""
    cfg = workloads.CONFIGS["ministral8b_128k"]
    seed = 6
    w = workloads.generate(cfg, 0, "cuda")
    s_np = _oracle_scores(oracle_mod, w, cfg)
    del w
    idx, p, count = ssa.ssa_select_strata(torch.from_numpy(s_np).cuda(), ssa.ssa.STRATA_UNIFORM, cfg.top_k, 0.0,
                                          cfg.budget, seed)
    idx, p, count = idx.cpu().numpy(), p.cpu().numpy(), count.cpu().numpy()
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            o_idx, o_p = oracle_mod.select_unit_uniform(s_np[b, h], cfg.top_k, cfg.budget, seed, b, h)
            n = int(count[b, h])
            assert np.array_equal(idx[b, h, :n], o_idx) and np.array_equal(p[b, h, :n], o_p), (b, h)


def test_full_size_top_p_given_oracle_scores(oracle_mod):
    """The top-p stratum at the 128K workload in the automatic plan: the stratum's size and set against the
    oracle's (a size one off only where top_p falls within 2e-6 of the stratum's edge), the sampled lists as
    the oracle's SSA sampler draws them for that size."""
    cfg = workloads.CONFIGS["ministral8b_128k"]
    w = workloads.generate(cfg, 0, "cuda")
    s_np = _oracle_scores(oracle_mod, w, cfg)
    del w
    s = torch.from_numpy(s_np).cuda()
    top_p, seed = 0.9, 8
    i0, _, c0 = ssa.ssa_select_strata(s, ssa.STRATA_TOP_P, 0, top_p, 0.0, seed)
    idx, p, count = ssa.ssa_select_strata(s, ssa.STRATA_TOP_P, 0, top_p, cfg.budget, seed)
    i0, c0 = i0.cpu().numpy(), c0.cpu().numpy()
    idx, p, count = idx.cpu().numpy(), p.cpu().numpy(), count.cpu().numpy()
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            k_o, before, at = oracle_mod.top_p_shares(s_np[b, h], top_p)
            k = int(c0[b, h])
            assert k == k_o or (k == k_o - 1 and top_p - before <= 2e-6) or (k == k_o + 1 and at - top_p <= 2e-6)
            assert np.array_equal(i0[b, h, :k], oracle_mod.select_unit(s_np[b, h], k, 0.0, seed, b, h)[0])
            o_idx, o_p, m, Z, p_all = oracle_mod.select_unit(s_np[b, h], k, cfg.budget, seed, b, h, want_p_all=True)
            n = int(count[b, h])
            compare_unit_lists(idx[b, h, :n], p[b, h, :n], o_idx, o_p, p_all,
                               lambda j: oracle_mod.uniform(seed, j, h, b))
