"""S2O-style early stopping of the attention (ssa_attend_early_stop, ssa_decode_early_stop).

"S2O: early stopping for sparse attention via online permutation", technical
summary, Method section 2: blocks processed in descending estimated
importance, the marginal gain of each tracked, and the computation ended once
that gain falls below tau relative to the accumulated score.  Here the blocks
are 128 rows of a unit's selected list in descending score order.

* Stage parity: the oracle's own lists and scores go into
  ssa_attend_early_stop; the number of blocks kept must equal the oracle's,
  or differ by one only where the oracle's gain ratio at the deciding block
  lies within 1e-4 (relative) of tau (the kernel tests it in fp32); out / lse
  must match the oracle's attention over the kernel's block count within
  2e-3.
* The decode chain is the selection of ssa_decode followed by that stage:
  its result equals ssa_decode's lists and scores fed to
  ssa_attend_early_stop, bit for bit.
* Limits: tau = 0 keeps every block (ssa_attend's result up to summation
  order), tau > 1 only the first; empty lists; lists longer than the order
  kernel holds are flagged.
"""
import math

import numpy as np
import pytest
import torch

import long_context_decode_subset_b300 as ssa
import workloads
from _util import u16
from test_gpu_stages import SMALL, case, oracle_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
TAUS = [0.0, 1e-5, 1e-4, 1e-3, 1e-2, 0.05, 0.3, 2.0]


def _oracle_lists(oracle_mod, s_np, k, B, seed):
    Bt, Hkv, N = s_np.shape
    lists = {}
    cap = 1
    for b in range(Bt):
        for h in range(Hkv):
            o_idx, o_p, _, _ = oracle_mod.select_unit(s_np[b, h], k, B, seed, b, h)
            lists[b, h] = (o_idx, o_p)
            cap = max(cap, o_idx.size)
    idx = np.zeros((Bt, Hkv, cap), np.int32)
    p = np.ones((Bt, Hkv, cap), np.float32)
    count = np.zeros((Bt, Hkv), np.int32)
    for (b, h), (o_idx, o_p) in lists.items():
        idx[b, h, :o_idx.size] = o_idx
        p[b, h, :o_p.size] = o_p
        count[b, h] = o_idx.size
    return lists, idx, p, count


def _check_stage(oracle_mod, w, s_np, lists, idx, p, count, taus, stats):
    cfg = w["cfg"]
    G = cfg.group
    qh_all, K_all, V_all = u16(w["q"]), u16(w["K"]), u16(w["V"])
    t = lambda a: torch.from_numpy(a).to(DEV)
    for tau in taus:
        out, lse, blocks = ssa.ssa_attend_early_stop(w["q"], w["K"], w["V"], t(idx), t(p), t(count), t(s_np), tau,
                                                     cfg.scale)
        out, lse, blocks = out.cpu().numpy(), lse.cpu().numpy(), blocks.cpu().numpy()
        for (b, h), (o_idx, o_p) in lists.items():
            qh = qh_all[b, h * G:(h + 1) * G]
            s_rows = s_np[b, h][o_idx]
            _, _, used, ratios = oracle_mod.attend_unit_early_stop(qh, K_all[b, h], V_all[b, h], o_idx, o_p, s_rows,
                                                                   cfg.scale, tau)
            gb = int(blocks[b, h])
            if gb != used:
                # only a block whose gain ratio sits at tau may be decided the other way
                edge = min(gb, used)   # the block (1-based) one side stopped at
                r = float(ratios[edge - 1]) if edge >= 1 else 1.0
                assert abs(gb - used) == 1 and abs(r - tau) <= 1e-4 * tau, (b, h, tau, gb, used, r)
                stats["edge"] = stats.get("edge", 0) + 1
            o_out, o_lse, _, _ = oracle_mod.attend_unit_early_stop(qh, K_all[b, h], V_all[b, h], o_idx, o_p, s_rows,
                                                                   cfg.scale, tau, force_blocks=gb)
            og, lg = out[b, h * G:(h + 1) * G], lse[b, h * G:(h + 1) * G]
            assert np.allclose(og, o_out, atol=2e-3, rtol=2e-3), (b, h, tau, np.abs(og - o_out).max())
            if o_idx.size:
                assert np.allclose(lg, o_lse, atol=2e-3, rtol=2e-3), (b, h, tau)
            else:
                assert gb == 0 and np.all(og == 0) and np.all(np.isneginf(lg))
            stats["blocks"] = stats.get("blocks", 0) + gb


@pytest.mark.parametrize("name", ["g4_d128", "g8_d128", "g1_d64", "g2_d128_s16"])
def test_attend_early_stop_matches_the_oracle(oracle_mod, name):
    w = case(name)
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    s_np = oracle_mod.score(q, Ks, sel, cfg.scale)
    # a larger stratum than the config's so that units have several blocks
    k, B = min(cfg.ctx_len, 6 * cfg.top_k + 5), 4.0 * cfg.budget
    lists, idx, p, count = _oracle_lists(oracle_mod, s_np, k, B, 3)
    stats = {}
    _check_stage(oracle_mod, w, s_np, lists, idx, p, count, TAUS, stats)
    print(name, stats)


def test_attend_early_stop_limits_and_empty_lists(oracle_mod):
    w = case("g4_d128")
    cfg = w["cfg"]
    q, K, V, Ks, sel = oracle_inputs(w)
    s_np = oracle_mod.score(q, Ks, sel, cfg.scale)
    lists, idx, p, count = _oracle_lists(oracle_mod, s_np, 700, 300.0, 5)
    count[0, 1] = 0   # an empty list
    lists[0, 1] = (np.zeros(0, np.int32), np.zeros(0, np.float32))
    t = lambda a: torch.from_numpy(a).to(DEV)
    out0, lse0, b0 = ssa.ssa_attend_early_stop(w["q"], w["K"], w["V"], t(idx), t(p), t(count), t(s_np), 0.0,
                                               cfg.scale)
    ref_out, ref_lse = ssa.ssa_attend(w["q"], w["K"], w["V"], t(idx), t(p), t(count), cfg.scale)
    assert torch.allclose(out0, ref_out, atol=1e-5, rtol=1e-5) and torch.allclose(lse0, ref_lse, atol=1e-5, rtol=1e-5)
    assert torch.equal(b0.cpu(), torch.from_numpy((count + 127) // 128))
    _, _, b2 = ssa.ssa_attend_early_stop(w["q"], w["K"], w["V"], t(idx), t(p), t(count), t(s_np), 2.0, cfg.scale)
    assert torch.equal(b2.cpu(), torch.from_numpy(np.minimum(count, 1)))
    _, _, binf = ssa.ssa_attend_early_stop(w["q"], w["K"], w["V"], t(idx), t(p), t(count), t(s_np), math.inf,
                                           cfg.scale)
    assert torch.equal(binf, b2)
    stats = {}
    _check_stage(oracle_mod, w, s_np, lists, idx, p, count, [0.0, 1e-3, 2.0], stats)


def test_order_capacity_is_flagged():
    cfg = workloads.make_config("ministral8b_32k", batch=1, n_q_heads=4, n_kv_heads=1, ctx_len=40000,
                                top_k=10, budget=10.0, n_needles=4)
    w = workloads.generate(cfg, 0, DEV)
    s = torch.randn((1, 1, cfg.ctx_len), device=DEV)
    n = 33000   # past the 32768 rows the order kernel holds
    idx = torch.arange(n, dtype=torch.int32, device=DEV).view(1, 1, n)
    p = torch.ones((1, 1, n), device=DEV)
    count = torch.full((1, 1), n, dtype=torch.int32, device=DEV)
    ws = ssa.workspace(ssa.shape_of(w["q"], w["K"]), n)
    out, lse, blocks = ssa.ssa_attend_early_stop(w["q"], w["K"], w["V"], idx, p, count, s, 0.0, cfg.scale, ws=ws)
    st, flags = ssa.ssa_get_device_status(ws)
    assert st == 5 and flags & ssa.ssa.DEV_OVERFLOW
    assert int(blocks[0, 0]) == 32768 // 128 and torch.isfinite(out).all()


@pytest.mark.parametrize("name", ["g4_d128", "g8_d128", "g2_d128_s16"])
def test_decode_early_stop_is_the_selection_then_the_stage(name):
    w = case(name)
    cfg = w["cfg"]
    q, K, V, Ks, sel = w["q"], w["K"], w["V"], w["Ks"], w["sel_ch"]
    Bt, Hkv, N = cfg.batch, cfg.n_kv_heads, cfg.ctx_len
    for k, B, seed in ((cfg.top_k, cfg.budget, 1), (4 * cfg.top_k, 3 * cfg.budget, 2), (cfg.top_k, math.inf, 0)):
        s_hat = torch.empty((Bt, Hkv, N), device=DEV)
        idx = torch.empty((Bt, Hkv, N), dtype=torch.int32, device=DEV)
        p = torch.empty((Bt, Hkv, N), device=DEV)
        count = torch.empty((Bt, Hkv), dtype=torch.int32, device=DEV)
        ssa.ssa_decode(q, K, V, Ks, sel, k, B, seed, cfg.scale, s_hat=s_hat, idx=idx, p=p, count=count, list_cap=N)
        for tau in (0.0, 1e-3, 0.05):
            out, lse, blocks = ssa.ssa_decode_early_stop(q, K, V, Ks, sel, k, B, seed, cfg.scale, tau)
            r_out, r_lse, r_blocks = ssa.ssa_attend_early_stop(q, K, V, idx, p, count, s_hat, tau, cfg.scale)
            torch.cuda.synchronize()
            assert torch.equal(blocks, r_blocks) and torch.equal(out, r_out) and torch.equal(lse, r_lse), (k, B, tau)
    # tau = 0 is the plain step up to the order of the sums
    d_out, d_lse = ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 7, cfg.scale)
    e_out, e_lse, _ = ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 7, cfg.scale, 0.0)
    assert torch.allclose(e_out, d_out, atol=1e-5, rtol=1e-5) and torch.allclose(e_lse, d_lse, atol=1e-5, rtol=1e-5)


def test_early_stop_full_size_128k(oracle_mod):
    """The 128K workload: the decode chain equals selection + stage; the stage matches the oracle on its own
    lists and scores for sampled units."""
    cfg = workloads.CONFIGS["ministral8b_128k"]
    w = workloads.generate(cfg, 0, DEV)
    w["Ks"] = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    q, K, V, Ks, sel = w["q"], w["K"], w["V"], w["Ks"], w["sel_ch"]
    Bt, Hkv, N = cfg.batch, cfg.n_kv_heads, cfg.ctx_len
    seed, tau = 3, 1e-3
    s_hat = torch.empty((Bt, Hkv, N), device=DEV)
    idx = torch.empty((Bt, Hkv, N), dtype=torch.int32, device=DEV)
    p = torch.empty((Bt, Hkv, N), device=DEV)
    count = torch.empty((Bt, Hkv), dtype=torch.int32, device=DEV)
    ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, seed, cfg.scale, s_hat=s_hat, idx=idx, p=p, count=count,
                   list_cap=N)
    out, lse, blocks = ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, seed, cfg.scale, tau)
    r_out, r_lse, r_blocks = ssa.ssa_attend_early_stop(q, K, V, idx, p, count, s_hat, tau, cfg.scale)
    assert torch.equal(blocks, r_blocks) and torch.equal(out, r_out) and torch.equal(lse, r_lse)
    nb = (count + 127) // 128
    assert torch.all(blocks >= 1) and torch.all(blocks <= nb)
    print("blocks kept", blocks.cpu().tolist(), "of", nb.cpu().tolist())
    # stage parity on the oracle's own inputs for two units
    qn, Kn, Vn, Ksn, seln = oracle_inputs(dict(w, cfg=cfg))
    s_np = oracle_mod.score(qn, Ksn, seln, cfg.scale)
    lists, o_idx, o_p, o_count = _oracle_lists(oracle_mod, s_np, cfg.top_k, cfg.budget, seed)
    keep = {(0, 0), (1, 5)}
    for key in list(lists):
        if key not in keep:
            o_count[key] = 0
            lists[key] = (np.zeros(0, np.int32), np.zeros(0, np.float32))
    stats = {}
    _check_stage(oracle_mod, dict(w, cfg=cfg), s_np, lists, o_idx, o_p, o_count, [1e-4, 1e-3, 1e-2], stats)
    print(stats)
