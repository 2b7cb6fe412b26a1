"""The paged, variable-length cache (ssa_decode_paged).

A serving batch keeps each sequence's K, V and key summary in fixed-size pages
of shared pools, found through a block table, and its sequences have
different lengths.  The step for unit (b, h) is the method's step over that
sequence's own tokens ("Stratified Sparse Attention speeds up decoding 2.96x
on a 1M context", problem statement: query, KV cache, k, B, seed; the Philox
counter of a token is its position in its sequence).

* Same data, every length = ctx_len: the pools only move rows, so out, lse,
  scores, lists and counts must equal the contiguous ssa_decode's bit for bit,
  for page sizes from 16 tokens (32 pages per 512-token stage of the score
  kernel) to larger than a stage.
* Ragged lengths (empty, one token, shorter than k, the full bound, and ends
  inside a page): every unit against the oracle over its own tokens
  (gpu_e2e.check_unit), with pool slots and block-table entries outside the
  sequences filled with junk that must not be read.
* The fused append writes each sequence's new token into its page.
* A bad page id or length is flagged, not faulted on.
"""
import os

import numpy as np
import pytest
import torch

import long_context_decode_subset_b300 as ssa
import workloads
from gpu_e2e import check_unit

pytestmark = pytest.mark.gpu

SMALL = workloads.make_config("ministral8b_32k", batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=5000,
                              top_k=50, budget=50.0, n_needles=8)
SMALL64 = workloads.make_config("tiny", batch=3, n_q_heads=8, n_kv_heads=2, ctx_len=3000, top_k=40, budget=40.0,
                                n_needles=4)


def _workload(cfg, seed):
    w = workloads.generate(cfg, seed, "cuda")
    w["Ks"] = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    return w


def _outputs(Bt, Hq, Hkv, d, N, cap):
    dev = "cuda"
    return dict(s_hat=torch.full((Bt, Hkv, N), float("nan"), device=dev),
                idx=torch.full((Bt, Hkv, cap), -1, dtype=torch.int32, device=dev),
                p=torch.full((Bt, Hkv, cap), float("nan"), device=dev),
                count=torch.full((Bt, Hkv), -1, dtype=torch.int32, device=dev))


def _paged_decode(w, pg, k, B, seed, N, k_new=None, v_new=None):
    q = w["q"]
    Bt, Hq, d = q.shape
    Hkv = w["K"].shape[1]
    cap = max(N, 1)
    o = _outputs(Bt, Hq, Hkv, d, N, cap)
    shape = ssa.paged_shape(q, pg["K_pool"], pg["Ks_pool"], N)
    ws = ssa.workspace(shape, cap)
    out, lse = ssa.ssa_decode_paged(q, pg["K_pool"], pg["V_pool"], pg["Ks_pool"], pg["block_table"], pg["seq_lens"],
                                    w["sel_ch"], k, B, seed, w["scale"], N, k_new=k_new, v_new=v_new, list_cap=cap,
                                    ws=ws, **o)
    st, flags = ssa.ssa_get_device_status(ws)
    return dict(out=out, lse=lse, status=st, flags=flags, **o)


def _contig_decode(w, k, B, seed, N):
    q = w["q"]
    Bt, Hq, d = q.shape
    Hkv = w["K"].shape[1]
    cap = max(N, 1)
    o = _outputs(Bt, Hq, Hkv, d, N, cap)
    out, lse = ssa.ssa_decode(q, w["K"], w["V"], w["Ks"], w["sel_ch"], k, B, seed, w["scale"], list_cap=cap, **o)
    torch.cuda.synchronize()
    return dict(out=out, lse=lse, **o)


@pytest.mark.parametrize("cfg", [SMALL, SMALL64], ids=["d128", "d64"])
@pytest.mark.parametrize("page_size", [16, 64, 256, 2048])
def test_paged_equals_contiguous_bit_for_bit(cfg, page_size):
    w = _workload(cfg, 1)
    N = cfg.ctx_len
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], [N] * cfg.batch, page_size, seed=3)
    for k, B, seed in ((cfg.top_k, cfg.budget, 7), (0, 2.0 * cfg.budget, 8), (cfg.top_k, float("inf"), 0)):
        g = _paged_decode(w, pg, k, B, seed, N)
        r = _contig_decode(w, k, B, seed, N)
        assert g["status"] == 0, hex(g["flags"])
        for key in ("out", "lse", "s_hat", "count"):
            assert torch.equal(g[key], r[key]), (key, k, B)
        c = r["count"]
        for b in range(cfg.batch):
            for h in range(cfg.n_kv_heads):
                n = int(c[b, h])
                assert torch.equal(g["idx"][b, h, :n], r["idx"][b, h, :n])
                assert torch.equal(g["p"][b, h, :n], r["p"][b, h, :n])


def _ragged(cfg, page_size):
    N, k = cfg.ctx_len, cfg.top_k
    lens = [N, 0, 1, k - 1, k + 1, N // 3 + 17, page_size * 3, 2 * page_size + 5, 513, N - 1]
    return [min(max(n, 0), N) for n in lens][:cfg.batch]


@pytest.mark.parametrize("split", [None, 3])
@pytest.mark.parametrize("page_size", [16, 128, 1024])
def test_paged_ragged_lengths_match_the_oracle(oracle_mod, page_size, split, monkeypatch):
    if split is not None:
        monkeypatch.setenv("SSA_FORCE_SPLIT", str(split))
    cfg = workloads.make_config("ministral8b_32k", batch=10, n_q_heads=8, n_kv_heads=2, ctx_len=4500,
                                top_k=45, budget=45.0, n_needles=8)
    w = _workload(cfg, 2)
    lens = _ragged(cfg, page_size)
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], lens, page_size, seed=5)
    seed = 11
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, seed, cfg.ctx_len)
    assert g["status"] == 0, hex(g["flags"])
    stats = {}
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            n = lens[b]
            if n == 0:
                G = cfg.group
                assert int(g["count"][b, h]) == 0
                assert torch.all(g["out"][b, h * G:(h + 1) * G] == 0)
                assert torch.all(torch.isneginf(g["lse"][b, h * G:(h + 1) * G]))
                continue
            if n <= cfg.top_k:   # the whole sequence is the stratum
                assert int(g["count"][b, h]) == n
                assert torch.equal(g["idx"][b, h, :n].cpu(), torch.arange(n, dtype=torch.int32))
                assert torch.all(g["p"][b, h, :n] == 1)
            check_unit(oracle_mod, w, g, b, h, cfg.top_k, cfg.budget, seed, stats, n=n)
    print(page_size, split, stats)


def test_paged_ragged_dense_limit(oracle_mod):
    """budget = +inf: every token of every sequence with p = 1 (the oracle's dense attention per sequence)."""
    cfg = SMALL64
    w = _workload(cfg, 4)
    lens = [cfg.ctx_len, 700, 0]
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], lens, 64, seed=1)
    g = _paged_decode(w, pg, cfg.top_k, float("inf"), 0, cfg.ctx_len)
    assert g["status"] == 0, hex(g["flags"])
    stats = {}
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            if lens[b]:
                check_unit(oracle_mod, w, g, b, h, cfg.top_k, float("inf"), 0, stats, n=lens[b])
    assert stats["units"] == 4


def test_paged_append_writes_each_sequence_in_its_page():
    cfg = SMALL
    w = _workload(cfg, 6)
    N = cfg.ctx_len
    dev = "cuda"
    k_new = torch.randn((cfg.batch, cfg.n_kv_heads, cfg.head_dim), device=dev).to(torch.bfloat16)
    v_new = torch.randn((cfg.batch, cfg.n_kv_heads, cfg.head_dim), device=dev).to(torch.bfloat16)
    # every sequence full: the same step as the contiguous fused append
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], [N] * cfg.batch, 64, seed=2)
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, 3, N, k_new=k_new, v_new=v_new)
    assert g["status"] == 0, hex(g["flags"])
    Kc, Vc, Ksc = w["K"].clone(), w["V"].clone(), w["Ks"].clone()
    out_r, lse_r = ssa.ssa_decode_append(w["q"], k_new, v_new, Kc, Vc, Ksc, w["sel_ch"], cfg.top_k, cfg.budget, 3,
                                         w["scale"])
    torch.cuda.synchronize()
    assert torch.equal(g["out"], out_r) and torch.equal(g["lse"], lse_r)
    # ragged: the new row lands at seq_lens[b] - 1 of each non-empty sequence, in its page
    lens = [N // 2 + 3, 0]
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], lens, 64, seed=4)
    before = {k: pg[k].clone() for k in ("K_pool", "V_pool", "Ks_pool")}
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, 3, N, k_new=k_new, v_new=v_new)
    assert g["status"] == 0, hex(g["flags"])
    pos = lens[0] - 1
    page = int(pg["block_table"][0, pos // 64])
    sel = w["sel_ch"].long()
    assert torch.equal(pg["K_pool"][page, :, pos % 64], k_new[0])
    assert torch.equal(pg["V_pool"][page, :, pos % 64], v_new[0])
    for h in range(cfg.n_kv_heads):
        assert torch.equal(pg["Ks_pool"][page, h, pos % 64], k_new[0, h, sel[h]])
    changed = [(before[k] != pg[k]).any(dim=-1).nonzero().tolist() for k in ("K_pool", "V_pool")]
    for c in changed:   # nothing else was written
        assert all(p == page and s == pos % 64 for p, _, s in c), c


def test_paged_bad_page_or_length_is_flagged():
    cfg = SMALL64
    w = _workload(cfg, 0)
    N = cfg.ctx_len
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], [N, 900, 5], 64, seed=0)
    pg["block_table"][1, 3] = pg["K_pool"].shape[0] + 7       # a page of sequence 1 past the pool
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, 0, N)
    assert g["status"] == 8 and g["flags"] & ssa.ssa.DEV_BAD_INDEX
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], [N, 900, 5], 64, seed=0)
    pg["block_table"][2, 0] = -3
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, 0, N)
    assert g["status"] == 8
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], [N, 900, 5], 64, seed=0)
    pg["seq_lens"][1] = N + 1                                   # longer than the bound
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, 0, N)
    assert g["status"] == 8
    # the next step on the same data is clean again
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], [N, 900, 5], 64, seed=0)
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, 0, N)
    assert g["status"] == 0


@pytest.mark.parametrize("name", ["ministral8b_128k"])
def test_paged_full_size_ragged(oracle_mod, name):
    """The 128K workload as a paged batch (256-token pages) with one full and one ragged sequence, in the
    automatic plan: sampled units against the oracle, the rest through properties."""
    cfg = workloads.CONFIGS[name]
    w = _workload(cfg, 0)
    N = cfg.ctx_len
    lens = [N, N // 2 + 1234]
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], lens, 256, seed=9)
    seed = 5
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, seed, N)
    assert g["status"] == 0, hex(g["flags"])
    count = g["count"].cpu().numpy()
    for b in range(cfg.batch):
        assert np.all(count[b] >= min(cfg.top_k, lens[b]))
    stats = {}
    for b, h in ((0, 0), (0, 5), (1, 2), (1, 7)):
        check_unit(oracle_mod, w, g, b, h, cfg.top_k, cfg.budget, seed, stats, n=lens[b])
    print(stats)
    # with both sequences full the paged step equals the contiguous one bit for bit
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], [N, N], 256, seed=9)
    g = _paged_decode(w, pg, cfg.top_k, cfg.budget, seed, N)
    r = _contig_decode(w, cfg.top_k, cfg.budget, seed, N)
    assert torch.equal(g["out"], r["out"]) and torch.equal(g["lse"], r["lse"])
    assert torch.equal(g["count"], r["count"])
