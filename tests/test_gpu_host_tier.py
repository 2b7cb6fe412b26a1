"""The host-resident memory tier ("FASA: Frequency-Aware Sparse Attention",
section 3, Variants, FASA-M: the dominant-channel summary stays in GPU memory,
the full K and V rows are offloaded to host memory and fetched only for the
selected tokens).

K and V are pinned host tensors (mapped into the device's address space at the
same address); the key summary, the query and the workspace stay on the
device.  The step runs the same kernels, so its results must equal the
device-resident step's bit for bit.  Pageable host memory is refused before
anything is launched.
"""
import pytest
import torch

import long_context_decode_subset_b300 as ssa
import workloads

pytestmark = pytest.mark.gpu

SMALL = workloads.make_config("ministral8b_32k", batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=5000,
                              top_k=50, budget=50.0, n_needles=8)


def _pinned(t):
    return t.cpu().pin_memory()


@pytest.mark.parametrize("name", ["small", "ministral8b_32k"])
def test_host_resident_kv_matches_device_resident(name):
    cfg = SMALL if name == "small" else workloads.CONFIGS[name]
    w = workloads.generate(cfg, 1, "cuda")
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    Ks = ssa.ssa_pack_summary(K, sel)
    Kh, Vh = _pinned(K), _pinned(V)
    for seed in (3, 4):
        out_d, lse_d = ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, seed, cfg.scale)
        out_h, lse_h = ssa.ssa_decode(q, Kh, Vh, Ks, sel, cfg.top_k, cfg.budget, seed, cfg.scale)
        torch.cuda.synchronize()
        assert torch.equal(out_h, out_d) and torch.equal(lse_h, lse_d)
    # the dense limit and the attention entry point read the host rows too
    out_d, _ = ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, float("inf"), 0, cfg.scale)
    out_h, _ = ssa.ssa_decode(q, Kh, Vh, Ks, sel, cfg.top_k, float("inf"), 0, cfg.scale)
    assert torch.equal(out_h, out_d)
    Bt, Hkv = cfg.batch, cfg.n_kv_heads
    idx = torch.arange(0, cfg.ctx_len, 7, dtype=torch.int32, device="cuda").repeat(Bt, Hkv, 1)
    p = torch.full(idx.shape, 0.5, device="cuda")
    count = torch.full((Bt, Hkv), idx.shape[-1], dtype=torch.int32, device="cuda")
    a_d, _ = ssa.ssa_attend(q, K, V, idx, p, count, cfg.scale)
    a_h, _ = ssa.ssa_attend(q, Kh, Vh, idx, p, count, cfg.scale)
    assert torch.equal(a_h, a_d)


def test_host_resident_append_step():
    """The serving form with the cache in host memory: the new token's K/V rows are written to host memory
    by the chain's first kernel, and the step equals the device-resident one."""
    cfg = SMALL
    w = workloads.generate(cfg, 2, "cuda")
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    N = cfg.ctx_len
    k_new = torch.randn((cfg.batch, cfg.n_kv_heads, cfg.head_dim), device="cuda").to(torch.bfloat16)
    v_new = torch.randn((cfg.batch, cfg.n_kv_heads, cfg.head_dim), device="cuda").to(torch.bfloat16)
    Kd, Vd = K.clone(), V.clone()
    Ksd = ssa.ssa_pack_summary(Kd, sel)
    Kh, Vh = _pinned(K), _pinned(V)
    Ksh = Ksd.clone()
    out_d, lse_d = ssa.ssa_decode_append(q, k_new, v_new, Kd, Vd, Ksd, sel, cfg.top_k, cfg.budget, 5, cfg.scale)
    out_h, lse_h = ssa.ssa_decode_append(q, k_new, v_new, Kh, Vh, Ksh, sel, cfg.top_k, cfg.budget, 5, cfg.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d) and torch.equal(lse_h, lse_d)
    assert torch.equal(Kh[:, :, N - 1], k_new.cpu()) and torch.equal(Vh[:, :, N - 1], v_new.cpu())
    assert torch.equal(Ksh, Ksd)


def test_pageable_host_memory_is_refused():
    cfg = SMALL
    w = workloads.generate(cfg, 0, "cuda")
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    Ks = ssa.ssa_pack_summary(K, sel)
    Kp = K.cpu()   # pageable: the device cannot read it
    assert not Kp.is_pinned()
    with pytest.raises(ssa.SsaError) as e:
        ssa.ssa_decode(q, Kp, V, Ks, sel, cfg.top_k, cfg.budget, 0, cfg.scale)
    assert e.value.status == 1
    with pytest.raises(ssa.SsaError) as e:   # the summary must be device memory
        ssa.ssa_decode(q, K, V, Ks.cpu().pin_memory(), sel, cfg.top_k, cfg.budget, 0, cfg.scale)
    assert e.value.status == 1


def test_host_resident_paged_pools():
    """The paged serving layout with its K and V pools in pinned host memory (the summary pool in HBM): the
    step equals the device-resident paged step bit for bit, ragged lengths included."""
    cfg = SMALL
    w = workloads.generate(cfg, 3, "cuda")
    Ks = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    N = cfg.ctx_len
    pg = workloads.to_paged(w["K"], w["V"], Ks, [N, N // 3 + 5], 128, seed=4)
    Kh, Vh = _pinned(pg["K_pool"]), _pinned(pg["V_pool"])
    args = (pg["Ks_pool"], pg["block_table"], pg["seq_lens"], w["sel_ch"], cfg.top_k, cfg.budget, 7, cfg.scale, N)
    out_d, lse_d = ssa.ssa_decode_paged(w["q"], pg["K_pool"], pg["V_pool"], *args)
    out_h, lse_h = ssa.ssa_decode_paged(w["q"], Kh, Vh, *args)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d) and torch.equal(lse_h, lse_d)
