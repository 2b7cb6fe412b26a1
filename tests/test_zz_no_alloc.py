"""ssa_decode_static: the decode step for callers that cannot allocate.

Some callers of this library own no device allocator: an inference engine
that reserves all HBM for its KV cache at start-up and forbids allocation
inside its decode loop, or a plugin interface that passes inputs and outputs
but no workspace.  ssa_decode_static serves them: its scratch is one fixed
array inside the library instead of a caller workspace.

The tests call it through the C ABI and compare it with ssa_decode (caller
workspace) on the same inputs.  Both run the same kernels with the same plan,
so the results must be identical bit for bit: a difference could only come
from the array's leftovers, which is what two calls in a row (the second one
finding the first one's contents) are there to catch.  The array's limit is
covered from both sides: a shape whose scratch just fits runs and matches, a
shape just past it is rejected.  This file is collected last so that a run
that stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import long_context_decode_subset_b300 as ssa
import workloads

pytestmark = pytest.mark.gpu

STATIC_BYTES = 64 << 20   # SSA_STATIC_SCRATCH_BYTES in include/ssa.h


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_decode(lib, q, K, V, Ks, sel, top_k, budget, seed, scale, shape, flags):
    Bt, Hq, d = q.shape
    out = torch.full((Bt, Hq, d), float("nan"), device="cuda")
    lse = torch.full((Bt, Hq), float("nan"), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.ssa_decode_static(_p(q), _p(K), _p(V), _p(Ks), _p(sel), top_k, budget, seed, scale, _p(out), _p(lse),
                               _p(flags), ctypes.byref(shape), stream)
    assert rc == 0, rc
    return out, lse


def test_static_scratch_decode_matches_workspace_decode():
    cfg = workloads.make_config("ministral8b_32k", batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=6000,
                                top_k=60, budget=60.0, n_needles=8)
    w = workloads.generate(cfg, 3, "cuda")
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    Ks = ssa.ssa_pack_summary(K, sel)
    lib = ssa.load_library()
    shape = ssa.shape_of(q, K, Ks)
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    previous = None
    for seed in (11, 12):
        out_s, lse_s = _static_decode(lib, q, K, V, Ks, sel, cfg.top_k, cfg.budget, seed, cfg.scale, shape, flags)
        out_r, lse_r = ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, seed, cfg.scale)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        assert torch.equal(out_s, out_r), (out_s - out_r).abs().max()
        assert torch.equal(lse_s, lse_r), (lse_s - lse_r).abs().max()
        if previous is not None:  # a new seed draws a new sample: not a stale result
            assert not torch.equal(out_s, previous)
        previous = out_s.clone()


def _largest_ctx_that_fits(Bt, Hq, Hkv, d, d_sel):
    """The largest context (a multiple of 1024) whose scratch fits the static array."""
    lo, hi = 1024, 1 << 24
    assert ssa.ssa_workspace_bytes(ssa.make_shape(Bt, Hq, Hkv, d, d_sel, lo)) <= STATIC_BYTES
    assert ssa.ssa_workspace_bytes(ssa.make_shape(Bt, Hq, Hkv, d, d_sel, hi)) > STATIC_BYTES
    while hi - lo > 1024:
        mid = (lo + hi) // 2 // 1024 * 1024
        if ssa.ssa_workspace_bytes(ssa.make_shape(Bt, Hq, Hkv, d, d_sel, mid)) <= STATIC_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_static_scratch_runs_a_shape_just_under_its_size():
    Bt, Hq, Hkv, d, d_sel = 1, 8, 2, 128, 32
    N = _largest_ctx_that_fits(Bt, Hq, Hkv, d, d_sel)
    shape = ssa.make_shape(Bt, Hq, Hkv, d, d_sel, N)
    assert ssa.ssa_workspace_bytes(shape) <= STATIC_BYTES
    assert ssa.ssa_workspace_bytes(ssa.make_shape(Bt, Hq, Hkv, d, d_sel, N + 1024)) > STATIC_BYTES
    g = torch.Generator(device="cuda").manual_seed(5)
    K = torch.randn((Bt, Hkv, N, d), generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn((Bt, Hkv, N, d), generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((Bt, Hq, d), generator=g, device="cuda").to(torch.bfloat16)
    sel = torch.stack([torch.randperm(d, generator=torch.Generator().manual_seed(h))[:d_sel].sort().values
                       for h in range(Hkv)]).to(torch.int32).cuda()
    Ks = ssa.ssa_pack_summary(K, sel)
    lib = ssa.load_library()
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    k, B, scale = N // 100, float(N // 100), d ** -0.5
    for seed in (1, 2):
        out_s, lse_s = _static_decode(lib, q, K, V, Ks, sel, k, B, seed, scale, shape, flags)
        out_r, lse_r = ssa.ssa_decode(q, K, V, Ks, sel, k, B, seed, scale)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        assert torch.equal(out_s, out_r) and torch.equal(lse_s, lse_r)
    del K, V, Ks
    torch.cuda.empty_cache()


def test_static_scratch_rejects_shapes_beyond_its_size():
    lib = ssa.load_library()
    Bt, Hq, Hkv, d, d_sel = 1, 8, 2, 128, 32
    N = _largest_ctx_that_fits(Bt, Hq, Hkv, d, d_sel) + 1024   # the next size up no longer fits
    for shape in (ssa.make_shape(Bt, Hq, Hkv, d, d_sel, N), ssa.make_shape(8, 32, 16, 128, 32, 1 << 20)):
        assert ssa.ssa_workspace_bytes(shape) > STATIC_BYTES
        fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
        rc = lib.ssa_decode_static(fake, fake, fake, fake, fake, 10, 10.0, 0, 0.1, fake, fake, None,
                                   ctypes.byref(shape), None)
        assert rc == 3  # SSA_ERR_WORKSPACE
