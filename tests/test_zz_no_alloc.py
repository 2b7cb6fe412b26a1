"""ssa_decode_static: the decode step for callers that cannot allocate.

Some callers of this library own no device allocator: an inference engine
that reserves all HBM for its KV cache at start-up and forbids allocation
inside its decode loop, or a plugin interface that passes inputs and outputs
but no workspace.  ssa_decode_static serves them: its scratch is one fixed
array inside the library instead of a caller workspace.

The test calls it through the C ABI twice in a row -- the second call finds
the first call's leftovers in the shared array -- and compares each result
with ssa_decode (caller-provided workspace) on the same inputs, within the
2e-3 tolerance the other parity tests use.  This file is collected last so a
run that stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import long_context_decode_subset_b300 as ssa
import workloads

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_static_scratch_decode_matches_workspace_decode():
    cfg = workloads.make_config("ministral8b_32k", batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=6000,
                                top_k=60, budget=60.0, n_needles=8)
    w = workloads.generate(cfg, 3, "cuda")
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    Ks = ssa.ssa_pack_summary(K, sel)
    lib = ssa.load_library()
    shape = ssa.shape_of(q, K, Ks)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    previous = None
    for seed in (11, 12):
        out_s = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), device="cuda")
        lse_s = torch.full((cfg.batch, cfg.n_q_heads), float("nan"), device="cuda")
        rc = lib.ssa_decode_static(_p(q), _p(K), _p(V), _p(Ks), _p(sel), cfg.top_k, cfg.budget, seed, cfg.scale,
                                   _p(out_s), _p(lse_s), _p(flags), ctypes.byref(shape), stream)
        assert rc == 0, rc
        out_r, lse_r = ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, seed, cfg.scale)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        assert torch.allclose(out_s, out_r, atol=2e-3, rtol=2e-3), (out_s - out_r).abs().max()
        assert torch.allclose(lse_s, lse_r, atol=2e-3, rtol=2e-3), (lse_s - lse_r).abs().max()
        if previous is not None:  # a new seed draws a new sample: not a stale result
            assert not torch.equal(out_s, previous)
        previous = out_s.clone()


def test_static_scratch_rejects_shapes_beyond_its_size():
    lib = ssa.load_library()
    shape = ssa.make_shape(8, 32, 16, 128, 32, 1 << 20)  # needs far more than the static array holds
    assert ssa.ssa_workspace_bytes(shape) > lib.ssa_workspace_bytes(ctypes.byref(ssa.make_shape(1, 4, 1, 64, 16, 8)), 0)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = lib.ssa_decode_static(fake, fake, fake, fake, fake, 10, 10.0, 0, 0.1, fake, fake, None,
                               ctypes.byref(shape), None)
    assert rc == 3  # SSA_ERR_WORKSPACE
