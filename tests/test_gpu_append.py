"""GPU append step.  ssa_append is bit-exact against the oracle's append, and
the fused ssa_decode_append (the new token written by the chain's first
kernel) leaves the cache equal to the appended one and returns exactly what
ssa_decode returns on that cache (same kernels, fixed reduction orders), which
the decode parity tests pin against the oracle.  The caches here have spare
capacity: the step runs on a prefix of a larger buffer, as in a serving loop."""
import math

import numpy as np
import pytest
import torch

import long_context_decode_subset_b300 as ssa
from gpu_e2e import check_unit, gpu_decode
from test_gpu_stages import SMALL, case
from _util import u16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    """Bit patterns of an fp32 tensor (equal bits: equal values, -0 and NaN included)."""
    return t.contiguous().view(torch.int32)


def _with_capacity(t, n_valid, extra, garbage_row, seed):
    """t [Bt][Hkv][N][w] copied into a buffer of N + extra tokens; row garbage_row is overwritten with
    other finite values.  Returns (buffer, view of its first n_valid tokens)."""
    Bt, Hkv, N, wdt = t.shape
    buf = torch.zeros((Bt, Hkv, N + extra, wdt), dtype=t.dtype, device=DEV)
    buf[:, :, :N] = t
    if garbage_row is not None:
        g = torch.Generator(device=DEV).manual_seed(seed)
        buf[:, :, garbage_row] = torch.randn((Bt, Hkv, wdt), generator=g, device=DEV).to(t.dtype)
    return buf, buf[:, :, :n_valid]


@pytest.mark.parametrize("name", list(SMALL))
def test_append_bit_exact(oracle_mod, name):
    w = case(name)
    Bt, Hkv, N, d = w["K"].shape
    _, K = _with_capacity(w["K"], N, 5, None, 0)
    _, V = _with_capacity(w["V"], N, 5, None, 0)
    _, Ks = _with_capacity(w["Ks"], N, 5, None, 0)
    sel = w["sel_ch"]
    g = torch.Generator(device=DEV).manual_seed(11)
    for pos in (0, N // 3, N - 1):
        k_new = torch.randn((Bt, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
        v_new = torch.randn((Bt, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
        want = oracle_mod.append(u16(K), u16(V), u16(Ks), u16(k_new), u16(v_new), sel.cpu().numpy(), pos)
        ssa.ssa_append(k_new, v_new, sel, pos, K, V, Ks)
        torch.cuda.synchronize()
        for got, exp in zip((K, V, Ks), want):
            assert np.array_equal(u16(got), exp), (name, pos)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("dense", [False, True])
def test_decode_append_equals_decode_on_the_appended_cache(oracle_mod, name, dense):
    w = case(name)
    cfg = w["cfg"]
    Bt, Hkv, N, d = w["K"].shape
    B = math.inf if dense else cfg.budget
    _, K = _with_capacity(w["K"], N, 7, N - 1, 1)
    _, V = _with_capacity(w["V"], N, 7, N - 1, 2)
    _, Ks = _with_capacity(w["Ks"], N, 7, N - 1, 3)
    k_new = w["K"][:, :, N - 1].contiguous()
    v_new = w["V"][:, :, N - 1].contiguous()
    shape = ssa.shape_of(w["q"], K, Ks)
    ws = ssa.workspace(shape, 0, DEV)
    out, lse = ssa.ssa_decode_append(w["q"], k_new, v_new, K, V, Ks, w["sel_ch"], cfg.top_k, B, 1, cfg.scale,
                                     ws=ws)
    st, flags = ssa.ssa_get_device_status(ws)
    assert st == 0, hex(flags)
    # the cache now holds the appended token
    want = oracle_mod.append(u16(w["K"]), u16(w["V"]), u16(w["Ks"]), u16(k_new), u16(v_new),
                             w["sel_ch"].cpu().numpy(), N - 1)
    for got, exp in zip((K, V, Ks), want):
        assert np.array_equal(u16(got), exp)
    # and the step equals ssa_decode on that cache, bit for bit
    ref = gpu_decode(w, cfg.top_k, B, 1)
    assert ref["status"] == 0
    assert torch.equal(_bits(out), _bits(ref["out"])), name
    assert torch.equal(_bits(lse), _bits(ref["lse"])), name
    if not dense and name in ("tiny", "g4_d128"):
        stats = {}
        for b in range(cfg.batch):
            for h in range(cfg.n_kv_heads):
                check_unit(oracle_mod, w, ref, b, h, cfg.top_k, B, 1, stats)
