"""Shared helpers for the tests (comparison logic only; no method arithmetic)."""
import numpy as np
import torch


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_values(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def score_bound(q_u16, Ks_u16, sel_ch, scale):
    """Per-token tolerance for s: 1e-5 * scale * max_g sum_j |q_g[S_j] Ks[i][j]| (+ tiny absolute)."""
    Bt, Hq, d = q_u16.shape
    _, Hkv, N, d_sel = Ks_u16.shape
    G = Hq // Hkv
    qv = bf16_values(q_u16).astype(np.float64)
    kv = np.abs(bf16_values(Ks_u16).astype(np.float64))
    out = np.zeros((Bt, Hkv, N))
    for b in range(Bt):
        for h in range(Hkv):
            qs = np.abs(qv[b, h * G:(h + 1) * G][:, sel_ch[h]])       # [G][d_sel]
            out[b, h] = (kv[b, h] @ qs.T).max(axis=1)
    return 1e-5 * scale * out + 1e-30


def ulp_diff_f32(a, b):
    ai = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(ai - bi)


def compare_unit_lists(g_idx, g_p, o_idx, o_p, o_p_all, u_of, tol_abs=1e-6, tol_rel=0.0, p_ulps=4):
    """Compare one unit's GPU selection with the oracle's.

    Tokens selected by exactly one side must be boundary cases |u - p| <= tol (u from the
    oracle's generator, p the oracle's); tokens selected by both must agree in p to p_ulps.
    Returns (n_boundary, n_common)."""
    g = dict(zip(g_idx.tolist(), g_p.tolist()))
    o = dict(zip(o_idx.tolist(), o_p.tolist()))
    diff = set(g) ^ set(o)
    for j in diff:
        u = u_of(j)
        pj = float(o_p_all[j])
        assert abs(u - pj) <= tol_abs + tol_rel * pj, f"token {j}: u={u} p={pj} selected only by {'gpu' if j in g else 'oracle'}"
    common = sorted(set(g) & set(o))
    if common:
        gp = np.array([g[j] for j in common], np.float32)
        op = np.array([o[j] for j in common], np.float32)
        bad = ulp_diff_f32(gp, op) > p_ulps
        assert not bad.any(), f"p differs beyond {p_ulps} ulp at tokens {np.array(common)[bad][:10]}"
    return len(diff), len(common)
