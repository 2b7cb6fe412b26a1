"""End-to-end comparison of one GPU decode step with the oracle, unit by unit.

The GPU computes the scores in fp32 on the tensor cores, the oracle in double
(from its own packed key summary), so the two may differ by rounding.  The
checks, per unit:
  * scores within the score bound (1e-5 * scale * max_g sum_j |q_g[S_j] Ks_ij|);
  * the selection: a token selected by one side only must be a boundary case,
    either at the top-k edge (its oracle score within twice the bound of the
    oracle's k-th score) or at the sampling edge (|u - p| <= 1e-6 + 2 delta p,
    delta being the largest score difference of the unit: p depends on the
    scores through exp(s_j - m) / Z, so a score error of delta moves p by at
    most 2 delta relative);
  * p on the common tokens within 2 delta relative + 4 ulp;
  * out and lse within 2e-3 abs + 2e-3 rel of the oracle's attention.  When the
    lists agree that is the oracle's own list.  When they differ (only at
    boundary tokens, checked above) the reference is the oracle's attention
    over the GPU's index set with the ORACLE's inclusion probabilities (p = 1
    for a top-k-edge token the GPU placed in the stratum): which side of an
    ambiguous decision a token falls on is taken from the GPU, every value the
    oracle computes with is its own.  No unit goes unchecked.
"""
import numpy as np
import torch

import long_context_decode_subset_b300 as ssa
from _util import score_bound, u16, ulp_diff_f32

EPS = 2.0 ** -24


def gpu_decode(w, k, B, seed, Ks=None, list_cap=0):
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    Ks = w["Ks"] if Ks is None else Ks
    Bt, Hkv, N, _ = K.shape
    cap = list_cap or max(N, 1)
    dev = q.device
    s_hat = torch.empty((Bt, Hkv, N), dtype=torch.float32, device=dev)
    idx = torch.empty((Bt, Hkv, cap), dtype=torch.int32, device=dev)
    p = torch.empty((Bt, Hkv, cap), dtype=torch.float32, device=dev)
    count = torch.empty((Bt, Hkv), dtype=torch.int32, device=dev)
    shape = ssa.shape_of(q, K, Ks)
    ws = ssa.workspace(shape, cap, dev)
    out, lse = ssa.ssa_decode(q, K, V, Ks, sel, k, B, seed, w["scale"], s_hat=s_hat, idx=idx, p=p, count=count,
                              list_cap=cap, ws=ws)
    st, flags = ssa.ssa_get_device_status(ws)
    return dict(out=out, lse=lse, s_hat=s_hat, idx=idx, p=p, count=count, status=st, flags=flags)


def unit_arrays(oracle_mod, w, b, h, n=None):
    """Host copies of one unit's inputs (q heads, its first n (default: all) K and V rows, the oracle's own key
    summary of them, channels)."""
    G = w["q"].shape[1] // w["K"].shape[1]
    n = w["K"].shape[2] if n is None else n
    Kb = u16(w["K"][b, h, :n])
    sel_h = w["sel_ch"][h].cpu().numpy()
    Ksb = oracle_mod.pack_summary(Kb[None, None], sel_h[None], sel_h.size)[0, 0]
    return u16(w["q"][b, h * G:(h + 1) * G]), Kb, u16(w["V"][b, h, :n]), Ksb, sel_h


def check_unit(oracle_mod, w, g, b, h, k, B, seed, stats, n=None):
    """Oracle for unit (b, h) over its first n tokens (default: all) computed from scratch; compare with the GPU's
    results."""
    qh, Kb, Vb, Ksb, sel_h = unit_arrays(oracle_mod, w, b, h, n)
    G, d = qh.shape
    N = Kb.shape[0]
    scale = w["scale"]
    s_ora = oracle_mod.score(qh[None], Ksb[None, None], sel_h[None], scale)[0, 0]
    tol = score_bound(qh[None], Ksb[None, None], sel_h[None], scale)[0, 0]
    s_gpu = g["s_hat"][b, h, :N].cpu().numpy()
    err = np.abs(s_gpu.astype(np.float64) - s_ora.astype(np.float64))
    assert np.all(err <= tol), f"unit ({b},{h}) score error {np.max(err / tol):.2f} x tol"
    delta = float(err.max()) if N else 0.0
    o_idx, o_p, m, Z, p_all = oracle_mod.select_unit(s_ora, k, B, seed, b, h, want_p_all=True)
    n = int(g["count"][b, h])
    cap = g["idx"].shape[-1]
    g_idx = g["idx"][b, h, :min(n, cap)].cpu().numpy()
    g_p = g["p"][b, h, :min(n, cap)].cpu().numpy()
    gd = dict(zip(g_idx.tolist(), g_p.tolist()))
    od = dict(zip(o_idx.tolist(), o_p.tolist()))
    diff = set(gd) ^ set(od)
    kth = float(np.sort(s_ora)[::-1][min(max(k, 1), N) - 1]) if N else 0.0
    topk_edge = set()
    for j in diff:
        u = oracle_mod.uniform(seed, j, h, b)
        pj = float(p_all[j])
        at_topk = abs(float(s_ora[j]) - kth) <= 2 * float(tol[j]) + 1e-30
        at_samp = abs(u - pj) <= 1e-6 + 2 * delta * pj
        assert at_topk or at_samp, f"unit ({b},{h}) token {j}: u={u} p={pj} s={s_ora[j]} kth={kth}"
        if at_topk:
            topk_edge.add(j)
    common = sorted(set(gd) & set(od))
    if common:
        gp = np.array([gd[j] for j in common], np.float64)
        op = np.array([od[j] for j in common], np.float64)
        near_edge = np.array([abs(float(s_ora[j]) - kth) <= 2 * float(tol[j]) + 1e-30 for j in common])
        bound = op * (2 * delta + 4 * EPS) + 1e-45
        ok = (np.abs(gp - op) <= bound) | near_edge
        assert ok.all(), f"unit ({b},{h}) p differs beyond 2 delta + 4 ulp at {np.array(common)[~ok][:8]}"
        if delta == 0.0:
            assert np.all(ulp_diff_f32(gp[~near_edge], op[~near_edge]) <= 4)
    stats["boundary"] = stats.get("boundary", 0) + len(diff)
    stats["units"] = stats.get("units", 0) + 1
    if diff:
        stats["units_differing"] = stats.get("units_differing", 0) + 1
        # the GPU's index set, the oracle's inclusion probabilities
        r_idx = np.array(sorted(gd), np.int32)
        r_p = np.array([1.0 if (j in topk_edge and gd[j] == 1.0) else float(p_all[j]) for j in r_idx.tolist()],
                       np.float32)
    else:
        r_idx, r_p = o_idx, o_p
    out_o, lse_o = oracle_mod.attend_unit(qh, Kb, Vb, r_idx, r_p, scale)
    out_g = g["out"][b, h * G:(h + 1) * G].cpu().numpy()
    lse_g = g["lse"][b, h * G:(h + 1) * G].cpu().numpy()
    assert np.allclose(out_g, out_o, atol=2e-3, rtol=2e-3), f"unit ({b},{h}) out err {np.abs(out_g - out_o).max()}"
    if r_idx.size:
        assert np.allclose(lse_g, lse_o, atol=2e-3, rtol=2e-3), f"unit ({b},{h}) lse err {np.abs(lse_g - lse_o).max()}"
    else:
        assert np.all(np.isneginf(lse_g)) and np.all(out_g == 0)
    stats["max_out_err"] = max(stats.get("max_out_err", 0.0), float(np.abs(out_g - out_o).max()))
