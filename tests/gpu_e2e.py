"""End-to-end comparison of one GPU decode step with the oracle, unit by unit.

The GPU computes the scores in fp32, the oracle in double, so the two may
differ by rounding; the selection can then differ only at its boundaries:
  * top-k boundary: a token whose oracle score is within twice the score
    tolerance of the oracle's k-th largest score;
  * sampling boundary: |u - p| <= 1e-6 + 3e-5 p (a score perturbation of the
    tolerance moves p by that relative amount).
Units whose lists agree exactly must agree in out / lse within 2e-3 abs +
2e-3 rel.  Nothing here feeds a GPU result into the oracle.
"""
import numpy as np
import torch

import long_context_decode_subset_b300 as ssa
from _util import score_bound, u16, ulp_diff_f32


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


def unit_arrays(w, b, h):
    """Host copies of one unit's inputs (q heads, K, V, Ks) for per-unit oracle calls."""
    G = w["q"].shape[1] // w["K"].shape[1]
    return (u16(w["q"][b, h * G:(h + 1) * G]), u16(w["K"][b, h]), u16(w["V"][b, h]), u16(w["Ks"][b, h]),
            w["sel_ch"][h].cpu().numpy())


def check_unit(oracle_mod, w, g, b, h, k, B, seed, stats):
    """Oracle for unit (b, h) computed from scratch; compare with the GPU's results."""
    qh, Kb, Vb, Ksb, sel_h = unit_arrays(w, b, h)
    G, d = qh.shape
    N = Kb.shape[0]
    scale = w["scale"]
    s_ora = oracle_mod.score(qh[None], Ksb[None, None], sel_h[None], scale)[0, 0]
    tol = score_bound(qh[None], Ksb[None, None], sel_h[None], scale)[0, 0]
    s_gpu = g["s_hat"][b, h].cpu().numpy()
    err = np.abs(s_gpu - s_ora)
    assert np.all(err <= tol), f"unit ({b},{h}) score error {np.max(err / tol):.2f} x tol"
    o_idx, o_p, m, Z, p_all = oracle_mod.select_unit(s_ora, k, B, seed, b, h, want_p_all=True)
    n = int(g["count"][b, h])
    cap = g["idx"].shape[-1]
    g_idx = g["idx"][b, h, :min(n, cap)].cpu().numpy()
    g_p = g["p"][b, h, :min(n, cap)].cpu().numpy()
    gd = dict(zip(g_idx.tolist(), g_p.tolist()))
    od = dict(zip(o_idx.tolist(), o_p.tolist()))
    diff = set(gd) ^ set(od)
    kth = float(np.sort(s_ora)[::-1][min(max(k, 1), N) - 1]) if N else 0.0
    for j in diff:
        u = oracle_mod.uniform(seed, j, h, b)
        pj = float(p_all[j])
        topk_edge = abs(float(s_ora[j]) - kth) <= 2 * float(tol[j]) + 1e-30
        samp_edge = abs(u - pj) <= 1e-6 + 3e-5 * pj
        assert topk_edge or samp_edge, f"unit ({b},{h}) token {j}: u={u} p={pj} s={s_ora[j]} kth={kth}"
    stats["boundary"] = stats.get("boundary", 0) + len(diff)
    stats["units"] = stats.get("units", 0) + 1
    if diff:
        stats["units_differing"] = stats.get("units_differing", 0) + 1
        return
    if o_idx.size:
        gp = np.array([gd[j] for j in o_idx.tolist()], np.float32)
        assert np.all(ulp_diff_f32(gp, o_p) <= 64), f"unit ({b},{h}) p differs"
    out_o, lse_o = oracle_mod.attend_unit(qh, Kb, Vb, o_idx, o_p, scale)
    out_g = g["out"][b, h * G:(h + 1) * G].cpu().numpy()
    lse_g = g["lse"][b, h * G:(h + 1) * G].cpu().numpy()
    assert np.allclose(out_g, out_o, atol=2e-3, rtol=2e-3), f"unit ({b},{h}) out err {np.abs(out_g - out_o).max()}"
    if o_idx.size:
        assert np.allclose(lse_g, lse_o, atol=2e-3, rtol=2e-3), f"unit ({b},{h}) lse err {np.abs(lse_g - lse_o).max()}"
    else:
        assert np.all(np.isneginf(lse_g)) and np.all(out_g == 0)
    stats["max_out_err"] = max(stats.get("max_out_err", 0.0), float(np.abs(out_g - out_o).max()))
