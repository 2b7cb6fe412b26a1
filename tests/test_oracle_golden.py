"""The oracle still reproduces its stored tiny-case output (tests/golden/tiny_seed0.json)."""
import json
import os

import numpy as np
import torch

import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_tiny_golden(oracle_mod):
    doc = json.load(open(os.path.join(HERE, "golden", "tiny_seed0.json")))
    cfg = workloads.CONFIGS["tiny"]
    w = workloads.generate(cfg, 0, "cpu")
    sel = w["sel_ch"].numpy()
    Ks = oracle_mod.pack_summary(u16(w["K"]), sel, cfg.d_sel)
    r = oracle_mod.decode(u16(w["q"]), u16(w["K"]), u16(w["V"]), Ks, sel, cfg.top_k, cfg.budget, 0, cfg.scale)
    n = int(r["count"][0, 0])
    assert n == doc["count"]
    assert r["idx"][0, 0, :n].tolist() == doc["idx"]
    assert r["p"][0, 0, :n].view(np.uint32).tolist() == doc["p_bits"]
    assert int(r["m"].view(np.uint32)[0, 0]) == doc["m_bits"]
    assert int(r["Z"].view(np.uint32)[0, 0]) == doc["Z_bits"]
    assert np.allclose(r["lse"][0], doc["lse"], rtol=1e-6)
    assert np.allclose(r["out"][0, 0, :8], doc["out_first8"], rtol=1e-5, atol=1e-7)
