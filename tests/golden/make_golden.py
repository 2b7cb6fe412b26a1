"""Writes tests/golden/tiny_seed0.json from the oracle alone.

The pages print no worked numeric example for the method, so the stored
values here are the oracle's own output on the tiny synthetic case (seed 0);
they pin the oracle against accidental drift, not against the pages.  Run:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads  # noqa: E402


def u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def main():
    cfg = workloads.CONFIGS["tiny"]
    w = workloads.generate(cfg, 0, "cpu")
    sel = w["sel_ch"].numpy()
    Ks = oracle.pack_summary(u16(w["K"]), sel, cfg.d_sel)
    r = oracle.decode(u16(w["q"]), u16(w["K"]), u16(w["V"]), Ks, sel, cfg.top_k, cfg.budget, 0, cfg.scale)
    n = int(r["count"][0, 0])
    doc = {
        "what": "oracle decode of the tiny synthetic case, seed 0 (regression pin of the oracle)",
        "config": "tiny",
        "count": n,
        "idx": r["idx"][0, 0, :n].tolist(),
        "p_bits": r["p"][0, 0, :n].view(np.uint32).tolist(),
        "m_bits": int(r["m"].view(np.uint32)[0, 0]),
        "Z_bits": int(r["Z"].view(np.uint32)[0, 0]),
        "lse": r["lse"][0].tolist(),
        "out_l2": float(np.linalg.norm(r["out"])),
        "out_first8": r["out"][0, 0, :8].tolist(),
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_seed0.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
