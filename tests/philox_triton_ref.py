"""Independent Philox4x32-10 evaluated by Triton's CPU interpreter.

Run as a subprocess (TRITON_INTERPRET must be set before Triton is imported).
Reads JSON [[c0, c1, c2, c3, k0, k1], ...] on stdin; prints JSON [[x0, x1, x2, x3], ...].
Used only to pin the oracle's Philox against a second implementation of the
published generator.
"""
import json
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"

import numpy as np  # noqa: E402
import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _philox_kernel(ctr_ptr, key_ptr, out_ptr, BLOCK: tl.constexpr):
    i = tl.arange(0, BLOCK)
    c0 = tl.load(ctr_ptr + i * 4 + 0).to(tl.uint32, bitcast=True)
    c1 = tl.load(ctr_ptr + i * 4 + 1).to(tl.uint32, bitcast=True)
    c2 = tl.load(ctr_ptr + i * 4 + 2).to(tl.uint32, bitcast=True)
    c3 = tl.load(ctr_ptr + i * 4 + 3).to(tl.uint32, bitcast=True)
    k0 = tl.load(key_ptr + i * 2 + 0).to(tl.uint32, bitcast=True)
    k1 = tl.load(key_ptr + i * 2 + 1).to(tl.uint32, bitcast=True)
    y0, y1, y2, y3 = tl.random.philox_impl(c0, c1, c2, c3, k0, k1, 10)
    tl.store(out_ptr + i * 4 + 0, y0.to(tl.int32, bitcast=True))
    tl.store(out_ptr + i * 4 + 1, y1.to(tl.int32, bitcast=True))
    tl.store(out_ptr + i * 4 + 2, y2.to(tl.int32, bitcast=True))
    tl.store(out_ptr + i * 4 + 3, y3.to(tl.int32, bitcast=True))


def main():
    rows = json.load(sys.stdin)
    n = len(rows)
    block = 1
    while block < n:
        block *= 2
    arr = np.zeros((block, 6), np.uint32)
    arr[:n] = np.array(rows, dtype=np.uint64).astype(np.uint32)
    ctr = torch.from_numpy(arr[:, :4].copy().view(np.int32))
    key = torch.from_numpy(arr[:, 4:].copy().view(np.int32))
    out = torch.zeros((block, 4), dtype=torch.int32)
    _philox_kernel[(1,)](ctr, key, out, BLOCK=block)
    res = out.numpy().view(np.uint32)[:n].astype(np.uint64).tolist()
    json.dump(res, sys.stdout)


if __name__ == "__main__":
    main()
