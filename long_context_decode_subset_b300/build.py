"""Builds libssa.so (the CUDA library behind include/ssa.h) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libssa.so")
SOURCES = ["ssa_api.cu"]
DEPS = ["ssa_api.cu", "common.cuh", "k_score.cuh", "k_select.cuh", "k_attend.cuh", "ptx.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
    "-Xptxas", "-v",
]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(INCLUDE, "ssa.h")]
    return any(os.path.getmtime(d) > t for d in deps)


CEILING_SRC = os.path.join(PKG, "read_ceiling.cu")
CEILING = os.path.join(PKG, "read_ceiling")


def build_ceiling(force: bool = False) -> str:
    """Builds the read-ceiling probe the benchmark places the score pass against (read_ceiling.cu)."""
    if not force and os.path.exists(CEILING) and os.path.getmtime(CEILING) >= os.path.getmtime(CEILING_SRC):
        return CEILING
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = CEILING + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", tmp, CEILING_SRC]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stderr[-4000:])
        raise RuntimeError("nvcc failed on read_ceiling.cu")
    os.replace(tmp, CEILING)
    return CEILING


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-o", tmp,
           *[os.path.join(CSRC, s) for s in SOURCES]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(PKG, "build.log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        sys.stderr.write(res.stderr[-6000:])
        raise RuntimeError(f"nvcc failed (see {log})")
    if verbose:
        sys.stdout.write(res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    build_ceiling(force="--force" in sys.argv)
    print(LIB)
