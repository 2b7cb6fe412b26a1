"""The C-ABI library loads, exports every symbol include/ssa.h declares, and
rejects bad arguments on the host (no GPU needed: validation precedes any
CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

import long_context_decode_subset_b300 as ssa
from long_context_decode_subset_b300 import ssa as binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ssa.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", ssa.LIB_PATH], capture_output=True, text=True).stdout
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} not exported"


def test_library_is_built_for_sm_103a():
    """The build compiles for sm_103a only, and the library in the tree came from that command (the build
    writes its command line to build.log beside the library)."""
    from long_context_decode_subset_b300 import build
    flags = " ".join(build.NVCC_FLAGS)
    assert "arch=compute_103a,code=sm_103a" in flags
    assert flags.count("-gencode") == 1
    log = os.path.join(os.path.dirname(ssa.LIB_PATH), "build.log")
    if not os.path.exists(log):
        pytest.skip("the library was not built by the package's build step here")
    cmd = open(log).readline()
    assert "arch=compute_103a,code=sm_103a" in cmd and cmd.count("-gencode") == 1


def test_status_strings_and_version():
    lib = ssa.load_library()
    assert lib.ssa_status_string(0) == b"ok"
    assert lib.ssa_status_string(3).startswith(b"workspace")
    assert ssa.ssa_version() >= 100


def _shape(**kw):
    base = dict(batch=2, n_q_heads=32, n_kv_heads=8, head_dim=128, d_sel=32, ctx_len=4096)
    base.update(kw)
    return ssa.make_shape(**base)


def test_workspace_bytes():
    s = _shape()
    n = ssa.ssa_workspace_bytes(s)
    units, N = 16, 4096
    # scores, candidate and selection lists, 16-bit Philox prefixes: at least 22 bytes per token
    assert n >= units * N * 22
    # the internal lists are sized for the worst case, so the list capacity does not matter
    assert ssa.ssa_workspace_bytes(s, 100) == n
    assert ssa.ssa_workspace_bytes(_shape(ctx_len=8192)) > n
    assert ssa.ssa_workspace_bytes(_shape(head_dim=96)) == 0
    assert ssa.ssa_workspace_bytes(_shape(n_q_heads=24)) == 0      # G = 3
    assert ssa.ssa_workspace_bytes(_shape(ctx_len=-1)) == 0


P = ctypes.c_void_p


def _decode(lib, shape, **over):
    fake = 1 << 20  # never dereferenced: every call below must fail validation first
    args = dict(q=fake, K=fake, V=fake, Ks=fake, sel=fake, k=10, B=10.0, seed=0, scale=0.1, out=fake, lse=fake,
                ws=fake, ws_bytes=1 << 40)
    args.update(over)
    return lib.ssa_decode(P(args["q"]), P(args["K"]), P(args["V"]), P(args["Ks"]), P(args["sel"]), args["k"],
                          args["B"], args["seed"], args["scale"], P(args["out"]), P(args["lse"]), None, None, None,
                          None, 0, P(args["ws"]), args["ws_bytes"], ctypes.byref(shape), None)


def test_decode_validation_statuses():
    lib = ssa.load_library()
    s = _shape()
    assert _decode(lib, s, q=0) == 1
    assert _decode(lib, s, k=-1) == 1
    assert _decode(lib, s, B=-1.0) == 1
    assert _decode(lib, s, B=float("nan")) == 1
    assert _decode(lib, s, scale=0.0) == 1
    assert _decode(lib, s, K=(1 << 20) + 2) == 1                    # misaligned
    assert _decode(lib, _shape(head_dim=80)) == 2
    assert _decode(lib, _shape(d_sel=24)) == 2
    assert _decode(lib, _shape(n_q_heads=48, n_kv_heads=4)) == 2   # G = 12
    assert _decode(lib, s, ws_bytes=1000) == 3
    assert _decode(lib, s, ws=(1 << 20) + 16) == 3                  # workspace not 256-aligned
    bad = _shape()
    bad.kv_stride_h = 100
    assert _decode(lib, bad) == 1
    bad = _shape()
    bad.reserved = 1
    assert _decode(lib, bad) == 1


def test_other_entry_points_validate():
    lib = ssa.load_library()
    s = _shape()
    f = P(1 << 20)
    cap = 0
    assert lib.ssa_select(None, 5, 1.0, 0, f, f, f, cap, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_select(f, -5, 1.0, 0, f, f, f, cap, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_select(f, 5, 1.0, 0, f, f, f, cap, f, 16, ctypes.byref(s), None) == 3
    assert lib.ssa_score(f, f, f, 0.1, None, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_score(f, f, f, float("inf"), f, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_attend(f, f, f, f, f, None, cap, 0.1, f, f, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_pack_summary(None, f, f, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_decode_host(None, f, f, f, f, 5, 1.0, 0, 0.1, f, f, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_get_device_status(None, None, None) == 3
    assert lib.ssa_query_plan(None, None, None, None) == 1
    assert lib.ssa_select_capacity(ctypes.byref(s)) == s.ctx_len
    assert lib.ssa_select_capacity(None) == 0
    # strata: an unknown kind or a negative / NaN top_p is invalid
    assert lib.ssa_select_strata(f, 3, 5, 0.0, 1.0, 0, f, f, f, cap, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_select_strata(f, -1, 5, 0.0, 1.0, 0, f, f, f, cap, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_select_strata(f, 1, 5, float("nan"), 1.0, 0, f, f, f, cap, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_select_strata(f, 2, 5, -0.5, 1.0, 0, f, f, f, cap, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_select_strata(f, 2, 5, 0.9, 1.0, 0, f, f, f, cap, f, 16, ctypes.byref(s), None) == 3
    assert lib.ssa_decode_strata(f, f, f, f, f, 7, 5, 0.0, 1.0, 0, 0.1, f, f, None, None, None, None, cap, f, 1 << 40,
                                 ctypes.byref(s), None) == 1
    assert lib.ssa_decode_strata(f, f, f, f, f, 2, 5, float("nan"), 1.0, 0, 0.1, f, f, None, None, None, None, cap, f,
                                 1 << 40, ctypes.byref(s), None) == 1


def test_binding_requires_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        binding.load_library()


def test_append_entry_points_validate():
    lib = ssa.load_library()
    s = _shape()
    f = P(1 << 20)
    n = s.ctx_len
    assert lib.ssa_append(None, f, f, 0, f, f, f, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_append(f, f, f, -1, f, f, f, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_append(f, f, f, n, f, f, f, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_append(f, f, f, 0, P((1 << 20) + 2), f, f, f, 1 << 40, ctypes.byref(s), None) == 1
    assert lib.ssa_append(f, f, f, 0, f, f, f, f, 16, ctypes.byref(s), None) == 3
    assert lib.ssa_append(f, f, f, 0, f, f, f, f, 1 << 40, ctypes.byref(_shape(head_dim=80)), None) == 2
    assert lib.ssa_decode_append(f, None, f, f, f, f, f, 5, 1.0, 0, 0.1, f, f, f, 1 << 40, ctypes.byref(s),
                                 None) == 1
    assert lib.ssa_decode_append(f, f, f, f, f, f, f, 5, 1.0, 0, 0.1, f, f, f, 1 << 40,
                                 ctypes.byref(_shape(ctx_len=0)), None) == 1
    assert lib.ssa_decode_append(f, P((1 << 20) + 8), f, f, f, f, f, 5, 1.0, 0, 0.1, f, f, f, 1 << 40,
                                 ctypes.byref(s), None) == 1
    assert lib.ssa_decode_append(f, f, f, f, f, f, f, -5, 1.0, 0, 0.1, f, f, f, 1 << 40, ctypes.byref(s),
                                 None) == 1


def test_header_is_plain_c_and_the_library_links_from_c(tmp_path):
    """include/ssa.h compiles as C99 with warnings as errors, and a C program linked against libssa.so
    gets the host-side validation statuses (no GPU needed)."""
    src = tmp_path / "use.c"
    src.write_text(r'''
#include "ssa.h"
#include <stdio.h>
int main(void) {
    ssa_shape s = {2, 32, 8, 128, 32, 0, 4096, 8 * 4096 * 128, 4096 * 128, 8 * 4096 * 32, 4096 * 32};
    size_t n = ssa_workspace_bytes(&s, 0);
    ssa_status st = ssa_decode(NULL, NULL, NULL, NULL, NULL, 5, 1.0f, 0, 0.1f, NULL, NULL, NULL, NULL, NULL,
                               NULL, 0, NULL, 0, &s, 0);
    printf("%zu %d %s\n", n, (int)st, ssa_status_string(st));
    return (n > 0 && st == SSA_ERR_INVALID_ARG) ? 0 : 1;
}
''')
    exe = tmp_path / "use"
    libdir = os.path.dirname(binding.LIB_PATH)
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, "-o", str(exe), str(src), "-L", libdir, "-lssa", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "invalid argument" in r.stdout


def _paged_call(lib, shape, pages, **over):
    f = 1 << 20  # never dereferenced: every call below must fail validation first
    args = dict(q=f, k_new=None, v_new=None, K=f, V=f, Ks=f, sel=f, k=10, B=10.0, ws=f, ws_bytes=1 << 40)
    args.update(over)
    return lib.ssa_decode_paged(P(args["q"]), P(args["k_new"]), P(args["v_new"]), P(args["K"]), P(args["V"]),
                                P(args["Ks"]), ctypes.byref(pages) if pages is not None else None, P(args["sel"]),
                                args["k"], args["B"], 0, 0.1, P(f), P(f), None, None, None, None, 0, P(args["ws"]),
                                args["ws_bytes"], ctypes.byref(shape), None)


def test_paged_entry_point_validates():
    lib = ssa.load_library()
    s = binding.ssa_shape(2, 32, 8, 128, 32, 0, 4096, 0, 0, 0, 0)   # a paged step's shape: strides 0
    f = 1 << 20

    def pages(**kw):
        d = dict(page_size=64, max_pages=64, num_pages=200, block_table=f, seq_lens=f)
        d.update(kw)
        return binding.ssa_paged_kv(d["page_size"], d["max_pages"], d["num_pages"], d["block_table"], d["seq_lens"])

    # the sizing calls take the stride-free shape
    assert ssa.ssa_workspace_bytes(s) == ssa.ssa_workspace_bytes(_shape())
    assert lib.ssa_select_capacity(ctypes.byref(s)) == 4096
    assert _paged_call(lib, s, pages(), ws_bytes=16) == 3                  # the checks pass up to the workspace
    assert _paged_call(lib, s, None) == 1                                   # no page description
    assert _paged_call(lib, s, pages(block_table=0)) == 1
    assert _paged_call(lib, s, pages(seq_lens=0)) == 1
    for bad_ps in (0, 8, 24, 100, 1 << 21):
        assert _paged_call(lib, s, pages(page_size=bad_ps)) == 1, bad_ps
    assert _paged_call(lib, s, pages(max_pages=63)) == 1                    # 63 * 64 < ctx_len
    assert _paged_call(lib, s, pages(max_pages=0)) == 1
    assert _paged_call(lib, s, pages(num_pages=0)) == 1
    assert _paged_call(lib, s, pages(num_pages=(1 << 31) // 64)) == 1       # pool tokens past 2^31 - 1
    assert _paged_call(lib, s, pages(num_pages=(1 << 31) // 64 - 1), ws_bytes=16) == 3
    assert _paged_call(lib, s, pages(), k_new=f) == 1                       # k_new without v_new
    assert _paged_call(lib, s, pages(), k_new=f + 2, v_new=f) == 1          # misaligned
    assert _paged_call(lib, s, pages(), K=f + 2) == 1
    assert _paged_call(lib, s, pages(), k=-1) == 1
    strided = _shape()                                                      # a contiguous shape's strides
    assert _paged_call(lib, strided, pages()) == 1
    assert _decode(lib, s) == 1                                             # ... and ssa_decode wants them


def test_early_stop_entry_points_validate():
    lib = ssa.load_library()
    s = _shape()
    f = P(1 << 20)
    cap = 0
    for tau in (-1.0, float("nan")):
        assert lib.ssa_attend_early_stop(f, f, f, f, f, f, cap, f, tau, 0.1, f, f, None, f, 1 << 40,
                                         ctypes.byref(s), None) == 1
        assert lib.ssa_decode_early_stop(f, f, f, f, f, 5, 1.0, 0, 0.1, tau, f, f, None, f, 1 << 40,
                                         ctypes.byref(s), None) == 1
    assert lib.ssa_attend_early_stop(f, f, f, f, f, f, cap, None, 0.1, 0.1, f, f, None, f, 1 << 40,
                                     ctypes.byref(s), None) == 1          # no scores to order by
    assert lib.ssa_attend_early_stop(f, f, f, f, f, f, cap, f, 0.1, 0.0, f, f, None, f, 1 << 40,
                                     ctypes.byref(s), None) == 1          # scale
    assert lib.ssa_attend_early_stop(f, f, f, f, f, f, cap, f, float("inf"), 0.1, f, f, None, f, 16,
                                     ctypes.byref(s), None) == 3          # +inf passes, the workspace does not
    assert lib.ssa_decode_early_stop(f, f, f, f, f, -1, 1.0, 0, 0.1, 0.1, f, f, None, f, 1 << 40,
                                     ctypes.byref(s), None) == 1
    assert lib.ssa_decode_early_stop(f, f, f, f, f, 5, 1.0, 0, 0.1, 0.1, f, f, None, f, 16,
                                     ctypes.byref(s), None) == 3


@pytest.mark.parametrize("tile,split", [(None, None), (None, 1), (None, 5), (None, 64), (512, 64), (1024, 7),
                                        (4096, 2)])
def test_workspace_size_does_not_depend_on_the_tiling(monkeypatch, tile, split):
    """ssa_workspace_bytes is the size every call checks against, whatever tiling the plan picks: the layout
    is sized for the largest tiling."""
    if tile:
        monkeypatch.setenv("SSA_FORCE_TILE", str(tile))
    if split:
        monkeypatch.setenv("SSA_FORCE_SPLIT", str(split))
    lib = ssa.load_library()
    for shp in (_shape(), _shape(batch=1, n_q_heads=2, n_kv_heads=2, head_dim=64, d_sel=16, ctx_len=1500),
                _shape(batch=8, n_q_heads=32, n_kv_heads=16, ctx_len=131072)):
        n = ssa.ssa_workspace_bytes(shp)
        # the checks pass up to the workspace; then the fake pointers are refused (1), never the size (3)
        assert _decode(lib, shp, ws_bytes=n) == 1
        assert _decode(lib, shp, ws_bytes=n - 256) == 3
