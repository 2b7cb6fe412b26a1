"""Python binding of libssa (include/ssa.h): argument marshalling only.

Every computation runs in the CUDA library ``libssa.so`` built in-tree for
sm_103a; this module only turns torch tensors into pointers, sizes, strides
and the current CUDA stream.  If the library is missing it raises instead
of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssa.so")

SSA_OK = 0
STATUS_NAMES = {
    0: "SSA_OK", 1: "SSA_ERR_INVALID_ARG", 2: "SSA_ERR_UNSUPPORTED", 3: "SSA_ERR_WORKSPACE",
    4: "SSA_ERR_CUDA", 5: "SSA_ERR_OVERFLOW", 6: "SSA_ERR_NONFINITE", 7: "SSA_ERR_DEVICE_TIMEOUT",
    8: "SSA_ERR_BAD_INDEX",
}
DEV_NONFINITE, DEV_OVERFLOW, DEV_TIMEOUT, DEV_BAD_INDEX = 0x1, 0x2, 0x4, 0x8

EXPORTS = [
    "ssa_status_string", "ssa_version", "ssa_workspace_bytes", "ssa_pack_summary", "ssa_score",
    "ssa_select", "ssa_attend", "ssa_decode", "ssa_decode_host", "ssa_get_device_status",
    "ssa_query_plan", "ssa_decode_static", "ssa_append", "ssa_decode_append", "ssa_select_capacity",
    "ssa_select_strata", "ssa_decode_strata", "ssa_decode_paged", "ssa_attend_early_stop",
    "ssa_decode_early_stop",
]
STRATA_SSA, STRATA_UNIFORM, STRATA_TOP_P = 0, 1, 2


class SsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({_status_string(status)})")


class ssa_shape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("d_sel", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("ctx_len", ctypes.c_int64), ("kv_stride_b", ctypes.c_int64), ("kv_stride_h", ctypes.c_int64),
        ("ks_stride_b", ctypes.c_int64), ("ks_stride_h", ctypes.c_int64),
    ]


class ssa_paged_kv(ctypes.Structure):
    _fields_ = [
        ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
    ]


_lib = None


def load_library():
    """Load libssa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libssa.so not found at {LIB_PATH}; build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                 ctypes.c_float, ctypes.c_size_t)
    SP = ctypes.POINTER(ssa_shape)
    sig = {
        "ssa_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "ssa_version": ([], ctypes.c_int),
        "ssa_workspace_bytes": ([SP, i64], sz),
        "ssa_select_capacity": ([SP], sz),
        "ssa_pack_summary": ([P, P, P, P, sz, SP, P], ctypes.c_int),
        "ssa_append": ([P, P, P, i64, P, P, P, P, sz, SP, P], ctypes.c_int),
        "ssa_decode_append": ([P, P, P, P, P, P, P, i64, f32, u64, f32, P, P, P, sz, SP, P], ctypes.c_int),
        "ssa_score": ([P, P, P, f32, P, P, sz, SP, P], ctypes.c_int),
        "ssa_select": ([P, i64, f32, u64, P, P, P, i64, P, sz, SP, P], ctypes.c_int),
        "ssa_select_strata": ([P, ctypes.c_int, i64, f32, f32, u64, P, P, P, i64, P, sz, SP, P], ctypes.c_int),
        "ssa_decode_strata": ([P, P, P, P, P, ctypes.c_int, i64, f32, f32, u64, f32, P, P, P, P, P, P, i64, P, sz, SP, P],
                              ctypes.c_int),
        "ssa_attend": ([P, P, P, P, P, P, i64, f32, P, P, P, sz, SP, P], ctypes.c_int),
        "ssa_decode": ([P, P, P, P, P, i64, f32, u64, f32, P, P, P, P, P, P, i64, P, sz, SP, P], ctypes.c_int),
        "ssa_decode_host": ([P, P, P, P, P, i64, f32, u64, f32, P, P, P, sz, SP, P], ctypes.c_int),
        "ssa_get_device_status": ([P, P, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
        "ssa_query_plan": ([SP, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)], ctypes.c_int),
        "ssa_decode_static": ([P, P, P, P, P, i64, f32, u64, f32, P, P, P, SP, P], ctypes.c_int),
        "ssa_decode_paged": ([P, P, P, P, P, P, ctypes.POINTER(ssa_paged_kv), P, i64, f32, u64, f32, P, P, P, P, P,
                              P, i64, P, sz, SP, P], ctypes.c_int),
        "ssa_attend_early_stop": ([P, P, P, P, P, P, i64, P, f32, f32, P, P, P, P, sz, SP, P], ctypes.c_int),
        "ssa_decode_early_stop": ([P, P, P, P, P, i64, f32, u64, f32, f32, P, P, P, P, sz, SP, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _status_string(status: int) -> str:
    try:
        return load_library().ssa_status_string(status).decode()
    except Exception:  # pragma: no cover - only used in error messages
        return "?"


def _check(status: int, what: str):
    if status != SSA_OK:
        raise SsaError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_shape(batch, n_q_heads, n_kv_heads, head_dim, d_sel, ctx_len, kv_strides=None, ks_strides=None) -> ssa_shape:
    kv_sh = ctx_len * head_dim
    ks_sh = ctx_len * d_sel
    kv_sb, kv_sh = kv_strides if kv_strides is not None else (n_kv_heads * kv_sh, kv_sh)
    ks_sb, ks_sh = ks_strides if ks_strides is not None else (n_kv_heads * ks_sh, ks_sh)
    return ssa_shape(batch, n_q_heads, n_kv_heads, head_dim, d_sel, 0, ctx_len, kv_sb, kv_sh, ks_sb, ks_sh)


def shape_of(q: torch.Tensor, K: torch.Tensor, Ks: Optional[torch.Tensor] = None, d_sel: Optional[int] = None) -> ssa_shape:
    """Shape from q [Bt][Hq][d], K [Bt][Hkv][N][d] and (optionally) Ks [Bt][Hkv][N][d_sel]."""
    Bt, Hq, d = q.shape
    _, Hkv, N, _ = K.shape
    if K.stride(3) != 1 or (N > 1 and K.stride(2) != d):
        raise ValueError("K/V rows must be contiguous with token stride head_dim")
    if Ks is not None:
        d_sel = Ks.shape[-1]
        if Ks.stride(3) != 1 or (N > 1 and Ks.stride(2) != d_sel):
            raise ValueError("Ks rows must be contiguous with token stride d_sel")
        ks = (Ks.stride(0), Ks.stride(1))
    else:
        d_sel = 32 if d_sel is None else d_sel
        ks = None
    return make_shape(Bt, Hq, Hkv, d, d_sel, N, (K.stride(0), K.stride(1)), ks)


def _scores_shape(s_hat: torch.Tensor) -> ssa_shape:
    Bt, Hkv, N = s_hat.shape
    return make_shape(Bt, Hkv, Hkv, 64, 16, N)


def ssa_version() -> int:
    return int(load_library().ssa_version())


def ssa_workspace_bytes(shape: ssa_shape, list_cap: int = 0) -> int:
    return int(load_library().ssa_workspace_bytes(ctypes.byref(shape), int(list_cap)))


def ssa_select_capacity(shape: ssa_shape) -> int:
    """Worst-case selected rows per unit (ctx_len): a list capacity that never overflows."""
    return int(load_library().ssa_select_capacity(ctypes.byref(shape)))


def workspace(shape: ssa_shape, list_cap: int = 0, device="cuda") -> torch.Tensor:
    n = ssa_workspace_bytes(shape, list_cap)
    if n == 0:
        raise SsaError(1, "ssa_workspace_bytes")
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def ssa_pack_summary(K: torch.Tensor, sel_ch: torch.Tensor, Ks: Optional[torch.Tensor] = None,
                     ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    Bt, Hkv, N, d = K.shape
    d_sel = sel_ch.shape[-1]
    if Ks is None:
        Ks = torch.empty((Bt, Hkv, N, d_sel), dtype=K.dtype, device=K.device)
    shape = make_shape(Bt, Hkv, Hkv, d, d_sel, N, (K.stride(0), K.stride(1)), (Ks.stride(0), Ks.stride(1)))
    if ws is None:
        ws = workspace(shape, 0, K.device)
    _check(load_library().ssa_pack_summary(_ptr(K), _ptr(sel_ch), _ptr(Ks), _ptr(ws), ws.numel(),
                                           ctypes.byref(shape), _stream(stream)), "ssa_pack_summary")
    return Ks


def ssa_score(q, Ks, sel_ch, scale: float, s_hat=None, ws=None, stream=None, K_like=None) -> torch.Tensor:
    Bt, Hq, d = q.shape
    _, Hkv, N, d_sel = Ks.shape
    shape = make_shape(Bt, Hq, Hkv, d, d_sel, N, None, (Ks.stride(0), Ks.stride(1)))
    if s_hat is None:
        s_hat = torch.empty((Bt, Hkv, N), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(shape, 0, q.device)
    _check(load_library().ssa_score(_ptr(q), _ptr(Ks), _ptr(sel_ch), float(scale), _ptr(s_hat), _ptr(ws),
                                    ws.numel(), ctypes.byref(shape), _stream(stream)), "ssa_score")
    return s_hat


def ssa_select(s_hat: torch.Tensor, top_k: int, budget: float, seed: int, idx=None, p=None, count=None,
               list_cap: int = 0, ws=None, stream=None):
    """Returns (idx [Bt][Hkv][cap] int32, p [Bt][Hkv][cap] fp32, count [Bt][Hkv] int32)."""
    Bt, Hkv, N = s_hat.shape
    shape = _scores_shape(s_hat)
    cap = list_cap if list_cap > 0 else max(N, 1)
    if idx is None:
        idx = torch.empty((Bt, Hkv, cap), dtype=torch.int32, device=s_hat.device)
    if p is None:
        p = torch.empty((Bt, Hkv, cap), dtype=torch.float32, device=s_hat.device)
    if count is None:
        count = torch.empty((Bt, Hkv), dtype=torch.int32, device=s_hat.device)
    if ws is None:
        ws = workspace(shape, cap, s_hat.device)
    _check(load_library().ssa_select(_ptr(s_hat), int(top_k), float(budget), int(seed) & (2**64 - 1),
                                     _ptr(idx), _ptr(p), _ptr(count), int(cap), _ptr(ws), ws.numel(),
                                     ctypes.byref(shape), _stream(stream)), "ssa_select")
    return idx, p, count


def ssa_select_strata(s_hat: torch.Tensor, strata: int, top_k: int, top_p: float, budget: float, seed: int,
                      idx=None, p=None, count=None, list_cap: int = 0, ws=None, stream=None):
    """ssa_select with a choice of strata (STRATA_SSA, STRATA_UNIFORM, STRATA_TOP_P)."""
    Bt, Hkv, N = s_hat.shape
    shape = _scores_shape(s_hat)
    cap = list_cap if list_cap > 0 else max(N, 1)
    if idx is None:
        idx = torch.empty((Bt, Hkv, cap), dtype=torch.int32, device=s_hat.device)
    if p is None:
        p = torch.empty((Bt, Hkv, cap), dtype=torch.float32, device=s_hat.device)
    if count is None:
        count = torch.empty((Bt, Hkv), dtype=torch.int32, device=s_hat.device)
    if ws is None:
        ws = workspace(shape, cap, s_hat.device)
    _check(load_library().ssa_select_strata(_ptr(s_hat), int(strata), int(top_k), float(top_p), float(budget),
                                            int(seed) & (2**64 - 1), _ptr(idx), _ptr(p), _ptr(count), int(cap),
                                            _ptr(ws), ws.numel(), ctypes.byref(shape), _stream(stream)),
           "ssa_select_strata")
    return idx, p, count


def ssa_attend(q, K, V, idx, p, count, scale: float, out=None, lse=None, ws=None, stream=None):
    """Returns (out [Bt][Hq][d] fp32, lse [Bt][Hq] fp32)."""
    shape = shape_of(q, K, d_sel=16)
    cap = idx.shape[-1]
    Bt, Hq, d = q.shape
    if out is None:
        out = torch.empty((Bt, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Bt, Hq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(shape, cap, q.device)
    _check(load_library().ssa_attend(_ptr(q), _ptr(K), _ptr(V), _ptr(idx), _ptr(p), _ptr(count), int(cap),
                                     float(scale), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                     ctypes.byref(shape), _stream(stream)), "ssa_attend")
    return out, lse


def ssa_attend_early_stop(q, K, V, idx, p, count, s_hat, tau: float, scale: float, out=None, lse=None, blocks=None,
                          ws=None, stream=None):
    """Corrected attention with S2O-style early stopping; returns (out, lse, blocks kept [Bt][Hkv])."""
    shape = shape_of(q, K)
    Bt, Hq, d = q.shape
    Hkv = K.shape[1]
    if out is None:
        out = torch.empty((Bt, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Bt, Hq), dtype=torch.float32, device=q.device)
    if blocks is None:
        blocks = torch.empty((Bt, Hkv), dtype=torch.int32, device=q.device)
    if ws is None:
        ws = workspace(shape, idx.shape[-1], q.device)
    _check(load_library().ssa_attend_early_stop(_ptr(q), _ptr(K), _ptr(V), _ptr(idx), _ptr(p), _ptr(count),
                                                int(idx.shape[-1]), _ptr(s_hat), float(tau), float(scale), _ptr(out),
                                                _ptr(lse), _ptr(blocks), _ptr(ws), ws.numel(), ctypes.byref(shape),
                                                _stream(stream)), "ssa_attend_early_stop")
    return out, lse, blocks


def ssa_decode_early_stop(q, K, V, Ks, sel_ch, top_k: int, budget: float, seed: int, scale: float, tau: float,
                          out=None, lse=None, blocks=None, ws=None, stream=None):
    """The step with early-stopping attention; returns (out, lse, blocks kept [Bt][Hkv])."""
    shape = shape_of(q, K, Ks)
    Bt, Hq, d = q.shape
    Hkv = K.shape[1]
    if out is None:
        out = torch.empty((Bt, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Bt, Hq), dtype=torch.float32, device=q.device)
    if blocks is None:
        blocks = torch.empty((Bt, Hkv), dtype=torch.int32, device=q.device)
    if ws is None:
        ws = workspace(shape, 0, q.device)
    _check(load_library().ssa_decode_early_stop(_ptr(q), _ptr(K), _ptr(V), _ptr(Ks), _ptr(sel_ch), int(top_k),
                                                float(budget), int(seed) & (2**64 - 1), float(scale), float(tau),
                                                _ptr(out), _ptr(lse), _ptr(blocks), _ptr(ws), ws.numel(),
                                                ctypes.byref(shape), _stream(stream)), "ssa_decode_early_stop")
    return out, lse, blocks


def ssa_decode(q, K, V, Ks, sel_ch, top_k: int, budget: float, seed: int, scale: float, out=None, lse=None,
               s_hat=None, idx=None, p=None, count=None, list_cap: int = 0, ws=None, stream=None):
    """The whole step; returns (out, lse).  s_hat / idx / p / count receive intermediates when given."""
    shape = shape_of(q, K, Ks)
    Bt, Hq, d = q.shape
    if out is None:
        out = torch.empty((Bt, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Bt, Hq), dtype=torch.float32, device=q.device)
    cap = list_cap if list_cap > 0 else (idx.shape[-1] if idx is not None else 0)
    if ws is None:
        ws = workspace(shape, cap, q.device)
    _check(load_library().ssa_decode(_ptr(q), _ptr(K), _ptr(V), _ptr(Ks), _ptr(sel_ch), int(top_k),
                                     float(budget), int(seed) & (2**64 - 1), float(scale), _ptr(out),
                                     _ptr(lse), _ptr(s_hat), _ptr(idx), _ptr(p), _ptr(count), int(cap),
                                     _ptr(ws), ws.numel(), ctypes.byref(shape), _stream(stream)), "ssa_decode")
    return out, lse


def ssa_decode_strata(q, K, V, Ks, sel_ch, strata: int, top_k: int, top_p: float, budget: float, seed: int,
                      scale: float, out=None, lse=None, s_hat=None, idx=None, p=None, count=None, list_cap: int = 0,
                      ws=None, stream=None):
    """ssa_decode with a choice of strata; returns (out, lse)."""
    shape = shape_of(q, K, Ks)
    Bt, Hq, d = q.shape
    if out is None:
        out = torch.empty((Bt, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Bt, Hq), dtype=torch.float32, device=q.device)
    cap = list_cap if list_cap > 0 else (idx.shape[-1] if idx is not None else 0)
    if ws is None:
        ws = workspace(shape, cap, q.device)
    _check(load_library().ssa_decode_strata(_ptr(q), _ptr(K), _ptr(V), _ptr(Ks), _ptr(sel_ch), int(strata),
                                            int(top_k), float(top_p), float(budget), int(seed) & (2**64 - 1),
                                            float(scale), _ptr(out), _ptr(lse), _ptr(s_hat), _ptr(idx), _ptr(p),
                                            _ptr(count), int(cap), _ptr(ws), ws.numel(), ctypes.byref(shape),
                                            _stream(stream)), "ssa_decode_strata")
    return out, lse


def ssa_append(k_new, v_new, sel_ch, pos: int, K, V, Ks, ws=None, stream=None):
    """Write the new token's rows (k_new, v_new [Bt][Hkv][d]) at position pos of K, V and its summary row of Ks."""
    Bt, Hkv, N, d = K.shape
    if tuple(k_new.shape) != (Bt, Hkv, d) or tuple(v_new.shape) != (Bt, Hkv, d):
        raise ValueError("k_new / v_new must be [Bt][Hkv][head_dim]")
    if not (k_new.is_contiguous() and v_new.is_contiguous()):
        raise ValueError("k_new / v_new must be contiguous")
    shape = make_shape(Bt, Hkv, Hkv, d, Ks.shape[-1], N, (K.stride(0), K.stride(1)), (Ks.stride(0), Ks.stride(1)))
    if ws is None:
        ws = workspace(shape, 0, K.device)
    _check(load_library().ssa_append(_ptr(k_new), _ptr(v_new), _ptr(sel_ch), int(pos), _ptr(K), _ptr(V), _ptr(Ks),
                                     _ptr(ws), ws.numel(), ctypes.byref(shape), _stream(stream)), "ssa_append")


def ssa_decode_append(q, k_new, v_new, K, V, Ks, sel_ch, top_k: int, budget: float, seed: int, scale: float,
                      out=None, lse=None, ws=None, stream=None):
    """Append the new token at position ctx_len - 1 of K, V, Ks, then decode over all ctx_len tokens."""
    shape = shape_of(q, K, Ks)
    Bt, Hq, d = q.shape
    _, Hkv, _, _ = K.shape
    if tuple(k_new.shape) != (Bt, Hkv, d) or tuple(v_new.shape) != (Bt, Hkv, d):
        raise ValueError("k_new / v_new must be [Bt][Hkv][head_dim]")
    if not (k_new.is_contiguous() and v_new.is_contiguous()):
        raise ValueError("k_new / v_new must be contiguous")
    if out is None:
        out = torch.empty((Bt, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Bt, Hq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(shape, 0, q.device)
    _check(load_library().ssa_decode_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(K), _ptr(V), _ptr(Ks),
                                            _ptr(sel_ch), int(top_k), float(budget), int(seed) & (2**64 - 1),
                                            float(scale), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                            ctypes.byref(shape), _stream(stream)), "ssa_decode_append")
    return out, lse


def paged_shape(q: torch.Tensor, K_pool: torch.Tensor, Ks_pool: torch.Tensor, ctx_len: int) -> ssa_shape:
    """Shape of a paged step: q [Bt][Hq][d], pools [num_pages][Hkv][page_size][d / d_sel], longest sequence ctx_len
    (the stride fields are 0)."""
    Bt, Hq, d = q.shape
    _, Hkv, _, _ = K_pool.shape
    return ssa_shape(Bt, Hq, Hkv, d, Ks_pool.shape[-1], 0, int(ctx_len), 0, 0, 0, 0)


def ssa_decode_paged(q, K_pool, V_pool, Ks_pool, block_table, seq_lens, sel_ch, top_k: int, budget: float, seed: int,
                     scale: float, ctx_len: int, k_new=None, v_new=None, out=None, lse=None, s_hat=None, idx=None,
                     p=None, count=None, list_cap: int = 0, ws=None, stream=None):
    """The step over a paged, variable-length cache; returns (out, lse).

    K_pool, V_pool [num_pages][Hkv][page_size][d] and Ks_pool [num_pages][Hkv][page_size][d_sel] (contiguous),
    block_table [Bt][max_pages] and seq_lens [Bt] int32 on the device, ctx_len >= every seq_lens[b].  With k_new /
    v_new [Bt][Hkv][d] the new token is first written at position seq_lens[b] - 1 of each sequence."""
    for t in (K_pool, V_pool, Ks_pool, block_table, seq_lens):
        if not t.is_contiguous():
            raise ValueError("pools, block table and lengths must be contiguous")
    num_pages, Hkv, page_size, d = K_pool.shape
    Bt, Hq, _ = q.shape
    if tuple(block_table.shape[:1]) != (Bt,) or tuple(seq_lens.shape) != (Bt,):
        raise ValueError("block_table must be [Bt][max_pages] and seq_lens [Bt]")
    shape = paged_shape(q, K_pool, Ks_pool, ctx_len)
    pages = ssa_paged_kv(page_size, block_table.shape[1], num_pages, block_table.data_ptr(), seq_lens.data_ptr())
    if out is None:
        out = torch.empty((Bt, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Bt, Hq), dtype=torch.float32, device=q.device)
    cap = list_cap if list_cap > 0 else (idx.shape[-1] if idx is not None else 0)
    if ws is None:
        ws = workspace(shape, cap, q.device)
    _check(load_library().ssa_decode_paged(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(K_pool), _ptr(V_pool),
                                           _ptr(Ks_pool), ctypes.byref(pages), _ptr(sel_ch), int(top_k),
                                           float(budget), int(seed) & (2**64 - 1), float(scale), _ptr(out),
                                           _ptr(lse), _ptr(s_hat), _ptr(idx), _ptr(p), _ptr(count), int(cap),
                                           _ptr(ws), ws.numel(), ctypes.byref(shape), _stream(stream)),
           "ssa_decode_paged")
    return out, lse


def ssa_decode_host(q_host, K, V, Ks, sel_ch, top_k: int, budget: float, seed: int, scale: float,
                    out_host, lse_host, ws, stream=None):
    """Enqueue H2D(q) -> decode -> D2H(out, lse) on the stream; the caller synchronises."""
    shape = shape_of(q_host, K, Ks)
    _check(load_library().ssa_decode_host(_ptr(q_host), _ptr(K), _ptr(V), _ptr(Ks), _ptr(sel_ch), int(top_k),
                                          float(budget), int(seed) & (2**64 - 1), float(scale),
                                          _ptr(out_host), _ptr(lse_host), _ptr(ws), ws.numel(),
                                          ctypes.byref(shape), _stream(stream)), "ssa_decode_host")


def ssa_get_device_status(ws: torch.Tensor, stream=None):
    """Synchronise, read and clear the device status bits.  Returns (status, flags)."""
    flags = ctypes.c_uint32(0)
    st = load_library().ssa_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


def ssa_query_plan(shape: ssa_shape):
    """(score-kernel CTAs, selection tiles per unit, attention CTAs per unit)."""
    c, r, s = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().ssa_query_plan(ctypes.byref(shape), ctypes.byref(c), ctypes.byref(r), ctypes.byref(s)),
           "ssa_query_plan")
    return c.value, r.value, s.value


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
