"""CPU oracle for Stratified Sparse Attention decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library never
loads it and shares no code with it: ``ssa_oracle.c`` is a plain, slow
restatement of the method (see its header for the sources and readings),
compiled with gcc into ``oracle/libssa_oracle.so``.

bf16 tensors cross this interface as ``numpy.uint16`` arrays holding the raw
bit patterns.  Every function here is pinned in ``tests/test_oracle_*.py``
against something other than itself (an independent Philox, exact rational
sums, brute-force enumeration, closed forms and special cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssa_oracle.c")
_LIB = os.path.join(_HERE, "libssa_oracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_OK = 0
ORACLE_ERR_ARG = 1
ORACLE_ERR_OVERFLOW = 5
ORACLE_ERR_NONFINITE = 6


def build(force: bool = False) -> str:
    """Compile ssa_oracle.c with gcc -O2 -fopenmp into libssa_oracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, u64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
            lib.oracle_orderkey.argtypes = [f32]
            lib.oracle_orderkey.restype = ctypes.c_uint32
            lib.oracle_bucket_floor.argtypes = [f32]
            lib.oracle_bucket_floor.restype = f32
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_uniform.argtypes = [u64, i64, i32, i32]
            lib.oracle_uniform.restype = f32
            lib.oracle_exact_sum_f32.argtypes = [P, i64]
            lib.oracle_exact_sum_f32.restype = f32
            lib.oracle_pack_summary.argtypes = [P, P, P, i32, i32, i32, i32, i64, i64, i64, i64, i64]
            lib.oracle_pack_summary.restype = None
            lib.oracle_score.argtypes = [P, P, P, i32, i32, i32, i32, i32, i64, i64, i64, f32, P]
            lib.oracle_score.restype = None
            lib.oracle_select_unit_m.argtypes = [P, i64, i64, f32, u64, i32, i32, P, P, i64, P, P, P, i32]
            lib.oracle_select_unit_m.restype = i64
            lib.oracle_attend_unit.argtypes = [P, P, P, i32, i32, P, P, i64, f32, P, P]
            lib.oracle_attend_unit.restype = None
            lib.oracle_attend_unit_early_stop.argtypes = [P, P, P, i32, i32, P, P, P, i64, f32, f32, i64, i64,
                                                          P, P, P]
            lib.oracle_attend_unit_early_stop.restype = i64
            lib.oracle_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i64, i64, i64, i64,
                                          i64, i64, f32, u64, f32, P, P, P, P, P, P, i64, P, P]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_dense_attention.argtypes = [P, P, P, i32, i32, i32, i32, i64, i64, i64, f32, P, P]
            lib.oracle_dense_attention.restype = None
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_threads(n: int) -> int:
    """Host threads for later calls (timing runs use 1 for the single-thread figure); returns the count."""
    return int(_load().oracle_set_threads(int(n)))


def orderkey(x: float) -> int:
    return int(_load().oracle_orderkey(float(x)))


def bucket_floor(x: float) -> np.float32:
    """Lower edge of the bucket of binary32 values sharing x's top 12 order-key bits."""
    return np.float32(_load().oracle_bucket_floor(float(x)))


def philox4x32_10(ctr, key) -> np.ndarray:
    """One Philox4x32-10 block: ctr = 4 uint32 words, key = 2 uint32 words."""
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, j: int, h_kv: int, b: int) -> float:
    return float(_load().oracle_uniform(seed, j, h_kv, b))


def exact_sum_f32(x) -> np.float32:
    a = _c(x, np.float32)
    return np.float32(_load().oracle_exact_sum_f32(_ptr(a), a.size))


def pack_summary(K: np.ndarray, sel_ch: np.ndarray, d_sel: int) -> np.ndarray:
    """K: uint16 [Bt][Hkv][N][d] -> Ks: uint16 [Bt][Hkv][N][d_sel]."""
    K = _c(K, np.uint16)
    sel = _c(sel_ch, np.int32)
    Bt, Hkv, N, d = K.shape
    Ks = np.zeros((Bt, Hkv, N, d_sel), np.uint16)
    _load().oracle_pack_summary(_ptr(K), _ptr(sel), _ptr(Ks), Bt, Hkv, d, d_sel, N,
                                Hkv * N * d, N * d, Hkv * N * d_sel, N * d_sel)
    return Ks


def append(K: np.ndarray, V: np.ndarray, Ks: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
           sel_ch: np.ndarray, pos: int):
    """The append step, the plain definition ("FASA: Frequency-Aware Sparse
    Attention", section 3, Stage 1: a token's dominant channels are stored
    contiguously when it is appended).  Returns new arrays with row pos of
    every (b, h_kv) replaced:  K[b][h][pos] = k_new[b][h],
    V[b][h][pos] = v_new[b][h],  Ks[b][h][pos][j] = k_new[b][h][sel_ch[h][j]]."""
    K = np.array(K, np.uint16, copy=True)
    V = np.array(V, np.uint16, copy=True)
    Ks = np.array(Ks, np.uint16, copy=True)
    k_new = np.asarray(k_new, np.uint16)
    v_new = np.asarray(v_new, np.uint16)
    sel = np.asarray(sel_ch, np.int64)
    Bt, Hkv, N, d = K.shape
    if not 0 <= pos < N:
        raise ValueError(f"pos {pos} outside the cache of {N} tokens")
    for b in range(Bt):
        for h in range(Hkv):
            K[b, h, pos, :] = k_new[b, h, :]
            V[b, h, pos, :] = v_new[b, h, :]
            for j in range(Ks.shape[-1]):
                Ks[b, h, pos, j] = k_new[b, h, sel[h, j]]
    return K, V, Ks


def score(q: np.ndarray, Ks: np.ndarray, sel_ch: np.ndarray, scale: float) -> np.ndarray:
    """q: uint16 [Bt][Hq][d]; Ks: uint16 [Bt][Hkv][N][d_sel] -> s_hat fp32 [Bt][Hkv][N]."""
    q = _c(q, np.uint16)
    Ks = _c(Ks, np.uint16)
    sel = _c(sel_ch, np.int32)
    Bt, Hq, d = q.shape
    _, Hkv, N, d_sel = Ks.shape
    s = np.zeros((Bt, Hkv, N), np.float32)
    _load().oracle_score(_ptr(q), _ptr(Ks), _ptr(sel), Bt, Hq, Hkv, d, d_sel, N,
                         Hkv * N * d_sel, N * d_sel, float(scale), _ptr(s))
    return s


def select_unit(s: np.ndarray, top_k: int, budget: float, seed: int, b: int, h_kv: int,
                cap: int | None = None, want_p_all: bool = False, m_at_kth: bool = False):
    """Selection for one unit.  Returns (idx int32, p fp32, m, Z[, p_all]) or raises.

    m_at_kth=False (the library's reading): the reference point m of the
    exponentials is the lower edge of the 12-bit order-key bucket of the k-th
    score; True: m is the k-th score itself.  p does not depend on m in exact
    arithmetic; the pins compare the two readings."""
    s = _c(s, np.float32)
    N = s.size
    cap = N if cap is None else cap
    idx = np.zeros(max(cap, 1), np.int32)
    p = np.zeros(max(cap, 1), np.float32)
    m = ctypes.c_float()
    z = ctypes.c_float()
    p_all = np.zeros(max(N, 1), np.float32) if want_p_all else None
    cnt = _load().oracle_select_unit_m(_ptr(s), N, int(top_k), float(budget), int(seed), int(b),
                                       int(h_kv), _ptr(idx), _ptr(p), cap,
                                       ctypes.addressof(m), ctypes.addressof(z), _ptr(p_all),
                                       1 if m_at_kth else 0)
    if cnt == -1:
        raise FloatingPointError("non-finite score")
    if cnt == -2:
        raise OverflowError("selection exceeds cap")
    res = (idx[:cnt].copy(), p[:cnt].copy(), np.float32(m.value), np.float32(z.value))
    if want_p_all:
        res = res + (p_all[:N].copy(),)
    return res


def select_unit_uniform(s: np.ndarray, top_k: int, budget: float, seed: int, b: int, h_kv: int):
    """The top-k + uniform hybrid ("Stratified Sparse Attention speeds up
    decoding 2.96x on a 1M context", section "How SSA splits the cache into
    strata": top-k and hybrids are special cases of the strata).  T is the
    same top-k stratum as select_unit; every other token j is kept with the
    same probability p = min(1, fl32(B / fl32(N - k))) (p = 1 for B = +inf),
    drawn with the same Philox uniform u_j < p.  Returns (idx int32
    ascending, p fp32)."""
    s = _c(s, np.float32)
    N = s.size
    t_idx = select_unit(s, top_k, 0.0, seed, b, h_kv)[0]
    n_r = N - t_idx.size
    if n_r == 0:
        return t_idx, np.ones(t_idx.size, np.float32)
    if np.isinf(budget):
        p_r = np.float32(1.0)
    else:
        p_r = min(np.float32(1.0), np.float32(np.float32(budget) / np.float32(n_r)))
    in_t = np.zeros(N, bool)
    in_t[t_idx] = True
    keep = [j for j in range(N) if in_t[j] or uniform(seed, j, h_kv, b) < p_r]
    idx = np.array(keep, np.int32)
    return idx, np.where(in_t[idx], np.float32(1.0), p_r).astype(np.float32)


def top_p_count(s: np.ndarray, top_p: float) -> int:
    """Size of the top-p stratum (same section: top-p is another special
    case): the fewest tokens, taken in the top-k order (score descending,
    then index ascending), whose share of the softmax of s over all N tokens
    (computed in double) reaches top_p.  0 for top_p <= 0, N for top_p >= 1."""
    s = _c(s, np.float32)
    N = s.size
    if top_p <= 0.0 or N == 0:
        return 0
    if top_p >= 1.0:
        return N
    if not np.all(np.isfinite(s)):
        raise FloatingPointError("non-finite score")
    bits = s.view(np.uint32).astype(np.uint64)
    key = np.where(bits >> 31, (~bits) & 0xFFFFFFFF, bits | 0x80000000)   # order key, -0 below +0
    order = np.lexsort((np.arange(N), -key.astype(np.int64)))
    w = np.exp(s.astype(np.float64) - float(np.max(s)))
    mass = np.cumsum(w[order]) / np.sum(w)
    return int(min(N, np.searchsorted(mass, top_p, side="left") + 1))


def top_p_shares(s: np.ndarray, top_p: float):
    """(k, share of the first k - 1 tokens, share of the first k tokens) for k = top_p_count(s, top_p),
    the shares computed as top_p_count computes them: how close top_p falls to the stratum's edges."""
    s = _c(s, np.float32)
    N = s.size
    k = top_p_count(s, top_p)
    if N == 0 or k == 0:
        return k, 0.0, 0.0
    bits = s.view(np.uint32).astype(np.uint64)
    key = np.where(bits >> 31, (~bits) & 0xFFFFFFFF, bits | 0x80000000)
    order = np.lexsort((np.arange(N), -key.astype(np.int64)))
    w = np.exp(s.astype(np.float64) - float(np.max(s)))
    mass = np.cumsum(w[order]) / np.sum(w)
    return k, (float(mass[k - 2]) if k >= 2 else 0.0), float(mass[k - 1])


def select_unit_top_p(s: np.ndarray, top_p: float, budget: float, seed: int, b: int, h_kv: int):
    """The top-p stratum with the SSA sampler on the rest: T is the top-p set
    (top_p_count tokens in the top-k order, i.e. the top-k stratum with
    k = top_p_count) and the remainder is sampled exactly as select_unit
    samples it.  Returns (idx, p, m, Z) as select_unit does."""
    return select_unit(s, top_p_count(s, top_p), budget, seed, b, h_kv)


def attend_unit(q_heads, Kb, Vb, idx, p, scale: float):
    """q_heads uint16 [G][d]; Kb/Vb uint16 [N][d]; idx/p lists -> out fp32 [G][d], lse fp32 [G]."""
    q_heads = _c(q_heads, np.uint16)
    Kb = _c(Kb, np.uint16)
    Vb = _c(Vb, np.uint16)
    idx = _c(idx, np.int32)
    p = _c(p, np.float32)
    G, d = q_heads.shape
    out = np.zeros((G, d), np.float32)
    lse = np.zeros(G, np.float32)
    _load().oracle_attend_unit(_ptr(q_heads), _ptr(Kb), _ptr(Vb), G, d, _ptr(idx), _ptr(p),
                               idx.size, float(scale), _ptr(out), _ptr(lse))
    return out, lse


def attend_unit_early_stop(q_heads, Kb, Vb, idx, p, s, scale: float, tau: float, block: int = 128,
                           force_blocks: int = -1):
    """Corrected attention over one unit's selected rows with S2O-style early stopping ("S2O ...", technical
    summary, Method section 2): rows ordered by s descending (ties by list position), blocks of `block` rows,
    stop after the first block whose gain is below tau times the accumulated denominator for every head.
    Returns (out fp32 [G][d], lse fp32 [G], blocks processed, per-block max gain ratio)."""
    q_heads = _c(q_heads, np.uint16)
    Kb = _c(Kb, np.uint16)
    Vb = _c(Vb, np.uint16)
    idx = _c(idx, np.int32)
    p = _c(p, np.float32)
    s = _c(s, np.float32)
    G, d = q_heads.shape
    n = idx.size
    out = np.zeros((G, d), np.float32)
    lse = np.zeros(G, np.float32)
    ratios = np.zeros(max(1, -(-n // block)), np.float32)
    used = _load().oracle_attend_unit_early_stop(_ptr(q_heads), _ptr(Kb), _ptr(Vb), G, d, _ptr(idx), _ptr(p),
                                                 _ptr(s), n, float(scale), float(tau), int(block),
                                                 int(force_blocks), _ptr(out), _ptr(lse), _ptr(ratios))
    return out, lse, int(used), ratios[:-(-n // block)]


def decode(q, K, V, Ks, sel_ch, top_k: int, budget: float, seed: int, scale: float,
           want_lists: bool = True):
    """The whole step.  Returns a dict with out, lse, s_hat and (optionally) idx, p, count, m, Z."""
    q = _c(q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    Ks = _c(Ks, np.uint16)
    sel = _c(sel_ch, np.int32)
    Bt, Hq, d = q.shape
    _, Hkv, N, _ = K.shape
    d_sel = Ks.shape[-1]
    out = np.zeros((Bt, Hq, d), np.float32)
    lse = np.zeros((Bt, Hq), np.float32)
    s_hat = np.zeros((Bt, Hkv, N), np.float32)
    cap = max(N, 1)
    idx = np.zeros((Bt, Hkv, cap), np.int32) if want_lists else None
    p = np.zeros((Bt, Hkv, cap), np.float32) if want_lists else None
    count = np.zeros((Bt, Hkv), np.int64)
    m = np.zeros((Bt, Hkv), np.float32)
    Z = np.zeros((Bt, Hkv), np.float32)
    rc = _load().oracle_decode(_ptr(q), _ptr(K), _ptr(V), _ptr(Ks), _ptr(sel), Bt, Hq, Hkv, d,
                               d_sel, N, Hkv * N * d, N * d, Hkv * N * d_sel, N * d_sel,
                               int(top_k), float(budget), int(seed), float(scale),
                               _ptr(out), _ptr(lse), _ptr(s_hat), _ptr(idx), _ptr(p), _ptr(count),
                               cap, _ptr(m), _ptr(Z))
    if rc != ORACLE_OK:
        raise RuntimeError(f"oracle_decode failed with code {rc}")
    res = dict(out=out, lse=lse, s_hat=s_hat, count=count, m=m, Z=Z)
    if want_lists:
        res.update(idx=idx, p=p)
    return res


def dense_attention(q, K, V, scale: float):
    q = _c(q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    Bt, Hq, d = q.shape
    _, Hkv, N, _ = K.shape
    out = np.zeros((Bt, Hq, d), np.float32)
    lse = np.zeros((Bt, Hq), np.float32)
    _load().oracle_dense_attention(_ptr(q), _ptr(K), _ptr(V), Bt, Hq, Hkv, d, N, Hkv * N * d,
                                   N * d, float(scale), _ptr(out), _ptr(lse))
    return out, lse
