"""Synthetic long-context decode workloads with the shapes of the models the pages name.

The pages evaluate on RULER / LongBench / LOFT / AIME with real models
(Ministral-3-8B and a 27B model, "Numbers and speedup" on the Stratified
Sparse Attention news page).  Neither the suites nor the weights are
available, so seeded synthetic layers with those shapes stand in for them:

* keys: N(0, 1) per channel; the 8 channels of the 4 lowest-frequency RoPE
  pairs scaled x5 (outlier channels); RoPE (half-split pairs (j, j + d/2),
  theta_j = base^(-2j/d)) applied at position i.  This gives the "frequency
  chunk" structure of "FASA: Frequency-Aware Sparse Attention", section 2:
  low-frequency chunks carry the position-independent (semantic) signal.
* values: N(0, 1).
* needles: per (b, h_kv) a set of planted positions; every query head of the
  group is q = RoPE(z, N) + alpha * mean(rotated needle keys), z ~ N(0, I),
  so the needles are the tokens that matter.
* the tiny case has no RoPE, sinks at positions 0-3 (keys x2; sinks are the
  always-attended first tokens of the sparse-attention glossary, "Common
  patterns") and 8 needles over [4, N).
* the summary channels ``sel_ch`` (the dominant chunks of FASA section 3,
  Stage 1, calibrated offline on data the pages do not give) come from a
  synthetic calibration: 64 calibration queries (seed + 1000) score every
  RoPE pair by the mean over queries of sum_i |q_c . k_{i,c}| over the first
  min(N, 32768) keys of batch 0; the top d_sel/2 pairs (both channels, in
  ascending order) are kept.  The tiny case uses channels 0..15.

All values are drawn in fp32 and rounded to bf16 (round to nearest even).
Random streams are torch generators seeded from (seed, stream tag), on the
device the tensors are made on (CPU and CUDA streams differ; each side of a
comparison reads the same bytes).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx_len: int
    d_sel: int
    top_k: int
    budget: float
    n_needles: int
    alpha: float
    rope: bool = True
    rope_base: float = 1e6
    sinks: bool = False
    needles_even: bool = False
    seeds: tuple = (0,)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def units(self) -> int:
        return self.batch * self.n_kv_heads


def budget_split(ctx_len: int, sparsity: int):
    """Total budget floor(N / s), split as top-k = ceil(half), B = floor(half)."""
    total = ctx_len // sparsity
    return (total + 1) // 2, float(total // 2)


def _ministral(name, batch, ctx_len, n_needles=16, needles_even=False, seeds=(0,), sparsity=50):
    k, B = budget_split(ctx_len, sparsity)
    return WorkloadConfig(name, batch, 32, 8, 128, ctx_len, 32, k, B, n_needles, 2.0,
                          needles_even=needles_even, seeds=seeds)


def _gemma27(name, sparsity: Optional[int]):
    if sparsity is None:  # dense limit: B covers every non-top-k token
        k, B = budget_split(131072, 50)[0], math.inf
    else:
        k, B = budget_split(131072, sparsity)
    return WorkloadConfig(name, 8, 32, 16, 128, 131072, 32, k, B, 16, 2.0)


CONFIGS = {
    "tiny": WorkloadConfig("tiny", 1, 4, 1, 64, 2048, 16, 32, 32.0, 8, 3.0, rope=False, sinks=True),
    "ministral8b_32k": _ministral("ministral8b_32k", 4, 32768),
    "ministral8b_128k": _ministral("ministral8b_128k", 2, 131072, seeds=tuple(range(10))),
    "ministral8b_1m": _ministral("ministral8b_1m", 1, 1048576, n_needles=64, needles_even=True),
    "27b_128k_10x": _gemma27("27b_128k_10x", 10),
    "27b_128k_20x": _gemma27("27b_128k_20x", 20),
    "27b_128k_50x": _gemma27("27b_128k_50x", 50),
    "27b_128k_100x": _gemma27("27b_128k_100x", 100),
    "27b_128k_dense": _gemma27("27b_128k_dense", None),
}


def make_config(base: str = "ministral8b_32k", **overrides) -> WorkloadConfig:
    """A named config with some fields replaced (used for small parity cases)."""
    cfg = dataclasses.replace(CONFIGS[base], **overrides)
    if "name" not in overrides:
        cfg = dataclasses.replace(cfg, name=base + "+" + ",".join(f"{k}={v}" for k, v in overrides.items()))
    return cfg


def _generator(device, seed: int, tag: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tag * 7919 + 12345) % (2**63 - 1))
    return g


def _rope_tables(positions: torch.Tensor, d: int, base: float):
    """cos/sin [len(positions)][d/2] in fp32, angles formed in fp64."""
    j = torch.arange(d // 2, device=positions.device, dtype=torch.float64)
    theta = base ** (-2.0 * j / d)
    ang = positions.to(torch.float64)[:, None] * theta[None, :]
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)


def _rotate(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor) -> torch.Tensor:
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    return torch.cat([a * cos - b * sin, a * sin + b * cos], dim=-1)


def _outlier_channels(d: int):
    """The 8 channels of the 4 lowest-frequency half-split RoPE pairs."""
    h = d // 2
    pairs = list(range(h - 4, h))
    return pairs + [p + h for p in pairs]


def _keys_for_head(cfg: WorkloadConfig, seed: int, b: int, h: int, device, chunk: int = 1 << 18):
    """fp32 keys [N][d] of one (b, h_kv), after outliers, sinks and RoPE."""
    N, d = cfg.ctx_len, cfg.head_dim
    gen = _generator(device, seed, 1000 + b * 4096 + h)
    K = torch.randn((N, d), generator=gen, device=device, dtype=torch.float32)
    if cfg.rope:
        K[:, _outlier_channels(d)] *= 5.0
        for s in range(0, N, chunk):
            e = min(N, s + chunk)
            cos, sin = _rope_tables(torch.arange(s, e, device=device), d, cfg.rope_base)
            K[s:e] = _rotate(K[s:e], cos, sin)
    if cfg.sinks:
        K[:4] *= 2.0
    return K


def _needle_positions(cfg: WorkloadConfig, seed: int, b: int, h: int, device):
    N, n = cfg.ctx_len, cfg.n_needles
    if cfg.needles_even:
        return torch.tensor([int((j + 0.5) * N / n) for j in range(n)], device=device, dtype=torch.long)
    lo = 4 if cfg.sinks else 0
    gen = _generator(device, seed, 2000 + b * 4096 + h)
    perm = torch.randperm(N - lo, generator=gen, device=device)[:n]
    return torch.sort(perm + lo).values


def _calibrate_sel_ch(cfg: WorkloadConfig, seed: int, h: int, K0: torch.Tensor, device) -> torch.Tensor:
    d, half = cfg.head_dim, cfg.head_dim // 2
    if not cfg.rope:
        return torch.arange(cfg.d_sel, device=device, dtype=torch.int32)
    gen = _generator(device, seed + 1000, 3000 + h)
    Tn = min(cfg.ctx_len, 32768)
    zq = torch.randn((64, d), generator=gen, device=device, dtype=torch.float32)
    cos, sin = _rope_tables(torch.tensor([cfg.ctx_len], device=device), d, cfg.rope_base)
    qc = _rotate(zq, cos, sin)
    keys = K0[:Tn]
    score = torch.empty(half, device=device, dtype=torch.float64)
    for j in range(half):
        qp = qc[:, [j, j + half]]                     # [64][2]
        kp = keys[:, [j, j + half]]                   # [Tn][2]
        score[j] = (qp @ kp.T).abs().sum(dim=1).to(torch.float64).mean()
    # top d_sel/2 pairs, ties to the lower pair index
    order = sorted(range(half), key=lambda j: (-float(score[j]), j))[: cfg.d_sel // 2]
    ch = sorted(order + [j + half for j in order])
    return torch.tensor(ch, device=device, dtype=torch.int32)


def generate(cfg: WorkloadConfig, seed: int = 0, device="cpu") -> dict:
    """Build one workload: q [Bt][Hq][d], K/V [Bt][Hkv][N][d] (bf16), sel_ch [Hkv][d_sel] (int32).

    Also returns the config's scalars (scale, top_k, budget, seed) and the needle positions."""
    device = torch.device(device)
    Bt, Hq, Hkv, d, N, G = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ctx_len, cfg.group
    K = torch.empty((Bt, Hkv, N, d), device=device, dtype=torch.bfloat16)
    V = torch.empty((Bt, Hkv, N, d), device=device, dtype=torch.bfloat16)
    q = torch.empty((Bt, Hq, d), device=device, dtype=torch.bfloat16)
    sel_ch = torch.empty((Hkv, cfg.d_sel), device=device, dtype=torch.int32)
    needles = torch.empty((Bt, Hkv, cfg.n_needles), device=device, dtype=torch.long)
    if cfg.rope:
        qcos, qsin = _rope_tables(torch.tensor([N], device=device), d, cfg.rope_base)
    for b in range(Bt):
        for h in range(Hkv):
            Kf = _keys_for_head(cfg, seed, b, h, device)
            if b == 0:
                sel_ch[h] = _calibrate_sel_ch(cfg, seed, h, Kf, device)
            pos = _needle_positions(cfg, seed, b, h, device) if cfg.n_needles > 0 else None
            gen_q = _generator(device, seed, 4000 + b * 4096 + h)
            z = torch.randn((G, d), generator=gen_q, device=device, dtype=torch.float32)
            if cfg.rope:
                z = _rotate(z, qcos, qsin)
            if pos is not None:
                needles[b, h] = pos
                z = z + cfg.alpha * Kf[pos].mean(dim=0, keepdim=True)
            q[b, h * G:(h + 1) * G] = z.to(torch.bfloat16)
            K[b, h] = Kf.to(torch.bfloat16)
            del Kf
            gen_v = _generator(device, seed, 5000 + b * 4096 + h)
            V[b, h] = torch.randn((N, d), generator=gen_v, device=device, dtype=torch.float32).to(torch.bfloat16)
    return dict(cfg=cfg, q=q, K=K, V=V, sel_ch=sel_ch, needles=needles, scale=cfg.scale,
                top_k=cfg.top_k, budget=cfg.budget, seed=seed)


def to_paged(K: torch.Tensor, V: torch.Tensor, Ks: torch.Tensor, lens, page_size: int, seed: int = 0,
             spare_pages: int = 2) -> dict:
    """A paged, variable-length copy of a contiguous cache (the serving layout of a batch of sequences).

    Sequence b keeps its first lens[b] tokens, cut into pages of page_size tokens; the pages of all sequences are
    placed in a random order in pools K_pool / V_pool [num_pages][Hkv][page_size][d] and Ks_pool [..][d_sel].  Slots
    past a sequence's end and `spare_pages` unused pages hold random values, and the block-table entries past a
    sequence's pages hold an out-of-range page id: none of them may be read.  Layout only: no value is computed."""
    Bt, Hkv, N, d = K.shape
    dsel = Ks.shape[-1]
    dev = K.device
    need = [(int(n) + page_size - 1) // page_size for n in lens]
    max_pages = max(1, (N + page_size - 1) // page_size)
    num_pages = sum(need) + spare_pages
    g = torch.Generator().manual_seed(seed * 7919 + page_size)
    order = torch.randperm(num_pages, generator=g).tolist()
    gd = torch.Generator(device=dev).manual_seed(seed * 104729 + page_size)

    def noise(*shape):
        return torch.randn(shape, generator=gd, device=dev).to(torch.bfloat16)

    K_pool, V_pool = noise(num_pages, Hkv, page_size, d), noise(num_pages, Hkv, page_size, d)
    Ks_pool = noise(num_pages, Hkv, page_size, dsel)
    table = torch.full((Bt, max_pages), 2**31 - 1, dtype=torch.int32)
    i = 0
    for b in range(Bt):
        for pi in range(need[b]):
            pg = order[i]
            i += 1
            t0, t1 = pi * page_size, min(int(lens[b]), (pi + 1) * page_size)
            K_pool[pg, :, :t1 - t0] = K[b, :, t0:t1]
            V_pool[pg, :, :t1 - t0] = V[b, :, t0:t1]
            Ks_pool[pg, :, :t1 - t0] = Ks[b, :, t0:t1]
            table[b, pi] = pg
    return dict(K_pool=K_pool, V_pool=V_pool, Ks_pool=Ks_pool, block_table=table.to(dev),
                seq_lens=torch.tensor([int(n) for n in lens], dtype=torch.int32, device=dev), page_size=page_size)
