#!/usr/bin/env python
"""Benchmark: microseconds per Stratified Sparse Attention decode step.

Default workload: the Ministral-8B-shaped layer at 128K context (batch 2,
32 query / 8 KV heads, d = 128, d_sel = 32, 50x sparsity: top-k 1311,
budget 1310), seeded synthetic inputs resident in HBM.  A step is one
ssa_decode call (three kernels: initialise, score, and the unit kernel that
selects, samples, attends and merges);
the seed changes every step.  L2 is flushed (a 256 MiB write) before every
timed step and each step is timed alone with CUDA events on its stream.

Prints one JSON line (rank 0): value (us per step), graph (the median of
graph-replayed steps, one step per CUDA graph), roofline (the score
pass alone against the measured copy bandwidth, with the DRAM traffic
recorded for these kernel sources and the read ceiling of the same bytes
timed the same way), e2e (through ssa_decode_host, host
memory in and out), append_step (ssa_decode_append, the serving form),
secondary (the 1M-context workload), configs (the 32K workload and the 27B
sweep points: us per step, graph-replayed median, achieved GB/s and roofline
fraction each, and the oracle on a bounded sample of units, on every host
thread and on one), host_tier (the 32K step with K/V in pinned host memory),
cpu_baseline (the oracle on the host cores, with a single-thread figure) and
cpu_dense (dense attention on the same cores), and error_vs_dense (relative
L2 error per head against dense attention, over the workload's seeds).  --impl reference
times the CPU oracle instead (the reference arm for this method has no
runnable upstream code).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per sparse decode step at 128K/1M ctx; achieved HBM GB/s vs B300 peak"
UNIT = "us/step"
FLUSH_BYTES = 256 << 20
CSRC = os.path.join(ROOT, "long_context_decode_subset_b300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ministral8b_128k")
    ap.add_argument("--secondary", default="ministral8b_1m", help="second workload reported beside ('' = none)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-error-stats", dest="error_stats", action="store_false",
                    help="skip the error-against-dense record of the main workload")
    ap.add_argument("--sweep", default="ministral8b_32k,27b_128k_10x,27b_128k_20x,27b_128k_50x,27b_128k_100x,"
                    "27b_128k_dense", help="further workloads timed for the per-config records ('' = none)")
    ap.add_argument("--host-tier", default="ministral8b_32k",
                    help="workload timed with K/V in pinned host memory ('' = none)")
    ap.add_argument("--paged", type=int, default=256,
                    help="page size of the paged-cache records of the main workload (0 = none)")
    ap.add_argument("--early-stop", default="1e-3,1e-2",
                    help="tau values of the early-stopping step records of the main workload ('' = none)")
    ap.add_argument("--plain-early-stop", type=float, default=None,
                    help="with --plain-steps: run ssa_decode_early_stop with this tau instead of ssa_decode")
    ap.add_argument("--plain-steps", type=int, default=0,
                    help="only run this many decode steps of --workload, then as many ssa_score launches (L2 "
                         "flushed before each), and exit: the program the ncu summaries under profiles/ capture")
    return ap.parse_args()


def _code_only(src: str) -> str:
    """C/CUDA source with its comments removed and whitespace runs collapsed (string and character
    literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_sha() -> str:
    """Hash of the kernel sources, comments and layout excluded: any change that can alter the compiled
    kernels changes it, a comment does not.  Keys the DRAM traffic recorded in profiles/traffic.json."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


class ClockSampler:
    """Samples SM clock and clock-event reasons while running: NVML through
    pynvml when it initialises, else an `nvidia-smi -lms` subprocess."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clocks"}

    def __init__(self, index: int, period: float = 0.01):
        self.index = index
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.source = None
        self._stop = threading.Event()
        self._period = period
        self._handle = None
        self._proc = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nvml = pynvml
            self._handle = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._handle, pynvml.NVML_CLOCK_SM)
            self.source = "nvml"
        except Exception:
            self._handle = None
        self._thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self._nvml.nvmlDeviceGetClockInfo(self._handle, self._nvml.NVML_CLOCK_SM))
                try:
                    r = self._nvml.nvmlDeviceGetCurrentClocksEventReasons(self._handle)
                except AttributeError:
                    r = self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons(self._handle)
                self.reasons |= int(r) & ~0x1
            except Exception:
                pass
            time.sleep(self._period)

    def __enter__(self):
        if self._handle is not None:
            self._thread.start()
        else:
            import subprocess
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                time.sleep(0.3)
            except Exception:
                self._proc = None
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._handle is not None:
            self._thread.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            for line in out.splitlines():
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 3:
                    continue
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                    self.reasons |= int(parts[2], 16) & ~0x1
                except ValueError:
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if self.reasons & b], "samples": len(self.samples),
                "source": self.source}


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over the ranks (the slowest rank's time is the job's time);
    the values themselves when there is one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_figures(step_us: float, e2e_us: float, world: int, device):
    """The job's figures for `world` replicas each timing its own steps: the step time is the slowest
    rank's (a replica's step takes that long; it is not divided by the replica count), and the aggregate
    throughput is `world` steps per that time."""
    step_us, e2e_us = max_over_ranks([step_us, e2e_us], device)
    return {"step_us": step_us, "e2e_us": e2e_us, "aggregate_steps_per_s": world * 1e6 / step_us,
            "aggregate_e2e_steps_per_s": world * 1e6 / e2e_us}


def algorithmic_bytes(cfg, rows_selected: float) -> float:
    """Key summary + selected K and V rows + q in + out/lse out (bytes per step)."""
    summary = cfg.batch * cfg.n_kv_heads * cfg.ctx_len * cfg.d_sel * 2
    rows = rows_selected * cfg.head_dim * 2 * 2
    io = cfg.batch * cfg.n_q_heads * (cfg.head_dim * 2 + cfg.head_dim * 4 + 4)
    return float(summary + rows + io)


def traffic_for(workload: str):
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_sha") == source_sha():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def read_ceiling(byte_counts):
    """The read-only ceiling for each byte count: the same bytes read once by plain loads and by a bulk-copy
    ring (read_ceiling.cu), each launch timed alone with CUDA events after an L2 flush, as the score pass is.
    {bytes: (plain_us, ring_us)}, or None if the probe is missing or fails."""
    import subprocess
    try:
        from long_context_decode_subset_b300 import build
        exe = build.build_ceiling()   # built with the library; compiled here if it is missing
    except Exception:
        return None
    try:
        res = subprocess.run([exe, *[str(int(b)) for b in byte_counts]], capture_output=True, text=True,
                             timeout=120)
        if res.returncode != 0:
            return None
        out = {}
        for ln in res.stdout.splitlines():
            d = json.loads(ln)
            out[int(d["bytes"])] = (float(d["plain_loads_us"]), float(d["bulk_ring_us"]))
        return out
    except Exception:
        return None


def ceiling_record(ceil, nbytes: float, kernel_us: float):
    """The score pass placed against the read ceiling of its own bytes (ceil from read_ceiling)."""
    if not ceil or int(nbytes) not in ceil:
        return None
    plain, ring = ceil[int(nbytes)]
    best = min(plain, ring)
    return {"plain_loads_us": plain, "bulk_ring_us": ring,
            "gbs": round(nbytes / (best * 1e-6) / 1e9, 1), "kernel_frac": round(best / kernel_us, 4),
            "note": "the same bytes read once with nothing else to do (plain loads; a 6 x 32 KB bulk-copy ring), "
                    "each launch timed alone after an L2 flush: kernel_frac = ceiling time / score-pass time"}


def u16(t):
    import numpy as np
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_host_inputs(w, cfg):
    """Host copies of a workload for the oracle, its key summary packed by the oracle itself (nothing the
    oracle reads comes from the CUDA library)."""
    import oracle
    K = u16(w["K"])
    sel = w["sel_ch"].cpu().numpy()
    return dict(q=u16(w["q"]), K=K, V=u16(w["V"]), Ks=oracle.pack_summary(K, sel, cfg.d_sel), sel=sel)


def time_oracle(h, cfg, seconds: float, max_steps: int | None = None):
    """Time oracle.decode steps (all units, all host threads) for about `seconds`."""
    import oracle
    times = []
    t_end = time.perf_counter() + seconds
    step = 0
    while True:
        t0 = time.perf_counter()
        oracle.decode(h["q"], h["K"], h["V"], h["Ks"], h["sel"], cfg.top_k, cfg.budget, step, cfg.scale,
                      want_lists=False)
        times.append(time.perf_counter() - t0)
        step += 1
        if (max_steps is not None and step >= max_steps) or (max_steps is None and time.perf_counter() > t_end):
            break
    return times, oracle.num_threads()


def cpu_threads() -> int:
    """Host threads the oracle runs on (OpenMP's default: every core of this host)."""
    import oracle
    return oracle.num_threads()


def oracle_sample(w, cfg, cores: int):
    """The oracle on a bounded sample of workload `cfg`: calls over the first batch rows that hold at least
    `cores` units (every host thread busy), and calls over one unit on one thread, each scaled to the whole
    step by its unit count.  Returns the per-config "oracle" record."""
    import oracle

    Hkv, G = cfg.n_kv_heads, cfg.group
    nb = min(cfg.batch, -(-min(cfg.units, cores) // Hkv))

    def host(nbatch, nheads):
        K = u16(w["K"][:nbatch, :nheads])
        sel = w["sel_ch"][:nheads].cpu().numpy()
        return dict(q=u16(w["q"][:nbatch, :nheads * G]), K=K, V=u16(w["V"][:nbatch, :nheads]),
                    Ks=oracle.pack_summary(K, sel, cfg.d_sel), sel=sel)

    h = host(nb, Hkv)
    t_all, threads = time_oracle(h, cfg, 0.0, max_steps=3)
    del h
    h1 = host(1, 1)
    oracle.set_threads(1)
    try:
        t_one, _ = time_oracle(h1, cfg, 0.0, max_steps=3)
    finally:
        oracle.set_threads(threads)
    return {"us_per_step": round(statistics.median(t_all) * cfg.units / (nb * Hkv) * 1e6, 1), "threads": threads,
            "single_thread_us_per_step": round(statistics.median(t_one) * cfg.units * 1e6, 1),
            "sample": f"median of 3 calls over {nb * Hkv} units ({nb} batch rows, {threads} threads) and of 3 calls "
                      f"over one unit (1 thread), each scaled by the step's {cfg.units} units"}


def error_vs_dense(cfg, dev):
    """Relative L2 error per query head of the step's output against dense attention (the library's dense
    limit, B = +inf), mean / p50 / p99 over heads and the workload's seeds, for SSA and, at the same total
    budget k + B, for pure top-k and the top-k + uniform hybrid."""
    import numpy as np
    import torch

    import long_context_decode_subset_b300 as ssa
    import workloads

    k, B = cfg.top_k, cfg.budget
    errs = {"ssa": [], "topk_same_budget": [], "uniform_hybrid_same_budget": []}

    def rel(out, ref):
        num = torch.linalg.vector_norm(out - ref, dim=-1)
        return (num / torch.linalg.vector_norm(ref, dim=-1).clamp_min(1e-30)).flatten().cpu().numpy()

    for seed in cfg.seeds:
        w = workloads.generate(cfg, seed, dev)
        q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
        Ks = ssa.ssa_pack_summary(K, sel)
        dense, _ = ssa.ssa_decode(q, K, V, Ks, sel, k, math.inf, seed, cfg.scale)
        errs["ssa"].append(rel(ssa.ssa_decode(q, K, V, Ks, sel, k, B, seed, cfg.scale)[0], dense))
        errs["topk_same_budget"].append(rel(ssa.ssa_decode(q, K, V, Ks, sel, k + int(B), 0.0, seed, cfg.scale)[0],
                                            dense))
        errs["uniform_hybrid_same_budget"].append(
            rel(ssa.ssa_decode_strata(q, K, V, Ks, sel, ssa.STRATA_UNIFORM, k, 0.0, B, seed, cfg.scale)[0], dense))
        del w, q, K, V, Ks, dense
        torch.cuda.empty_cache()
    rec = {}
    for name, v in errs.items():
        x = np.concatenate(v)
        rec[name] = {"mean": round(float(np.mean(x)), 5), "p50": round(float(np.percentile(x, 50)), 5),
                     "p99": round(float(np.percentile(x, 99)), 5)}
    rec.update(workload=cfg.name, seeds=list(cfg.seeds), heads_per_seed=cfg.batch * cfg.n_q_heads,
               reference="dense attention over every token (the library's B = +inf limit, pinned to the oracle)")
    return rec


def graph_replay_us(decode, replays: int, flush, seeds: int = 4):
    """Median and mean us of `replays` replays of CUDA graphs that each hold one decode step (`seeds` graphs,
    seeds 0.. in turn), L2 flushed before every replay.  decode(seed) enqueues one step on the current stream."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # eager warm-up on a side stream, as capture wants
        for sd in range(seeds):
            decode(sd)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graphs = []
    for sd in range(seeds):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            decode(sd)
        graphs.append(g)
    stream = torch.cuda.current_stream()
    for i in range(2 * seeds):
        flush.fill_(i & 0xff)
        graphs[i % seeds].replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
    torch.cuda._sleep(20_000_000)
    for i in range(replays):
        flush.fill_(i & 0xff)
        ev[i][0].record(stream)
        graphs[i % seeds].replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) * 1e3 for a, b in ev]
    del graphs
    return statistics.median(times), statistics.fmean(times)


def measure_ours(cfg, steps: int, warmup: int, dev, with_e2e: bool = True):
    import torch

    import long_context_decode_subset_b300 as ssa
    import workloads

    w = workloads.generate(cfg, 0, dev)
    Ks = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    shape = ssa.shape_of(q, K, Ks)
    ws = ssa.workspace(shape, 0, dev)
    units = cfg.batch * cfg.n_kv_heads
    out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
    lse = torch.empty((cfg.batch, cfg.n_q_heads), dtype=torch.float32, device=dev)
    counts = torch.zeros((steps, units), dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i, count_buf=None):
        ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, out=out, lse=lse,
                       count=count_buf, ws=ws, stream=stream)

    for i in range(warmup):
        flush.fill_(i & 0xff)
        step(1_000_000 + i)
    torch.cuda.synchronize()
    st, flags = ssa.ssa_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x}")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(dev.index or 0) as clk:
        torch.cuda._sleep(50_000_000)  # give the host a head start so launches queue up
        for i in range(steps):
            flush.fill_(i & 0xff)
            ev[i][0].record(stream)
            step(i, counts[i])
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    times_us = [a.elapsed_time(b) * 1e3 for a, b in ev]
    st, flags = ssa.ssa_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x}")
    rows = counts.sum(dim=1).double().mean().item()
    res = dict(times_us=times_us, rows=rows, clocks=clk.summary(), w=w, Ks=Ks)
    res["graph_replays"] = max(100, min(steps, 1000))
    res["graph_us"] = graph_replay_us(
        lambda sd: ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, sd, cfg.scale, out=out, lse=lse, ws=ws),
        res["graph_replays"], flush)
    st, flags = ssa.ssa_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x}")

    # the dominant kernel alone: ssa_score launches the score kernel (TMA + tcgen05) after the
    # one-launch initialiser that zeroes its stage queue
    s_hat = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.ctx_len), dtype=torch.float32, device=dev)
    for i in range(warmup):
        flush.fill_(i & 0xff)
        ssa.ssa_score(q, Ks, sel, cfg.scale, s_hat=s_hat, ws=ws, stream=stream)
    torch.cuda.synchronize()
    n1 = min(steps, 500)
    ev1 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n1)]
    torch.cuda._sleep(50_000_000)
    for i in range(n1):
        flush.fill_(i & 0xff)
        ev1[i][0].record(stream)
        ssa.ssa_score(q, Ks, sel, cfg.scale, s_hat=s_hat, ws=ws, stream=stream)
        ev1[i][1].record(stream)
    torch.cuda.synchronize()
    res["score_us"] = [a.elapsed_time(b) * 1e3 for a, b in ev1]
    del s_hat

    if with_e2e:
        q_host = q.cpu().pin_memory()
        out_h = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(warmup):
            ssa.ssa_decode_host(q_host, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, out_h, lse_h, ws,
                                stream=stream)
        torch.cuda.synchronize()
        torch.cuda._sleep(50_000_000)
        for i in range(steps):
            flush.fill_(i & 0xff)
            ev2[i][0].record(stream)
            ssa.ssa_decode_host(q_host, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, out_h, lse_h, ws,
                                stream=stream)
            ev2[i][1].record(stream)
        torch.cuda.synchronize()
        res["e2e_us"] = [a.elapsed_time(b) * 1e3 for a, b in ev2]
        res["h2d"] = q_host.numel() * 2
        res["d2h"] = out_h.numel() * 4 + lse_h.numel() * 4

        # the serving form of the step: the new token's K/V rows and summary row appended by the chain's
        # first kernel (ssa_decode_append).  The appended row is the cache's last one, so the cache keeps
        # its values from step to step.
        N = cfg.ctx_len
        k_new = K[:, :, N - 1].contiguous()
        v_new = V[:, :, N - 1].contiguous()
        ev3 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(warmup):
            ssa.ssa_decode_append(q, k_new, v_new, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, out=out,
                                  lse=lse, ws=ws, stream=stream)
        torch.cuda.synchronize()
        torch.cuda._sleep(50_000_000)
        for i in range(steps):
            flush.fill_(i & 0xff)
            ev3[i][0].record(stream)
            ssa.ssa_decode_append(q, k_new, v_new, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, out=out,
                                  lse=lse, ws=ws, stream=stream)
            ev3[i][1].record(stream)
        torch.cuda.synchronize()
        st, flags = ssa.ssa_get_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {st} flags {flags:#x}")
        res["append_us"] = [a.elapsed_time(b) * 1e3 for a, b in ev3]
    del flush
    return res


def time_steps(cfg, steps: int, warmup: int, dev, host_kv: bool = False, cores: int = 0):
    """Mean us per ssa_decode step of workload `cfg` (L2 flushed before every step, seed = step index), the
    mean rows selected, the clocks, and extras: the median of graph-replayed steps and, with cores > 0, the
    oracle on a bounded sample.  With host_kv the K and V rows sit in pinned host memory."""
    import torch

    import long_context_decode_subset_b300 as ssa
    import workloads

    w = workloads.generate(cfg, 0, dev)
    Ks = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    if host_kv:
        K, V = K.cpu().pin_memory(), V.cpu().pin_memory()
        del w["K"], w["V"]
    shape = ssa.shape_of(q, K, Ks)
    ws = ssa.workspace(shape, 0, dev)
    out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
    lse = torch.empty((cfg.batch, cfg.n_q_heads), dtype=torch.float32, device=dev)
    counts = torch.zeros((steps, cfg.units), dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        flush.fill_(i & 0xff)
        ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 1_000_000 + i, cfg.scale, out=out, lse=lse, ws=ws,
                       stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(dev.index or 0) as clk:
        torch.cuda._sleep(20_000_000)
        for i in range(steps):
            flush.fill_(i & 0xff)
            ev[i][0].record(stream)
            ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, out=out, lse=lse, count=counts[i],
                           ws=ws, stream=stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    st, flags = ssa.ssa_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x}")
    us = statistics.fmean(a.elapsed_time(b) * 1e3 for a, b in ev)
    rows = counts.sum(dim=1).double().mean().item()
    extra = {}
    if not host_kv:
        med, mean = graph_replay_us(
            lambda sd: ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, sd, cfg.scale, out=out, lse=lse,
                                      ws=ws), 100, flush)
        extra["graph"] = {"median_us": round(med, 3), "mean_us": round(mean, 3), "replays": 100}
        st, flags = ssa.ssa_get_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {st} flags {flags:#x}")
    if cores > 0:
        del flush, ws
        torch.cuda.empty_cache()
        extra["oracle"] = oracle_sample(w, cfg, cores)
    return us, rows, clk.summary(), extra


def time_paged(cfg, steps: int, warmup: int, dev, page_size: int, lens):
    """Mean us per ssa_decode_paged step of workload `cfg` laid out in pages of `page_size` tokens with sequence
    lengths `lens` (L2 flushed before every step, seed = step index), and the mean rows selected."""
    import torch

    import long_context_decode_subset_b300 as ssa
    import workloads

    w = workloads.generate(cfg, 0, dev)
    Ks = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    pg = workloads.to_paged(w["K"], w["V"], Ks, lens, page_size, seed=1)
    q, sel = w["q"], w["sel_ch"]
    del w, Ks
    shape = ssa.paged_shape(q, pg["K_pool"], pg["Ks_pool"], cfg.ctx_len)
    ws = ssa.workspace(shape, 0, dev)
    out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
    lse = torch.empty((cfg.batch, cfg.n_q_heads), dtype=torch.float32, device=dev)
    counts = torch.zeros((steps, cfg.units), dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i, count=None):
        ssa.ssa_decode_paged(q, pg["K_pool"], pg["V_pool"], pg["Ks_pool"], pg["block_table"], pg["seq_lens"], sel,
                             cfg.top_k, cfg.budget, i, cfg.scale, cfg.ctx_len, out=out, lse=lse, count=count, ws=ws,
                             stream=stream)
    for i in range(warmup):
        flush.fill_(i & 0xff)
        step(1_000_000 + i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(dev.index or 0) as clk:
        torch.cuda._sleep(20_000_000)
        for i in range(steps):
            flush.fill_(i & 0xff)
            ev[i][0].record(stream)
            step(i, counts[i])
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    st, flags = ssa.ssa_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x}")
    us = statistics.fmean(a.elapsed_time(b) * 1e3 for a, b in ev)
    rows = counts.sum(dim=1).double().mean().item()
    return us, rows, clk.summary()


def time_early_stop(cfg, steps: int, warmup: int, dev, tau: float):
    """Mean us per ssa_decode_early_stop step of workload `cfg` (L2 flushed before every step, seed = step
    index), and the mean fraction of the selected rows' 128-row blocks the attention kept."""
    import torch

    import long_context_decode_subset_b300 as ssa
    import workloads

    w = workloads.generate(cfg, 0, dev)
    Ks = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    ws = ssa.workspace(ssa.shape_of(q, K, Ks), 0, dev)
    out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
    lse = torch.empty((cfg.batch, cfg.n_q_heads), dtype=torch.float32, device=dev)
    blocks = torch.zeros((steps, cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device=dev)
    all_blocks = torch.zeros((4, cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        flush.fill_(i & 0xff)
        ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 1_000_000 + i, cfg.scale, tau, out=out,
                                  lse=lse, ws=ws, stream=stream)
    for i in range(4):   # every block (tau = 0): the denominator of the kept fraction
        ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, 0.0, out=out, lse=lse,
                                  blocks=all_blocks[i], ws=ws, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(dev.index or 0) as clk:
        torch.cuda._sleep(20_000_000)
        for i in range(steps):
            flush.fill_(i & 0xff)
            ev[i][0].record(stream)
            ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, tau, out=out, lse=lse,
                                      blocks=blocks[i], ws=ws, stream=stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    st, flags = ssa.ssa_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x}")
    us = statistics.fmean(a.elapsed_time(b) * 1e3 for a, b in ev)
    frac = blocks[:4].double().sum().item() / max(1.0, all_blocks.double().sum().item())
    return us, frac, clk.summary()


def config_record(cfg, us, rows, peak, clocks):
    ab = algorithmic_bytes(cfg, rows)
    gbs = ab / (us * 1e-6) / 1e9
    return {"workload": cfg.name, "value": round(us, 3), "unit": UNIT, "rows_selected_per_step": round(rows, 1),
            "algorithmic_bytes_per_step": int(ab), "achieved_gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
            "frac_of_8000": round(gbs / 8000.0, 4), "clocks": clocks}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    cfg = workloads.CONFIGS[args.workload]

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    m = measure_ours(cfg, args.steps, args.warmup, dev)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t0

    rep = replica_figures(statistics.fmean(m["times_us"]), statistics.fmean(m["e2e_us"]), world, dev)
    mean_us, e2e_us = rep["step_us"], rep["e2e_us"]
    peak, peak_kind = measured_peaks()
    abytes = algorithmic_bytes(cfg, m["rows"])
    achieved = abytes / (mean_us * 1e-6) / 1e9
    score_us = statistics.fmean(m["score_us"])
    score_bytes = float(cfg.batch * cfg.n_kv_heads * cfg.ctx_len * cfg.d_sel * 2)
    score_gbs = score_bytes / (score_us * 1e-6) / 1e9
    line = {
        "metric": METRIC,
        "value": round(mean_us, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_us / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; shapes of a Ministral-8B layer, generator in workloads/)",
        "config": {
            "workload": cfg.name, "batch": cfg.batch, "n_q_heads": cfg.n_q_heads, "n_kv_heads": cfg.n_kv_heads,
            "head_dim": cfg.head_dim, "ctx_len": cfg.ctx_len, "d_sel": cfg.d_sel, "top_k": cfg.top_k,
            "budget": cfg.budget, "inputs": "bf16 q/K/V/summary, fp32 scores and accumulation",
            "l2": "flushed before every timed step (256 MiB write)", "seed": "step index",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "us_per_step_median": round(statistics.median(m["times_us"]), 3),
        "graph": {"median_us": round(m["graph_us"][0], 3), "mean_us": round(m["graph_us"][1], 3),
                  "replays": m["graph_replays"],
                  "note": "one ssa_decode step per CUDA graph (4 graphs, seeds 0..3 in turn), L2 flushed before "
                          "every replay"},
        "us_per_step_p10_p90": [round(sorted(m["times_us"])[len(m["times_us"]) // 10], 3),
                                round(sorted(m["times_us"])[(9 * len(m["times_us"])) // 10], 3)],
        "rows_selected_per_step": round(m["rows"], 1),
        "algorithmic_bytes_per_step": int(abytes),
        "roofline": {
            "bound": "hbm", "achieved": round(score_gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(score_gbs / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth (burst, kernel timed alone)",
            "frac_of_8000": round(score_gbs / 8000.0, 4),
            "traffic": traffic_for(cfg.name),
            "kernel": "ssa::score_kernel (TMA + tcgen05 scorer) with its initialiser, launched by ssa_score",
            "kernel_us": round(score_us, 3),
            "algorithmic_bytes_per_launch": int(score_bytes),
            "step": {"achieved": round(achieved, 1), "frac": round(achieved / peak, 4),
                     "frac_of_8000": round(achieved / 8000.0, 4),
                     "note": "whole decode step: summary + selected K/V rows + q/out over the step time"},
        },
        "aggregate_steps_per_s": round(rep["aggregate_steps_per_s"], 1),
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": m["h2d"],
                "aggregate_steps_per_s": round(rep["aggregate_e2e_steps_per_s"], 1),
                "d2h_bytes_per_step": m["d2h"],
                "api": "ssa_decode_host: the kernels read q from pinned host memory and write out/lse into it"},
        "append_step": {"value": round(statistics.fmean(m["append_us"]), 3), "unit": UNIT,
                        "api": "ssa_decode_append (the new token's K/V and summary rows written by the chain's "
                               "first kernel, then the step over all tokens)"},
        "gpu_launches": 3 * args.steps,   # per timed step: the initialiser, the score kernel, the unit kernel
        "clocks": m["clocks"],
        "wall_s": round(wall, 2),
    }
    if rank == 0:
        sizes = [score_bytes]
        if args.secondary:
            c2 = workloads.CONFIGS[args.secondary]
            sizes.append(float(c2.batch * c2.n_kv_heads * c2.ctx_len * c2.d_sel * 2))
        ceil = read_ceiling(sizes)
        line["roofline"]["read_ceiling"] = ceiling_record(ceil, score_bytes, score_us)
    if rank == 0 and args.secondary:
        cfg2 = workloads.CONFIGS[args.secondary]
        del m
        torch.cuda.empty_cache()
        steps2 = max(20, min(args.steps, 300))
        m2 = measure_ours(cfg2, steps2, max(3, min(args.warmup, 10)), dev, with_e2e=False)
        us2 = statistics.fmean(m2["times_us"])
        oracle2 = None
        if not args.no_cpu_baseline:
            m2["Ks"] = None
            torch.cuda.empty_cache()
            oracle2 = oracle_sample(m2["w"], cfg2, cpu_threads())
        ab2 = algorithmic_bytes(cfg2, m2["rows"])
        line["secondary"] = {
            "workload": cfg2.name, "value": round(us2, 3), "unit": UNIT, "steps": steps2,
            "algorithmic_bytes_per_step": int(ab2), "achieved_gbs": round(ab2 / (us2 * 1e-6) / 1e9, 1),
            "frac": round(ab2 / (us2 * 1e-6) / 1e9 / peak, 4),
            "frac_of_8000": round(ab2 / (us2 * 1e-6) / 1e9 / 8000.0, 4),
            "traffic": traffic_for(cfg2.name), "clocks": m2["clocks"],
            "score_pass": {"kernel_us": round(statistics.fmean(m2["score_us"]), 3),
                           "read_ceiling": ceiling_record(
                               ceil, float(cfg2.batch * cfg2.n_kv_heads * cfg2.ctx_len * cfg2.d_sel * 2),
                               statistics.fmean(m2["score_us"]))},
            "graph": {"median_us": round(m2["graph_us"][0], 3), "mean_us": round(m2["graph_us"][1], 3),
                      "replays": m2["graph_replays"]},
        }
        if oracle2 is not None:
            line["secondary"]["oracle"] = oracle2
        del m2
        torch.cuda.empty_cache()
        m = None
    if rank == 0 and args.error_stats:
        line["error_vs_dense"] = error_vs_dense(cfg, dev)
        torch.cuda.empty_cache()
    if rank == 0 and args.sweep:
        # the other workloads' steps (the per-config records of the measurement plan)
        line["configs"] = []
        for name in [x for x in args.sweep.split(",") if x]:
            cfgx = workloads.CONFIGS[name]
            steps_x = max(20, min(args.steps, 200))
            us, rows, clk, extra = time_steps(cfgx, steps_x, max(3, min(args.warmup, 10)), dev,
                                              cores=0 if args.no_cpu_baseline else cpu_threads())
            rec = config_record(cfgx, us, rows, peak, clk)
            rec["steps"] = steps_x
            rec.update(extra)
            line["configs"].append(rec)
            torch.cuda.empty_cache()
    if rank == 0 and args.host_tier:
        # the host-resident tier: K and V in pinned host memory, the summary in HBM; the selected rows cross
        # the host link
        cfgh = workloads.CONFIGS[args.host_tier]
        steps_h = max(20, min(args.steps, 100))
        us, rows, clk, _ = time_steps(cfgh, steps_h, 3, dev, host_kv=True)
        rec = config_record(cfgh, us, rows, peak, clk)
        rec.update(steps=steps_h, kv="pinned host memory (mapped), summary in HBM",
                   row_bytes_per_step=int(rows * cfgh.head_dim * 2 * 2),
                   host_link_gbs=round(rows * cfgh.head_dim * 4 / (us * 1e-6) / 1e9, 1))
        line["host_tier"] = rec
        torch.cuda.empty_cache()
    if rank == 0 and args.paged:
        # the same workload as a paged cache (pool pages in a random order): every sequence full (the contiguous
        # step's work), then ragged lengths; bytes are counted over the tokens the sequences hold
        line["paged"] = []
        steps_p = max(20, min(args.steps, 300))
        n = cfg.ctx_len
        for kind, lens in (("full", [n] * cfg.batch),
                           ("ragged", [max(1, (n * (i + 1)) // (cfg.batch + 1)) for i in range(cfg.batch)])):
            us, rows, clk = time_paged(cfg, steps_p, max(3, min(args.warmup, 10)), dev, args.paged, lens)
            summary = cfg.n_kv_heads * sum(lens) * cfg.d_sel * 2
            ab = summary + rows * cfg.head_dim * 4 + cfg.batch * cfg.n_q_heads * (cfg.head_dim * 6 + 4)
            gbs = ab / (us * 1e-6) / 1e9
            line["paged"].append({
                "workload": cfg.name, "lengths": kind, "seq_lens": lens, "page_size": args.paged,
                "value": round(us, 3), "unit": UNIT, "steps": steps_p, "rows_selected_per_step": round(rows, 1),
                "algorithmic_bytes_per_step": int(ab), "achieved_gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                "clocks": clk, "api": "ssa_decode_paged"})
            torch.cuda.empty_cache()
    if rank == 0 and args.early_stop:
        # the step with S2O-style early stopping of the attention (ssa_decode_early_stop)
        line["early_stop"] = []
        for tau in [float(x) for x in args.early_stop.split(",") if x]:
            steps_e = max(20, min(args.steps, 300))
            us, frac, clk = time_early_stop(cfg, steps_e, max(3, min(args.warmup, 10)), dev, tau)
            line["early_stop"].append({"workload": cfg.name, "tau": tau, "value": round(us, 3), "unit": UNIT,
                                       "steps": steps_e, "blocks_kept_frac": round(frac, 4), "clocks": clk,
                                       "api": "ssa_decode_early_stop"})
            torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle as it stands, on this host's cores, on a bounded sample of the same workload
        w = workloads.generate(cfg, 0, dev)
        h = oracle_host_inputs(w, cfg)
        one = oracle_sample(w, cfg, cpu_threads())
        del w
        times, cores = time_oracle(h, cfg, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": round(statistics.fmean(times) * 1e6, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} full decode steps of {cfg.name} (all {cfg.units} units), seeds 0..{len(times) - 1}",
            "single_thread": {"value": one["single_thread_us_per_step"], "unit": UNIT, "cores": 1,
                              "sample": "median of 3 calls over one unit on one thread, scaled by the step's "
                                        f"{cfg.units} units"},
        }
        # and dense attention over every cached token on the same cores, for context
        import oracle
        dense = []
        t_end = time.perf_counter() + min(5.0, args.cpu_seconds)
        while not dense or (time.perf_counter() < t_end and len(dense) < 20):
            t1 = time.perf_counter()
            oracle.dense_attention(h["q"], h["K"], h["V"], cfg.scale)
            dense.append(time.perf_counter() - t1)
        line["cpu_dense"] = {
            "value": round(statistics.fmean(dense) * 1e6, 1), "unit": UNIT, "cores": cores,
            "kind": "oracle dense attention (every token, double accumulation)",
            "sample": f"{len(dense)} full steps of {cfg.name}",
        }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_plain(args):
    """args.plain_steps decode steps of the workload, nothing timed (for ncu)."""
    import torch

    import long_context_decode_subset_b300 as ssa
    import workloads

    cfg = workloads.CONFIGS[args.workload]
    dev = torch.device("cuda", 0)
    w = workloads.generate(cfg, 0, dev)
    Ks = ssa.ssa_pack_summary(w["K"], w["sel_ch"])
    q, K, V, sel = w["q"], w["K"], w["V"], w["sel_ch"]
    ws = ssa.workspace(ssa.shape_of(q, K, Ks), 0, dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for i in range(args.plain_steps):
        flush.fill_(i & 0xff)
        if args.plain_early_stop is not None:
            ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, args.plain_early_stop,
                                      ws=ws)
        else:
            ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, i, cfg.scale, ws=ws)
    # then as many launches of the roofline kernel as the bench times it (ssa_score alone)
    s_hat = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.ctx_len), dtype=torch.float32, device=dev)
    for i in range(args.plain_steps):
        flush.fill_(i & 0xff)
        ssa.ssa_score(q, Ks, sel, cfg.scale, s_hat=s_hat, ws=ws)
    st, flags = ssa.ssa_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x}")
    print(json.dumps({"plain_steps": args.plain_steps, "workload": cfg.name}), flush=True)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    import workloads

    cfg = workloads.CONFIGS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = workloads.generate(cfg, 0, dev)
    import oracle
    oracle.build()
    h = oracle_host_inputs(w, cfg)
    del w
    # one untimed step to estimate the cost, then K timed steps within a few minutes:
    # if K full steps would take too long, each step runs the oracle on a subset of
    # units and is scaled to the full step.
    t_est, cores = time_oracle(h, cfg, 0.0, max_steps=1)
    budget_s = 150.0
    n_units = cfg.units
    units_per_step = n_units
    if t_est[0] * (args.steps + args.warmup) > budget_s:
        units_per_step = max(1, int(n_units * budget_s / (t_est[0] * (args.steps + args.warmup))))
    G = cfg.group
    sub = []
    for u in range(units_per_step):
        b, hh = divmod(u, cfg.n_kv_heads)
        sub.append(dict(q=h["q"][b:b + 1, hh * G:(hh + 1) * G], K=h["K"][b:b + 1, hh:hh + 1],
                        V=h["V"][b:b + 1, hh:hh + 1], Ks=h["Ks"][b:b + 1, hh:hh + 1], sel=h["sel"][hh:hh + 1]))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        if units_per_step == n_units:
            oracle.decode(h["q"], h["K"], h["V"], h["Ks"], h["sel"], cfg.top_k, cfg.budget, i, cfg.scale,
                          want_lists=False)
        else:
            for s in sub:
                oracle.decode(s["q"], s["K"], s["V"], s["Ks"], s["sel"], cfg.top_k, cfg.budget, i, cfg.scale,
                              want_lists=False)
        dt = (time.perf_counter() - t0) * n_units / units_per_step
        if i >= args.warmup:
            times.append(dt)
    us = statistics.fmean(times) * 1e6
    sample = (f"full steps (all {n_units} units)" if units_per_step == n_units else
              f"{units_per_step} of {n_units} units per step, scaled to the full step (one unit per thread at most)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "batch": cfg.batch, "n_q_heads": cfg.n_q_heads,
                   "n_kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim, "ctx_len": cfg.ctx_len,
                   "d_sel": cfg.d_sel, "top_k": cfg.top_k, "budget": cfg.budget},
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "no runnable upstream implementation exists; the reference arm is the CPU oracle (C, OpenMP)",
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.plain_steps > 0:
        run_plain(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
