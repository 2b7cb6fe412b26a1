"""bench.py's reference arm (the CPU oracle, the one arm that runs without a
GPU) prints the JSON line the benchmark contract asks for; the roofline
traffic figure is reported only for the kernel sources it was measured on."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1",
                        "--workload", "tiny"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["higher_is_better"] is False and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["config"]["workload"] == "tiny"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_traffic_is_reported_only_for_the_measured_sources(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"w": {"source_sha": bench.source_sha(), "dram_bytes_per_launch": 123.0},
                             "v": {"source_sha": "0" * 16, "dram_bytes_per_launch": 456.0}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.traffic_for("w") == 123.0
    assert bench.traffic_for("v") is None
    assert bench.traffic_for("missing") is None


def test_source_hash_ignores_comments_but_not_code():
    a = 'int f(int x) { return x + 1; } // one\n/* block\n comment */ const char* s = "a // b";\n'
    b = 'int f(int x)   {\n  return x + 1;   /* other */ }\nconst char* s = "a // b";'
    c = 'int f(int x) { return x + 2; }\nconst char* s = "a // b";'
    d = 'int f(int x) { return x + 1; }\nconst char* s = "a // c";'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only(a) != bench._code_only(d)


def _rank(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        q.put((rank, (bench.max_over_ranks([10.0 + rank, 5.0 - rank, 7.5], "cpu"),
                      bench.replica_figures(40.0 + 10.0 * rank, 50.0 - 2.0 * rank, world, "cpu"))))
    finally:
        dist.destroy_process_group()


def test_times_are_the_maximum_over_ranks():
    """The multi-rank bench reports the slowest rank's times as the step time and world / that time as
    the aggregate throughput (gloo on CPU, world size 2)."""
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        times, rep = got[r]
        assert times == [11.0, 5.0, 7.5]
        # the replicas' step time is the slowest rank's, never divided by the replica count; the aggregate
        # throughput counts every replica's steps
        assert rep == {"step_us": 50.0, "e2e_us": 50.0, "aggregate_steps_per_s": 2 * 1e6 / 50.0,
                       "aggregate_e2e_steps_per_s": 2 * 1e6 / 50.0}
    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]   # no process group: unchanged


def test_oracle_result_does_not_depend_on_its_thread_count():
    """The single-thread timing runs the same computation: one host thread gives the all-threads result bit for
    bit (units are independent; no sum crosses units)."""
    import numpy as np
    import oracle
    import workloads
    cfg = workloads.make_config("ministral8b_32k", batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=2048, top_k=30,
                                budget=30.0)
    w = workloads.generate(cfg, 3, "cpu")
    h = bench.oracle_host_inputs(w, cfg)
    args = (h["q"], h["K"], h["V"], h["Ks"], h["sel"], cfg.top_k, cfg.budget, 3, cfg.scale)
    many = oracle.decode(*args)
    n = oracle.num_threads()
    oracle.set_threads(1)
    try:
        assert oracle.num_threads() == 1
        one = oracle.decode(*args)
    finally:
        oracle.set_threads(n)
    assert oracle.num_threads() == n
    for k in ("out", "lse", "s_hat", "count", "idx", "p"):
        assert np.array_equal(many[k], one[k]), k


def test_oracle_sample_record():
    import workloads
    cfg = workloads.make_config("ministral8b_32k", batch=3, n_q_heads=8, n_kv_heads=2, ctx_len=1024, top_k=20,
                                budget=20.0)
    w = workloads.generate(cfg, 0, "cpu")
    rec = bench.oracle_sample(w, cfg, 4)
    # four threads' worth of units: two batch rows of two heads, scaled by 6 / 4
    assert "over 4 units (2 batch rows" in rec["sample"] and "6 units" in rec["sample"]
    assert rec["us_per_step"] > 0 and rec["single_thread_us_per_step"] > 0
    assert rec["threads"] == bench.cpu_threads()


def test_read_ceiling_record():
    """The score pass is placed against the faster of the two read-only probes of its own byte count; a size the
    probe did not measure, or no probe at all, gives no record."""
    ceil = {134217728: (30.0, 32.0)}
    rec = bench.ceiling_record(ceil, 134217728.0, 40.0)
    assert rec["plain_loads_us"] == 30.0 and rec["bulk_ring_us"] == 32.0
    assert rec["kernel_frac"] == 0.75
    assert abs(rec["gbs"] - 134217728 / 30e-6 / 1e9) < 0.1
    assert bench.ceiling_record(ceil, 1024.0, 40.0) is None
    assert bench.ceiling_record(None, 134217728.0, 40.0) is None


def test_read_ceiling_without_a_gpu_reports_nothing():
    import pytest
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the probe runs")
    # the probe either is not built or finds no device: either way no figure, and no exception
    assert bench.read_ceiling([32768]) is None


def test_read_ceiling_probe_rejects_sizes_that_are_not_whole_chunks():
    """The probe checks its arguments before it touches a device."""
    from long_context_decode_subset_b300 import build
    exe = build.build_ceiling()
    for arg in ("1000", "0", "x"):
        r = subprocess.run([exe, arg], capture_output=True, text=True, timeout=60)
        assert r.returncode == 2 and "multiple" in r.stderr, (arg, r.returncode, r.stderr)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 2 and "usage" in r.stderr
