"""bench.py on the host, no GPU: the reference arm's JSON line, the rank
aggregation of replicas over a 2-process gloo group, rank-0-only output under
torchrun, the clock-sample window, and the traffic record's source check."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["unit"] == "GB/s" and d["value"] > 0
    assert d["config"]["workload"] == "w4a16_decode"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def _ranks_worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(1.5 + rank, "cpu", world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    """Each replica times its own steps; the line reports the slowest rank."""
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ranks_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {0: 2.5, 1: 2.5}
    assert bench.max_over_ranks(3.0, "cpu", 1) == 3.0


def test_reference_arm_step_size_is_bounded():
    """At any K the reference arm's steps fit its time budget: whole GEMVs
    while they fit, else a block of output columns (a multiple of 32)."""
    import bench
    assert bench.ref_columns(20, 2.6e-3) == bench.DEC_N
    for steps in (50000, 200000, 10 ** 7):
        cols = bench.ref_columns(steps, 2.6e-3)
        assert cols % 32 == 0 and 32 <= cols < bench.DEC_N
        assert steps * 2.6e-3 * cols / bench.DEC_N <= bench.REF_BUDGET_S or cols == 32


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                          "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
                          "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300, check=True).stdout
    assert len([ln for ln in out.splitlines() if ln.startswith("{")]) == 1


def test_clock_sampler_window_and_reasons():
    c = bench.ClockSampler(0)
    c.lines = [(1.0, "1000, 2070, 500, 0x0, Not Active, Not Active, Not Active, Not Active"),
               (2.0, "2070, 2070, 900, 0x4, Not Active, Not Active, Not Active, Active"),
               (3.0, "2060, 2070, 880, 0x0, Not Active, Not Active, Not Active, Not Active"),
               (9.0, "300, 2070, 90, 0x0, Not Active, Active, Not Active, Not Active")]
    s = c.summary(1.5, 3.5)
    assert s["samples"] == 2 and s["sm_mhz"] == 2065.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler(0).summary()["samples"] == 0


def test_traffic_reported_only_for_the_captured_source(monkeypatch):
    monkeypatch.setitem(bench.TRAFFIC, "probe", (123, "0000000000000000", "w4a16.cu"))
    assert bench._traffic("probe") is None
    sha = bench._sha(os.path.join(ROOT, "int4_weight_quantized_w4_gb300", "csrc", "w4a16.cu"))
    monkeypatch.setitem(bench.TRAFFIC, "probe", (123, sha, "w4a16.cu"))
    assert bench._traffic("probe") == 123
    assert bench._traffic("no such kernel") is None


def test_line_order_and_summary():
    """The per-row detail leads the line and a compact summary of every row's
    headline figure ends it, so a reader that keeps only the end of the line
    still sees the W4A8, MoE and sweep numbers."""
    line = {"metric": "m", "value": 1.0, "roofline": {"achieved": 3000.0, "frac": 0.44},
            "rows": {"w4a8_prefill": {"value": 700.0, "gemm_tops": 720.0, "quant_gbs": 4000.0,
                                      "roofline": {"frac": 0.38}},
                     "w4a8_prefill_sweep": {"points": {"M512_N4096": {"frac": 0.2}}},
                     "w4afp8_moe": {"value": 400.0, "gemm_tflops": 450.0, "roofline": {"frac": 0.12}},
                     "w4a16_sweep": {"points": {"M8_sym_fp16": {"frac": 0.36}}},
                     "lm_head_gemv": {"value": 3700.0, "roofline": {"frac": 0.55}}},
            "cpu_baseline": {"value": 0.2}}
    out = bench.ordered_line(line)
    keys = list(out)
    assert keys[0] == "rows" and keys[-1] == "summary" and keys.index("metric") < keys.index("cpu_baseline")
    sm = out["summary"]
    assert sm["w4a16_M1"] == {"gbs": 3000.0, "frac": 0.44}
    assert sm["w4a8_prefill"]["frac"] == 0.38 and sm["w4a8_sweep_frac"] == {"M512_N4096": 0.2}
    assert sm["w4afp8_moe"]["frac_fp8"] == 0.12 and sm["w4a16_sweep_frac"]["M8_sym_fp16"] == 0.36
    assert sm["lm_head_gemv"]["frac"] == 0.55
    assert len(json.dumps(sm)) < 1500
