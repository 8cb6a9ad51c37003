#!/usr/bin/env python3
"""Benchmark of the int4-weight linear layer on one node.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.

Headline workload: W4A16 decode, M=1 token, K=4096, N=14336, group 128, fp16
scales (symmetric). A step is one layer call at that token count: below 512
tokens the layer runs the W4A16 path, so one call of ``w4a16_gemm`` is the
whole hot path of a decode step. ``value`` is the weight bytes streamed per
second (GB/s) with inputs resident in HBM; 16 distinct weight copies (485 MB,
more than the 129 MB L2) rotate between calls, so every call reads HBM.
Calls are replayed from a CUDA graph so launch latency on the host does not
gate the GPU.

The other rows of the hot path are measured in the same run and reported
under ``rows``: per-token quantization + W4A8 GEMM on the prefill and
diffusion shapes, and the W4AFP8 grouped expert GEMMs.

Multi-GPU: the layer is replicated; each rank runs the same workload on its
own GPU with no collective in the data path (weak scaling). The timed region
is bracketed by a barrier and a synchronize, and rank 0 reports the maximum
time over ranks.

``--impl reference`` times the CPU oracle (numpy, float64) on the same
workload and metric, each step a bounded column sample of the decode GEMV.
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

L2_BYTES = 129 * 2 ** 20          # GB300 L2

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as S  # noqa: E402

METRIC = "W4A8 GEMM TOPS (% int8/fp8 peak); W4A16 M=1 weight GB/s (% HBM)"
DEC_M, DEC_K, DEC_N, DEC_G = 1, 4096, 14336, 128
N_COPIES = 16
GRAPH_CALLS = 200
FP8_PER_BF16 = 2.0            # dense fp8 : bf16 tensor rate (4.5 vs 2.25 PFLOP/s nominal)
MOE_KERNEL = "the two grouped GEMM calls (w4a8_tc_kernel in expert mode; gate_up with its fused gather-quant)"
BLOCK_CYCLES = 400_000        # ~0.2 ms at 2 GHz: longer than submitting the timed graph

# DRAM bytes (read + write) per launch from ncu, keyed by the SHA-256 of the
# kernel's source file at capture time; reported only while the source matches.
TRAFFIC = {
    # w4a16_kernel, M=1 K=4096 N=14336 g128, caches flushed: dram__bytes_read.sum + dram__bytes_write.sum
    # (30,329,856 + 0)
    "w4a16": (30329856, "746bc24064d2dbca", "w4a16.cu"),
    # w4a8_tc_kernel<2, fp16, last-wave split>, W4A8 diffusion M=16384 K=N=3072 g=-1 (105,709,824 + 68,560,640)
    "w4a8_diffusion": (174270464, "10e03aa25d9f1866", "w4a8.cu"),
    # lm_head_tc1_kernel, M=1 V=131072 D=2048 g128 (151,322,880 + 2,742,784)
    "lm_head": (154065664, "718ef95e1608b20c", "embed.cu"),
    # quantize_chunks_kernel<bf16, 16, 4>, N=14336 K=4096 g128 (117,464,064 + 14,775,040; the codes,
    # scales and zeros are partly still in L2 when the kernel ends)
    "quantize": (132239104, "13988ce8d7acefec", "tools.cu"),
    # w4a8_tc_kernel<2, e4m3> in expert mode, the MoE layer's two GEMMs: gate_up (257,933,568 + 150,066,432)
    # and down (141,715,200 + 90,804,736)
    "w4afp8_moe": (640519936, "10e03aa25d9f1866", "w4a8.cu"),
}


def _traffic(key):
    """ncu DRAM bytes per launch for `key` while its source is unchanged since the capture, else None."""
    rec = TRAFFIC.get(key)
    if not rec:
        return None
    src = os.path.join(ROOT, "int4_weight_quantized_w4_gb300", "csrc", rec[2])
    return rec[0] if rec[1] == _sha(src) else None


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def decode_bytes(M=DEC_M, K=DEC_K, N=DEC_N, G=DEC_G, zeros=False):
    """Algorithmic bytes of one W4A16 call: packed weights, scales (+zeros), x in, y out."""
    b = K * N // 2 + (K // G) * N * 2 + M * K * 2 + M * N * 2
    if zeros:
        b += (K // G) * N * 2
    return b


def max_over_ranks(value, device, world):
    """The largest of the ranks' values (every rank gets it), after a barrier;
    the value itself with one rank. Replicas: no data moves between ranks
    except this one number."""
    if world <= 1:
        return value
    import torch
    torch.distributed.barrier()
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []        # (host monotonic time the sample arrived, csv line)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def wait_first(self, timeout=5.0):
        """Block until nvidia-smi delivers its first sample (it takes a moment to start)."""
        t0 = time.monotonic()
        while self.proc is not None and not self.lines and time.monotonic() - t0 < timeout:
            time.sleep(0.01)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Samples that arrived within [t0, t1] (host monotonic), all if not given."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import int4_weight_quantized_w4_gb300 as w4

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w4.load()
    stream = torch.cuda.Stream(dev)
    hbm, bf16_tf, bf16_tf_sus, peak_kind = measured_peaks()

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    # --- inputs resident in HBM ---
    xb = S.activations_bf16(DEC_M, DEC_K, seed=0)
    x = bf16(xb)
    qws = [torch.from_numpy(S.random_words((DEC_K // 8, DEC_N), seed=1, tag=20 + i)).to(dev) for i in range(N_COPIES)]
    sws = [torch.from_numpy(S.scales_f16((DEC_K // DEC_G, DEC_N), seed=2, tag=30 + i)).to(dev) for i in range(N_COPIES)]
    y = torch.empty((DEC_M, DEC_N), dtype=torch.bfloat16, device=dev)

    def call(i, xin=x, yout=y):
        w4.w4a16_gemm(xin, qws[i % N_COPIES], sws[i % N_COPIES], DEC_G, y=yout, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3) * N_COPIES):
            call(i)
    torch.cuda.synchronize()

    # exactly K calls: a graph of up to GRAPH_CALLS calls (rotating weight
    # copies) replayed K // calls times, and a graph of the remainder
    steps = max(1, args.steps)
    calls = min(GRAPH_CALLS, steps)
    replays, rem = steps // calls, steps % calls
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(calls):
            call(i)
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                call(calls + i)
    with torch.cuda.stream(stream):          # replay() launches on the current stream
        for _ in range(max(args.warmup, 3)):
            g.replay()
            if g_rem is not None:
                g_rem.replay()
    torch.cuda.synchronize()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk, torch.cuda.stream(stream):
        clk.wait_first()
        t_begin = time.monotonic()
        # a blocking kernel ahead of the start event keeps the stream busy while
        # the host submits the event and the graph, so the events time the
        # steps on the GPU and not the host's launch latency
        torch.cuda._sleep(BLOCK_CYCLES)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t_end = time.monotonic()
        # nvidia-smi samples every 100 ms: when the timed region is shorter
        # than that, the same graph keeps running (untimed, one replay in
        # flight at a time) until 0.6 s have passed, so the samples see the
        # GPU under this load
        window = "timed region"
        if t_end - t_begin < 0.6:
            window = "timed region + untimed replays of the same graph up to 0.6 s"
            while time.monotonic() - t_begin < 0.6:
                g.replay()
                torch.cuda.synchronize()
            t_end = time.monotonic()
    ms = e0.elapsed_time(e1)
    clocks = clk.summary(t_begin, t_end)
    clocks["window"] = window
    ms = max_over_ranks(ms, dev, world)
    ms_per_step = ms / steps
    nbytes = decode_bytes()
    value = world * steps * nbytes / (ms * 1e-3) / 1e9
    gbs_per_launch = nbytes / (ms_per_step * 1e-3) / 1e9

    # --- end to end through the C ABI with host buffers: every step copies x
    # in from page-locked host memory, runs the GEMM and copies y back out
    # (w4a16_gemm_host queues all three on the stream) ---
    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.empty((DEC_M, DEC_N), dtype=torch.bfloat16).pin_memory()
    lib = w4.load()
    host_fn = lib.w4a16_gemm_host
    sp = stream.cuda_stream
    argsets = [(x_host.data_ptr(), x.data_ptr(), qws[c].data_ptr(), sws[c].data_ptr(), w4.W4_FP16, None, DEC_G,
                None, y.data_ptr(), y_host.data_ptr(), DEC_M, DEC_N, DEC_K, sp) for c in range(N_COPIES)]
    e2e_steps = min(steps, 20000)
    bad = 0
    for i in range(3 * N_COPIES):
        bad |= host_fn(*argsets[i % N_COPIES])
    stream.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        bad |= host_fn(*argsets[i % N_COPIES])
    stream.synchronize()
    e2e_s = time.perf_counter() - t0
    if bad:
        raise RuntimeError("w4a16_gemm_host failed: " + lib.w4_last_error().decode())
    e2e_value = world * e2e_steps * nbytes / e2e_s / 1e9

    traffic = _traffic("w4a16")

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 x int4 -> fp32 acc",
        "data": "synthetic (seeded SplitMix64: x~N(0,1) bf16, uniform int4 codes, fp16 scales U[0.005,0.02])",
        "config": {"workload": "w4a16_decode", "M": DEC_M, "K": DEC_K, "N": DEC_N, "group": DEC_G,
                   "scales": "fp16", "zeros": False, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {N_COPIES} rotating weight copies "
                         f"({N_COPIES * nbytes / 1e6:.0f} MB)",
                   "timing": f"CUDA graph of {calls} calls replayed {replays}x"
                             + (f" + a graph of {rem}" if rem else "")
                             + ", CUDA events on the launching stream behind a blocking kernel"},
        "roofline": {"bound": "hbm", "achieved": round(gbs_per_launch, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs_per_launch / hbm, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs", "kernel": "w4a16_kernel",
                     "algorithmic_bytes_per_launch": nbytes},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": DEC_M * DEC_K * 2,
                "d2h_bytes_per_step": DEC_M * DEC_N * 2, "steps": e2e_steps,
                "how": "per step one w4a16_gemm_host call (C ABI, host buffers): page-locked x in, the GEMM, y out "
                       "into page-locked memory (x copied by the call's L2-prefetch grid, y written by the GEMV); "
                       "host wall clock over all steps and the final sync"},
        "gpu_launches": 2 * steps,   # per call: the L2 prefetch grid and the GEMV grid
        "clocks": clocks,
        "sm_count": torch.cuda.get_device_properties(dev).multi_processor_count,
    }
    if not args.no_rows:
        only = set(args.rows.split(",")) if args.rows else None
        line["rows"] = bench_rows(dev, stream, bf16_tf, peak_kind, hbm, only)
    return line


# ---------------------------------------------------------------------------
# the other rows of the hot path (same run, own timing)
# ---------------------------------------------------------------------------

def _time_graph(torch, stream, fn, calls, replays, warmup=3):
    """Capture `calls` invocations of fn into a graph; return ms per invocation."""
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(calls):
            fn()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(BLOCK_CYCLES)   # hides the host's submission of the replays
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (calls * replays)


def bench_rows(dev, stream, bf16_tf, peak_kind, hbm_peak, only=None):
    """The other rows; ``only`` (a set of row names) limits which run."""
    import torch
    import int4_weight_quantized_w4_gb300 as w4

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def on(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    rows = {}

    def want(name):
        return only is None or name in only

    def dense(name, M, N, K, group, outliers):
        g = K if group == -1 else group
        x = bf16(S.activations_bf16(M, K, seed=0, outlier_frac=outliers))
        qw = on(S.random_words((K // 8, N), seed=1))
        sw = on(S.scales_f16((K // g, N), seed=2))
        q = torch.empty((M, K), dtype=torch.int8, device=dev)
        s = torch.empty((M,), dtype=torch.float32, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty((w4.w4_workspace_bytes(w4.W4_OP_W4A8, M, N, K, group),), dtype=torch.uint8, device=dev)

        def step():
            w4.w4_quant_act_per_token(x, "int8", q=q, scale=s, stream=stream)
            w4.w4a8_gemm(q, s, qw, sw, group, y=y, workspace=ws, stream=stream)

        def gemm():
            w4.w4a8_gemm(q, s, qw, sw, group, y=y, workspace=ws, stream=stream)

        # the quantizer alone on rotating copies of x, together larger than L2
        xq = [x] + [x.clone() for _ in range(max(1, -(-L2_BYTES * 2 // (M * K * 2))) - 1)]
        xq_next = itertools.cycle(xq)

        def quant():
            w4.w4_quant_act_per_token(next(xq_next), "int8", q=q, scale=s, stream=stream)

        def fused():
            w4.w4a8_gemm_bf16in(x, qw, sw, group, y=y, x_scale=s, workspace=ws, stream=stream)

        t_fused = _time_graph(torch, stream, fused, 5, 10)
        t_step = _time_graph(torch, stream, step, 5, 10)
        t_gemm = _time_graph(torch, stream, gemm, 5, 10)
        t_quant = _time_graph(torch, stream, quant, len(xq), 10)
        ops = 2.0 * M * N * K
        tops_gemm = ops / (t_gemm * 1e-3) / 1e12
        rows[name] = {
            "config": {"M": M, "N": N, "K": K, "group": group, "outlier_channels": outliers},
            "value": round(ops / (t_fused * 1e-3) / 1e12, 1), "unit": "TOPS",
            "ms_per_step": t_fused, "step": "w4a8_gemm_bf16in (per-token int8 quantization fused into the GEMM)",
            "unfused_ms": t_step, "unfused_tops": round(ops / (t_step * 1e-3) / 1e12, 1),
            "unfused_step": "w4_quant_act_per_token + w4a8_gemm",
            "gemm_ms": t_gemm, "gemm_tops": round(tops_gemm, 1),
            "quant_ms": t_quant, "quant_gbs": round(3.0 * M * K / (t_quant * 1e-3) / 1e9, 1),
            "quant_l2": f"{len(xq)} rotating copies of x ({len(xq) * M * K * 2 / 1e6:.0f} MB)",
            "roofline": {"bound": "tensor", "achieved": round(tops_gemm, 1), "peak": bf16_tf, "unit": "TFLOP/s",
                         "frac": round(tops_gemm / bf16_tf, 4), "traffic": _traffic(name),
                         "peak_source": f"{peak_kind} bf16_tflops (the exact int8 x int4 products run on the "
                                        "fp16 tensor datapath; sm_103a has no int8 tcgen05 MMA)",
                         "kernel": "w4a8_gemm call = widen_kernel + w4a8_tc_kernel"},
            "l2": "inputs + outputs per step larger than L2",
        }

    if want("w4a8_prefill"):
        dense("w4a8_prefill", 4096, 11008, 4096, 128, 0.01)
    if want("w4a8_diffusion"):
        dense("w4a8_diffusion", 16384, 3072, 3072, -1, 0.0)

    if want("w4a8_prefill_sweep"):
        # the prefill sweep M x N at K = 4096, g128, 1% outlier channels; weight
        # copies rotate so that every point's working set exceeds L2
        K = 4096
        xs_all = bf16(S.activations_bf16(4096, K, seed=0, outlier_frac=0.01))
        points = {}
        for N in (4096, 11008):
            wbytes = K * N // 2 + (K // 128) * N * 2
            copies = max(2, -(-256 * 2**20 // wbytes))
            qws = [on(S.random_words((K // 8, N), seed=1, tag=20 + c)) for c in range(copies)]
            sws = [on(S.scales_f16((K // 128, N), seed=2, tag=30 + c)) for c in range(copies)]
            for M in (512, 1024, 2048, 4096):
                x = xs_all[:M]
                y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                sx = torch.empty((M,), dtype=torch.float32, device=dev)
                ws = torch.empty((w4.w4_workspace_bytes(w4.W4_OP_W4A8, M, N, K, 128),), dtype=torch.uint8,
                                 device=dev)
                it = [0]

                def call(x=x, y=y, sx=sx, ws=ws, it=it, qws=qws, sws=sws):
                    c = it[0] % len(qws)
                    it[0] += 1
                    w4.w4a8_gemm_bf16in(x, qws[c], sws[c], 128, y=y, x_scale=sx, workspace=ws, stream=stream)

                t = _time_graph(torch, stream, call, copies, 3)
                tops = 2.0 * M * N * K / (t * 1e-3) / 1e12
                points[f"M{M}_N{N}"] = {"ms": round(t, 5), "tops": round(tops, 1), "frac": round(tops / bf16_tf, 4)}
            del qws, sws
        rows["w4a8_prefill_sweep"] = {
            "config": {"M": [512, 1024, 2048, 4096], "N": [4096, 11008], "K": K, "group": 128,
                       "outlier_channels": 0.01},
            "unit": "TOPS", "step": "w4a8_gemm_bf16in", "points": points,
            "peak": bf16_tf, "peak_source": f"{peak_kind} bf16_tflops",
            "l2": "weight copies rotate: at least 256 MB of distinct weights per point",
        }
    if want("w4a16_sweep"):
        # decode at M = 1, 4, 8: symmetric fp16 scales, symmetric bf16 scales, and
        # the asymmetric variant with bf16 zeros; 16 rotating weight copies (> L2)
        K, N, g = DEC_K, DEC_N, DEC_G
        qws = [on(S.random_words((K // 8, N), seed=1, tag=20 + c)) for c in range(N_COPIES)]
        sfs = [on(S.scales_f16((K // g, N), seed=2, tag=30 + c)) for c in range(N_COPIES)]
        sbs = [bf16(S.to_bf16_bits(S.scales_f16((K // g, N), seed=2, tag=30 + c).astype(np.float32)))
               for c in range(N_COPIES)]
        zs = [bf16(S.to_bf16_bits(0.01 * S.normal(3, 40 + c, (K // g) * N).reshape(K // g, N)))
              for c in range(N_COPIES)]
        points = {}
        for M in (1, 4, 8):
            x = bf16(S.activations_bf16(M, K, seed=0))
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            for variant in ("sym_fp16", "sym_bf16", "asym_fp16_zeros"):
                sc = sbs if variant == "sym_bf16" else sfs
                zz = zs if variant.startswith("asym") else None
                it = [0]

                def call(x=x, y=y, sc=sc, zz=zz, it=it):
                    c = it[0] % N_COPIES
                    it[0] += 1
                    w4.w4a16_gemm(x, qws[c], sc[c], g, zeros=None if zz is None else zz[c], y=y, stream=stream)

                t = _time_graph(torch, stream, call, 4 * N_COPIES, 20)
                nbytes = K * N // 2 + (K // g) * N * 2 * (2 if zz is not None else 1) + M * K * 2 + M * N * 2
                gbs = nbytes / (t * 1e-3) / 1e9
                points[f"M{M}_{variant}"] = {"ms": round(t, 5), "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4)}
        rows["w4a16_sweep"] = {
            "config": {"M": [1, 4, 8], "K": K, "N": N, "group": g,
                       "variants": ["sym_fp16", "sym_bf16", "asym_fp16_zeros"]},
            "unit": "GB/s", "step": "w4a16_gemm (prefetch grid + GEMV grid)", "points": points,
            "peak": hbm_peak, "l2": f"{N_COPIES} rotating weight copies",
        }
    if want('w4afp8_moe'):
        # the routed MoE layer: 4096 tokens, hidden 2048, 64 experts, top-8,
        # intermediate 1408 (gate_up N = 2816, down K = 1408)
        T, E, top, g, Hd, I = 4096, 64, 8, 128, 2048, 1408
        R = T * top
        lg = on(S.router_logits(T, E, seed=5))
        xt = bf16(S.activations_bf16(T, Hd, seed=0))
        w1, s1 = on(S.random_words((E, 2 * I, Hd // 8), seed=1)), on(S.scales_f16((E, 2 * I, Hd // g), seed=2))
        w2 = on(S.random_words((E, Hd, I // 8), seed=1, tag=21))
        s2 = on(S.scales_f16((E, Hd, I // g), seed=2, tag=31))
        route = w4.w4_moe_route(lg, top, True)
        ids, wts, off, rt, ro = route
        h1 = torch.empty((R, 2 * I), dtype=torch.bfloat16, device=dev)
        sx1 = torch.empty((R,), dtype=torch.float32, device=dev)
        qa = torch.empty((R, I), dtype=torch.float8_e4m3fn, device=dev)
        sa = torch.empty((R,), dtype=torch.float32, device=dev)
        y2 = torch.empty((R, Hd), dtype=torch.bfloat16, device=dev)
        out = torch.empty((T, Hd), dtype=torch.bfloat16, device=dev)
        ws = torch.empty((max(w4.w4_workspace_bytes(w4.W4_OP_W4AFP8_MOE, R, 2 * I, Hd, g),
                              w4.w4_workspace_bytes(w4.W4_OP_W4AFP8_MOE, R, Hd, I, g)),), dtype=torch.uint8, device=dev)
        rws = torch.empty((max(16, w4.w4_workspace_bytes(w4.W4_OP_MOE_ROUTE, T, E, 1, 0)),), dtype=torch.uint8,
                          device=dev)

        def st_route():
            w4.w4_moe_route(lg, top, True, out=route, workspace=rws, stream=stream)

        def st_gate_up():
            w4.w4afp8_moe_gemm_bf16in(xt, rt, off, w1, s1, g, y=h1, x_scale=sx1, workspace=ws, stream=stream)

        def st_act():
            w4.w4_moe_silu_mul_quant_fp8(h1, q=qa, scale=sa, stream=stream)

        def st_down():
            w4.w4afp8_moe_grouped_gemm(qa, sa, off, w2, s2, g, y=y2, workspace=ws, stream=stream)

        def st_combine():
            w4.w4_moe_combine(y2, wts, ro, out=out, stream=stream)

        def moe_layer():
            st_route()
            st_gate_up()
            st_act()
            st_down()
            st_combine()

        t_layer = _time_graph(torch, stream, moe_layer, 3, 10)
        t_st = {nm: _time_graph(torch, stream, fn, 3, 10) for nm, fn in
                (("route", st_route), ("gate_up", st_gate_up), ("act", st_act), ("down", st_down),
                 ("combine", st_combine))}
        flops = 2.0 * R * (2 * I) * Hd + 2.0 * R * Hd * I
        t_gemm = t_st["gate_up"] + t_st["down"]
        tf_gemm = flops / (t_gemm * 1e-3) / 1e12
        act_bytes = R * 2 * I * 2 + R * I + R * 4
        comb_bytes = R * Hd * 2 + T * top * 8 + T * Hd * 2
        rows["w4afp8_moe"] = {
            "config": {"tokens": T, "hidden": Hd, "experts": E, "top_k": top, "intermediate": I, "rows": R,
                       "gate_up": [Hd, 2 * I], "down": [I, Hd], "group": g, "renormalize": True},
            "value": round(flops / (t_layer * 1e-3) / 1e12, 1), "unit": "TFLOP/s", "ms_per_step": t_layer,
            "step": "the whole routed layer: route, gather + fp8 quant + gate_up GEMM, SiLU*up + fp8 requant, "
                    "down GEMM, weighted combine",
            "stage_ms": {k: round(v, 5) for k, v in t_st.items()},
            "gemm_tflops": round(tf_gemm, 1),
            "act_gbs": round(act_bytes / (t_st["act"] * 1e-3) / 1e9, 1),
            "combine_gbs": round(comb_bytes / (t_st["combine"] * 1e-3) / 1e9, 1),
            "roofline": {"bound": "tensor", "achieved": round(tf_gemm, 1), "peak": round(FP8_PER_BF16 * bf16_tf, 1),
                         "unit": "TFLOP/s", "frac": round(tf_gemm / (FP8_PER_BF16 * bf16_tf), 4),
                         "traffic": _traffic("w4afp8_moe"),
                         "peak_source": f"dense fp8 peak = {FP8_PER_BF16:g} x {peak_kind} bf16_tflops "
                                        "(the nominal fp8:bf16 ratio of 4.5:2.25 PFLOP/s)",
                         "kernel": MOE_KERNEL},
        }
    if want('weight_quantize_groupwise'):
        # weight-side tool (load time): the group quantizer on a 14336 x 4096 bf16 weight
        Nq, Kq, gq = 14336, 4096, 128
        blk = S.to_bf16_bits(S.normal(0, 90, 1024 * Kq).reshape(1024, Kq) * 0.05)
        wq = bf16(np.tile(blk, (Nq // 1024, 1)))
        pk = torch.empty((Nq, Kq // 2), dtype=torch.uint8, device=dev)
        sq = torch.empty((Nq, Kq // gq), dtype=torch.float32, device=dev)
        zq = torch.empty((Nq, Kq // gq), dtype=torch.float32, device=dev)
        t_q = _time_graph(torch, stream, lambda: w4.w4_quantize_groupwise(wq, gq, pk, sq, zq, stream=stream), 5, 10)
        qbytes = Nq * Kq * 2 + Nq * Kq // 2 + 2 * Nq * (Kq // gq) * 4
        rows["weight_quantize_groupwise"] = {
            "config": {"N": Nq, "K": Kq, "group": gq, "w": "bf16"}, "value": round(qbytes / (t_q * 1e-3) / 1e9, 1),
            "unit": "GB/s", "ms_per_step": t_q,
            "roofline": {"bound": "hbm", "achieved": round(qbytes / (t_q * 1e-3) / 1e9, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(qbytes / (t_q * 1e-3) / 1e9 / hbm_peak, 4),
                         "traffic": _traffic("quantize"),
                         "kernel": "quantize_chunks_kernel", "algorithmic_bytes_per_launch": qbytes},
        }
    if want('lm_head_gemv'):
        # tied embedding table used as the decode output head: one token against a
        # 131072 x 2048 group-128 table (4 rotating copies, 604 MB, more than L2)
        V, D, gh = 131072, 2048, 128
        tabs = []
        for c in range(4):
            pk = on(np.tile(S.raw_u64(c, 97, 1024 * D // 16).view(np.uint8).reshape(1024, D // 2), (V // 1024, 1)))
            scl = on(np.tile((0.002 + 0.001 * S.uniform(c, 98, 1024 * D // gh)).astype(np.float32).reshape(1024, D // gh),
                             (V // 1024, 1)))
            zr = on(np.tile((0.01 * S.normal(c, 99, 1024 * D // gh)).astype(np.float32).reshape(1024, D // gh),
                            (V // 1024, 1)))
            tabs.append((pk, scl, zr))
        hh = bf16(S.activations_bf16(1, D, seed=0))
        yh = torch.empty((1, V), dtype=torch.bfloat16, device=dev)
        it = [0]

        def head():
            pk, scl, zr = tabs[it[0] % 4]
            it[0] += 1
            w4.w4_lm_head_gemv(hh, pk, scl, zr, gh, y=yh, stream=stream)

        t_h = _time_graph(torch, stream, head, 8, 10)
        hbytes = V * D // 2 + 2 * V * (D // gh) * 4 + D * 2 + V * 2
        rows["lm_head_gemv"] = {
            "config": {"M": 1, "V": V, "D": D, "group": gh, "scale_zero": "f32", "l2": "4 rotating tables (604 MB)"},
            "value": round(hbytes / (t_h * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": t_h,
            "roofline": {"bound": "hbm", "achieved": round(hbytes / (t_h * 1e-3) / 1e9, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(hbytes / (t_h * 1e-3) / 1e9 / hbm_peak, 4),
                         "traffic": _traffic("lm_head"),
                         "kernel": "lm_head_tc1_kernel", "algorithmic_bytes_per_launch": hbytes},
        }
    if want('s4_repack_uint4b8'):
        # weight-side tool (load time): the XOR 0x88 repack of a 64-expert [E, N, K/2] int4 tensor
        rb = 64 * 2816 * 1024
        s4 = on((S.raw_u64(8, 80, rb // 8).view(np.uint8)))
        s4o = torch.empty_like(s4)
        t_r = _time_graph(torch, stream, lambda: w4.w4_repack_s4_to_uint4b8(s4, s4o, stream=stream), 5, 10)
        rows["s4_repack_uint4b8"] = {
            "config": {"bytes": rb, "layout": "[64, 2816, 1024] int8 -> int32 [64, 2816, 256]"},
            "value": round(2 * rb / (t_r * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": t_r,
            "roofline": {"bound": "hbm", "achieved": round(2 * rb / (t_r * 1e-3) / 1e9, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(2 * rb / (t_r * 1e-3) / 1e9 / hbm_peak, 4), "traffic": None,
                         "kernel": "xor88_kernel", "algorithmic_bytes_per_launch": 2 * rb},
        }
    return rows


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------

def oracle_decode_sample(cols, seed=0):
    """Inputs for the decode GEMV restricted to a column block (same generator streams)."""
    xb = S.activations_bf16(DEC_M, DEC_K, seed=seed)
    qw = S.random_words((DEC_K // 8, DEC_N), seed=1, tag=20)[:, cols]
    sw = S.scales_f16((DEC_K // DEC_G, DEC_N), seed=2, tag=30)[:, cols]
    return xb, np.ascontiguousarray(qw), np.ascontiguousarray(sw)


def cpu_baseline(budget_s=10.0):
    """Time the C oracle's W4A16 (plain loops in float64, threads over the output
    columns) on the whole M=1 decode GEMV, repeated for ~budget_s."""
    from oracle import c_oracle as C
    xb, qw, sw = oracle_decode_sample(np.arange(DEC_N))
    C.w4a16_linear(xb, qw, sw, DEC_G)   # warm (and build)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        C.w4a16_linear(xb, qw, sw, DEC_G)
        n += 1
    dt = time.perf_counter() - t0
    nbytes = decode_bytes()
    return {"value": round(n * nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": C.threads(), "kind": "oracle",
            "sample": f"{n} calls of the C oracle (oracle/w4_oracle_c.c, float64, {C.threads()} threads) on the whole "
                      f"M=1 decode GEMV (K=4096, N=14336, group 128), {dt:.1f} s"}


REF_BUDGET_S = 60.0   # the reference arm's timed steps, whatever K is


def ref_columns(steps, t_full, budget_s=REF_BUDGET_S):
    """Output columns per reference step: all of them when `steps` whole calls
    (t_full seconds each) fit in budget_s, else the largest multiple of 32
    (at least 32) that keeps the steps within it."""
    if steps * t_full <= budget_s:
        return DEC_N
    return max(32, int(DEC_N * budget_s / (steps * t_full)) // 32 * 32)


def run_reference(args, rank, world):
    """The C oracle on the decode GEMV, K steps. A step is the whole GEMV when
    K of them fit in REF_BUDGET_S; otherwise a block of its output columns
    (a multiple of 32) sized from one timed whole call, so that the run ends
    within minutes at any K."""
    if rank != 0:
        return None
    from oracle import c_oracle as C
    xb, qw, sw = oracle_decode_sample(np.arange(DEC_N))
    t0 = time.perf_counter()
    C.w4a16_linear(xb, qw, sw, DEC_G)
    t_full = max(time.perf_counter() - t0, 1e-6)
    steps = max(1, args.steps)
    cols = ref_columns(steps, t_full)
    if cols < DEC_N:
        xb, qw, sw = oracle_decode_sample(np.arange(cols))
    for _ in range(max(args.warmup, 3)):
        C.w4a16_linear(xb, qw, sw, DEC_G)
    t0 = time.perf_counter()
    for _ in range(steps):
        C.w4a16_linear(xb, qw, sw, DEC_G)
    dt = time.perf_counter() - t0
    nbytes = decode_bytes(N=cols)
    value = steps * nbytes / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same generator as the GPU arm)",
        "config": {"workload": "w4a16_decode", "M": DEC_M, "K": DEC_K, "N": DEC_N, "group": DEC_G,
                   "scales": "fp16", "zeros": False,
                   "sample": ("each step: the C oracle on the whole decode GEMV" if cols == DEC_N else
                              f"each step: the C oracle on output columns 0..{cols - 1} of the decode GEMV")},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": C.threads(), "kind": "oracle",
                         "sample": f"{steps} steps, each the C oracle (float64, {C.threads()} threads) on "
                                   + ("the whole M=1 decode GEMV" if cols == DEC_N else
                                      f"{cols} of the {DEC_N} output columns of the M=1 decode GEMV")},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def summarize(line):
    """The headline figure of every row in a few hundred bytes: TOPS / GB/s and
    the fraction of the measured peak, so that the end of the line carries them."""
    rows = line.get("rows") or {}
    rf = line["roofline"]
    out = {"w4a16_M1": {"gbs": rf["achieved"], "frac": rf["frac"]}}
    for nm in ("w4a8_prefill", "w4a8_diffusion"):
        r = rows.get(nm)
        if r:
            out[nm] = {"tops": r["value"], "gemm_tops": r["gemm_tops"], "frac": r["roofline"]["frac"],
                       "quant_gbs": r["quant_gbs"]}
    sw = rows.get("w4a8_prefill_sweep")
    if sw:
        out["w4a8_sweep_frac"] = {k: v["frac"] for k, v in sw["points"].items()}
    m = rows.get("w4afp8_moe")
    if m:
        out["w4afp8_moe"] = {"layer_tflops": m["value"], "gemm_tflops": m["gemm_tflops"],
                             "frac_fp8": m["roofline"]["frac"]}
    ws = rows.get("w4a16_sweep")
    if ws:
        out["w4a16_sweep_frac"] = {k: v["frac"] for k, v in ws["points"].items()}
    for nm in ("lm_head_gemv", "weight_quantize_groupwise", "s4_repack_uint4b8"):
        r = rows.get(nm)
        if r:
            out[nm] = {"gbs": r["value"], "frac": r["roofline"]["frac"]}
    return out


def ordered_line(line):
    """The bulky per-row detail first, the headline keys after it and the
    compact summary last."""
    out = {}
    if "rows" in line:
        out["rows"] = line["rows"]
    for k, v in line.items():
        if k != "rows":
            out[k] = v
    out["summary"] = summarize(line)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="time only the headline workload")
    ap.add_argument("--rows", default="", help="comma-separated names of the other rows to run (default: all)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(ordered_line(line)), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
