"""Benchmark of the fused attention forward + JVP (jvp_attn_fwd_dual).

One step = one fwd_dual call (the whole hot path) over the bf16 workload
B=4, H=16, N=2048, D=128 with no mask, inputs resident in HBM.  Timed with
CUDA events on the launching stream around each call; a 256 MiB buffer is
written between timed calls so every step starts with a cold L2.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs the same
workload on its own GPU (replicas, weak scaling, no collective on the data
path); `value` is all ranks' FLOPs over the slowest rank's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the float64 CPU oracle, timed on host cores
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+JVP attention TFLOP/s & % of GB300 tensor peak (bf16, N=2048)"
DEFAULT_WORKLOAD = "bf16_b4h16n2048d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
TC_SOURCES = ["forward_mode_flash_gb300/csrc/fwd_dual_tc.cuh",
              "forward_mode_flash_gb300/csrc/sm103_ptx.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target length of the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-causal", action="store_true",
                    help="skip the causal companion timing of the default workload")
    ap.add_argument("--mode", default="fwd_dual",
                    choices=["fwd_dual", "fwd", "bwd_dual", "bwd", "sweep", "memory"],
                    help="fwd_dual (the headline), the forward without tangents (fwd), the "
                         "backward of the dual computation (bwd_dual) "
                         "or of attention without tangents (bwd), the "
                         "sequence-length sweep (one JSON line per configuration) or the "
                         "memory-scaling report (one JSON line per N)")
    ap.add_argument("--sweep-dtypes", default="bf16,f16")
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="(batch, head) groups of the host-buffer entry point in the e2e run")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """The source without comments and blank lines, each line stripped.

    A comment-only edit does not change the compiled kernel, so it should not
    invalidate counters recorded for it.  (Scans for // and /* */ outside
    string and character literals.)
    """
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.strip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def source_hash() -> str:
    """Hash of the tensor-core kernel's code (comments and layout excluded)."""
    h = hashlib.sha256()
    for rel in TC_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it matches the source."""
    path = os.path.join(ROOT, "profiles", f"fwd_dual_tc_{workload}_traffic.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_hash") != source_hash():
        return None  # the kernel changed since the counters were taken
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region.

    A reader thread collects nvidia-smi's lines (one per 100 ms).  Entering
    waits for the first sample, and leaving waits for one more sample taken
    after the region ends, so even a region shorter than the sampling period
    is bracketed by samples taken under the same load conditions."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.out = ""

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def _wait_for(self, n, timeout):
        t_end = time.time() + timeout
        while len(self.lines) < n and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.005)

    def __enter__(self):
        import threading

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        self._wait_for(1, 3.0)
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            return
        self._wait_for(len(self.lines) + 1, 1.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        self.out = "".join(self.lines)

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v and
                          "Not" not in v})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def cpu_baseline(workload, target_s: float):
    """The float64 oracle on a bounded sample of rows of the same workload."""
    import numpy as np

    import oracle
    from forward_mode_flash_gb300 import metrics, synth

    w = synth.WORKLOADS[workload]
    inp = synth.make_inputs(w)
    f64 = [x.double().numpy() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    kind = w.mask
    m = None
    if w.mask == "bool":
        m = inp.mask.numpy()
    elif w.mask == "additive":
        m = inp.mask.double().numpy()
    total = w.B * w.H * w.N
    rng = np.random.default_rng(0)
    cores = oracle.default_threads()
    n = max(cores, 16)
    t0 = time.perf_counter()
    oracle.fwd_dual_rows(*f64, rng.integers(0, total, n), kind, m)
    dt = time.perf_counter() - t0
    n = int(min(total, max(n, n * target_s / max(dt, 1e-3))))
    rows = rng.integers(0, total, n)
    t0 = time.perf_counter()
    oracle.fwd_dual_rows(*f64, rows, kind, m)
    dt = time.perf_counter() - t0
    causal = w.mask == "causal"
    if causal:
        keys = float(np.sum(np.minimum(rows % w.N + 1, w.N)))
        flops = 12.0 * keys * w.D
    else:
        flops = metrics.flops_fwd_dual(1, 1, n, w.N, w.D)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} random query rows of {workload} (every key of each row), float64 "
                      f"dual-number oracle, {dt:.1f} s wall"}, dt


def timed_steps(step, steps, flush, stream, local):
    """Times `steps` calls of step() with CUDA events on `stream`, writing the
    L2-flush buffer before each call (outside the events); returns the
    per-call milliseconds and the clocks sampled meanwhile."""
    import torch

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # Two untimed steps right before the timed ones: the device may have
        # idled (and lowered its clock) while the sampler started, and they
        # give the host a head start, so that no stall before the first timed
        # call is timed as device time.
        for _ in range(2):
            flush.fill_(0.0)
            step()
        with torch.cuda.nvtx.range(f"timed region: {steps} steps"):
            for s in range(steps):
                flush.fill_(float(s))  # evict L2 between timed steps (outside the events)
                starts[s].record(stream)
                with torch.cuda.nvtx.range("step"):
                    step()
                ends[s].record(stream)
            torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], clocks


CAUSAL_WORKLOAD = "bf16_b4h16n2048d128_causal"


def causal_companion(args, dev, world, flush, stream, local, peak, pk_src):
    """The headline shape with the causal mask, timed like the headline: the
    same number of steps, after its own warm-up, with its own clock record."""
    import torch

    from forward_mode_flash_gb300 import api, metrics, replicas, synth

    w = synth.WORKLOADS[CAUSAL_WORKLOAD]
    inp = synth.make_inputs(w, device=str(dev))
    g = [inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv]
    out = (torch.empty_like(g[0]), torch.empty_like(g[0]))

    def step():
        return api.fwd_dual(*g, is_causal=True, out=out)

    for _ in range(max(3, args.warmup)):
        step()
    per_ms, clocks = timed_steps(step, args.steps, flush, stream, local)
    if api.last_path() not in api.TENSOR_CORE_PATHS:
        raise SystemExit("the tensor-core path did not run for the causal workload")
    total_ms = replicas.max_over_ranks(sum(per_ms), device=dev)
    ms_step = total_ms / args.steps
    flops = metrics.flops_fwd_dual(w.B, w.H, w.N, w.N, w.D, True)
    value = replicas.aggregate_throughput(world, flops, args.steps, total_ms * 1e-3) / 1e12
    achieved = flops / (ms_step * 1e-3) / 1e12
    return {"workload": CAUSAL_WORKLOAD, "ms_per_step": ms_step, "value": value,
            "unit": "TFLOP/s", "steps": args.steps, "flops_per_step": flops,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": recorded_traffic(CAUSAL_WORKLOAD),
                         "peak_source": f"{pk_src} bf16_tflops (burst; kernel timed alone)",
                         "kernel": "fwd_dual_tc_kernel"},
            "clocks": clocks.summary(), "gpu_launches": args.steps,
            "per_step_ms": {"min": min(per_ms), "median": statistics.median(per_ms),
                            "max": max(per_ms), "max_at": per_ms.index(max(per_ms))}}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from forward_mode_flash_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    vals, times = [], []
    per_step = max(1.0, min(10.0, 60.0 / max(1, args.steps + args.warmup)))
    for s in range(args.warmup + args.steps):
        cb, dt = cpu_baseline(args.workload, per_step)
        if s >= args.warmup:
            vals.append(cb["value"])
            times.append(dt)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                       "mask": w.mask, "input_dtype": w.dtype},
            "cpu_baseline": dict(cb, value=v),
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


FP32_LANES_PER_SM = 128  # CUDA-core fp32 FMA lanes per SM (4 partitions x 32)


def run_bwd(args, rank, world, local):
    """Times jvp_attn_bwd_dual (--mode bwd_dual) or jvp_attn_bwd, the backward
    of attention without tangents (--mode bwd), on one workload.

    fp16/bf16 inputs with D in {64, 128} run the row pre-pass and the tcgen05
    kernels (query-major, then key-major: one launch at D = 64 and for the
    primal, value and key parts for the dual at D = 128); other shapes run
    three CUDA-core kernels."""
    primal = args.mode == "bwd"
    import numpy as np
    import torch

    import oracle
    from forward_mode_flash_gb300 import api, build, replicas, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    name = args.workload
    w = synth.WORKLOADS[name]
    causal = w.mask == "causal"
    inp = synth.make_inputs(w, with_cotangents=True, device=str(dev))
    g = [inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv]
    ws = torch.empty(max(1, api.bwd_dual_workspace_size(w.B, w.H, w.N, w.N, w.D)),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if primal:
        o, lse = api.attention(*g[:3], attn_mask=inp.mask, is_causal=causal, return_lse=True)

        def step():
            return api.bwd(*g[:3], o, lse, inp.g_o, attn_mask=inp.mask, is_causal=causal,
                           workspace=ws)
    else:
        o, t_o, lse, mu = api.fwd_dual(*g, attn_mask=inp.mask, is_causal=causal,
                                       return_stats=True)

        def step():
            return api.bwd_dual(*g, o, t_o, lse, mu, inp.g_o, inp.g_to, attn_mask=inp.mask,
                                is_causal=causal, workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    tensor_core = api.last_path() == 1
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        for _ in range(2):  # untimed steps right before the timed ones (see timed_steps)
            flush.fill_(0.0)
            step()
        with torch.cuda.nvtx.range(f"{args.mode} timed region: {args.steps} steps"):
            for s in range(args.steps):
                flush.fill_(float(s))
                starts[s].record(stream)
                with torch.cuda.nvtx.range("step"):
                    step()
                ends[s].record(stream)
            torch.cuda.synchronize()
    per_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = replicas.max_over_ranks(sum(per_ms), device=dev)
    ms_step = total_ms / args.steps
    half = 0.5 if causal else 1.0
    bhnnd = w.B * w.H * w.N * w.N * w.D * half
    if primal:
        alg_flops = 8.0 * bhnnd    # gO V^T, gS K, gS^T Q, P^T gO
        exec_flops = 14.0 * bhnnd  # S and gO V^T formed in both kernels
    else:
        alg_flops = 30.0 * bhnnd   # the 15 N x N x D products of the reverse mode
        # Products executed (scores recomputed): 21 per (row, key, d) in the
        # CUDA-core kernels and in the tensor-core kernels at D = 64; the D = 128
        # key-major split recomputes the three score products once more (24).
        exec_flops = (48.0 if (tensor_core and w.D == 128) else 42.0) * bhnnd
    value = replicas.aggregate_throughput(world, alg_flops, args.steps, total_ms * 1e-3) / 1e12
    pk, pk_src = peaks()
    clk = pk.get("sm_max_mhz", 2070.0) * 1e6
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    achieved = alg_flops / (ms_step * 1e-3) / 1e12
    achieved_exec = exec_flops / (ms_step * 1e-3) / 1e12
    if tensor_core:
        tc_peak = float(pk.get("bf16_tflops", 1900.0))  # fp16 and bf16 share the dense rate
        launches = 3 if (w.D == 64 or primal) else 4
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": achieved / tc_peak, "traffic": None,
                    "flops": ("algorithmic: 8 B H Nq Nk D (half for causal), the four N x N x D "
                              "products of the backward" if primal else
                              "algorithmic: 30 B H Nq Nk D (half for causal), the 15 N x N x D "
                              "products of the reverse mode"),
                    "achieved_executed": achieved_exec, "frac_executed": achieved_exec / tc_peak,
                    "peak_source": f"{pk_src} bf16 dense (cuBLAS burst)",
                    "kernel": "whole step: bwd_rows_kernel + bwd_q_tc_kernel + bwd_k_tc_kernel"
                              + (" x2 (value, key parts)" if (w.D == 128 and not primal) else "")}
    else:
        alu_peak = n_sms * FP32_LANES_PER_SM * 2 * clk / 1e12
        launches = 3
        roofline = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                    "frac": achieved / alu_peak, "traffic": None,
                    "achieved_executed": achieved_exec, "frac_executed": achieved_exec / alu_peak,
                    "peak_source": f"{n_sms} SMs x {FP32_LANES_PER_SM} fp32 FMA lanes x 2 x "
                                   f"{clk / 1e6:.0f} MHz (CUDA-core fp32)",
                    "kernel": "bwd_keys_kernel + bwd_queries_kernel + bwd_rows_kernel"}
    line = {
        "metric": ("bwd (backward of attention without tangents) TFLOP/s" if primal else
                   "bwd_dual (reverse mode of fwd+JVP attention) TFLOP/s"), "mode": args.mode,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": f"{w.dtype} (fp32 accumulate)" if tensor_core else "f32", "data": "synthetic",
        "config": {"workload": name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "mask": w.mask,
                   "input_dtype": w.dtype, "algorithmic_flops_per_step": alg_flops,
                   "executed_flops_per_step": exec_flops,
                   "l2": "flushed: 256 MiB written between timed steps (outside the events)"},
        "roofline": roofline,
        "clocks": clocks.summary(), "gpu_launches": launches * args.steps, "e2e": None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # The float64 oracle's reverse mode on one whole head of the same workload.
        x = [t[:1, :1].double().cpu().numpy() for t in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv,
                                                         inp.g_o, inp.g_to)]
        if primal:  # zero tangents and tangent cotangent: the primal backward
            x = x[:3] + [np.zeros_like(a) for a in x[3:6]] + [x[6], np.zeros_like(x[7])]
        t0 = time.perf_counter()
        oracle.bwd_dual(*x, w.mask, None)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": alg_flops / (w.B * w.H) / dt / 1e12,
                                "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                "sample": f"one (b, h) head of {name}, float64 reverse mode, "
                                          f"{dt:.1f} s wall (the oracle threads over heads)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_fwd(args, rank, world, local):
    """Times jvp_attn_fwd, the forward of attention without tangents (O and the
    log-sum-exp), on one workload (--mode fwd): the plain attention forward of
    jvp_attention outside torch.func.jvp."""
    import torch

    import oracle
    from forward_mode_flash_gb300 import api, build, metrics, replicas, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    name = args.workload
    w = synth.WORKLOADS[name]
    causal = w.mask == "causal"
    inp = synth.make_inputs(w, device=str(dev))
    o = torch.empty_like(inp.q)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        return api.attention(inp.q, inp.k, inp.v, attn_mask=inp.mask, is_causal=causal,
                             return_lse=True, out=o)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    tensor_core = api.last_path() == 1
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        for _ in range(2):  # untimed steps right before the timed ones (see timed_steps)
            flush.fill_(0.0)
            step()
        with torch.cuda.nvtx.range(f"fwd timed region: {args.steps} steps"):
            for s in range(args.steps):
                flush.fill_(float(s))
                starts[s].record(stream)
                with torch.cuda.nvtx.range("step"):
                    step()
                ends[s].record(stream)
            torch.cuda.synchronize()
    per_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = replicas.max_over_ranks(sum(per_ms), device=dev)
    ms_step = total_ms / args.steps
    flops = metrics.flops_fwd(w.B, w.H, w.N, w.N, w.D, causal)
    value = replicas.aggregate_throughput(world, flops, args.steps, total_ms * 1e-3) / 1e12
    pk, pk_src = peaks()
    achieved = flops / (ms_step * 1e-3) / 1e12
    if tensor_core:
        tc_peak = float(pk.get("bf16_tflops", 1900.0))  # fp16 and bf16 share the dense rate
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": achieved / tc_peak, "traffic": None,
                    "flops": "algorithmic: 4 B H Nq Nk D (half for causal), Q K^T and P V",
                    "peak_source": f"{pk_src} bf16 dense (cuBLAS burst)",
                    "kernel": "fwd_dual_tc_kernel without tangents"}
    else:
        clk = pk.get("sm_max_mhz", 2070.0) * 1e6
        n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = n_sms * FP32_LANES_PER_SM * 2 * clk / 1e12
        roofline = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                    "frac": achieved / alu_peak, "traffic": None,
                    "peak_source": f"{n_sms} SMs x {FP32_LANES_PER_SM} fp32 FMA lanes x 2 x "
                                   f"{clk / 1e6:.0f} MHz (CUDA-core fp32)",
                    "kernel": "fwd_dual_simt_kernel without tangents"}
    line = {
        "metric": "fwd (attention forward without tangents) TFLOP/s", "mode": args.mode,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": f"{w.dtype} (fp32 accumulate)" if tensor_core else "f32", "data": "synthetic",
        "config": {"workload": name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "mask": w.mask,
                   "input_dtype": w.dtype, "algorithmic_flops_per_step": flops,
                   "l2": "flushed: 256 MiB written between timed steps (outside the events)"},
        "roofline": roofline,
        "clocks": clocks.summary(), "gpu_launches": args.steps, "e2e": None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # The float64 oracle on one whole head of the same workload (zero tangents).
        x = [t[:1, :1].double().cpu().numpy() for t in (inp.q, inp.k, inp.v)]
        m = inp.mask
        kind, mm = w.mask, None
        if m is not None:
            mm = m[:1, :1].double().cpu().numpy() if w.mask == "additive" else m[:1, :1].cpu().numpy()
        t0 = time.perf_counter()
        oracle.fwd_dual(*x, mask_kind=kind, mask=mm)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": flops / (w.B * w.H) / dt / 1e12,
                                "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                "sample": f"one (b, h) head of {name}, float64 forward "
                                          f"(the oracle's dual evaluation with zero tangents), "
                                          f"{dt:.1f} s wall (the oracle threads over heads)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_report(args, rank, world, local):
    """The sequence-length sweep or the memory-scaling report (rank 0 only)."""
    import torch

    from forward_mode_flash_gb300 import build, report

    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    build.build()
    pk, pk_src = peaks()
    if args.mode == "sweep":
        for row in report.sweep(dtypes=tuple(args.sweep_dtypes.split(",")),
                                peak_tflops=float(pk.get("bf16_tflops", 1900.0)),
                                peak_gbs=float(pk.get("hbm_gbs", 6800.0))):
            print(json.dumps({"mode": "sweep", "peaks": pk_src, **row}), flush=True)
    else:
        for row in report.memory_scaling():
            print(json.dumps({"mode": "memory", **row}), flush=True)
    return 0


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist

    from forward_mode_flash_gb300 import api, build, metrics, replicas, synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if args.mode in ("sweep", "memory"):
        return run_report(args, rank, world, local)
    if args.mode in ("bwd_dual", "bwd", "fwd"):
        rc = (run_fwd if args.mode == "fwd" else run_bwd)(args, rank, world, local)
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return rc
    build.build()

    w = synth.WORKLOADS[args.workload]
    causal = w.mask == "causal"
    inp = synth.make_inputs(w, device=str(dev))
    g = [inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv]
    mask = inp.mask
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flops = metrics.flops_fwd_dual(w.B, w.H, w.N, w.N, w.D, causal)
    elem = g[0].element_size()
    out = (torch.empty_like(g[0]), torch.empty_like(g[0]))

    def step():
        return api.fwd_dual(*g, attn_mask=mask, is_causal=causal, out=out)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if api.last_path() not in api.TENSOR_CORE_PATHS:
        raise SystemExit("the tensor-core path did not run for the benchmark workload")
    if world > 1:
        dist.barrier()
    stream = torch.cuda.current_stream()
    per_ms, clocks = timed_steps(step, args.steps, flush, stream, local)
    if world > 1:
        dist.barrier()
    total_ms = replicas.max_over_ranks(sum(per_ms), device=dev)
    ms_step = total_ms / args.steps
    value = replicas.aggregate_throughput(world, flops, args.steps, total_ms * 1e-3) / 1e12
    launches = args.steps  # one fwd_dual kernel per step

    # End to end through the public API: pinned host inputs -> device -> kernel -> host.
    # (api.fwd_dual_host, which overlaps chunked copies with the kernel, measured slower
    # here: the host link, not the kernel, sets the pace.)
    e2e = None
    if not args.no_e2e:
        host_in = [x.cpu().pin_memory() for x in g]
        host_mask = mask.cpu().pin_memory() if mask is not None else None
        dev_in = [torch.empty_like(x) for x in g]
        dev_mask = torch.empty_like(mask) if mask is not None else None
        host_out = [torch.empty(out[0].shape, dtype=out[0].dtype).pin_memory() for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in host_in)
        if host_mask is not None:
            h2d += host_mask.numel() * host_mask.element_size()
        d2h = sum(x.numel() * x.element_size() for x in host_out)

        # Through the host-buffer entry point (copies pipelined with the kernels
        # over chunks of (batch, head) pairs) when no per-batch mask is involved;
        # otherwise plain copies around fwd_dual.
        host_api = mask is None or mask.shape[0] == 1
        ws_host = None
        if host_api:
            ws_host = torch.empty(max(1, api.fwd_dual_host_workspace_size(
                w.B, w.H, w.N, w.N, w.D, g[0].dtype, args.e2e_chunks)), dtype=torch.uint8,
                device=dev)

        def e2e_step():
            if host_api:
                api.fwd_dual_host(*host_in, attn_mask=host_mask, is_causal=causal,
                                  chunks=args.e2e_chunks, out=host_out, workspace=ws_host)
                return
            for d, hsrc in zip(dev_in, host_in):
                d.copy_(hsrc, non_blocking=True)
            if dev_mask is not None:
                dev_mask.copy_(host_mask, non_blocking=True)
            o, t_o = api.fwd_dual(*dev_in, attn_mask=dev_mask, is_causal=causal, out=out)
            host_out[0].copy_(o, non_blocking=True)
            host_out[1].copy_(t_o, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        k_e2e = max(3, min(args.steps, 10))
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.nvtx.range(f"e2e timed region: {k_e2e} steps"):
            for _ in range(k_e2e):
                e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = replicas.max_over_ranks(a.elapsed_time(b) / k_e2e, device=dev)
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": k_e2e,
               "gpu_launches": k_e2e * (min(args.e2e_chunks, w.B * w.H) if host_api else 1),
               "path": (f"jvp_attn_fwd_dual_host, {args.e2e_chunks} chunks" if host_api
                        else "copies + jvp_attn_fwd_dual"),
               "h2d_plus_d2h_gbs": (h2d + d2h) / (e2e_ms * 1e-3) / 1e9}

    pk, pk_src = peaks()
    peak = float(pk["bf16_tflops"])
    achieved = flops / (ms_step * 1e-3) / 1e12
    traffic = recorded_traffic(args.workload)
    alg_bytes = metrics.bytes_fwd_dual(w.B, w.H, w.N, w.N, w.D, elem, w.mask, w.B)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else w.dtype, "data": "synthetic",
        "config": {"workload": args.workload, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "mask": w.mask, "flops_per_step": flops, "algorithmic_bytes_per_step": alg_bytes,
                   "l2": "flushed: 256 MiB written between timed steps (outside the events)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{pk_src} bf16_tflops (burst; kernel timed alone)",
                     "kernel": "fwd_dual_tc_kernel"},
        "clocks": clocks.summary(),
        "gpu_launches": launches,
        "e2e": e2e,
        "per_step_ms": {"min": min(per_ms), "median": statistics.median(per_ms),
                        "max": max(per_ms), "max_at": per_ms.index(max(per_ms))},
    }
    if args.workload == DEFAULT_WORKLOAD and not args.no_causal:
        line["causal"] = causal_companion(args, dev, world, flush, stream, local, peak, pk_src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], _ = cpu_baseline(args.workload, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
