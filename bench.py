#!/usr/bin/env python3
"""Benchmark of the fused SwiGLU up-projection Y = SiLU(A x W1) (.) (A x W2).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload LABEL] [--dtype bf16|fp8] [--split replicas|columns]

One step = one call of swiglu_up_forward (the whole fused path: both GEMMs,
the activation and the BF16 store) over one batch of M tokens. Default
workload: the largest single-GPU configuration, the Qwen-2.5-72B-shaped
up-projection with M=8192 tokens (K=8192, N=29568). Its inputs are the
seeded synthetic data of workloads/ (numpy PCG64), generated once and
resident in HBM before the timed region. Consecutive steps rotate over
several copies of A, the packed weights and Y whose total exceeds twice the
L2 size, so no step finds its operands in L2. `--dtype fp8` runs
swiglu_up_forward_fp8 on the E4M3 quantization of the same draws
(per-tensor scales, BF16 Y); its tensor roofline is the measured BF16 peak
times the nominal FP8/BF16 ratio of 2.

Besides the headline it measures, in the same process:
  * `sweep`: every workload of workloads.WORKLOADS (the metric is "vs M"),
    each timed over a window of graph-replayed launches with the clocks of
    that window; inputs drawn on the GPU from torch's seeded generator with
    the workloads' distributions;
  * `context_sustained`: the headline launch replayed for >= 1 s, against
    the sustained BF16 peak, with the clocks of that window;
  * `e2e`: the same metric through the public call with a pinned-host copy
    of A in and of Y out inside every step;
  * context only: L2-warm launches, the unfused cuBLAS path, the whole gated
    MLP, and the CPU oracle on a bounded row sample (`cpu_baseline`).

Prints one JSON line (rank 0). `--gpus N` with N > 1 starts N ranks itself
(torch.distributed.run on this node) unless it already runs under torchrun.
`--split replicas` (default): every rank runs the whole workload on its own
GPU (weak scaling); `--split columns`: rank r packs its slice of W1 and W2's
columns and writes Y[:, slice] (column-parallel, strong scaling). Neither
needs a collective on the data path; `value` is the FLOPs of all ranks over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused SwiGLU up-proj TFLOP/s and % of GB300 BF16/HBM roofline vs M"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "11"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
REFERENCE_BUDGET_S = 120.0
TILE_COLS = 128          # output columns of one tile: the column-split granule


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def device_info(dev) -> dict:
    """Name, SM count and L2 size of the GPU the step ran on."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    return {"name": torch.cuda.get_device_name(dev), "sm_count": props.multi_processor_count,
            "l2_bytes": getattr(props, "L2_cache_size", None)}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_swiglu_mlp_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_label: str, dtype: str = "bf16"):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    only if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    key = workload_label if dtype == "bf16" else "%s/%s" % (workload_label, dtype)
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get("workloads", {}).get(key)
        if rec and d.get("kernel_source_hash") == kernel_source_hash():
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


FP8_OVER_BF16 = 2.0      # nominal dense tensor rate ratio (4.5 vs 2.25 PFLOP/s)


def tensor_peak(peaks, dtype: str, key: str = "bf16_tflops") -> float:
    return peaks[key] * (FP8_OVER_BF16 if dtype == "fp8" else 1.0)


def algorithmic_bytes(w, dtype: str) -> int:
    """Compulsory HBM bytes of one launch: A and both weights read once, Y
    written once (element size 1 for FP8 inputs, 2 for BF16; Y is BF16)."""
    if dtype == "fp8":
        return w.M * w.K + 2 * w.K * w.N + 2 * w.M * w.N
    return w.roofline_bytes


def roofline_us(w, peaks, dtype: str = "bf16", key: str = "bf16_tflops"):
    return max(w.flops / (tensor_peak(peaks, dtype, key) * 1e12),
               algorithmic_bytes(w, dtype) / (peaks["hbm_gbs"] * 1e9)) * 1e6


def bound_of(w, peaks, dtype: str = "bf16") -> str:
    t_tc = w.flops / (tensor_peak(peaks, dtype) * 1e12)
    t_hbm = algorithmic_bytes(w, dtype) / (peaks["hbm_gbs"] * 1e9)
    return "tensor" if t_tc >= t_hbm else "hbm"


def roofline_entry(w, peaks, dtype: str, launch_s: float) -> dict:
    """The roofline numbers of one launch duration: the binding resource, the
    achieved rate against its measured peak (burst peak for a tensor-bound
    launch, also against the sustained one), and the fraction of roofline
    time (the slower of the tensor and HBM bounds)."""
    bound = bound_of(w, peaks, dtype)
    tflops = w.flops / launch_s / 1e12
    gbs = algorithmic_bytes(w, dtype) / launch_s / 1e9
    e = {"us_per_launch": launch_s * 1e6, "tflops": tflops, "bound": bound,
         "achieved_gbs": gbs, "frac_of_roofline_time": roofline_us(w, peaks, dtype) * 1e-6 / launch_s}
    if bound == "tensor":
        e["frac"] = tflops / tensor_peak(peaks, dtype)
        e["frac_of_sustained"] = tflops / tensor_peak(peaks, dtype, "bf16_tflops_sustained")
    else:
        e["frac"] = gbs / peaks["hbm_gbs"]
    return e


class ClockSampler:
    """Samples SM clock, power and throttle reasons with nvidia-smi while
    running; summaries are taken over any wall-clock window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 25):
        self.samples = []
        self.proc = None
        self.period_ms = period_ms
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                self.samples.append({
                    "t": time.time(), "sm": float(parts[2]), "sm_max": float(parts[3]),
                    "power": float(parts[4]), "hw": parts[6], "hw_thermal": parts[7],
                    "sw_thermal": parts[8], "sw_power_cap": parts[9]})
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0=None, t1=None, min_samples: int = 3):
        """Clocks over the wall-clock window [t0, t1]; with fewer than
        `min_samples` samples inside it, over the run so far (and says so)."""
        samples = list(self.samples)
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        window = "timed"
        sel = [s for s in samples if t0 is not None and t0 <= s["t"] <= t1]
        if len(sel) < min_samples:
            window = "whole run (fewer than %d samples inside the timed window)" % min_samples
            sel = samples[1:] or samples
        active = lambda v: v.lower() in ("active", "1", "yes")
        reasons = set()
        for s in sel:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
                if active(s[key]):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s["sm"] for s in sel),
                "sm_max_mhz": max(s["sm_max"] for s in sel),
                "power_w_median": statistics.median(s["power"] for s in sel),
                "power_w_max": max(s["power"] for s in sel),
                "samples": len(sel), "period_ms": self.period_ms, "window": window,
                "reasons": sorted(reasons)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a scalar over all ranks (identity for a single process)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world <= 1:
        return
    import torch
    import torch.distributed as dist
    t = torch.zeros(1, device=device)
    dist.all_reduce(t)


def aggregate_value(flops_per_step: float, steps: int, world: int, elapsed_max_s: float) -> float:
    """Whole-job TFLOP/s of replicas: every rank's FLOPs over the slowest
    rank's time."""
    return flops_per_step * steps * world / elapsed_max_s / 1e12


def column_slice(N: int, world: int, rank: int, granule: int = TILE_COLS):
    """Columns [c0, c1) of Y (and of W1, W2) that rank `rank` computes in the
    column-parallel split: whole 128-column tiles dealt out as evenly as
    possible, the last slice ending at N. Every slice width is a multiple of
    8 (N is), so each rank's problem meets the library's requirements."""
    tiles = -(-N // granule)
    if world > tiles:
        raise ValueError("column split: %d ranks for %d column tiles" % (world, tiles))
    t0 = rank * tiles // world
    t1 = (rank + 1) * tiles // world
    return t0 * granule, min(t1 * granule, N)


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun_command(n: int, argv) -> list:
    """The command that starts n ranks of this script on this node, one
    process per GPU (rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            "--nproc-per-node=%d" % n, "--master-addr", "127.0.0.1",
            "--master-port", str(free_port()), os.path.abspath(__file__)] + list(argv)


# ----------------------------------------------------------------------------- CPU oracle legs
def oracle_inputs(w, dtype: str):
    """The workload's inputs as the oracle takes them: (A, W1, W2) BF16 bits,
    or (A8, W1_8, W2_8, s_a, s_w1, s_w2) for FP8."""
    import workloads
    return workloads.make_inputs_fp8(w) if dtype == "fp8" else workloads.make_inputs(w)


def oracle_sample_rate(w, inputs, rows: int, cols: int, threads: int = 0):
    """Times the oracle on `rows` rows x `cols` columns; returns (seconds, flops)."""
    import numpy as np

    import oracle
    rng = np.random.Generator(np.random.PCG64(77))
    r = np.sort(rng.choice(w.M, size=min(rows, w.M), replace=False))
    fn = oracle.swiglu_up_fp8 if len(inputs) == 6 else oracle.swiglu_up
    t0 = time.perf_counter()
    fn(*inputs, rows=r, cols=(0, cols), nthreads=threads)
    dt = time.perf_counter() - t0
    return dt, 4.0 * len(r) * cols * w.K


def cpu_baseline(w, inputs, target_s: float = 12.0):
    """The oracle as it stands, on every host core, on a bounded row sample."""
    cores = len(os.sched_getaffinity(0))
    dt, fl = oracle_sample_rate(w, inputs, rows=cores, cols=w.N)
    rows_per_s = cores / dt
    rows = int(min(w.M, max(cores, (target_s - dt) * rows_per_s)))
    rows = max(cores, rows // cores * cores)
    dt2, fl2 = oracle_sample_rate(w, inputs, rows=rows, cols=w.N)
    return {"value": fl2 / dt2 / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d of %d rows x all %d columns (K=%d), %.1f s" % (rows, w.M, w.N, w.K, dt2)}


def run_reference(args, w):
    """Reference arm: the CPU oracle timed on this host's cores, one bounded
    sample of the workload per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    inputs = oracle_inputs(w, args.dtype)
    cores = len(os.sched_getaffinity(0))
    rows = min(cores, w.M)
    # size the per-step column block so that warmup + steps fit the budget
    dt, _ = oracle_sample_rate(w, inputs, rows=rows, cols=min(w.N, 256))
    per_col = dt / min(w.N, 256)
    budget = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    cols = int(max(8, min(w.N, budget / max(per_col, 1e-9))) // 8 * 8)
    for _ in range(args.warmup):
        oracle_sample_rate(w, inputs, rows=rows, cols=cols)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        _, fl = oracle_sample_rate(w, inputs, rows=rows, cols=cols)
        flops += fl
    el = time.perf_counter() - t0
    value = flops / el / 1e12
    sample = "%d rows x %d columns (K=%d) of the %dx%d output per step" % (rows, cols, w.K, w.M, w.N)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, None, args.dtype),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def fusion_efficiency(w, t_unfused_s: float, t_fused_s: float, hbm_gbs: float) -> float:
    """Time the fusion saved over the time the HBM traffic it removes would
    take at the measured copy bandwidth. The removed traffic is the pages'
    count ("Tile-Level Activation Overlap for Efficient LLM Inference",
    technical summary, contributions and results): Gate and Up each written
    and read once in BF16, 8*M*N bytes. Above 1 means the fused kernel also
    gains from overlap (the summary reports this for its Kernel-2)."""
    return (t_unfused_s - t_fused_s) / (8.0 * w.M * w.N / (hbm_gbs * 1e9))


# ----------------------------------------------------------------------------- GPU pieces
class Problem:
    """One workload resident on the GPU: R rotating sets of A, packed weights,
    Y and workspace (R sized so the sets exceed twice the L2), and the
    forward call over set j. `n_cols` < N: this rank's column slice."""

    def __init__(self, sg, w, dtype, dev, A_d, Wp, scales=None, n_cols=None):
        import torch
        self.sg, self.w, self.dtype, self.dev = sg, w, dtype, dev
        self.fp8 = dtype == "fp8"
        self.N = w.N if n_cols is None else n_cols
        self.scales = scales
        a_elem = 1 if self.fp8 else 2
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        per_set = w.M * w.K * a_elem + Wp.numel() + w.M * self.N * 2
        self.R = max(2, -(-2 * l2 // per_set))
        self.As = [A_d] + [A_d.clone() for _ in range(self.R - 1)]
        self.Wps = [Wp] + [Wp.clone() for _ in range(self.R - 1)]
        self.Ys = [torch.empty(w.M, self.N, dtype=torch.bfloat16, device=dev) for _ in range(self.R)]
        ws = (sg.swiglu_workspace_bytes_fp8 if self.fp8 else sg.swiglu_workspace_bytes)(
            w.M, self.N, w.K)
        self.Wss = [torch.zeros(max(ws, 16), dtype=torch.uint8, device=dev) if ws else None
                    for _ in range(self.R)]
        self.l2_note = "rotating %d input sets (%.0f MB total, > 2x the %.0f MB L2)" % (
            self.R, self.R * per_set / 1e6, l2 / 1e6)

    def forward(self, j, stream):
        j %= self.R
        if self.fp8:
            s_a, s_w1, s_w2 = self.scales
            self.sg.swiglu_up_forward_fp8(self.As[j], self.Wps[j], self.N, s_a, s_w1, s_w2,
                                          Y=self.Ys[j], workspace=self.Wss[j], stream=stream)
        else:
            self.sg.swiglu_up_forward(self.As[j], self.Wps[j], self.N, Y=self.Ys[j],
                                      workspace=self.Wss[j], stream=stream)

    def capture(self, n, dev):
        """A CUDA graph of n forward calls over the rotating sets (the calls
        go through the same public entry point)."""
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream(dev)
            for i in range(n):
                self.forward(i, cs)
        return g


def pack_problem(sg, w, dtype, dev, inputs, split=None):
    """Device copies of the inputs, packed weights (of this rank's column
    slice when `split` = (c0, c1)) and the rotating sets. `inputs` are host
    arrays (workloads' recipe) or device tensors (make_inputs_device)."""
    import numpy as np
    import torch
    from tests.parity import to_device_bf16
    fp8 = dtype == "fp8"
    c0, c1 = split if split else (0, w.N)
    if fp8:
        A, W1, W2, s_a, s_w1, s_w2 = inputs
        if isinstance(A, np.ndarray):
            A_d = torch.from_numpy(A).to(dev)
            W1d, W2d = torch.from_numpy(W1).to(dev), torch.from_numpy(W2).to(dev)
        else:
            A_d, W1d, W2d = A, W1, W2
        Wp = sg.swiglu_pack_weights_fp8(W1d[:, c0:c1].contiguous(), W2d[:, c0:c1].contiguous())
        scales = (s_a, s_w1, s_w2)
    else:
        A, W1, W2 = inputs
        if isinstance(A, np.ndarray):
            A_d, W1d, W2d = to_device_bf16(A, dev), to_device_bf16(W1, dev), to_device_bf16(W2, dev)
        else:
            A_d, W1d, W2d = A, W1, W2
        Wp = sg.swiglu_pack_weights(W1d[:, c0:c1].contiguous(), W2d[:, c0:c1].contiguous())
        scales = None
    del W1d, W2d
    return Problem(sg, w, dtype, dev, A_d, Wp, scales, n_cols=c1 - c0)


def replay_window(graphs, stream, dev, min_s: float):
    """Replays `graphs` (a list replayed in order = one round) until at least
    `min_s` seconds of GPU time have passed; the number of rounds is fixed
    from one untimed round first. Returns (seconds, rounds, wall t0, wall t1)."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for g in graphs:
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    one = max(e0.elapsed_time(e1) * 1e-3, 1e-7)
    rounds = max(1, int(-(-1.1 * min_s // one)))   # 10% margin: a round may run faster
    wall0 = time.time()
    e0.record(stream)
    for _ in range(rounds):
        for g in graphs:
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    return e0.elapsed_time(e1) * 1e-3, rounds, wall0, wall1


def graph_launches(R: int, launch_s: float, target_s: float = 2e-3, cap: int = 256) -> int:
    """Launches per captured graph: enough that one replay lasts about
    `target_s`, a multiple of the R rotating sets, at most `cap`."""
    n = max(1, int(target_s / max(launch_s, 1e-7)))
    n = max(R, -(-n // R) * R)
    return min(n, max(R, cap // R * R))


def sweep(sg, peaks, dtype, dev, stream, sampler, window_s: float, labels):
    """Every workload timed on its own: inputs drawn on the GPU (seeded, the
    workloads' distributions), packed, R rotating sets, a CUDA graph of
    launches replayed for `window_s` seconds; one entry per workload."""
    import torch

    import workloads
    out = []
    for label in labels:
        w = workloads.BY_LABEL[label]
        inputs = workloads.make_inputs_device(w, dev, fp8=dtype == "fp8")
        p = pack_problem(sg, w, dtype, dev, inputs)
        del inputs
        for i in range(3):
            p.forward(i, stream)
        torch.cuda.synchronize(dev)
        sg.swiglu_check_device_status(stream)
        n = graph_launches(p.R, roofline_us(w, peaks, dtype) * 1e-6)
        g = p.capture(n, dev)
        el, rounds, t0, t1 = replay_window([g], stream, dev, window_s)
        sg.swiglu_check_device_status(stream)
        e = {"workload": label, "name": w.name, "M": w.M, "K": w.K, "N": w.N,
             "variant": w.variant, "launches": n * rounds}
        e.update(roofline_entry(w, peaks, dtype, el / (n * rounds)))
        e["clocks"] = sampler.summary(t0, t1, min_samples=2)
        out.append(e)
        del g, p
        torch.cuda.empty_cache()
    return out


DOWN_SWEEP_LABELS = ("0", "1", "3", "5", "6", "7", "9", "10", "11")


def down_sweep(sg, dev, stream, sampler, window_s: float, labels=DOWN_SWEEP_LABELS):
    """The down-projection out = Y W3 (Y [M, N], W3 [N, K]) of the gated MLP
    at the workloads' shapes, this library's kernel (whichever it picks)
    against cuBLAS (torch.matmul) on the same rotating inputs (Y ~ N(0, 1),
    W3 ~ N(0, 1/N), drawn on the GPU, seeded): CUDA graphs replayed for
    `window_s` seconds each, in the order ours, cuBLAS, ours, cuBLAS, so that
    neither side gets the cooler GPU; each side's number is its faster
    window, with the SM clock of that window. BF16."""
    import torch

    import workloads
    out = []
    for label in labels:
        w = workloads.BY_LABEL[label]
        M, N, K = w.M, w.N, w.K
        per = 2 * (M * N + N * K + M * K)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        R = max(2, min(8, int(2.5 * l2 // per) + 1))   # the sets exceed twice the L2
        g = torch.Generator(device=dev)
        g.manual_seed(7000 + w.seed_index)
        Ys = [torch.randn(M, N, generator=g, device=dev).to(torch.bfloat16) for _ in range(R)]
        W3s = [(torch.randn(N, K, generator=g, device=dev) * N ** -0.5).to(torch.bfloat16)
               for _ in range(R)]
        W3ps = [sg.swiglu_pack_down_weights(x) for x in W3s]
        Os = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        ws = sg.swiglu_down_workspace_bytes(M, N, K)
        Wss = [torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev) for _ in range(R)]

        def ours(i, st):
            j = i % R
            sg.swiglu_down_forward(Ys[j], W3ps[j], K, out=Os[j],
                                   workspace=Wss[j] if ws else None, stream=st)

        def cublas(i, st):
            j = i % R
            torch.matmul(Ys[j], W3s[j], out=Os[j])

        flops = 2.0 * M * N * K
        graphs = {}
        for name, fn in (("ours", ours), ("cublas", cublas)):
            with torch.cuda.stream(stream):
                for i in range(R):
                    fn(i, stream)
            torch.cuda.synchronize(dev)
            est = max(flops / 1.5e15, per / R / 6e12)
            n = graph_launches(R, est)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                cs = torch.cuda.current_stream(dev)
                for i in range(n):
                    fn(i, cs)
            graphs[name] = (gr, n)
        best = {}
        for name in ("ours", "cublas", "ours", "cublas"):
            gr, n = graphs[name]
            el, rounds, t0, t1 = replay_window([gr], stream, dev, window_s)
            us = el / (n * rounds) * 1e6
            if name not in best or us < best[name][0]:
                best[name] = (us, sampler.summary(t0, t1, min_samples=2))
        sg.swiglu_check_device_status(stream)
        e = {"workload": label, "name": w.name, "M": M, "N": N, "K": K}
        for name in ("ours", "cublas"):
            us, clk = best[name]
            e[name] = {"us": us, "tflops": flops / (us * 1e-6) / 1e12, "clocks": clk}
        e["ours_over_cublas_time"] = best["ours"][0] / best["cublas"][0]
        out.append(e)
        del graphs, Ys, W3s, W3ps, Os, Wss
        torch.cuda.empty_cache()
    return out


def mlp_decode_context(sg, peaks, dev, stream, sampler, window_s: float, label: str = "3"):
    """The whole gated MLP at a decode shape (default the 7B workload with 16
    tokens): out = (SiLU(A W1) * (A W2)) W3, a stream of the three weight
    matrices. This library's whole-MLP call (the fused up-projection, then
    the decode down-projection kernel), the fused up-projection followed by
    torch.matmul (cuBLAS), and eager PyTorch (three cuBLAS GEMMs and
    silu * mul), each as a CUDA graph of launches over rotating inputs
    (seeded, drawn on the GPU: A ~ N(0, 1), W1 and W2 ~ N(0, 1/K), W3 ~
    N(0, 1/N)) replayed for `window_s` seconds, in two alternating rounds,
    the faster window of each with its SM clock; plus the HBM roofline of
    the weight stream (3 K N BF16 values) at the measured copy rate. BF16."""
    import torch
    import torch.nn.functional as F

    import workloads
    w = workloads.BY_LABEL[label]
    M, K, N = w.M, w.K, w.N
    per = 2 * (M * K + 3 * K * N + 2 * M * N + M * K)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, min(8, int(2.5 * l2 // per) + 1))   # the sets exceed twice the L2
    g = torch.Generator(device=dev)
    g.manual_seed(9000 + w.seed_index)

    def rnd(rows, cols, scale):
        return (torch.randn(rows, cols, generator=g, device=dev) * scale).to(torch.bfloat16)

    As = [rnd(M, K, 1.0) for _ in range(R)]
    W1s = [rnd(K, N, K ** -0.5) for _ in range(R)]
    W2s = [rnd(K, N, K ** -0.5) for _ in range(R)]
    W3s = [rnd(N, K, N ** -0.5) for _ in range(R)]
    Wps = [sg.swiglu_pack_weights(W1s[j], W2s[j]) for j in range(R)]
    W3ps = [sg.swiglu_pack_down_weights(W3s[j]) for j in range(R)]
    Gs = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    Us = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    Ys = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    Os = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    mws = sg.swiglu_mlp_workspace_bytes(M, N, K)
    uws = sg.swiglu_workspace_bytes(M, N, K)
    MWs = [torch.zeros(max(mws, 256), dtype=torch.uint8, device=dev) for _ in range(R)]
    UWs = [torch.zeros(max(uws, 256), dtype=torch.uint8, device=dev) for _ in range(R)]

    def fused(i, st):
        j = i % R
        sg.swiglu_mlp_forward(As[j], Wps[j], W3ps[j], N, Y=Ys[j], out=Os[j],
                              workspace=MWs[j] if mws else None, stream=st)

    def fused_cublas_down(i, st):
        j = i % R
        sg.swiglu_up_forward(As[j], Wps[j], N, Y=Ys[j], workspace=UWs[j] if uws else None,
                             stream=st)
        torch.matmul(Ys[j], W3s[j], out=Os[j])

    def eager(i, st):
        j = i % R
        torch.matmul(As[j], W1s[j], out=Gs[j])
        torch.matmul(As[j], W2s[j], out=Us[j])
        torch.mul(F.silu(Gs[j]), Us[j], out=Ys[j])
        torch.matmul(Ys[j], W3s[j], out=Os[j])

    variants = (("fused", fused), ("fused_up_cublas_down", fused_cublas_down), ("eager", eager))
    weight_bytes = 3 * K * N * 2
    roof_us = weight_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    graphs = {}
    for name, fn in variants:
        with torch.cuda.stream(stream):
            for i in range(R):
                fn(i, stream)
        torch.cuda.synchronize(dev)
        n = graph_launches(R, roof_us * 1e-6)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            cs = torch.cuda.current_stream(dev)
            for i in range(n):
                fn(i, cs)
        graphs[name] = (gr, n)
    best = {}
    for _ in range(2):
        for name, _fn in variants:
            gr, n = graphs[name]
            el, rounds, t0, t1 = replay_window([gr], stream, dev, window_s)
            us = el / (n * rounds) * 1e6
            if name not in best or us < best[name][0]:
                best[name] = (us, sampler.summary(t0, t1, min_samples=2))
    sg.swiglu_check_device_status(stream)
    e = {"workload": label, "name": w.name, "M": M, "K": K, "N": N,
         "weight_bytes": weight_bytes, "hbm_roofline_us": roof_us}
    for name, _fn in variants:
        us, clk = best[name]
        e[name] = {"us": us, "frac_of_hbm_roofline": roof_us / us, "clocks": clk}
    e["mlp_speedup_over_eager"] = best["eager"][0] / best["fused"][0]
    e["what"] = ("whole gated MLP at a decode shape, CUDA graphs over rotating inputs; fused = "
                 "swiglu_mlp_forward (fused up-projection + decode down-projection kernel)")
    del graphs, As, W1s, W2s, W3s, Wps, W3ps, Gs, Us, Ys, Os, MWs, UWs
    torch.cuda.empty_cache()
    return e


ABLATION_FORMS = (
    # (packed layout, kernel variant, schedule form); "auto" = the library's choice
    [(layout, "auto", mode) for layout in ("blocked", "interleaved")
     for mode in ("auto", "dp", "split", "sk", "sk-tail")] +
    [(layout, variant, "auto") for layout in ("blocked", "interleaved") for variant in ("1sm", "2sm")])


def ablation(sg, peaks, dev, stream, sampler, window_s: float, labels, forms=ABLATION_FORMS):
    """The schedule ablation (the pages' Kernel-1 / Kernel-2 trade on this
    GPU): for every workload, each packed layout (blocked 128-row halves, or
    the pages' column interleave) x kernel (1-SM, CTA pairs) x work split
    (whole tiles, column sub-tiles for the last wave, stream-K), forced
    through SWIGLU_FUSED_VARIANT / SWIGLU_SCHEDULE, timed like the sweep on
    the same rotating inputs; plus the unfused cuBLAS path for the fusion
    efficiency. BF16."""
    import torch
    import torch.nn.functional as F

    import workloads
    out = []
    saved = {k: os.environ.get(k) for k in ("SWIGLU_FUSED_VARIANT", "SWIGLU_SCHEDULE")}
    try:
        for label in labels:
            w = workloads.BY_LABEL[label]
            A, W1, W2 = workloads.make_inputs_device(w, dev)
            l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            per_set = 2 * (w.M * w.K + 4 * w.K * w.N + w.M * w.N)
            R = max(2, -(-2 * l2 // per_set))
            As = [A] + [A.clone() for _ in range(R - 1)]
            Ys = [torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
            packed = {"blocked": sg.swiglu_pack_weights(W1, W2),
                      "interleaved": sg.swiglu_pack_weights_interleaved(W1, W2)}
            Wps = {k: [v] + [v.clone() for _ in range(R - 1)] for k, v in packed.items()}
            fwd = {"blocked": sg.swiglu_up_forward, "interleaved": sg.swiglu_up_forward_interleaved}
            entry = {"workload": label, "name": w.name, "M": w.M, "K": w.K, "N": w.N, "forms": []}
            for layout, variant, mode in forms:
                for k, v in (("SWIGLU_FUSED_VARIANT", variant), ("SWIGLU_SCHEDULE", mode)):
                    if v == "auto":
                        os.environ.pop(k, None)
                    else:
                        os.environ[k] = v
                ws = sg.swiglu_workspace_bytes(w.M, w.N, w.K)
                Wss = [torch.zeros(ws, dtype=torch.uint8, device=dev) if ws else None
                       for _ in range(R)]

                def one(i, st, layout=layout, Wss=Wss):
                    j = i % R
                    fwd[layout](As[j], Wps[layout][j], w.N, Y=Ys[j], workspace=Wss[j], stream=st)

                for i in range(3):
                    one(i, stream)
                torch.cuda.synchronize(dev)
                sg.swiglu_check_device_status(stream)
                n = graph_launches(R, roofline_us(w, peaks) * 1e-6)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    cs = torch.cuda.current_stream(dev)
                    for i in range(n):
                        one(i, cs)
                # untimed half window first: the clock settles under this
                # form's load before the timed window
                replay_window([g], stream, dev, window_s / 2)
                el, rounds, t0, t1 = replay_window([g], stream, dev, window_s)
                sg.swiglu_check_device_status(stream)
                f = {"layout": layout, "variant": variant, "schedule": mode,
                     "workspace_bytes": ws, "launches": n * rounds}
                f.update(roofline_entry(w, peaks, "bf16", el / (n * rounds)))
                clk = sampler.summary(t0, t1, min_samples=1)
                f["sm_mhz"] = clk.get("sm_mhz")
                f["clock_samples"] = clk.get("samples")
                if f["sm_mhz"]:
                    # launch time x SM clock: comparable across power-capped clocks
                    f["ms_x_ghz"] = f["us_per_launch"] * f["sm_mhz"] * 1e-6
                entry["forms"].append(f)
                del g, Wss
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
            # the unfused path on the same rotating inputs
            W1s = [W1] + [W1.clone() for _ in range(R - 1)]
            W2s = [W2] + [W2.clone() for _ in range(R - 1)]

            def unfused(i):
                j = i % R
                torch.mul(F.silu(torch.matmul(As[j], W1s[j])), torch.matmul(As[j], W2s[j]),
                          out=Ys[j])

            with torch.cuda.stream(stream):
                for i in range(3):
                    unfused(i)
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                t_est = max(roofline_us(w, peaks) * 1e-6, 1e-6)
                reps = max(R, int(window_s / (2 * t_est)))
                for i in range(reps):
                    unfused(i)
                e1.record(stream)
                torch.cuda.synchronize(dev)
            t_unf = e0.elapsed_time(e1) * 1e-3 / reps
            entry["unfused_us"] = t_unf * 1e6
            for f in entry["forms"]:
                f["fusion_efficiency"] = fusion_efficiency(w, t_unf, f["us_per_launch"] * 1e-6,
                                                           peaks["hbm_gbs"])
                f["speedup_vs_unfused"] = t_unf / (f["us_per_launch"] * 1e-6)
            out.append(entry)
            del As, Ys, packed, Wps, W1s, W2s, A, W1, W2
            torch.cuda.empty_cache()
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return out


def run_ablation(args):
    """`bench.py --ablation`: one JSON line with the ablation of every workload."""
    import torch
    world, rank, local = dist_env()
    if world != 1:
        raise SystemExit("--ablation runs on one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from gemm_swiglu_mlp_gb300 import build as lib_build
    lib_build.build()
    import gemm_swiglu_mlp_gb300 as sg

    import workloads
    peaks, peaks_src = load_peaks()
    sampler = ClockSampler(local)
    time.sleep(0.3)
    labels = args.ablation_workloads.split(",") if args.ablation_workloads else [
        x.c for x in workloads.WORKLOADS]
    res = ablation(sg, peaks, dev, torch.cuda.current_stream(dev), sampler, args.sweep_window_s,
                   labels)
    sampler.stop()
    print(json.dumps({"ablation": res, "peaks": peaks, "peaks_source": peaks_src,
                      "kernel_source_hash": kernel_source_hash(), "device": device_info(dev),
                      "window_s": args.sweep_window_s}), flush=True)
    return 0


def time_unfused_context(w, W1, W2, As, Ys, R, dev, stream, steps, fused_value, hbm_gbs):
    """Context only (not this library): the unfused PyTorch path the pages
    compare against ("Tile-Level Activation Overlap for Efficient LLM
    Inference", Section 1: two GEMMs that write Gate and Up to HBM, then the
    activation), timed on the same rotating inputs: torch.matmul x2 (cuBLAS),
    then silu(g) * u in BF16."""
    import torch
    import torch.nn.functional as F
    from tests.parity import to_device_bf16
    w1 = to_device_bf16(W1, dev)
    w2 = to_device_bf16(W2, dev)
    W1s = [w1] + [w1.clone() for _ in range(R - 1)]
    W2s = [w2] + [w2.clone() for _ in range(R - 1)]

    def unfused_step(i):
        j = i % R
        g = torch.matmul(As[j], W1s[j])
        u = torch.matmul(As[j], W2s[j])
        torch.mul(F.silu(g), u, out=Ys[j])

    with torch.cuda.stream(stream):
        for i in range(5):
            unfused_step(i)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            unfused_step(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    el = e0.elapsed_time(e1) * 1e-3
    v = w.flops * steps / el / 1e12
    del W1s, W2s
    return {"value": v, "unit": UNIT, "ms_per_step": el / steps * 1e3, "steps": steps,
            "fused_speedup": fused_value / v,
            "fusion_efficiency": fusion_efficiency(w, el / steps, w.flops / (fused_value * 1e12),
                                                   hbm_gbs),
            "what": "torch.matmul(A, W1), torch.matmul(A, W2) (cuBLAS, Gate/Up written to HBM "
                    "in BF16), then silu(Gate) * Up in BF16; same rotating inputs"}


def time_mlp_context(w, W1, W2, sg, p, dev, stream, steps):
    """Context for the pages' Figure 1 ("Tile-Level Activation Overlap for
    Efficient LLM Inference", Section 1: SwiGLU and its intermediates as a
    share of MLP time): the whole gated MLP out = Y W3 with a synthetic
    down-projection W3 [N, K]. Fused: this library's whole-MLP call (the
    fused up-projection, then its own down-projection kernel), and for
    comparison the fused up-projection followed by torch.matmul (cuBLAS).
    Eager: three cuBLAS GEMMs and silu * mul, each also timed alone for the
    activation's share."""
    import torch
    import torch.nn.functional as F

    import workloads
    from tests.parity import to_device_bf16
    R, As, Wps, Ys, Wss = p.R, p.As, p.Wps, p.Ys, p.Wss
    w3 = to_device_bf16(workloads.make_W3(w), dev)
    w1 = to_device_bf16(W1, dev)
    w2 = to_device_bf16(W2, dev)
    W1s = [w1] + [w1.clone() for _ in range(R - 1)]
    W2s = [w2] + [w2.clone() for _ in range(R - 1)]
    W3s = [w3] + [w3.clone() for _ in range(R - 1)]
    G = [torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    U = [torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    O = [torch.empty(w.M, w.K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    W3ps = [sg.swiglu_pack_down_weights(W3s[j]) for j in range(R)]
    mlp_ws = max(1, sg.swiglu_mlp_workspace_bytes(w.M, w.N, w.K))
    MWs = [torch.zeros(mlp_ws, dtype=torch.uint8, device=dev) for _ in range(R)]

    def timed(fn):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps):
                fn(i)
            e1.record(stream)
            torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps  # ms

    ops = {
        "gate_gemm": lambda i: torch.matmul(As[i % R], W1s[i % R], out=G[i % R]),
        "up_gemm": lambda i: torch.matmul(As[i % R], W2s[i % R], out=U[i % R]),
        "silu_mul": lambda i: torch.mul(F.silu(G[i % R]), U[i % R], out=Ys[i % R]),
        "down_gemm": lambda i: torch.matmul(Ys[i % R], W3s[i % R], out=O[i % R]),
    }
    op_ms = {k: timed(f) for k, f in ops.items()}

    def eager(i):
        for f in ops.values():
            f(i)

    def fused(i):
        j = i % R
        sg.swiglu_mlp_forward(As[j], Wps[j], W3ps[j], w.N, Y=Ys[j], out=O[j], workspace=MWs[j],
                              stream=stream)

    def fused_cublas_down(i):
        j = i % R
        sg.swiglu_up_forward(As[j], Wps[j], w.N, Y=Ys[j], workspace=Wss[j], stream=stream)
        torch.matmul(Ys[j], W3s[j], out=O[j])

    def down(i):
        j = i % R
        sg.swiglu_down_forward(Ys[j], W3ps[j], w.K, out=O[j], workspace=MWs[j], stream=stream)

    # The whole-MLP variants and the two down-projections in alternating
    # rounds, the faster of two rounds each: timed one after the other, the
    # later ones ran on a warmer GPU at a lower clock under the power cap.
    def down_cublas(i):
        ops["down_gemm"](i)

    variants = (("eager", eager), ("fused", fused), ("fused_cublas", fused_cublas_down),
                ("down", down), ("down_cublas", down_cublas))
    best = {}
    for _ in range(2):
        for name, fn in variants:
            t = timed(fn)
            best[name] = min(t, best.get(name, t))
    eager_ms, fused_ms, fused_cublas_ms = best["eager"], best["fused"], best["fused_cublas"]
    down_ms = best["down"]
    mlp_flops = w.flops + 2 * w.M * w.N * w.K
    down_flops = 2 * w.M * w.N * w.K
    del W1s, W2s, W3s, W3ps, MWs, G, U, O
    return {"eager_mlp_ms": eager_ms, "fused_mlp_ms": fused_ms,
            "mlp_speedup": eager_ms / fused_ms,
            "fused_mlp_tflops": mlp_flops / (fused_ms * 1e-3) / 1e12,
            "fused_up_cublas_down_mlp_ms": fused_cublas_ms,
            "down_ms": down_ms, "down_tflops": down_flops / (down_ms * 1e-3) / 1e12,
            "down_cublas_ms": best["down_cublas"],
            "eager_op_ms": op_ms,
            "activation_share_of_eager_mlp": op_ms["silu_mul"] / sum(op_ms.values()),
            "what": "out = (SiLU(A W1) * (A W2)) W3, W3 [N, K] ~ N(0, 1/N) synthetic; fused = this "
                    "library's swiglu_mlp_forward (fused up-projection + its down-projection "
                    "kernel); eager = 3 cuBLAS GEMMs + silu*mul (Figure 1 of the pages measures "
                    "this share on H100; eager_op_ms times each op alone, one after the other); "
                    "down_* = the down-projection alone, this library's kernel and cuBLAS; the "
                    "MLP variants and down_* in two alternating rounds, the faster of each"}


def config_of(w, l2_note, dtype: str = "bf16", split: str = "replicas", world: int = 1):
    io = ("FP8 E4M3 in (per-tensor amax/448 scales), BF16 out" if dtype == "fp8"
          else "BF16 in/out")
    c = {"workload": "%s: M=%d tokens, K=%d, N=%d, A~N(0,1), W1/W2~N(0,1/K), %s, FP32 accumulate"
                     % (w.name, w.M, w.K, w.N, io),
         "M": w.M, "K": w.K, "N": w.N,
         "parallelism": ("column-parallel x%d (each rank packs and computes its slice of the N "
                         "columns, no collective)" % world) if split == "columns" else
                        "replicas (each rank runs the whole workload, no collective)"}
    if l2_note:
        c["l2"] = l2_note
    return c


# ----------------------------------------------------------------------------- GPU arm
def run_gb300(args, w):
    import dataclasses

    import numpy as np
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from gemm_swiglu_mlp_gb300 import build as lib_build
    lib_build.build()
    import gemm_swiglu_mlp_gb300 as sg

    peaks, peaks_src = load_peaks()
    fp8 = args.dtype == "fp8"
    columns = args.split == "columns" and world > 1
    inputs = oracle_inputs(w, args.dtype)
    split = column_slice(w.N, world, rank) if columns else None
    p = pack_problem(sg, w, args.dtype, dev, inputs, split)
    # this rank's share of the work (its column slice, or the whole workload)
    w_rank = dataclasses.replace(w, N=p.N)
    job_flops_per_step = w.flops if columns else w.flops * world
    stream = torch.cuda.current_stream(dev)

    sampler = ClockSampler(local)
    time.sleep(0.3)
    for i in range(args.warmup):
        p.forward(i, stream)
    torch.cuda.synchronize(dev)
    sg.swiglu_check_device_status(stream)

    # ---- device-resident timed region: K launches back to back, one per step.
    # Events only at the two ends: the average launch duration is the region
    # over K (it includes any gap between launches, so it is conservative),
    # and nothing between launches keeps one call's launch from overlapping
    # the previous call's tail. By default the launches are replayed from CUDA
    # graphs (captured through the same public call, rotating over the same
    # buffers), so that the host's per-call cost does not set the pace of
    # launches shorter than it; `--launch direct` issues K calls instead.
    K = args.steps
    R = p.R
    graphs, timing, g_main, gl = [], "direct: %d calls" % K, None, 0
    if args.launch == "graph":
        try:
            gl = min(K, R * max(1, 256 // R))
            g_main = p.capture(gl, dev)
            graphs = [g_main] * (K // gl)
            if K % gl:
                graphs.append(p.capture(K % gl, dev))
            g_main.replay()                      # one untimed replay
            torch.cuda.synchronize(dev)
            sg.swiglu_check_device_status(stream)
            timing = "CUDA graph of %d launches replayed %d times%s" % (
                gl, K // gl, (" + one of %d" % (K % gl)) if K % gl else "")
        except Exception as exc:               # capture unavailable: direct calls
            graphs, timing, g_main = [], "direct: %d calls (graph capture failed: %s)" % (K, exc), None
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_begin.record(stream)
    if graphs:
        for g in graphs:
            g.replay()
    else:
        for i in range(K):
            p.forward(i, stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(world, dev)
    elapsed = t_begin.elapsed_time(t_end) * 1e-3
    sg.swiglu_check_device_status(stream)
    elapsed_max = max_over_ranks(elapsed, world, dev)
    value = job_flops_per_step * K / elapsed_max / 1e12
    avg_launch = elapsed / K
    clocks_timed = sampler.summary(wall0, wall1)

    # ---- sustained: the headline launch replayed for >= args.sustained_s
    # seconds, so that the clocks settle under the power cap and the sampler
    # sees the load; reported against the sustained BF16 peak as well.
    sustained = None
    if g_main is not None and args.sustained_s > 0:
        el, rounds, s0, s1 = replay_window([g_main], stream, dev, args.sustained_s)
        sg.swiglu_check_device_status(stream)
        n_l = rounds * gl
        sustained = roofline_entry(w_rank, peaks, args.dtype, el / n_l)
        sustained.update({"launches": n_l, "seconds": el, "clocks": sampler.summary(s0, s1, 10),
                          "what": "the timed region's CUDA graph replayed back to back for "
                                  ">= %.1f s of GPU time" % args.sustained_s})

    # ---- L2-warm context: the same launches on one input set, so A and the
    # weights stay in L2 from call to call when they fit (not the headline).
    Kw = min(K, 2000)
    w0 = torch.cuda.Event(enable_timing=True)
    w1_ = torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        p.forward(0, stream)
    w0.record(stream)
    for _ in range(Kw):
        p.forward(0, stream)
    w1_.record(stream)
    torch.cuda.synchronize(dev)
    warm_s = w0.elapsed_time(w1_) * 1e-3 / Kw
    l2_warm = {"avg_launch_us": warm_s * 1e6, "tflops": w_rank.flops / warm_s / 1e12, "steps": Kw,
               "what": "one input set reused every call (operands L2-resident when they fit)"}

    # ---- end to end through the public API, as a serving loop runs it: every
    # step copies its A from pinned host memory, runs the forward and copies
    # its Y back to pinned host memory. Copy-in, compute and copy-out of
    # consecutive steps overlap on three streams; slot j's device buffers are
    # reused only after step j-R has finished with them (events).
    Ke = min(K, 2000)
    A_np = inputs[0]
    A_h = (torch.from_numpy(A_np) if fp8 else
           torch.from_numpy(A_np.view(np.int16)).view(torch.bfloat16)).pin_memory()
    Y_h = [torch.empty((w.M, p.N), dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(R)]
    ev_comp = [torch.cuda.Event() for _ in range(R)]
    ev_out = [torch.cuda.Event() for _ in range(R)]
    used = [False] * R

    def e2e_step(i):
        j = i % R
        if used[j]:
            s_in.wait_event(ev_comp[j])          # A slot free once its compute is done
        with torch.cuda.stream(s_in):
            p.As[j].copy_(A_h, non_blocking=True)
        ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        if used[j]:
            stream.wait_event(ev_out[j])         # Y slot free once its copy-out is done
        p.forward(j, stream)
        ev_comp[j].record(stream)
        s_out.wait_event(ev_comp[j])
        with torch.cuda.stream(s_out):
            Y_h[j].copy_(p.Ys[j], non_blocking=True)
        ev_out[j].record(s_out)
        used[j] = True

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    ew0 = time.time()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(Ke):
        e2e_step(i)
    for st_ in (s_in, s_out):
        done = torch.cuda.Event()
        done.record(st_)
        stream.wait_event(done)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ew1 = time.time()
    e2e_clocks = sampler.summary(ew0, ew1)
    barrier(world, dev)
    e_el = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world, dev)
    e2e_value = job_flops_per_step * Ke / e_el / 1e12
    sg.swiglu_check_device_status(stream)
    # the pipelined loop returned the right bytes: the last Y equals the device result
    y_check = Y_h[(Ke - 1) % R]
    if not torch.equal(y_check.to(dev), p.Ys[(Ke - 1) % R]):
        raise RuntimeError("e2e loop: copied-out Y differs from the device result")
    del Y_h, A_h

    unfused = mlp = None
    if not args.no_context and not fp8 and not columns:
        _, W1, W2 = inputs
        unfused = time_unfused_context(w, W1, W2, p.As, p.Ys, R, dev, stream, min(K, 2000),
                                       w.flops / avg_launch / 1e12, peaks["hbm_gbs"])
        mlp = time_mlp_context(w, W1, W2, sg, p, dev, stream, min(K, 500))
        torch.cuda.empty_cache()

    l2_note = p.l2_note
    sweep_out = None
    if world == 1 and not args.no_sweep:
        del p
        torch.cuda.empty_cache()
        import workloads
        labels = [x.c for x in workloads.WORKLOADS]
        sweep_out = sweep(sg, peaks, args.dtype, dev, stream, sampler, args.sweep_window_s, labels)
    down_out = mlp_decode = None
    if world == 1 and not args.no_context and not args.no_sweep and not fp8:
        down_out = down_sweep(sg, dev, stream, sampler, min(args.sweep_window_s, 0.15))
        mlp_decode = mlp_decode_context(sg, peaks, dev, stream, sampler,
                                        min(args.sweep_window_s, 0.15))
    sampler.stop()

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    # the roofline of the kernel as launched: the whole workload, or (column
    # split) this rank's slice of it
    bound = bound_of(w_rank, peaks, args.dtype)
    abytes = algorithmic_bytes(w_rank, args.dtype)
    if bound == "tensor":
        achieved = w_rank.flops / avg_launch / 1e12
        peak = tensor_peak(peaks, args.dtype)
        src = ("%s burst bf16 x %g (nominal fp8/bf16 ratio)" % (peaks_src, FP8_OVER_BF16) if fp8
               else "%s burst bf16" % peaks_src)
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": src,
                "frac_of_sustained": achieved / tensor_peak(peaks, args.dtype,
                                                            "bf16_tflops_sustained")}
    else:
        achieved = abytes / avg_launch / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": "%s copy bandwidth" % peaks_src}
    roof["traffic"] = recorded_traffic(w.c, args.dtype) if not columns else None
    roof["algorithmic_per_launch"] = w_rank.flops if bound == "tensor" else abytes
    roof["avg_launch_us"] = avg_launch * 1e6
    roof["frac_of_roofline_time"] = roofline_us(w_rank, peaks, args.dtype) * 1e-6 / avg_launch

    a_elem = 1 if fp8 else 2
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": elapsed_max / K * 1e3, "higher_is_better": True,
        "scaling": "strong" if columns else "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3" if fp8 else "bf16", "data": "synthetic",
        "config": dict(config_of(w, l2_note, args.dtype, "columns" if columns else "replicas",
                                 world), timing=timing),
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": w.M * w.K * a_elem,
                "d2h_bytes_per_step": w.M * w_rank.N * 2, "steps": Ke,
                "ms_per_step": e_el / Ke * 1e3,
                "how": "pinned host A -> device, forward, device Y -> pinned host, every step; "
                       "copy-in, compute and copy-out of consecutive steps overlap on 3 streams",
                "clocks": e2e_clocks},
        "gpu_launches": K, "clocks": clocks_timed, "context_l2_warm": l2_warm,
        "device": device_info(dev),
    }
    if sustained is not None:
        line["context_sustained"] = sustained
    if sweep_out is not None:
        line["sweep"] = sweep_out
    if unfused is not None:
        line["context_unfused_torch"] = unfused
    if mlp is not None:
        line["context_mlp"] = mlp
    if down_out is not None:
        line["context_down"] = down_out
    if mlp_decode is not None:
        line["context_mlp_decode"] = mlp_decode
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inputs)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   help="workload label (workloads.WORKLOADS), default 11 = Qwen-2.5-72B M=8192")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-context", action="store_true",
                   help="skip timing the unfused PyTorch path and the whole MLP (context only)")
    p.add_argument("--no-sweep", action="store_true", help="skip the per-workload sweep")
    p.add_argument("--sweep-window-s", type=float, default=0.25,
                   help="GPU seconds of replayed launches per sweep workload")
    p.add_argument("--sustained-s", type=float, default=1.0,
                   help="GPU seconds of the sustained window (0: skip)")
    p.add_argument("--launch", choices=("graph", "direct"), default="graph",
                   help="timed region: replay CUDA graphs of the calls (default) or call K times")
    p.add_argument("--dtype", choices=("bf16", "fp8"), default="bf16",
                   help="input type: bf16, or fp8 (E4M3 with per-tensor scales)")
    p.add_argument("--variant", choices=("auto", "1sm", "2sm"), default="auto",
                   help="fused kernel: auto (2-SM pairs for M >= 256), or force one (ablation)")
    p.add_argument("--ablation", action="store_true",
                   help="instead of the benchmark: time every workload under each packed layout, "
                        "kernel variant and schedule form (one JSON line)")
    p.add_argument("--ablation-workloads", default="",
                   help="comma-separated workload labels for --ablation (default: all)")
    p.add_argument("--split", choices=("replicas", "columns"), default="replicas",
                   help="N > 1: every rank runs the whole workload (replicas), or its slice of "
                        "the output columns (column-parallel)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.gpus < 1:
        p.error("--gpus must be at least 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return subprocess.call(torchrun_command(args.gpus, argv))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        p.error("--gpus %d but WORLD_SIZE=%d" % (args.gpus, world))
    import workloads
    w = workloads.BY_LABEL[args.workload]
    if args.variant != "auto":
        os.environ["SWIGLU_FUSED_VARIANT"] = args.variant
    if args.impl == "reference":
        return run_reference(args, w)
    if args.ablation:
        return run_ablation(args)
    return run_gb300(args, w)


if __name__ == "__main__":
    sys.exit(main())
