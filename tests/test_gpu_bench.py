"""bench.py on the GPU: the JSON line the benchmark contract asks for."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_bench_prints_one_contract_line(dtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "0", "--steps", "50",
           "--warmup", "3", "--no-cpu-baseline", "--no-context", "--dtype", dtype,
           "--sustained-s", "0.2", "--sweep-window-s", "0.05"]
    if dtype == "fp8":
        cmd.append("--no-sweep")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    r = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in r, key
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r["roofline"], key
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in r["e2e"], key
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in r["clocks"], key
    assert r["device"]["sm_count"] > 0 and r["device"]["name"]
    assert r["value"] > 0 and r["e2e"]["value"] > 0 and r["gpu_launches"] == 50
    assert r["roofline"]["bound"] == "hbm"          # the 0.5B shape streams weights
    assert r["dtype"] == ("fp8-e4m3" if dtype == "fp8" else "bf16")
    assert r["e2e"]["h2d_bytes_per_step"] == 128 * 896 * (1 if dtype == "fp8" else 2)
    assert r["e2e"]["d2h_bytes_per_step"] == 128 * 4864 * 2
    cs = r["context_sustained"]
    assert cs["seconds"] >= 0.2 and cs["launches"] % 50 == 0 and cs["us_per_launch"] > 0
    for key in ("sm_mhz", "samples", "reasons"):
        assert key in cs["clocks"], key
    if dtype == "fp8":
        assert "sweep" not in r
        return
    import workloads
    sw = r["sweep"]
    assert [e["workload"] for e in sw] == [w.c for w in workloads.WORKLOADS]
    for e, w in zip(sw, workloads.WORKLOADS):
        assert (e["M"], e["K"], e["N"], e["variant"]) == (w.M, w.K, w.N, w.variant)
        for key in ("us_per_launch", "tflops", "bound", "frac", "achieved_gbs", "clocks",
                    "launches", "frac_of_roofline_time"):
            assert key in e, (w.c, key)
        assert e["us_per_launch"] > 0 and 0 < e["frac"] < 1.5, e
        assert e["tflops"] == pytest.approx(w.flops / (e["us_per_launch"] * 1e-6) / 1e12)
        assert e["bound"] == ("hbm" if w.M <= 128 else "tensor"), e


def test_bench_context_down_projection():
    """With the context on: the whole MLP at the bench workload, the
    down-projection sweep (this library against cuBLAS at the workloads'
    down-projection shapes, alternating windows, clocks per window) and the
    whole MLP at a decode shape (graph-replayed, against eager cuBLAS)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "0", "--steps", "20",
           "--warmup", "3", "--no-cpu-baseline", "--sustained-s", "0", "--sweep-window-s", "0.03"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    r = json.loads(lines[0])
    import bench
    import workloads
    assert "context_mlp" in r and r["context_mlp"]["fused_mlp_ms"] > 0
    cd = r["context_down"]
    assert [e["workload"] for e in cd] == list(bench.DOWN_SWEEP_LABELS)
    for e in cd:
        w = workloads.BY_LABEL[e["workload"]]
        assert (e["M"], e["N"], e["K"]) == (w.M, w.N, w.K)
        for side in ("ours", "cublas"):
            assert e[side]["us"] > 0 and e[side]["tflops"] > 0, e
            assert "sm_mhz" in e[side]["clocks"], e
        assert e["ours_over_cublas_time"] == pytest.approx(e["ours"]["us"] / e["cublas"]["us"])
    md = r["context_mlp_decode"]
    w = workloads.BY_LABEL[md["workload"]]
    assert (md["M"], md["K"], md["N"]) == (w.M, w.K, w.N) and md["weight_bytes"] == 6 * w.K * w.N
    for side in ("fused", "fused_up_cublas_down", "eager"):
        assert md[side]["us"] > 0 and 0 < md[side]["frac_of_hbm_roofline"] < 1.5, md
        assert "sm_mhz" in md[side]["clocks"], md
    assert md["mlp_speedup_over_eager"] == pytest.approx(md["eager"]["us"] / md["fused"]["us"])


@pytest.mark.parametrize("world", [2, 3])
def test_column_split_ranks_reassemble_the_whole_forward(world, monkeypatch):
    """What each rank of `bench.py --split columns` runs, done here for every
    rank in turn on one GPU: its slice of W1/W2's columns packed and run
    through the public forward. Side by side, the slices are exactly the
    whole forward's Y (columns of Y are independent; whole tiles are forced
    so that every element is summed over k in the same order)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("SWIGLU_SCHEDULE", "dp")
    import numpy as np

    import bench
    import workloads
    from gemm_swiglu_mlp_gb300 import build
    build.build()
    import gemm_swiglu_mlp_gb300 as sg
    from tests.parity import from_device_bf16, to_device_bf16
    M, K, N = 520, 512, 1000
    w = workloads.Workload("t", "column-split-test", M, K, N)
    inputs = workloads.random_case(M, N, K, seed=55)
    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream(dev)
    A, W1, W2 = inputs
    whole = from_device_bf16(sg.swiglu_up_forward(
        to_device_bf16(A, dev),
        sg.swiglu_pack_weights(to_device_bf16(W1, dev), to_device_bf16(W2, dev)), N))
    parts = []
    for rank in range(world):
        c0, c1 = bench.column_slice(N, world, rank)
        p = bench.pack_problem(sg, w, "bf16", dev, inputs, split=(c0, c1))
        assert p.N == c1 - c0
        p.forward(0, st)
        torch.cuda.synchronize()
        parts.append(from_device_bf16(p.Ys[0]))
    sg.swiglu_check_device_status()
    assert np.array_equal(np.concatenate(parts, axis=1), whole)


def test_ablation_mode_prints_every_form():
    """`bench.py --ablation` on one workload: one JSON line with every packed
    layout x kernel x schedule form, each with its time, roofline fraction
    and fusion efficiency against the unfused cuBLAS path."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--ablation", "--ablation-workloads",
           "0", "--sweep-window-s", "0.02"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    r = json.loads(lines[0])
    (e,) = r["ablation"]
    assert (e["M"], e["K"], e["N"]) == (128, 896, 4864) and e["unfused_us"] > 0
    forms = {(f["layout"], f["variant"], f["schedule"]) for f in e["forms"]}
    assert forms == set(bench.ABLATION_FORMS)
    for f in e["forms"]:
        assert f["us_per_launch"] > 0 and f["bound"] == "hbm" and "fusion_efficiency" in f
        assert (f["workspace_bytes"] > 0) == (f["schedule"] in ("sk", "sk-tail")), f
