"""bench.py's roofline bookkeeping, checked by hand (no GPU)."""
import bench
import workloads


def test_algorithmic_bytes_by_hand():
    w = workloads.BY_LABEL["1"]                     # M=2048, K=1536, N=8960
    assert bench.algorithmic_bytes(w, "bf16") == 2 * (2048 * 1536 + 2 * 1536 * 8960 + 2048 * 8960)
    assert bench.algorithmic_bytes(w, "fp8") == 2048 * 1536 + 2 * 1536 * 8960 + 2 * 2048 * 8960


def test_fp8_peak_is_twice_bf16_and_moves_the_ridge():
    peaks = {"hbm_gbs": 7000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}
    assert bench.tensor_peak(peaks, "fp8") == 4000.0
    assert bench.tensor_peak(peaks, "fp8", "bf16_tflops_sustained") == 3600.0
    w = workloads.BY_LABEL["1"]
    assert bench.bound_of(w, peaks, "bf16") == "tensor"
    t = bench.roofline_us(w, peaks, "fp8")
    assert abs(t - max(w.flops / 4e15, bench.algorithmic_bytes(w, "fp8") / 7e12) * 1e6) < 1e-9
    decode = workloads.BY_LABEL["10"]
    assert bench.bound_of(decode, peaks, "fp8") == "hbm"


def test_fusion_efficiency_by_hand():
    w = workloads.BY_LABEL["0"]                     # M=128, N=4864
    removed_s = 8 * 128 * 4864 / 5000e9             # 8*M*N bytes at 5000 GB/s
    assert abs(bench.fusion_efficiency(w, 10e-6 + removed_s, 10e-6, 5000.0) - 1.0) < 1e-12
    assert abs(bench.fusion_efficiency(w, 10e-6 + 2 * removed_s, 10e-6, 5000.0) - 2.0) < 1e-12
    assert bench.fusion_efficiency(w, 10e-6, 10e-6, 5000.0) == 0.0


def test_reference_arm_prints_one_contract_line(monkeypatch, capsys):
    """The reference arm (the CPU oracle) on the small workload, one step:
    one JSON line with the contract's keys, on this host's cores."""
    import json
    import oracle
    oracle.build()
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)

    class Args:
        steps, warmup, dtype = 1, 3, "bf16"

    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 2.0)
    assert bench.run_reference(Args(), workloads.BY_LABEL["0"]) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    r = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in r, key
    assert r["impl"] == "reference" and r["metric"] == bench.METRIC and r["unit"] == "TFLOP/s"
    assert r["value"] > 0 and r["cpu_baseline"]["kind"] == "oracle"
    assert r["e2e"]["h2d_bytes_per_step"] == 0 and r["gpu_launches"] == 0
    assert r["config"]["M"] == 128 and r["config"]["N"] == 4864 and r["config"]["K"] == 896


def test_roofline_entry_by_hand():
    peaks = {"hbm_gbs": 5000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    big = workloads.BY_LABEL["11"]                  # tensor-bound
    t = big.flops / 1000e12                         # a launch at 1000 TFLOP/s
    e = bench.roofline_entry(big, peaks, "bf16", t)
    assert e["bound"] == "tensor"
    assert abs(e["tflops"] - 1000.0) < 1e-6 and abs(e["frac"] - 0.5) < 1e-9
    assert abs(e["frac_of_sustained"] - 1000.0 / 1600.0) < 1e-9
    assert abs(e["frac_of_roofline_time"] - (big.flops / 2000e12) / t) < 1e-9
    small = workloads.BY_LABEL["2"]                 # M=1: weight streaming
    t = small.roofline_bytes / 2500e9               # 2500 GB/s
    e = bench.roofline_entry(small, peaks, "bf16", t)
    assert e["bound"] == "hbm" and abs(e["achieved_gbs"] - 2500.0) < 1e-6
    assert abs(e["frac"] - 0.5) < 1e-9 and "frac_of_sustained" not in e


def test_graph_launches_rounds_to_the_rotation():
    # about 2 ms of launches per graph, a multiple of R, capped at 256
    assert bench.graph_launches(3, 1e-3) == 3            # 2 launches -> one rotation
    assert bench.graph_launches(2, 8e-6) == 250          # 250 = 2 ms / 8 us
    assert bench.graph_launches(3, 8e-6) == 252          # rounded up to a multiple of 3
    assert bench.graph_launches(2, 1e-6) == 256          # capped
    assert bench.graph_launches(3, 1e-6) == 255
    assert bench.graph_launches(2, 5e-3) == 2


def test_every_workload_is_in_the_sweep_labels():
    labels = [w.c for w in workloads.WORKLOADS]
    assert len(labels) == 13 and len(set(labels)) == 13
    assert bench.DEFAULT_WORKLOAD == "11"
    w = workloads.BY_LABEL[bench.DEFAULT_WORKLOAD]
    assert (w.M, w.K, w.N) == (8192, 8192, 29568)      # the largest single-GPU config
    assert max(workloads.WORKLOADS, key=lambda x: x.flops) is w
