"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small cases are compared in full, element by element; the Qwen-2.5-shaped
workloads are run at full size through the same entry point and launch
configuration the bench times, and compared in full where the oracle takes
seconds (every workload up to 6e11 flops), else on sampled rows (every
column of those rows; at least one row in every 128-row tile) that the
oracle computes one by one. Criteria (tests/parity.py):
zero mismatches (relative error > 1% with a 1e-3 floor) and every element
within 2 BF16 ulps + 1e-3 of the oracle's BF16 result.
"""
import numpy as np
import pytest

import workloads
from tests.parity import (compare, fp32_accumulation_bound, from_device_bf16, pack_reference,
                          to_device_bf16, unpack_reference)

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_swiglu_mlp_gb300 import build
    build.build()
    import gemm_swiglu_mlp_gb300 as mod
    torch.cuda.set_device(0)
    return mod


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def run_fused(sg, A, W1, W2, dev="cuda"):
    K, N = W1.shape
    Wp = sg.swiglu_pack_weights(to_device_bf16(W1, dev), to_device_bf16(W2, dev))
    Y = sg.swiglu_up_forward(to_device_bf16(A, dev), Wp, N)
    sg.swiglu_check_device_status()
    return from_device_bf16(Y), Wp


def assert_parity(got, want, label="", accum_bound=None):
    r = compare(got, want, accum_bound)
    assert r["nonfinite"] == 0, (label, r)
    assert r["mismatches"] == 0, (label, r)
    assert r["over_bound"] == 0, (label, r)
    return r


@pytest.mark.parametrize("K,N,seed", [(8, 8, 1), (64, 128, 2), (200, 264, 3), (896, 4864, 4),
                                        (72, 136, 5)])
def test_pack_is_the_documented_permutation(sg, K, N, seed):
    _, W1, W2 = workloads.random_case(1, N, K, seed)
    Wp = sg.swiglu_pack_weights(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    torch.cuda.synchronize()
    got = Wp.cpu().numpy().view(np.uint16).reshape(-1)
    want = pack_reference(W1, W2)
    assert got.shape == want.shape and np.array_equal(got, want)
    # unpack(pack(W)) == W
    u1, u2 = unpack_reference(got, K, N)
    assert np.array_equal(u1, W1) and np.array_equal(u2, W2)


@pytest.mark.parametrize("K,N,seed", [(8, 8, 11), (200, 264, 12), (896, 4864, 13)])
def test_pack_from_linear_layout_matches(sg, K, N, seed):
    # nn.Linear keeps W as [N, K]: packing W^T that way gives the same bytes
    _, W1, W2 = workloads.random_case(1, N, K, seed)
    a = sg.swiglu_pack_weights(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    b = sg.swiglu_pack_weights_nk(to_device_bf16(np.ascontiguousarray(W1.T), "cuda"),
                                  to_device_bf16(np.ascontiguousarray(W2.T), "cuda"))
    torch.cuda.synchronize()
    assert torch.equal(a, b)


SMALL = [
    (1, 8, 8),          # smallest legal problem: one partial tile everywhere
    (7, 136, 72),       # ragged M, N (128 + 8) and K (64 + 8)
    (64, 128, 64),      # exactly one tile, one k-block
    (129, 256, 128),    # one row into a second row-tile
    (300, 392, 200),    # several tiles, ragged in every dimension
    (256, 1024, 1024),  # more tiles than a single wave of row-tiles
    (128, 4864, 896),   # the Qwen-2.5-0.5B shape, checked in full (3-way split tiles)
    (70, 520, 1000),    # K split across 2 CTAs per tile; ragged M leaves a dead warp
    (33, 264, 2000),    # K split across 4 CTAs per tile; 33 rows
    (1, 136, 4096),     # one token, long K split many ways
    (2048, 392, 520),   # data-parallel tiles plus a stream-K tail
    (513, 136, 72),     # one row into a third 256-row pair tile
    (100, 4600, 200),   # 36 tiles on 152 SMs: 32-column sub-tiles, ragged last sub-tile
    (64, 9000, 136),    # 71 tiles: 64-column sub-tiles
    (1280, 11776, 64),  # whole-tile waves plus a column-split tail
    (64, 27648, 256),   # weight-streaming: one wave plus half-width tail units
]


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_forward_small_full_compare(sg, orc, monkeypatch, variant, M, N, K):
    # every kernel on every shape: the 1-SM kernel and the 2-SM (CTA pair) one
    # (rows past M in a 256-row pair tile are computed from zero-filled A and
    # not stored)
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    A, W1, W2 = workloads.random_case(M, N, K, seed=M * 7 + N * 3 + K)
    got, _ = run_fused(sg, A, W1, W2)
    want = orc.swiglu_up(A, W1, W2)["Y"]
    assert_parity(got, want, (variant, M, N, K))


SCHEDULE_MODES = ["dp", "split", "sk", "sk-tail"]


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
@pytest.mark.parametrize("mode", SCHEDULE_MODES)
def test_every_schedule_form_matches(sg, orc, monkeypatch, variant, mode):
    """Each work split the scheduler can choose, forced on one shape with more
    tiles than either kernel's grid (176 1-SM tiles, 96 pair tiles) and a
    stream-K remainder of several k-blocks per CTA: whole tiles, the
    column-split tail, stream-K over the last wave plus the remainder, and
    stream-K over the remainder alone."""
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    M, N, K = 1300, 2000, 2056
    A, W1, W2 = workloads.random_case(M, N, K, seed=91)
    got, _ = run_fused(sg, A, W1, W2)
    want = orc.swiglu_up(A, W1, W2)["Y"]
    assert_parity(got, want, (variant, mode))


@pytest.mark.parametrize("variant,mode", [("1sm", "auto"), ("2sm", "auto"), ("1sm", "sk"),
                                          ("2sm", "sk")])
def test_cuda_graph_replay_matches_direct_calls(sg, monkeypatch, variant, mode):
    """The forward captured in a CUDA graph (after one direct call has done
    the per-device set-up) replays to the same bytes as direct calls,
    including the stream-K path whose workspace counters must return to
    zero after every launch."""
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    if mode != "auto":
        monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    M, N, K = 520, 1160, 1032
    A, W1, W2 = workloads.random_case(M, N, K, seed=17)
    Ad = to_device_bf16(A, "cuda")
    Wp = sg.swiglu_pack_weights(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    ws_bytes = sg.swiglu_workspace_bytes(M, N, K)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    Y_direct = sg.swiglu_up_forward(Ad, Wp, N, workspace=ws)
    torch.cuda.synchronize()
    Ys = [torch.zeros((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for Y in Ys:
            sg.swiglu_up_forward(Ad, Wp, N, Y=Y, workspace=ws, stream=cs)
    for _ in range(2):
        for Y in Ys:
            Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert sg.swiglu_check_device_status() == 0
        for Y in Ys:
            assert torch.equal(Y.view(torch.int16), Y_direct.view(torch.int16))


def test_forward_saturating_inputs(sg, orc):
    # pre-activations with std ~8-16: SiLU at both saturated ends
    A, W1, W2 = workloads.random_case(200, 264, 512, seed=5, a_scale=12.0)
    got, _ = run_fused(sg, A, W1, W2)
    want = orc.swiglu_up(A, W1, W2)["Y"]
    assert_parity(got, want, "saturating")


def test_zero_gate_weight_gives_signed_zero(sg):
    A, W1, W2 = workloads.random_case(130, 136, 200, seed=6)
    W1[:] = 0
    got, _ = run_fused(sg, A, W1, W2)
    assert np.all((got == 0x0000) | (got == 0x8000))


def test_zero_up_weight_gives_signed_zero(sg):
    A, W1, W2 = workloads.random_case(130, 136, 200, seed=7)
    W2[:] = 0
    got, _ = run_fused(sg, A, W1, W2)
    assert np.all((got == 0x0000) | (got == 0x8000))


def test_rank_one_inputs(sg, orc):
    # one nonzero column of A: Gate and Up are single exact products
    M, N, K, k0 = 160, 200, 136, 77
    A, W1, W2 = workloads.random_case(M, N, K, seed=8, a_scale=3.0)
    A[:, :k0] = 0
    A[:, k0 + 1:] = 0
    got, _ = run_fused(sg, A, W1, W2)
    want = orc.swiglu_up(A, W1, W2)["Y"]
    r = assert_parity(got, want, "rank1")
    # products are exact in FP32: only SiLU's exp/divide can differ, by <= 1 ulp
    diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
    same_sign = (got & 0x8000) == (want & 0x8000)
    assert np.all(diff[same_sign] <= 1), r


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
def test_deterministic_bitwise(sg, monkeypatch, variant):
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    A, W1, W2 = workloads.random_case(300, 392, 520, seed=9)
    Wp = sg.swiglu_pack_weights(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    Ad = to_device_bf16(A, "cuda")
    y1 = from_device_bf16(sg.swiglu_up_forward(Ad, Wp, 392))
    y2 = from_device_bf16(sg.swiglu_up_forward(Ad, Wp, 392))
    assert np.array_equal(y1, y2)


def test_workspace_reused_across_shapes(sg, orc, monkeypatch):
    # the default workspace is shared by all calls on a stream: counters must
    # come back to zero after every call, whatever the split and the kernel
    cases = [(70, 520, 1000, 21), (33, 264, 2000, 22), (128, 4864, 896, 23), (70, 520, 1000, 24),
             (600, 392, 2000, 25), (70, 520, 1000, 26)]
    for M, N, K, seed in cases:
        monkeypatch.setenv("SWIGLU_FUSED_VARIANT", "2sm" if M >= 256 else "1sm")
        A, W1, W2 = workloads.random_case(M, N, K, seed=seed)
        got, _ = run_fused(sg, A, W1, W2)
        assert_parity(got, orc.swiglu_up(A, W1, W2)["Y"], (M, N, K, seed))


def test_output_rows_outside_m_untouched(sg):
    # Y is a view into a larger buffer: rows past M must not be written
    M, N, K = 70, 136, 64
    A, W1, W2 = workloads.random_case(M, N, K, seed=10)
    big = torch.full((M + 64, N), 7.0, dtype=torch.bfloat16, device="cuda")
    Wp = sg.swiglu_pack_weights(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    sg.swiglu_up_forward(to_device_bf16(A, "cuda"), Wp, N, Y=big[:M])
    torch.cuda.synchronize()
    assert torch.all(big[M:] == 7.0)


def test_device_status_clean_after_runs(sg):
    assert sg.swiglu_check_device_status() == 0


def _sample_rows(M, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    base = {0, M - 1, M // 2, min(127, M - 1), min(128, M - 1)}
    extra = rng.choice(M, size=min(M, 11), replace=False).tolist()
    return sorted(base | set(extra))


FULL_COMPARE_FLOPS = 6e11   # the oracle does this in well under a minute on the host cores


def _workload_rows(w, seed):
    """Every row where the oracle finishes in seconds; for the three largest
    prefill shapes, fixed and random rows plus one random row in every
    128-row tile (so every row tile of every CTA's work is checked)."""
    if w.flops <= FULL_COMPARE_FLOPS:
        return list(range(w.M))
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    per_tile = {int(t + rng.integers(0, min(128, w.M - t))) for t in range(0, w.M, 128)}
    return sorted(set(_sample_rows(w.M, seed)) | per_tile)


@pytest.mark.parametrize("label", [w.c for w in workloads.WORKLOADS])
def test_workload_full_size(sg, orc, label):
    w = workloads.BY_LABEL[label]
    A, W1, W2 = workloads.make_inputs(w)
    got, _ = run_fused(sg, A, W1, W2)
    rows = _workload_rows(w, 5000 + w.seed_index)
    ref = orc.swiglu_up(A, W1, W2, rows=rows, want_gate_up=True)
    E = fp32_accumulation_bound(A[rows], W1, W2, ref["G"], ref["U"])
    r = assert_parity(got[rows], ref["Y"], w.name, accum_bound=E)
    _report(w, rows, r)


def _report(w, rows, r):
    """Appends the parity figures to the JSON-lines file named by
    SWIGLU_PARITY_REPORT, if set (used to publish raw/exempt counts)."""
    import json
    import os
    path = os.environ.get("SWIGLU_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"workload": w.name, "M": w.M, "K": w.K, "N": w.N,
                                "rows_checked": len(rows), **r}) + "\n")


@pytest.mark.parametrize("label", ["1", "6", "10"])
def test_unfused_torch_context_mismatch_rate(sg, orc, label):
    """Context for the pages' accuracy claim (zero mismatches for the fused
    kernels against 4.5-11% for the cuBLAS path): the unfused PyTorch path
    rounds Gate and Up to BF16 in HBM before the activation. Its mismatch
    count is reported, not gated; the fused result must have none."""
    import torch.nn.functional as F
    w = workloads.BY_LABEL[label]
    A, W1, W2 = workloads.make_inputs(w)
    rows = _sample_rows(w.M, 6000 + w.seed_index)
    Ad = to_device_bf16(A, "cuda")
    g = torch.matmul(Ad, to_device_bf16(W1, "cuda"))
    u = torch.matmul(Ad, to_device_bf16(W2, "cuda"))
    unfused = from_device_bf16(F.silu(g) * u)[rows]
    fused, _ = run_fused(sg, A, W1, W2)
    ref = orc.swiglu_up(A, W1, W2, rows=rows, want_gate_up=True)
    E = fp32_accumulation_bound(A[rows], W1, W2, ref["G"], ref["U"])
    r_unfused = compare(unfused, ref["Y"], E)
    r_fused = assert_parity(fused[rows], ref["Y"], w.name, accum_bound=E)
    _report(w, rows, dict(r_unfused, path="unfused_torch"))
    assert r_fused["mismatches"] <= r_unfused["mismatches"]
