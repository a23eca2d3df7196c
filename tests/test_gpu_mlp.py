"""GPU parity of the down-projection (out = Y x W3, the CTA-pair kernel's
plain mode) and of the whole gated MLP (fused up-projection, then the
down-projection) against the oracle, through the C ABI.

Criteria as for the up-projection (tests/parity.py): zero mismatches (1%,
1e-3 floor, FP32-accumulation exemption) and every element within 2 BF16
ulps + 1e-3. The down-projection's FP32 accumulation scale is the plain
product's (c 2^-24 sqrt(N) ||y (.) w||).
"""
import numpy as np
import pytest

import workloads
from tests.parity import (beyond_scale_allowance, bits_to_f64, compare, fp32_accumulation_bound,
                          from_device_bf16, pack_down_reference, plain_accumulation_bound,
                          plain_certified_bound, to_device_bf16, ulp_bf16)

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


def _rand_bf16(seed, shape, scale):
    rng = np.random.Generator(np.random.PCG64(seed))
    return workloads.f32_to_bf16_bits(
        rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale))


def _down_case(M, N, K, seed):
    """Y [M, N] ~ N(0, 1) and W3 [N, K] ~ N(0, 1/N), BF16 bit patterns."""
    return _rand_bf16(seed, (M, N), 1.0), _rand_bf16(seed + 1, (N, K), N ** -0.5)


def _check_plain(got, want, Yb, W3b, label):
    r = compare(got, want, plain_accumulation_bound(Yb, W3b), plain_certified_bound(Yb, W3b))
    assert r["nonfinite"] == 0, (label, r)
    assert r["mismatches"] == 0 and r["over_bound"] == 0, (label, r)
    assert r["beyond_accum_scale"] <= beyond_scale_allowance(r["elements"]), (label, r)
    return r


def _down(sg, Yb, W3b, nk=False):
    N, K = W3b.shape
    if nk:
        Wd = sg.swiglu_pack_down_weights_nk(to_device_bf16(np.ascontiguousarray(W3b.T), "cuda"))
    else:
        Wd = sg.swiglu_pack_down_weights(to_device_bf16(W3b, "cuda"))
    out = sg.swiglu_down_forward(to_device_bf16(Yb, "cuda"), Wd, K)
    sg.swiglu_check_device_status()
    return from_device_bf16(out)


@pytest.mark.parametrize("N,K,seed", [(8, 8, 1), (136, 264, 2), (1000, 136, 3), (2056, 512, 4)])
def test_down_pack_is_the_documented_layout(sg, N, K, seed):
    _, W3 = _down_case(1, N, K, seed)
    ref = pack_down_reference(W3)
    for nk in (False, True):
        if nk:
            Wd = sg.swiglu_pack_down_weights_nk(to_device_bf16(np.ascontiguousarray(W3.T), "cuda"))
        else:
            Wd = sg.swiglu_pack_down_weights(to_device_bf16(W3, "cuda"))
        torch.cuda.synchronize()
        got = Wd.cpu().numpy().view(np.uint16)
        assert got.size == ref.size and np.array_equal(got, ref), nk


DOWN_SHAPES = [(1, 8, 8), (7, 136, 264), (129, 256, 512), (300, 392, 400), (513, 1000, 136),
               (2048, 528, 392), (100, 4600, 208), (256, 2056, 1024)]


@pytest.mark.parametrize("M,N,K", DOWN_SHAPES)
def test_down_small_full_compare(sg, orc, M, N, K):
    Yb, W3b = _down_case(M, N, K, M + 3 * N + 7 * K)
    got = _down(sg, Yb, W3b, nk=(M % 2 == 1))
    want = orc.matmul(Yb, W3b)["C"]
    _check_plain(got, want, Yb, W3b, (M, N, K))


@pytest.mark.parametrize("mode", ["dp", "sk", "sk-tail", "split"])
def test_down_every_schedule_form_matches(sg, orc, monkeypatch, mode):
    """Forced work splits (split is not offered for the plain product and
    falls back to the automatic choice)."""
    monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    M, N, K = 1300, 2056, 2000
    Yb, W3b = _down_case(M, N, K, 77)
    got = _down(sg, Yb, W3b)
    want = orc.matmul(Yb, W3b)["C"]
    _check_plain(got, want, Yb, W3b, mode)


def _sample_rows(M, per_block=4, block=128):
    rows = []
    for b0 in range(0, M, block):
        hi = min(M, b0 + block)
        rows += sorted({b0, hi - 1, (b0 + hi) // 2, min(hi - 1, b0 + 37)})[:per_block]
    return np.array(sorted(set(rows)), np.int64)


def _mlp_inputs(w):
    A, W1, W2 = workloads.make_inputs(w)
    return A, W1, W2, workloads.make_W3(w)


def _run_mlp(sg, A, W1, W2, W3, graph=False):
    M, K = A.shape
    N = W1.shape[1]
    Wp = sg.swiglu_pack_weights(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    Wd = sg.swiglu_pack_down_weights(to_device_bf16(W3, "cuda"))
    Ad = to_device_bf16(A, "cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    if not graph:
        sg.swiglu_mlp_forward(Ad, Wp, Wd, N, Y=Y, out=out)
    else:
        ws = torch.zeros(max(1, sg.swiglu_mlp_workspace_bytes(M, N, K)), dtype=torch.uint8,
                         device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            sg.swiglu_mlp_forward(Ad, Wp, Wd, N, Y=Y, out=out, workspace=ws, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        out.zero_()
        Y.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sg.swiglu_mlp_forward(Ad, Wp, Wd, N, Y=Y, out=out, workspace=ws,
                                  stream=torch.cuda.current_stream())
        for _ in range(3):
            g.replay()
    sg.swiglu_check_device_status()
    return from_device_bf16(Y), from_device_bf16(out)


def _check_mlp(orc, A, W1, W2, W3, Yg, outg, rows, label):
    """Y against the oracle's up-projection; out against the oracle's down
    product of the GPU's own Y (the down path alone, strict) and against the
    oracle's whole MLP (end to end). End to end, the intermediate Y is BF16
    on both sides and may differ by a rounding step where the FP32 and the
    binary64 Gate/Up fall on opposite sides of a BF16 midpoint (the Y check
    above allows exactly that); that difference, carried through W3
    (sum_n |dY_n| |W3_nh|), joins the accumulation scale for the 1%
    criterion and widens the 2-ulp + 1e-3 bound by the same amount. The
    down check before it (the GPU's Y on both sides) has neither."""
    up = orc.swiglu_up(A, W1, W2, rows=rows, want_gate_up=True)
    E = fp32_accumulation_bound(A[rows], W1, W2, up["G"], up["U"])
    r = compare(Yg[rows], up["Y"], E)
    assert r["nonfinite"] == 0 and r["mismatches"] == 0 and r["over_bound"] == 0, (label, "Y", r)
    own = orc.matmul(Yg[rows], W3)["C"]
    _check_plain(outg[rows], own, Yg[rows], W3, (label, "down"))
    end = orc.matmul(up["Y"], W3)["C"]
    dY = np.abs(bits_to_f64(Yg[rows]) - bits_to_f64(up["Y"]))
    carried = (dY.astype(np.float32) @ np.abs(bits_to_f64(W3)).astype(np.float32)).astype(np.float64)
    r = compare(outg[rows], end, plain_accumulation_bound(up["Y"], W3) + carried)
    assert r["nonfinite"] == 0 and r["mismatches"] == 0, (label, "mlp", r)
    want = bits_to_f64(end)
    err = np.abs(bits_to_f64(outg[rows]) - want)
    over = err > 2.0 * ulp_bf16(want) + 1e-3 + carried
    assert not over.any(), (label, "mlp bound", int(over.sum()), float(err[over].max()))


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (70, 520, 264), (300, 392, 400),
                                   (513, 1000, 1032)])
def test_mlp_small_full_compare(sg, orc, M, N, K):
    A, W1, W2 = workloads.random_case(M, N, K, seed=5 * M + N + K)
    W3 = _rand_bf16(900 + M, (N, K), N ** -0.5)
    Yg, outg = _run_mlp(sg, A, W1, W2, W3)
    _check_mlp(orc, A, W1, W2, W3, Yg, outg, np.arange(M, dtype=np.int64), (M, N, K))


@pytest.mark.parametrize("M,N,K", [(600, 1032, 520), (16, 4600, 1032)])
def test_mlp_in_a_cuda_graph(sg, orc, M, N, K):
    """The whole MLP captured in a CUDA graph: a prefill-sized shape (the
    CTA-pair kernels) and a decode-sized one (the down-projection on the
    decode kernel's clusters)."""
    A, W1, W2 = workloads.random_case(M, N, K, seed=31 + M)
    W3 = _rand_bf16(32 + M, (N, K), N ** -0.5)
    Yg, outg = _run_mlp(sg, A, W1, W2, W3, graph=True)
    _check_mlp(orc, A, W1, W2, W3, Yg, outg, np.arange(M, dtype=np.int64), ("graph", M))


@pytest.mark.parametrize("label,full", [("0", True), ("1", False), ("6", False), ("10", False)])
def test_mlp_workload_full_size(sg, orc, label, full):
    """The whole MLP at the 0.5B (every row), 1.5B and 7B prefill and 72B
    decode shapes (rows sampled from every 128-row block; each sampled row
    compared in every column). The 7B down-projection (112 output tiles on
    the CTA pairs) runs whole tiles plus stream-K over the tail."""
    w = workloads.BY_LABEL[label]
    A, W1, W2, W3 = _mlp_inputs(w)
    Yg, outg = _run_mlp(sg, A, W1, W2, W3)
    rows = np.arange(w.M, dtype=np.int64) if full else _sample_rows(w.M, 4 if w.M > 64 else 8)
    _check_mlp(orc, A, W1, W2, W3, Yg, outg, rows, w.name)


@pytest.mark.parametrize("mode", ["auto", "sk", "dp"])
def test_down_deterministic_bitwise(sg, monkeypatch, mode):
    """Stream-K partial sums are added in a fixed order: repeated calls give
    bit-identical results (the 1.5B down-projection shape, and a ragged one)."""
    if mode != "auto":
        monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    for M, N, K in [(2048, 8960, 1536), (1300, 2056, 2000)]:
        Yb, W3b = _down_case(M, N, K, 55)
        Wd = sg.swiglu_pack_down_weights(to_device_bf16(W3b, "cuda"))
        Yd = to_device_bf16(Yb, "cuda")
        first = sg.swiglu_down_forward(Yd, Wd, K)
        for _ in range(3):
            again = sg.swiglu_down_forward(Yd, Wd, K)
            assert torch.equal(first.view(torch.int16), again.view(torch.int16)), (mode, M, N, K)
        sg.swiglu_check_device_status()
