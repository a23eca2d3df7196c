"""GPU parity of the decode down-projection kernel (down_decode_kernel.cuh:
swapped operands, tiles of 128 output columns x all token rows, each tile's
K ranges on one cluster of CTAs, summed through distributed shared memory)
against the oracle, through the C ABI.

It is the automatic choice up to 128 rows; SWIGLU_DOWN_TILE=128 forces it
(up to 128 rows), SWIGLU_DECODE_SPLITS the K ranges per tile (the cluster
size). The shapes cover every token block (mt = 16 .. 128, M tails inside a
16-token group), output widths that end inside a 128-column tile and inside
the first half of a packed 256-column weight tile, ragged reductions and
uneven K ranges, clusters of 1 to 16 CTAs, more clusters than fit at once
(waves), ranges of a single k-block, and the decode down-projection shapes
of the 0.5B, 7B, 32B and 72B workloads in full. Criteria as in
tests/test_gpu_mlp.py (plain product).
"""
import numpy as np
import pytest

import workloads
from tests.parity import (beyond_scale_allowance, compare, from_device_bf16,
                          plain_accumulation_bound, plain_certified_bound, to_device_bf16)

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


def _case(M, N, K, seed):
    return _rand_bf16(seed, (M, N), 1.0), _rand_bf16(seed + 1, (N, K), N ** -0.5)


def _run(sg, Yb, W3b, reps=1):
    N, K = W3b.shape
    Wd = sg.swiglu_pack_down_weights(to_device_bf16(W3b, "cuda"))
    Yd = to_device_bf16(Yb, "cuda")
    outs = [sg.swiglu_down_forward(Yd, Wd, K) for _ in range(reps)]
    sg.swiglu_check_device_status()
    return [from_device_bf16(o) for o in outs]


def _check(got, want, Yb, W3b, label):
    r = compare(got, want, plain_accumulation_bound(Yb, W3b), plain_certified_bound(Yb, W3b))
    assert r["nonfinite"] == 0, (label, r)
    assert r["mismatches"] == 0 and r["over_bound"] == 0, (label, r)
    assert r["beyond_accum_scale"] <= beyond_scale_allowance(r["elements"]), (label, r)


# (M, N, K): out [M, K] = Y [M, N] x W3 [N, K]
DECODE_SHAPES = [
    (1, 8, 8),            # one row, one k-block, 8 of a tile's 128 columns
    (7, 136, 264),        # 3 tiles, the last inside the first half of a weight tile
    (16, 4600, 208),      # long reduction, two tiles: each split in 16
    (33, 1000, 1032),     # three 16-token parts, the last with one live row
    (100, 4600, 208),     # seven parts, split tiles
    (128, 1000, 1032),    # eight parts, 9 tiles
    (64, 27656, 136),     # 433 k-blocks, a 128-column and an 8-column tile
]


@pytest.mark.parametrize("M,N,K", DECODE_SHAPES)
def test_decode_full_compare(sg, orc, monkeypatch, M, N, K):
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "128")
    Yb, W3b = _case(M, N, K, 5 * M + 3 * N + K)
    got = _run(sg, Yb, W3b)[0]
    _check(got, orc.matmul(Yb, W3b)["C"], Yb, W3b, (M, N, K))


@pytest.mark.parametrize("splits", ["1", "2", "3", "5", "8", "13", "16"])
@pytest.mark.parametrize("M,N,K", [(40, 7000, 1304), (8, 1000, 20000)])
def test_decode_every_split(sg, orc, monkeypatch, splits, M, N, K):
    """11 tiles of 110 k-blocks in 1 to 16 K ranges (uneven: 110 / 3, / 8,
    / 13, / 16; 16 x 11 clusters are more CTAs than SMs, so clusters run in
    waves); 157 tiles of 16 k-blocks (more tiles than SMs: waves at any
    split; 16 ranges of a single k-block each)."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "128")
    monkeypatch.setenv("SWIGLU_DECODE_SPLITS", splits)
    Yb, W3b = _case(M, N, K, 31 + M)
    got = _run(sg, Yb, W3b)[0]
    _check(got, orc.matmul(Yb, W3b)["C"], Yb, W3b, (splits, M, N, K))


@pytest.mark.parametrize("label,splits", [
    ("0", None), ("2", None), ("3", None), ("4", None), ("8", None), ("10", None),
    ("8", "2"), ("10", "4"), ("3", "16"), ("0", "1"),
])
def test_decode_down_at_workload_shapes(sg, orc, monkeypatch, label, splits):
    """The automatic choice (this kernel, its automatic split) at the decode
    workloads' down-projection shapes, every element compared: 0.5B (M=128),
    7B (M = 1, 16, 128), 32B (M=64), 72B (M=32); and other splits there."""
    if splits:
        monkeypatch.setenv("SWIGLU_DECODE_SPLITS", splits)
    w = workloads.BY_LABEL[label]
    M, N, K = w.M, w.N, w.K
    Yb, W3b = _case(M, N, K, 500 + int(label))
    got = _run(sg, Yb, W3b)[0]
    _check(got, orc.matmul(Yb, W3b)["C"], Yb, W3b, (w.name, splits))


def test_decode_deterministic_bitwise(sg, monkeypatch):
    """Every slice sums the cluster's partials in rank (= K) order:
    repeated launches give bit-identical results."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "128")
    for M, N, K in [(16, 18944, 3584), (100, 4600, 208), (64, 27656, 136)]:
        Yb, W3b = _case(M, N, K, 59)
        outs = _run(sg, Yb, W3b, reps=4)
        for o in outs[1:]:
            assert np.array_equal(o, outs[0]), (M, N, K)


def test_decode_needs_no_workspace(sg, orc, monkeypatch):
    """Split tiles are summed inside their cluster: no workspace is asked for
    or used, split or not."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "128")
    for i, (M, N, K) in enumerate([(16, 4600, 208), (100, 4600, 208), (1, 18944, 3584)]):
        assert sg.swiglu_down_workspace_bytes(M, N, K) == 0
        Yb, W3b = _case(M, N, K, 800 + i)
        Wd = sg.swiglu_pack_down_weights(to_device_bf16(W3b, "cuda"))
        out = sg.swiglu_down_forward(to_device_bf16(Yb, "cuda"), Wd, K, workspace=None)
        sg.swiglu_check_device_status()
        _check(from_device_bf16(out), orc.matmul(Yb, W3b)["C"], Yb, W3b, (M, N, K))


def test_decode_and_slim_agree_with_the_oracle_on_one_input(sg, orc, monkeypatch):
    """The decode kernel and the 1-SM plain mode on the same input, each
    within the criteria (they may differ from each other by FP32 summation
    order only)."""
    M, N, K = 16, 18944, 3584
    Yb, W3b = _case(M, N, K, 61)
    want = orc.matmul(Yb, W3b)["C"]
    for tile in ("128", "64"):
        monkeypatch.setenv("SWIGLU_DOWN_TILE", tile)
        got = _run(sg, Yb, W3b)[0]
        _check(got, want, Yb, W3b, tile)


@pytest.mark.parametrize("M,N,K", [(16, 18944, 3584), (128, 4864, 896), (32, 4600, 1032)])
def test_decode_in_a_cuda_graph(sg, monkeypatch, M, N, K):
    """The decode kernel captured in a CUDA graph (clusters of 4, 16 and 2 at
    these shapes) replays to the bytes of direct calls: nothing carries over
    between launches."""
    Yb, W3b = _case(M, N, K, 71)
    Wd = sg.swiglu_pack_down_weights(to_device_bf16(W3b, "cuda"))
    Yd = to_device_bf16(Yb, "cuda")
    direct = sg.swiglu_down_forward(Yd, Wd, K)
    torch.cuda.synchronize()
    outs = [torch.zeros((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for o in outs:
            sg.swiglu_down_forward(Yd, Wd, K, out=o, stream=cs)
    for _ in range(2):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert sg.swiglu_check_device_status() == 0
        for o in outs:
            assert torch.equal(o.view(torch.int16), direct.view(torch.int16))
