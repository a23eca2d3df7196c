"""GPU parity of the 1-SM kernel's plain mode (tiles of 128 rows x 64 output
columns), the down-projection of decode-sized MLPs, against the oracle,
through the C ABI.

SWIGLU_DOWN_TILE=64 forces it at any M (the decode kernel took its place as
the automatic choice for decode-sized products), SWIGLU_SCHEDULE a work
split. The shapes cover M tails inside a
128-row tile, output widths that end inside a 64-column tile and inside a
256-column packed weight tile, ragged reductions, stream-K tiles split over
up to ~50 CTAs (the last contributor sums every partial), and the decode
down-projection shapes of the 7B, 32B and 72B workloads in full. Criteria as
in tests/test_gpu_mlp.py.
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


SLIM_SHAPES = [
    (1, 8, 8),            # one row, one k-block, 8 of a tile's 64 columns
    (7, 136, 264),        # output ends inside the second packed weight tile
    (100, 4600, 208),     # long reduction, four tiles: stream-K over many CTAs
    (128, 1000, 1032),    # a full 128-row tile, 17 tiles
    (300, 392, 400),      # three 128-row tiles, the last partly live
    (64, 27656, 136),     # 3 tiles, 433 k-blocks: ~50 CTAs per tile
]


@pytest.mark.parametrize("M,N,K", SLIM_SHAPES)
def test_slim_full_compare(sg, orc, monkeypatch, M, N, K):
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "64")
    Yb, W3b = _case(M, N, K, 3 * M + 7 * N + K)
    got = _run(sg, Yb, W3b)[0]
    _check(got, orc.matmul(Yb, W3b)["C"], Yb, W3b, (M, N, K))


@pytest.mark.parametrize("mode", ["dp", "sk", "sk-tail"])
def test_slim_every_schedule_form(sg, orc, monkeypatch, mode):
    """Whole tiles, stream-K over all tiles, stream-K over the tail (2600
    rows: 21 x 21 = 441 tiles, 2.9 waves on 152 SMs)."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "64")
    monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    M, N, K = 2600, 520, 1320
    Yb, W3b = _case(M, N, K, 17)
    got = _run(sg, Yb, W3b)[0]
    _check(got, orc.matmul(Yb, W3b)["C"], Yb, W3b, mode)


@pytest.mark.parametrize("label", ["0", "2", "3", "4", "8", "10"])
def test_slim_down_at_decode_workload_shapes(sg, orc, monkeypatch, label):
    """This kernel, forced, at the decode workloads' down-projection shapes,
    every element compared: the 0.5B shape (M=128, 896 output columns), and
    M = 1, 16, 128 for 7B, 64 for 32B and 32 for 72B."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "64")
    w = workloads.BY_LABEL[label]
    M, N, K = w.M, w.N, w.K
    Yb, W3b = _case(M, N, K, 400 + int(label))
    got = _run(sg, Yb, W3b)[0]
    _check(got, orc.matmul(Yb, W3b)["C"], Yb, W3b, w.name)


def test_slim_deterministic_bitwise(sg, monkeypatch):
    """Split tiles are summed in k order by whichever CTA arrives last:
    repeated launches give bit-identical results."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "64")
    for M, N, K in [(16, 18944, 3584), (100, 4600, 208)]:
        Yb, W3b = _case(M, N, K, 58)
        outs = _run(sg, Yb, W3b, reps=4)
        for o in outs[1:]:
            assert np.array_equal(o, outs[0]), (M, N, K)
