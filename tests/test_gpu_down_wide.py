"""GPU parity of the wide down-projection kernel (down_wide_kernel.cuh:
tiles of 256 rows x 512 output columns, one TMEM accumulator stage, split
tiles finished by the last participant to count in on each 128-column part)
against the oracle, through the C ABI.

SWIGLU_DOWN_TILE=512 forces it on every shape (it is the automatic choice
from 256 rows on); SWIGLU_SCHEDULE forces a work split. The shapes cover:
a ragged M tail inside a 256-row tile, an odd number of 256-column weight
tiles (the last wide tile has only its first half), ragged reductions, split
tiles among 2 to ~18 pairs (the finisher reading the other partials through
the idle operand ring when at most three others fit, from global memory
otherwise), pairs whose range spans two tiles, and the automatic plans of
the 1.5B, 7B and 72B down-projection shapes (rows sampled from every 128-row
block, each sampled row compared in every column). Criteria as in
tests/test_gpu_mlp.py (plain product: zero mismatches, 2 BF16 ulps + 1e-3).
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


def _sample_rows(M, per_block=4, block=128):
    rows = []
    for b0 in range(0, M, block):
        hi = min(M, b0 + block)
        rows += sorted({b0, hi - 1, (b0 + hi) // 2, min(hi - 1, b0 + 37)})[:per_block]
    return np.array(sorted(set(rows)), np.int64)


# (M, N, K): out [M, K] = Y [M, N] x W3 [N, K]
WIDE_SHAPES = [
    (1, 8, 8),            # one row, one k-block, the first half of one weight tile
    (7, 136, 264),        # two weight tiles, ragged reduction
    (129, 256, 512),      # rows in the second CTA's half only partly live
    (300, 392, 400),      # M tail in the second 256-row tile
    (513, 1000, 136),     # one weight tile (the wide tile's second half absent)
    (2048, 528, 392),     # 8 tiles of one wide column
    (100, 4600, 208),     # long reduction, few tiles: many pairs per split tile
    (1300, 2056, 2000),   # 24 tiles, each cut in three K ranges (72 pairs)
]


@pytest.mark.parametrize("M,N,K", WIDE_SHAPES)
def test_wide_full_compare(sg, orc, monkeypatch, M, N, K):
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "512")
    Yb, W3b = _case(M, N, K, 2 * M + 5 * N + 3 * K)
    got = _run(sg, Yb, W3b)[0]
    _check(got, orc.matmul(Yb, W3b)["C"], Yb, W3b, (M, N, K))


@pytest.mark.parametrize("mode", ["dp", "sk", "sk-tail", "sk-aligned"])
@pytest.mark.parametrize("M,N,K", [(1300, 2056, 2000), (513, 4104, 1800)])
def test_wide_every_schedule_form(sg, orc, monkeypatch, mode, M, N, K):
    """Whole tiles, stream-K over all tiles on all pairs (ranges spanning
    two tiles, 4-5 participants per tile), stream-K over the tail, and every
    tile cut into equal K ranges (24 tiles in three on 72 pairs; 12 tiles in
    six on 72 pairs: the finishers read five other partials from global
    memory)."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "512")
    monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    Yb, W3b = _case(M, N, K, 91 + M)
    got = _run(sg, Yb, W3b)[0]
    _check(got, orc.matmul(Yb, W3b)["C"], Yb, W3b, (mode, M, N, K))


@pytest.mark.parametrize("N", [4864, 2048])
def test_wide_split_tiles_and_whole_tiles_in_one_launch(sg, orc, monkeypatch, N):
    """84 tiles on 76 pairs, stream-K over the tail forced. N=4864 (76
    k-blocks): 76 whole tiles, then the other 8 split among all pairs (8
    k-blocks each, ~10 participants per tile: the finishers read the other
    partials from global memory). N=2048 (32 k-blocks): the remainder alone
    would give each pair too few k-blocks, so the last full wave joins it:
    ranges of ~35 k-blocks span up to three tiles, the middle one whole.
    Rows sampled."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "512")
    monkeypatch.setenv("SWIGLU_SCHEDULE", "sk-tail")
    M, K = 3072, 3584
    Yb, W3b = _case(M, N, K, 123)
    got = _run(sg, Yb, W3b)[0]
    rows = _sample_rows(M)
    _check(got[rows], orc.matmul(Yb, W3b, rows=rows)["C"], Yb[rows], W3b, "sk-tail")


@pytest.mark.parametrize("label,tile,mode", [
    ("1", "512", "sk-aligned"),   # 24 tiles, each in three K ranges on 72 pairs
    ("5", "512", "sk-aligned"),   # 14 tiles in five K ranges on 70 pairs
    ("6", "512", "sk"),           # 56 tiles, stream-K over all on 76 pairs
    ("9", "512", "sk-tail"),      # 160 tiles: two whole waves, stream-K over 8
    ("7", None, None),            # automatic: whole wide tiles (224 tiles, 2.95 waves)
    ("11", None, None),           # automatic: whole wide tiles (512 tiles, 6.7 waves)
])
def test_wide_down_at_workload_shapes(sg, orc, monkeypatch, label, tile, mode):
    """The wide kernel at the down-projection shapes of the workloads, in the
    form given (or the automatic choice, which takes the wide kernel there);
    W3 [N, K] ~ N(0, 1/N), Y ~ N(0, 1)."""
    if tile:
        monkeypatch.setenv("SWIGLU_DOWN_TILE", tile)
    if mode:
        monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    w = workloads.BY_LABEL[label]
    M, N, K = w.M, w.N, w.K
    Yb, W3b = _case(M, N, K, 300 + int(label))
    got = _run(sg, Yb, W3b)[0]
    rows = _sample_rows(M, 1 if M >= 8192 else (2 if M >= 4096 else 4))
    _check(got[rows], orc.matmul(Yb, W3b, rows=rows)["C"], Yb[rows], W3b, w.name)


@pytest.mark.parametrize("mode", ["sk-aligned", "sk"])
def test_wide_deterministic_bitwise(sg, monkeypatch, mode):
    """Whoever finishes a part, its partials are added in k order: repeated
    launches give bit-identical results."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "512")
    monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    for M, N, K in [(2048, 8960, 1536), (1300, 2056, 2000)]:
        Yb, W3b = _case(M, N, K, 56)
        outs = _run(sg, Yb, W3b, reps=4)
        for o in outs[1:]:
            assert np.array_equal(o, outs[0]), (mode, M, N, K)


def test_wide_and_narrow_agree_with_the_oracle_on_one_input(sg, orc, monkeypatch):
    """Both down-projection kernels on the same input (sampled rows), each
    within the criteria; they may differ from each other by FP32 summation
    order only."""
    M, N, K = 2048, 8960, 1536
    Yb, W3b = _case(M, N, K, 57)
    rows = _sample_rows(M)
    want = orc.matmul(Yb, W3b, rows=rows)["C"]
    for tile in ("256", "512"):
        monkeypatch.setenv("SWIGLU_DOWN_TILE", tile)
        got = _run(sg, Yb, W3b)[0]
        _check(got[rows], want, Yb[rows], W3b, tile)


def test_wide_workspace_reused_across_shapes(sg, orc, monkeypatch):
    """One workspace through split and whole-tile launches of different
    shapes: every launch leaves its counters at zero for the next."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "512")
    monkeypatch.setenv("SWIGLU_SCHEDULE", "sk-aligned")
    shapes = [(1300, 2056, 2000), (513, 4104, 1800), (2048, 528, 392), (1300, 2056, 2000)]
    need = max(sg.swiglu_down_workspace_bytes(*s) for s in shapes)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    for i, (M, N, K) in enumerate(shapes):
        Yb, W3b = _case(M, N, K, 700 + i)
        Wd = sg.swiglu_pack_down_weights(to_device_bf16(W3b, "cuda"))
        out = sg.swiglu_down_forward(to_device_bf16(Yb, "cuda"), Wd, K, workspace=ws)
        sg.swiglu_check_device_status()
        _check(from_device_bf16(out), orc.matmul(Yb, W3b)["C"], Yb, W3b, (M, N, K))
