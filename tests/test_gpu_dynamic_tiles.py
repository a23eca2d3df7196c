"""GPU parity of the CTA-pair kernel's dynamic tile order.

A launch of whole tiles and at least eight waves hands out the tiles past
the first wave at run time (a counter in the workspace, a ring of tile
indices shared by the pair's roles); SWIGLU_DYNAMIC_TILES=1 takes the
dynamic order from two waves on, which the small cases here use. Every tile is still computed whole by one pair,
summing k in order, so the result must be bit-identical to the static order
(SWIGLU_DYNAMIC_TILES=0) and meet the oracle criteria; the counter must be
back at zero after every launch, so back-to-back launches and a launch after
an aborted one are correct too.
"""
import numpy as np
import pytest

import workloads
from tests.parity import compare, from_device_bf16, to_device_bf16
from tests.test_gpu_parity import assert_parity

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


# (M, N, K): two and three waves of 256 x 128 pair tiles on 76 pairs, with
# 3 or 4 k-blocks per tile (short tiles: the producer runs far ahead, so the
# tile ring fills up), ragged M in the second
SHAPES = [(2048, 2432, 200), (3000, 2432, 136)]


def _forward(sg, layout, A, W1, W2):
    N = W1.shape[1]
    w1, w2, a = to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"), to_device_bf16(A, "cuda")
    if layout == "interleaved":
        Wp = sg.swiglu_pack_weights_interleaved(w1, w2)
        fwd = sg.swiglu_up_forward_interleaved
    else:
        Wp = sg.swiglu_pack_weights(w1, w2)
        fwd = sg.swiglu_up_forward
    ys = [from_device_bf16(fwd(a, Wp, N)) for _ in range(3)]   # back to back, one workspace
    sg.swiglu_check_device_status()
    return ys


@pytest.mark.parametrize("layout", ["blocked", "interleaved"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_dynamic_tiles_match_static_order_and_oracle(sg, orc, monkeypatch, layout, M, N, K):
    A, W1, W2 = workloads.random_case(M, N, K, seed=M + N + K)
    monkeypatch.delenv("SWIGLU_DYNAMIC_TILES", raising=False)
    assert sg.swiglu_workspace_bytes(M, N, K) == 0          # 2-3 waves: static by default
    monkeypatch.setenv("SWIGLU_DYNAMIC_TILES", "1")
    assert sg.swiglu_workspace_bytes(M, N, K) > 0          # the tile counters
    dyn = _forward(sg, layout, A, W1, W2)
    monkeypatch.setenv("SWIGLU_DYNAMIC_TILES", "0")
    assert sg.swiglu_workspace_bytes(M, N, K) == 0          # static whole tiles
    static = _forward(sg, layout, A, W1, W2)
    assert_parity(dyn[0], orc.swiglu_up(A, W1, W2)["Y"], (layout, M, N, K))
    for y in dyn + static[1:]:
        assert np.array_equal(y, static[0])


def test_dynamic_tiles_fp8(sg, orc, monkeypatch):
    M, N, K = 2048, 2432, 256
    A8, W18, W28, sa, s1, s2 = workloads.random_case_fp8(M, N, K, seed=41)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    Wp = sg.swiglu_pack_weights_fp8(dev(W18), dev(W28))

    def run():
        return from_device_bf16(sg.swiglu_up_forward_fp8(dev(A8), Wp, N, sa, s1, s2))

    monkeypatch.setenv("SWIGLU_DYNAMIC_TILES", "1")
    assert sg.swiglu_workspace_bytes_fp8(M, N, K) > 0
    y_dyn = run()
    monkeypatch.setenv("SWIGLU_DYNAMIC_TILES", "0")
    y_static = run()
    sg.swiglu_check_device_status()
    assert np.array_equal(y_dyn, y_static)
    r = compare(y_dyn, orc.swiglu_up_fp8(A8, W18, W28, sa, s1, s2)["Y"])
    assert r["mismatches"] == 0 and r["over_bound"] == 0, r


def test_dynamic_tiles_down_projection(sg, orc, monkeypatch):
    """The CTA-pair kernel's plain (down-projection) mode: 152 output tiles
    of 256 x 256 on 76 pairs, whole tiles (two waves, dynamic when asked
    for). The wide down-projection kernel, which would take this shape, has
    no dynamic order, so the CTA-pair kernel is forced."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", "256")
    M, N, K = 2048, 512, 4864
    rng = np.random.Generator(np.random.PCG64(42))
    Yb = workloads.f32_to_bf16_bits(rng.standard_normal(size=(M, N), dtype=np.float32))
    W3 = workloads.f32_to_bf16_bits(
        rng.standard_normal(size=(N, K), dtype=np.float32) * np.float32(N ** -0.5))
    W3p = sg.swiglu_pack_down_weights(to_device_bf16(W3, "cuda"))
    Yd = to_device_bf16(Yb, "cuda")
    monkeypatch.setenv("SWIGLU_DYNAMIC_TILES", "1")
    assert sg.swiglu_down_workspace_bytes(M, N, K) > 0
    outs = [from_device_bf16(sg.swiglu_down_forward(Yd, W3p, K)) for _ in range(2)]
    monkeypatch.setenv("SWIGLU_DYNAMIC_TILES", "0")
    ref = from_device_bf16(sg.swiglu_down_forward(Yd, W3p, K))
    sg.swiglu_check_device_status()
    for o in outs:
        assert np.array_equal(o, ref)
    r = compare(outs[0], orc.matmul(Yb, W3)["C"])
    assert r["mismatches"] == 0 and r["over_bound"] == 0, r


def test_dynamic_tiles_whole_workload(sg, orc, monkeypatch):
    """The 7B M=2048 prefill shape (1184 pair tiles, 15.6 waves: dynamic by
    default) as the bench runs it, checked on one row of every 256-row pair
    tile."""
    monkeypatch.delenv("SWIGLU_DYNAMIC_TILES", raising=False)
    w = workloads.BY_LABEL["6"]
    A, W1, W2 = workloads.make_inputs(w)
    assert sg.swiglu_workspace_bytes(w.M, w.N, w.K) > 0
    Wp = sg.swiglu_pack_weights(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    Y = from_device_bf16(sg.swiglu_up_forward(to_device_bf16(A, "cuda"), Wp, w.N))
    sg.swiglu_check_device_status()
    rows = np.arange(0, w.M, 256) + 97
    want = orc.swiglu_up(A, W1, W2, rows=rows)["Y"]
    assert_parity(Y[rows], want, "7b-m2048 dynamic")
