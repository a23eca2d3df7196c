"""GPU parity of the column-interleaved packing (the pages' Kernel-2
pairing: even packed rows Gate, odd rows Up) against the oracle, and against
the default blocked packing.

The interleaved path runs the same kernels with the epilogue pairing
accumulator columns 2i and 2i+1 instead of i and 128+i. Every accumulator
element is the same dot product either way, so the two layouts must give the
same Y bit for bit; each is also held to the oracle criteria on its own.
"""
import numpy as np
import pytest

import workloads
from tests.parity import (compare, from_device_bf16, pack_reference_interleaved,
                          to_device_bf16)
from tests.test_gpu_parity import SMALL, assert_parity

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


def _both(sg, A, W1, W2):
    """Y from the interleaved entry points and from the default ones."""
    N = W1.shape[1]
    w1, w2, a = to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"), to_device_bf16(A, "cuda")
    Wi = sg.swiglu_pack_weights_interleaved(w1, w2)
    Yi = sg.swiglu_up_forward_interleaved(a, Wi, N)
    Wb = sg.swiglu_pack_weights(w1, w2)
    Yb = sg.swiglu_up_forward(a, Wb, N)
    sg.swiglu_check_device_status()
    return from_device_bf16(Yi), from_device_bf16(Yb)


@pytest.mark.parametrize("K,N,seed", [(8, 8, 1), (200, 264, 3), (896, 4864, 4), (72, 136, 5)])
def test_interleaved_pack_is_the_documented_permutation(sg, K, N, seed):
    _, W1, W2 = workloads.random_case(1, N, K, seed)
    Wp = sg.swiglu_pack_weights_interleaved(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    torch.cuda.synchronize()
    got = Wp.cpu().numpy().view(np.uint16).reshape(-1)
    assert np.array_equal(got, pack_reference_interleaved(W1, W2))


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_interleaved_small_full_compare(sg, orc, monkeypatch, variant, M, N, K):
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    A, W1, W2 = workloads.random_case(M, N, K, seed=M * 7 + N * 3 + K)
    yi, yb = _both(sg, A, W1, W2)
    assert_parity(yi, orc.swiglu_up(A, W1, W2)["Y"], ("interleaved", variant, M, N, K))
    assert np.array_equal(yi, yb), int(np.count_nonzero(yi != yb))


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
@pytest.mark.parametrize("mode", ["dp", "split", "sk", "sk-tail"])
def test_interleaved_every_schedule_form(sg, orc, monkeypatch, variant, mode):
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    M, N, K = 1300, 2000, 2056
    A, W1, W2 = workloads.random_case(M, N, K, seed=91)
    yi, yb = _both(sg, A, W1, W2)
    assert_parity(yi, orc.swiglu_up(A, W1, W2)["Y"], ("interleaved", variant, mode))
    assert np.array_equal(yi, yb)


@pytest.mark.parametrize("label", ["0", "1"])
def test_interleaved_workload_full_size(sg, orc, label):
    """The 0.5B (weight-streaming, 32-column sub-tiles) and 1.5B (CTA pairs,
    64-column halves in the tail) shapes in full."""
    w = workloads.BY_LABEL[label]
    A, W1, W2 = workloads.make_inputs(w)
    yi, yb = _both(sg, A, W1, W2)
    r = compare(yi, orc.swiglu_up(A, W1, W2)["Y"])
    assert r["nonfinite"] == 0 and r["mismatches"] == 0 and r["over_bound"] == 0, r
    assert np.array_equal(yi, yb)
