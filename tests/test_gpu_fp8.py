"""GPU parity of the FP8 (E4M3, per-tensor scales) path against the oracle.

The inputs are FP8 bytes plus scales; the oracle computes the exact result
for those same inputs (Gate = s_a s_w1 sum A8 W1_8, etc.), so the same
criteria as the BF16 path apply: zero mismatches (1%, 1e-3 floor, FP32
accumulation exemption) and every element within 2 BF16 ulps + 1e-3.
"""
import numpy as np
import pytest

import workloads
from tests.parity import (compare, fp32_accumulation_bound, from_device_bf16,
                          pack_reference_fp8)

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _run(sg, A8, W18, W28, sa, s1, s2):
    N = W18.shape[1]
    Wp = sg.swiglu_pack_weights_fp8(_dev(W18), _dev(W28))
    Y = sg.swiglu_up_forward_fp8(_dev(A8), Wp, N, sa, s1, s2)
    sg.swiglu_check_device_status()
    return from_device_bf16(Y)


def _dequant(b, s):
    return workloads.e4m3_bits_to_f64(b) * s


def _check(got, ref, A8, W18, W28, sa, s1, s2, label):
    E = fp32_accumulation_bound(None, None, None, ref["G"], ref["U"],
                                values=(_dequant(A8, sa), _dequant(W18, s1), _dequant(W28, s2)))
    r = compare(got, ref["Y"], E)
    assert r["nonfinite"] == 0, (label, r)
    assert r["mismatches"] == 0 and r["over_bound"] == 0, (label, r)
    return r


@pytest.mark.parametrize("K,N,seed", [(16, 8, 1), (256, 136, 2), (1008, 264, 3)])
def test_fp8_pack_is_the_documented_permutation(sg, K, N, seed):
    _, W18, W28, _, _, _ = workloads.random_case_fp8(1, N, K, seed)
    Wp = sg.swiglu_pack_weights_fp8(_dev(W18), _dev(W28))
    torch.cuda.synchronize()
    assert np.array_equal(Wp.cpu().numpy(), pack_reference_fp8(W18, W28))


SHAPES = [(1, 8, 16), (7, 136, 144), (129, 256, 256), (300, 392, 400), (100, 4600, 208),
          (70, 520, 1008), (2048, 392, 528), (513, 136, 144)]


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fp8_forward_small_full_compare(sg, orc, monkeypatch, variant, M, N, K):
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    A8, W18, W28, sa, s1, s2 = workloads.random_case_fp8(M, N, K, seed=M + 3 * N + 7 * K)
    got = _run(sg, A8, W18, W28, sa, s1, s2)
    ref = orc.swiglu_up_fp8(A8, W18, W28, sa, s1, s2, want_gate_up=True)
    _check(got, ref, A8, W18, W28, sa, s1, s2, (variant, M, N, K))


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
@pytest.mark.parametrize("mode", ["dp", "split", "sk", "sk-tail"])
def test_fp8_every_schedule_form_matches(sg, orc, monkeypatch, variant, mode):
    """The FP8 path under each forced work split (k-blocks of 128 here)."""
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    M, N, K = 1300, 2000, 2064
    A8, W18, W28, sa, s1, s2 = workloads.random_case_fp8(M, N, K, seed=92)
    got = _run(sg, A8, W18, W28, sa, s1, s2)
    ref = orc.swiglu_up_fp8(A8, W18, W28, sa, s1, s2, want_gate_up=True)
    _check(got, ref, A8, W18, W28, sa, s1, s2, (variant, mode))


@pytest.mark.parametrize("label", ["1", "1s", "3", "6", "8", "10"])
def test_fp8_workload_full_size(sg, orc, label):
    """Full-size FP8 runs of the 1.5B prefill (also with the x8 stress input,
    pre-activations that saturate SiLU), 7B decode and prefill (M=2048),
    32B decode (1% outlier channels, which set the per-tensor scale) and 72B
    decode shapes, every output element compared."""
    w = workloads.BY_LABEL[label]
    A8, W18, W28, sa, s1, s2 = workloads.make_inputs_fp8(w)
    got = _run(sg, A8, W18, W28, sa, s1, s2)
    ref = orc.swiglu_up_fp8(A8, W18, W28, sa, s1, s2, want_gate_up=True)
    _check(got, ref, A8, W18, W28, sa, s1, s2, w.name)


def test_fp8_rejects_bad_scales(sg):
    lib = sg.load_library()
    fake = 1 << 20
    for bad in (0.0, -1.0, float("nan")):
        assert lib.swiglu_up_forward_fp8(fake, fake * 3, fake * 5, 16, 128, 128, bad, 1.0, 1.0,
                                         None, 0, None) == 1


def test_fp8_binding_checks_shapes(sg):
    """The binding rejects a Y of the wrong shape, an A that is not [M, K]
    and packed weights that are too small, before anything is launched."""
    M, N, K = 64, 136, 144
    A8, W18, W28, sa, s1, s2 = workloads.random_case_fp8(M, N, K, seed=5)
    Wp = sg.swiglu_pack_weights_fp8(_dev(W18), _dev(W28))
    Ad = _dev(A8)
    with pytest.raises(ValueError, match="Y must be"):
        sg.swiglu_up_forward_fp8(Ad, Wp, N, sa, s1, s2,
                                 Y=torch.empty((M, N + 8), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError, match="Y must be"):
        sg.swiglu_up_forward_fp8(Ad, Wp, N, sa, s1, s2,
                                 Y=torch.empty((M + 1, N), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError, match="A must be"):
        sg.swiglu_up_forward_fp8(Ad.view(-1), Wp, N, sa, s1, s2)
    with pytest.raises(ValueError, match="Wpacked"):
        sg.swiglu_up_forward_fp8(Ad, Wp[:-16], N, sa, s1, s2)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert sg.swiglu_up_forward_fp8(Ad, Wp, N, sa, s1, s2, Y=Y) is Y
    sg.swiglu_check_device_status()
