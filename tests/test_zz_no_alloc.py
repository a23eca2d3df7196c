"""The allocation-free entry point, swiglu_up_forward_noalloc.

It serves callers that cannot allocate device memory (a runtime that plans
all device memory at start-up and must not call cudaMalloc later, or a
plugin interface that gives a kernel no workspace). It is checked here
through the C ABI against the ordinary entry point, swiglu_up_forward, on
two calls in a row, with the tolerance the other parity tests use.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test. It needs nothing from the other
test files and passes alone in a fresh process.
"""
import numpy as np
import pytest

import workloads
from tests.parity import compare, from_device_bf16, to_device_bf16

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


# Shapes that split K across CTAs (so the scratch is used) and shapes that
# run whole tiles (no scratch), on both the 1-SM and the 2-SM kernel.
CASES = [(33, 264, 2000), (128, 4864, 896), (70, 520, 1000), (1, 136, 4096),
         (300, 392, 200), (2048, 392, 520)]


@pytest.mark.parametrize("M,N,K", CASES)
def test_noalloc_matches_forward_on_two_calls(sg, M, N, K):
    lib = sg.load_library()
    A, W1, W2 = workloads.random_case(M, N, K, seed=4000 + M + N + K)
    Ad = to_device_bf16(A, "cuda")
    Wp = sg.swiglu_pack_weights(to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda"))
    ref = from_device_bf16(sg.swiglu_up_forward(Ad, Wp, N))
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.swiglu_up_forward_noalloc(Ad.data_ptr(), Wp.data_ptr(), Y.data_ptr(),
                                           M, N, K, stream)
        assert st == 0, sg.swiglu_status_string(st)
        assert sg.swiglu_check_device_status() == 0
        r = compare(from_device_bf16(Y), ref)
        assert r["nonfinite"] == 0, (call, r)
        assert r["mismatches"] == 0 and r["over_bound"] == 0, (call, r)


def test_noalloc_rejects_problems_over_its_scratch(sg):
    lib = sg.load_library()
    # 200 rows, 30 column tiles, K = 8192: 60 tiles, or their column
    # sub-tiles, would leave most of the SMs idle, so K is split over every SM
    # and the workspace exceeds the 32 MiB scratch.
    M, N, K = 200, 3840, 8192
    need = sg.swiglu_workspace_bytes(M, N, K)
    assert need > 32 * 1024 * 1024
    fake = 1 << 20   # 16-byte aligned, never dereferenced: the call is rejected first
    st = lib.swiglu_up_forward_noalloc(fake, fake * 3, fake * 5, M, N, K, None)
    assert st == 2, sg.swiglu_status_string(st)   # SWIGLU_ERR_UNSUPPORTED
