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


# (M, N, K, forced schedule or None). The first group goes through the
# shared scratch array: three shapes split K across CTAs (stream-K) by the
# library's own choice on a 152-SM part, two are forced to stream-K (one per
# kernel) so that the scratch path is run whatever the automatic choice
# becomes, and one runs eight waves of whole tiles on CTA pairs, handed out
# at run time from a tile counter in the scratch. The last group runs one wave
# of whole tiles or column sub-tiles and needs no scratch.
SCRATCH_CASES = [(33, 264, 2000, None), (70, 520, 1000, None), (2048, 392, 520, None),
                 (300, 392, 1000, "sk"), (128, 4864, 896, "sk"), (2048, 9728, 136, None)]
PLAIN_CASES = [(128, 4864, 896, None), (512, 4864, 256, None), (1300, 2000, 256, None),
               (200, 9728, 256, None)]


@pytest.mark.parametrize("M,N,K,mode,uses_scratch",
                         [c + (True,) for c in SCRATCH_CASES] + [c + (False,) for c in PLAIN_CASES])
def test_noalloc_matches_forward_on_two_calls(sg, monkeypatch, M, N, K, mode, uses_scratch):
    """Two calls in a row give exactly the bytes of swiglu_up_forward on the
    same inputs (the second call finds the first call's partial sums still
    in the scratch array), and are within the oracle tolerance of it."""
    if mode is not None:
        monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    assert (sg.swiglu_workspace_bytes(M, N, K) > 0) == uses_scratch
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
        got = from_device_bf16(Y)
        r = compare(got, ref)
        assert r["nonfinite"] == 0, (call, r)
        assert r["mismatches"] == 0 and r["over_bound"] == 0, (call, r)
        # same kernel, same schedule, same k order of the partial sums
        assert np.array_equal(got, ref), (call, int(np.count_nonzero(got != ref)))


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
