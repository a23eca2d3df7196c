"""C-ABI checks that need no GPU: the library builds, loads without a driver,
exports every function include/swiglu.h declares, and rejects bad arguments
on the host before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

from tests import parity

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gemm_swiglu_mlp_gb300 import build
    build.build()
    import gemm_swiglu_mlp_gb300 as sg
    return sg.load_library()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(swiglu_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("swiglu_pack_weights", "swiglu_up_forward", "swiglu_packed_weight_bytes",
                     "swiglu_check_device_status", "swiglu_status_string",
                     "swiglu_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    import gemm_swiglu_mlp_gb300 as sg
    for name in _declared_functions():
        assert hasattr(lib, name), name          # dlsym succeeds
    assert set(_declared_functions()) <= set(sg.EXPORTED_SYMBOLS)


def test_binding_has_every_abi_name():
    import gemm_swiglu_mlp_gb300 as sg
    for name in _declared_functions():
        assert callable(getattr(sg, name, None)), name


def test_status_strings_and_version(lib):
    import gemm_swiglu_mlp_gb300 as sg
    assert sg.swiglu_status_string(0) == "SWIGLU_OK"
    assert sg.swiglu_status_string(4) == "SWIGLU_ERR_DEVICE_TIMEOUT"
    assert sg.swiglu_status_string(77) == "SWIGLU_ERR_UNKNOWN"
    assert sg.swiglu_version() >= 1


def test_packed_weight_bytes(lib):
    import gemm_swiglu_mlp_gb300 as sg
    assert sg.swiglu_packed_weight_bytes(4864, 896) == 2 * 4864 * 896 * 2
    assert sg.swiglu_packed_weight_bytes(136, 64) == 2 * 256 * 64 * 2    # padded to 256 columns
    assert sg.swiglu_packed_weight_bytes(128, 72) == 2 * 128 * 128 * 2   # K padded to 128
    assert sg.swiglu_packed_weight_bytes(0, 64) == 0
    assert sg.swiglu_packed_weight_bytes(8, -1) == 0


def test_workspace_query_is_consistent(lib):
    import gemm_swiglu_mlp_gb300 as sg
    for M, N, K in [(1, 18944, 3584), (2048, 8960, 1536), (8192, 29568, 8192)]:
        assert sg.swiglu_workspace_bytes(M, N, K) >= 0


P = 0x10000          # fake, 16-byte aligned "device" addresses: never dereferenced
Q = 0x40000000
R = 0x80000000


@pytest.mark.parametrize("args", [
    (0, Q, R, 4, 8, 8), (P, 0, R, 4, 8, 8), (P, Q, 0, 4, 8, 8),       # null pointers
    (P, Q, R, 0, 8, 8), (P, Q, R, -3, 8, 8),                          # M < 1
    (P, Q, R, 4, 12, 8), (P, Q, R, 4, 8, 12), (P, Q, R, 4, 0, 8),     # N, K not multiples of 8
    (P + 8, Q, R, 4, 8, 8), (P, Q + 2, R, 4, 8, 8), (P, Q, R + 4, 4, 8, 8),  # misaligned
    (P, Q, P, 4, 8, 8),                                               # Y aliases A
    (P, Q, R, 1 << 31, 8, 8),                                         # M too large
])
def test_forward_rejects_bad_arguments_on_host(lib, args):
    A, Wp, Y, M, N, K = args
    st = lib.swiglu_up_forward(A, Wp, Y, M, N, K, None, 0, None)
    assert st == 1, "expected SWIGLU_ERR_INVALID_ARG"


@pytest.mark.parametrize("args", [
    (0, Q, R, 64, 64), (P, Q, 0, 64, 64), (P, Q, R, 60, 64), (P, Q, R, 64, 4),
    (P + 2, Q, R, 64, 64), (P, Q, P, 64, 64),
])
def test_pack_rejects_bad_arguments_on_host(lib, args):
    W1, W2, Wp, K, N = args
    assert lib.swiglu_pack_weights(W1, W2, K, N, Wp, None) == 1
    assert lib.swiglu_pack_weights_nk(W1, W2, N, K, Wp, None) == 1


def test_fp8_sizes_and_host_validation(lib):
    import gemm_swiglu_mlp_gb300 as sg
    assert sg.swiglu_packed_weight_bytes_fp8(4864, 896) == 2 * 4864 * 896
    assert sg.swiglu_packed_weight_bytes_fp8(136, 64) == 2 * 256 * 128     # N -> 256, K -> 128
    assert sg.swiglu_packed_weight_bytes_fp8(0, 64) == 0
    assert sg.swiglu_workspace_bytes_fp8(2048, 8960, 1536) >= 0
    f = lib.swiglu_up_forward_fp8
    ok = (P, Q, R, 4, 8, 16)
    for bad in [(0, Q, R, 4, 8, 16), (P, Q, R, 4, 8, 8),               # null; K % 16 != 0
                (P, Q, R, 4, 12, 16), (P + 8, Q, R, 4, 8, 16), (P, Q, P, 4, 8, 16)]:
        assert f(*bad, 1.0, 1.0, 1.0, None, 0, None) == 1, bad
    for sa, s1, s2 in [(0.0, 1.0, 1.0), (1.0, -1.0, 1.0), (1.0, 1.0, float("nan")),
                       (float("inf"), 1.0, 1.0), (1e30, 1e30, 1.0), (1e-30, 1e-30, 1.0)]:
        assert f(*ok, sa, s1, s2, None, 0, None) == 1, (sa, s1, s2)
    for bad in [(0, Q, R, 64, 64), (P, Q, R, 64, 4), (P, Q, R, 8, 64), (P + 4, Q, R, 64, 64)]:
        W1, W2, Wp, K, N = bad
        assert lib.swiglu_pack_weights_fp8(W1, W2, K, N, Wp, None) == 1, bad


def test_valid_call_without_gpu_reports_error_not_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = lib.swiglu_up_forward(P, Q, R, 4, 8, 8, None, 0, None)
    assert st in (2, 3)                       # UNSUPPORTED or CUDA: no device here


def test_binding_fails_loudly_when_library_missing(tmp_path):
    import gemm_swiglu_mlp_gb300 as sg
    saved = sg._lib
    sg._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            sg.load_library(str(tmp_path / "missing.so"))
    finally:
        sg._lib = saved


def test_pack_reference_layout_by_hand():
    # K=2, N=3: one tile [256][64]; row r<3 holds W1[:, r] in its first 2
    # entries, row 128+r holds W2[:, r]; everything else is zero padding
    W1 = np.arange(6, dtype=np.uint16).reshape(2, 3)
    W2 = (100 + np.arange(6, dtype=np.uint16)).reshape(2, 3)
    P_ = parity.pack_reference(W1, W2).reshape(256, 64)
    assert P_[1, :2].tolist() == [1, 4] and P_[129, :2].tolist() == [101, 104]
    assert not P_[:, 2:].any() and not P_[3:128].any() and not P_[131:].any()
    # two k-blocks and two column blocks: element W1[70, 130] sits in tile
    # (j=1, b=1), row 2, column 6
    K, N = 72, 136
    A1 = np.arange(K * N, dtype=np.uint16).reshape(K, N)
    A2 = A1 + np.uint16(1)
    T = parity.pack_reference(A1, A2).reshape(2, 2, 256, 64)
    assert T[1, 1, 2, 6] == A1[70, 130] and T[1, 1, 130, 6] == A2[70, 130]
    u1, u2 = parity.unpack_reference(T.reshape(-1), K, N)
    assert np.array_equal(u1, A1) and np.array_equal(u2, A2)


def test_interleaved_pack_reference_layout_by_hand():
    # K=2, N=3: row 2i holds W1[:, i], row 2i+1 holds W2[:, i]
    W1 = np.arange(6, dtype=np.uint16).reshape(2, 3)
    W2 = (100 + np.arange(6, dtype=np.uint16)).reshape(2, 3)
    P_ = parity.pack_reference_interleaved(W1, W2).reshape(256, 64)
    assert P_[0, :2].tolist() == [0, 3] and P_[1, :2].tolist() == [100, 103]
    assert P_[4, :2].tolist() == [2, 5] and P_[5, :2].tolist() == [102, 105]
    assert not P_[:, 2:].any() and not P_[6:].any()
    # W1[70, 130] sits in tile (j=1, b=1), row 2*2, column 6; W2's in row 5
    K, N = 72, 136
    A1 = np.arange(K * N, dtype=np.uint16).reshape(K, N)
    A2 = A1 + np.uint16(1)
    T = parity.pack_reference_interleaved(A1, A2).reshape(2, 2, 256, 64)
    assert T[1, 1, 4, 6] == A1[70, 130] and T[1, 1, 5, 6] == A2[70, 130]
    # the same values as the blocked layout, rows permuted within each tile
    B = parity.pack_reference(A1, A2).reshape(2, 2, 256, 64)
    perm = np.empty(256, np.int64)
    perm[0::2] = np.arange(128)
    perm[1::2] = 128 + np.arange(128)
    assert np.array_equal(T, B[:, :, perm, :])


def test_parity_criteria_by_hand():
    import workloads
    want = workloads.f32_to_bf16_bits(np.array([1.0, 0.0, 100.0, 1e-4], np.float32))
    same = parity.compare(want, want)
    assert same["mismatches"] == 0 and same["over_bound"] == 0 and same["bit_exact_frac"] == 1.0
    # one BF16 ulp off at 100 (ulp 0.5) is within 2 ulps; 2% off is a mismatch
    got = workloads.f32_to_bf16_bits(np.array([1.0, 0.0, 100.5, 1e-4], np.float32))
    r = parity.compare(got, want)
    assert r["mismatches"] == 0 and r["over_bound"] == 0
    got = workloads.f32_to_bf16_bits(np.array([1.02, 0.0, 100.0, 1e-4], np.float32))
    r = parity.compare(got, want)
    assert r["mismatches"] == 1 and r["over_bound"] == 1
    # near zero the relative test is floored: 5e-6 <= 0.01 * 1e-3 is not a mismatch,
    # but it is one under the literal, unfloored reading
    got = workloads.f32_to_bf16_bits(np.array([1.0, 5e-6, 100.0, 1e-4], np.float32))
    r = parity.compare(got, want)
    assert r["mismatches"] == 0 and r["over_bound"] == 0 and r["literal_rel_mismatches"] == 1


def test_down_sizes_and_host_validation(lib):
    """The down-projection / whole-MLP entry points: packed size and
    argument checks made on the host before anything is launched."""
    import gemm_swiglu_mlp_gb300 as sg
    assert sg.swiglu_down_packed_weight_bytes(8960, 1536) == 1536 * 8960 * 2
    assert sg.swiglu_down_packed_weight_bytes(4864, 896) == 1024 * 4864 * 2   # K -> 4 x 256
    assert sg.swiglu_down_packed_weight_bytes(72, 8) == 256 * 128 * 2         # N -> 128
    assert sg.swiglu_down_packed_weight_bytes(0, 8) == 0
    assert sg.swiglu_down_workspace_bytes(2048, 8960, 1536) >= 0
    # up to 128 rows the decode kernel serves the call and sums its split
    # tiles inside a cluster: no workspace (7B M=16, the 0.5B shape); from
    # 129 rows on the CTA-pair kernel's stream-K needs one
    assert sg.swiglu_down_workspace_bytes(16, 18944, 3584) == 0
    assert sg.swiglu_down_workspace_bytes(128, 4864, 896) == 0
    assert sg.swiglu_down_workspace_bytes(129, 4864, 896) > 0
    assert sg.swiglu_mlp_workspace_bytes(2048, 8960, 1536) >= max(
        sg.swiglu_workspace_bytes(2048, 8960, 1536), sg.swiglu_down_workspace_bytes(2048, 8960, 1536))
    d = lib.swiglu_down_forward
    for bad in [(0, Q, R, 4, 8, 8), (P, 0, R, 4, 8, 8), (P, Q, 0, 4, 8, 8),   # null pointers
                (P, Q, R, 0, 8, 8), (P, Q, R, 4, 12, 8), (P, Q, R, 4, 8, 12),  # M, N, K
                (P + 8, Q, R, 4, 8, 8), (P, Q, R + 2, 4, 8, 8),                # misaligned
                (P, Q, P, 4, 8, 8), (P, Q, Q, 4, 8, 8)]:                       # out aliases Y, W3
        assert d(*bad, None, 0, None) == 1, bad
    m = lib.swiglu_mlp_forward
    S = 0xC0000000
    for bad in [(0, Q, R, S, P + 0x100000, 4, 8, 8),                          # null A
                (P, Q, R, S, S, 4, 8, 8),                                     # out aliases Y
                (P, Q, R, S, P, 4, 8, 8),                                     # out aliases A
                (P, Q, R, R, S, 4, 8, 8),                                     # Y aliases W3packed
                (P, Q, R, S, P + 0x100000, 4, 12, 8)]:                        # N % 8 != 0
        assert m(*bad, None, 0, None) == 1, bad
    for bad in [(0, 64, 64, R), (P, 60, 64, R), (P, 64, 4, R), (P + 2, 64, 64, R), (P, 64, 64, P)]:
        W, N, K, Wp = bad
        assert lib.swiglu_pack_down_weights(W, N, K, Wp, None) == 1, bad
        assert lib.swiglu_pack_down_weights_nk(W, K, N, Wp, None) == 1, bad


def test_binding_rejects_host_tensors_for_the_mlp_calls(lib):
    """The Python binding checks dtype, device and shape before any launch:
    CPU tensors or wrong shapes raise instead of reaching the C ABI."""
    import torch
    import gemm_swiglu_mlp_gb300 as sg
    Y = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(8, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        sg.swiglu_pack_down_weights(W)
    with pytest.raises(TypeError):
        sg.swiglu_pack_down_weights_nk(W)
    with pytest.raises(TypeError):
        sg.swiglu_down_forward(Y, torch.zeros(16, dtype=torch.uint8), 8)
    with pytest.raises(TypeError):
        sg.swiglu_mlp_forward(Y, torch.zeros(16, dtype=torch.uint8),
                              torch.zeros(16, dtype=torch.uint8), 8)
    with pytest.raises(TypeError):
        sg.swiglu_down_forward(torch.zeros(4, 8, dtype=torch.float32),
                               torch.zeros(16, dtype=torch.uint8), 8)


def test_pack_down_reference_layout_by_hand():
    # N=2 (reduction), K=3 (outputs): one tile [256][64]; packed row r < 3
    # holds W3[:, r] in its first 2 entries; everything else is zero padding
    from tests.parity import pack_down_reference
    W3 = np.arange(6, dtype=np.uint16).reshape(2, 3)
    P = pack_down_reference(W3).reshape(1, 1, 256, 64)
    assert P.shape == (1, 1, 256, 64)
    for r in range(3):
        assert list(P[0, 0, r, :2]) == [W3[0, r], W3[1, r]]
        assert not P[0, 0, r, 2:].any()
    assert not P[0, 0, 3:].any()
    import gemm_swiglu_mlp_gb300 as sg
    assert sg.swiglu_down_packed_weight_bytes(2, 3) == P.size * 2
