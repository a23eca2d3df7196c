"""Failure detection without a GPU fault.

Every wait inside the fused kernels is bounded. A test-only build of the same
sources (SWIGLU_TEST_FAULT_INJECTION, ~10 ms wait limit, never loaded by the
product binding) can leave the first pipeline stage unfilled, so the MMA
warp's wait for it (or a producer's wait for a stage that MMA never frees)
runs out. The kernel must then record the timeout in the
device status word, drain what is in flight, free its tensor memory and exit;
the host reads the status with swiglu_check_device_status, and the same CUDA
context must go on computing correct results. Nothing here traps, faults or
hangs a GPU: the only failure is a wait on a barrier that nothing completes.
"""
import ctypes
import os
import time

import numpy as np
import pytest

import workloads
from tests.parity import compare, from_device_bf16, to_device_bf16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TIMEOUT_STATUS = 4        # SWIGLU_ERR_DEVICE_TIMEOUT
PRODUCER_TIMEOUT_BIT = 1  # kStatusProducerTimeout
MMA_TIMEOUT_BIT = 2       # kStatusMmaTimeout


@pytest.fixture(scope="module")
def fi_lib(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_swiglu_mlp_gb300 import build
    path = str(tmp_path_factory.mktemp("fi") / "libswiglu_faultinject.so")
    build.build_fault_injection_library(path)
    lib = ctypes.CDLL(path)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.swiglu_test_set_fault_injection.argtypes = [ctypes.c_int]
    lib.swiglu_test_set_fault_injection.restype = None
    lib.swiglu_pack_weights.argtypes = [vp, vp, i64, i64, vp, vp]
    lib.swiglu_up_forward.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
    lib.swiglu_workspace_bytes.argtypes = [i64, i64, i64]
    lib.swiglu_workspace_bytes.restype = sz
    lib.swiglu_packed_weight_bytes.argtypes = [i64, i64]
    lib.swiglu_packed_weight_bytes.restype = sz
    lib.swiglu_check_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    torch.cuda.set_device(0)
    return lib


def _run(lib, A, Wp, M, N, K, stream):
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    ws_bytes = lib.swiglu_workspace_bytes(M, N, K)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    st = lib.swiglu_up_forward(A.data_ptr(), Wp.data_ptr(), Y.data_ptr(), M, N, K,
                               ws.data_ptr() if ws_bytes else None, ws_bytes, stream)
    assert st == 0
    raw = ctypes.c_uint32(0)
    status = lib.swiglu_check_device_status(stream, ctypes.byref(raw))
    return Y, status, raw.value


@pytest.mark.parametrize("variant,M,N,K", [("1sm", 128, 256, 512), ("2sm", 512, 256, 512)])
def test_wait_timeout_is_reported_and_context_survives(fi_lib, monkeypatch, variant, M, N, K):
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", variant)
    import oracle
    A, W1, W2 = workloads.random_case(M, N, K, seed=77)
    Ad = to_device_bf16(A, "cuda")
    W1d, W2d = to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda")
    Wp = torch.empty(fi_lib.swiglu_packed_weight_bytes(N, K), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert fi_lib.swiglu_pack_weights(W1d.data_ptr(), W2d.data_ptr(), K, N, Wp.data_ptr(),
                                      stream) == 0

    # 1) a launch whose first stage is never filled: the bounded wait runs out
    fi_lib.swiglu_test_set_fault_injection(1)
    try:
        _, status, raw = _run(fi_lib, Ad, Wp, M, N, K, stream)
    finally:
        fi_lib.swiglu_test_set_fault_injection(0)
    assert status == TIMEOUT_STATUS
    # The MMA waits for the stage that is never filled; the producers then
    # wait for stages that its MMAs never free. Whichever bounded wait runs
    # out first reports.
    assert raw & (MMA_TIMEOUT_BIT | PRODUCER_TIMEOUT_BIT)

    # 2) the word was cleared by the read, and the context still works
    Y, status, raw = _run(fi_lib, Ad, Wp, M, N, K, stream)
    assert status == 0 and raw == 0
    r = compare(from_device_bf16(Y), oracle.swiglu_up(A, W1, W2)["Y"])
    assert r["mismatches"] == 0 and r["over_bound"] == 0, r


@pytest.mark.parametrize("tile,mode,M,N,K", [
    (t, mode, M, N, K) for t in ("64", "256", "512")
    for mode, M, N, K in (("auto", 512, 2048, 512), ("dp", 512, 512, 512))
] + [("128", "auto", 16, 2048, 512), ("128", "dp", 64, 512, 512)])
def test_down_projection_wait_timeout(fi_lib, monkeypatch, tile, mode, M, N, K):
    """The same for the down-projection, on each of its kernels (the 1-SM
    kernel's plain mode, tile 64, the CTA-pair kernel's plain mode, tile 256,
    the wide kernel, tile 512, and the decode kernel, tile 128), with
    stream-K split tiles (auto: 4 or 2 output tiles on many pairs; the decode
    kernel: 4 tiles of 128 columns, each in 8 K ranges on a cluster) and with
    whole tiles: the timeout is reported and the next call is correct."""
    monkeypatch.setenv("SWIGLU_DOWN_TILE", tile)
    if mode != "auto":
        monkeypatch.setenv("SWIGLU_SCHEDULE", mode)
    elif tile == "512":
        monkeypatch.setenv("SWIGLU_SCHEDULE", "sk")   # the wide kernel's split tiles
    import oracle
    lib = fi_lib
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.swiglu_pack_down_weights.argtypes = [vp, i64, i64, vp, vp]
    lib.swiglu_down_packed_weight_bytes.argtypes = [i64, i64]
    lib.swiglu_down_packed_weight_bytes.restype = sz
    lib.swiglu_down_workspace_bytes.argtypes = [i64, i64, i64]
    lib.swiglu_down_workspace_bytes.restype = sz
    lib.swiglu_down_forward.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
    rng = np.random.Generator(np.random.PCG64(78))
    Yb = workloads.f32_to_bf16_bits(rng.standard_normal(size=(M, N), dtype=np.float32))
    W3 = workloads.f32_to_bf16_bits(
        rng.standard_normal(size=(N, K), dtype=np.float32) * np.float32(N ** -0.5))
    Yd, W3d = to_device_bf16(Yb, "cuda"), to_device_bf16(W3, "cuda")
    W3p = torch.empty(lib.swiglu_down_packed_weight_bytes(N, K), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.swiglu_pack_down_weights(W3d.data_ptr(), N, K, W3p.data_ptr(), stream) == 0
    ws_bytes = lib.swiglu_down_workspace_bytes(M, N, K)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")

    def run():
        out = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        assert lib.swiglu_down_forward(Yd.data_ptr(), W3p.data_ptr(), out.data_ptr(), M, N, K,
                                       ws.data_ptr() if ws_bytes else None, ws_bytes,
                                       stream) == 0
        raw = ctypes.c_uint32(0)
        return out, lib.swiglu_check_device_status(stream, ctypes.byref(raw)), raw.value

    lib.swiglu_test_set_fault_injection(1)
    try:
        _, status, raw = run()
    finally:
        lib.swiglu_test_set_fault_injection(0)
    assert status == TIMEOUT_STATUS and raw & (MMA_TIMEOUT_BIT | PRODUCER_TIMEOUT_BIT), raw
    # an aborted launch may leave partial counts behind: zero the workspace again
    ws.zero_()
    out, status, raw = run()
    assert status == 0 and raw == 0
    r = compare(from_device_bf16(out), oracle.matmul(Yb, W3)["C"])
    assert r["mismatches"] == 0 and r["over_bound"] == 0, r


def _busy_and_run(lib, op, n_busy=120, busy_ns=300_000_000):
    """Other work holds `n_busy` SMs for `busy_ns` on another stream while
    `op(stream)` runs on this one. Returns (op status word, raw word,
    whether the busy kernel was still running when op's stream finished)."""
    lib.swiglu_test_busy_sms.argtypes = [ctypes.c_int, ctypes.c_ulonglong, ctypes.c_void_p]
    busy_stream = torch.cuda.Stream()
    busy_done = torch.cuda.Event()
    assert lib.swiglu_test_busy_sms(n_busy, busy_ns, busy_stream.cuda_stream) == 0
    busy_done.record(busy_stream)
    time.sleep(0.02)                                  # the busy blocks are resident by now
    stream = torch.cuda.current_stream()
    out = op(stream.cuda_stream)
    stream.synchronize()
    still_busy = not busy_done.query()
    raw = ctypes.c_uint32(0)
    status = lib.swiglu_check_device_status(stream.cuda_stream, ctypes.byref(raw))
    busy_stream.synchronize()
    return out, status, raw.value, still_busy


@pytest.mark.parametrize("kind", ["down", "down-wide", "down-decode", "up"])
def test_split_tiles_finish_while_other_work_holds_sms(fi_lib, monkeypatch, kind):
    """A K-split launch while a kernel on another stream holds 120 of the
    SMs for 300 ms: only some of its pairs can run at first. In the CTA-pair
    kernel a split tile's owner waits only for pairs that started before it
    (worker numbers follow the start order); in the wide down-projection
    kernel nobody waits (the last to count in on a part finishes it); in the
    decode kernel a CTA waits only for the CTAs of its own cluster, which are
    scheduled together. Either
    way the call completes on the free SMs, well within this build's ~10 ms
    wait limit, and is correct. (Were owners to wait for pairs not yet
    started, they would hold their SMs until the limit and report
    SWIGLU_ERR_DEVICE_TIMEOUT.)"""
    import oracle
    lib = fi_lib
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    if kind.startswith("down"):
        # CTA-pair kernel: 8 output tiles of 256 x 256, 64 k-blocks each,
        # stream-K over 64 pairs; wide kernel: 4 tiles of 256 x 512,
        # stream-K forced, on 32 pairs; decode kernel (16 rows): 8 tiles of
        # 128 columns, each in two K ranges on a cluster of 2 (a cluster
        # needs its CTAs' SMs free at once: pairs fit beside the busy kernel)
        tile = {"down-wide": "512", "down-decode": "128"}.get(kind, "256")
        monkeypatch.setenv("SWIGLU_DOWN_TILE", tile)
        if kind == "down-wide":
            monkeypatch.setenv("SWIGLU_SCHEDULE", "sk")
        if kind == "down-decode":
            monkeypatch.setenv("SWIGLU_DECODE_SPLITS", "2")
        M, N, K = (16 if kind == "down-decode" else 512), 4096, 1024
        lib.swiglu_pack_down_weights.argtypes = [vp, i64, i64, vp, vp]
        lib.swiglu_down_packed_weight_bytes.argtypes = [i64, i64]
        lib.swiglu_down_packed_weight_bytes.restype = sz
        lib.swiglu_down_workspace_bytes.argtypes = [i64, i64, i64]
        lib.swiglu_down_workspace_bytes.restype = sz
        lib.swiglu_down_forward.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
        rng = np.random.Generator(np.random.PCG64(79))
        Yb = workloads.f32_to_bf16_bits(rng.standard_normal(size=(M, N), dtype=np.float32))
        W3 = workloads.f32_to_bf16_bits(
            rng.standard_normal(size=(N, K), dtype=np.float32) * np.float32(N ** -0.5))
        Yd, W3d = to_device_bf16(Yb, "cuda"), to_device_bf16(W3, "cuda")
        W3p = torch.empty(lib.swiglu_down_packed_weight_bytes(N, K), dtype=torch.uint8,
                          device="cuda")
        st0 = torch.cuda.current_stream().cuda_stream
        assert lib.swiglu_pack_down_weights(W3d.data_ptr(), N, K, W3p.data_ptr(), st0) == 0
        ws_bytes = lib.swiglu_down_workspace_bytes(M, N, K)
        # the K split is planned (the decode kernel sums inside its clusters)
        assert (ws_bytes == 0) if kind == "down-decode" else (ws_bytes > 0)
        ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()

        def op(stream):
            out = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
            assert lib.swiglu_down_forward(Yd.data_ptr(), W3p.data_ptr(), out.data_ptr(), M, N,
                                           K, ws.data_ptr() if ws_bytes else None, ws_bytes,
                                           stream) == 0
            return out

        out, status, raw, still_busy = _busy_and_run(lib, op)
        assert status == 0 and raw == 0, raw
        want = oracle.matmul(Yb, W3)["C"]
    else:
        # forced stream-K on the CTA-pair kernel: 16 tiles, 64 k-blocks each
        monkeypatch.setenv("SWIGLU_FUSED_VARIANT", "2sm")
        monkeypatch.setenv("SWIGLU_SCHEDULE", "sk")
        M, N, K = 512, 1024, 4096
        A, W1, W2 = workloads.random_case(M, N, K, seed=80)
        Ad = to_device_bf16(A, "cuda")
        W1d, W2d = to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda")
        Wp = torch.empty(lib.swiglu_packed_weight_bytes(N, K), dtype=torch.uint8, device="cuda")
        st0 = torch.cuda.current_stream().cuda_stream
        assert lib.swiglu_pack_weights(W1d.data_ptr(), W2d.data_ptr(), K, N, Wp.data_ptr(),
                                       st0) == 0
        ws_bytes = lib.swiglu_workspace_bytes(M, N, K)
        assert ws_bytes > 0
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()

        def op(stream):
            Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
            assert lib.swiglu_up_forward(Ad.data_ptr(), Wp.data_ptr(), Y.data_ptr(), M, N, K,
                                         ws.data_ptr(), ws_bytes, stream) == 0
            return Y

        out, status, raw, still_busy = _busy_and_run(lib, op)
        assert status == 0 and raw == 0, raw
        want = oracle.swiglu_up(A, W1, W2)["Y"]
    # the call ran beside the busy kernel, not after it
    assert still_busy
    r = compare(from_device_bf16(out), want)
    assert r["mismatches"] == 0 and r["over_bound"] == 0, r


def test_dynamic_tile_counter_survives_a_timeout(fi_lib, monkeypatch):
    """A whole-tile launch of several waves on CTA pairs hands out tiles from
    a counter in the workspace. After a launch that times out, the same
    workspace (not zeroed again) must serve the next launch correctly: every
    pair counts itself out on its way through teardown, and the last one
    resets the counter."""
    monkeypatch.setenv("SWIGLU_FUSED_VARIANT", "2sm")
    monkeypatch.setenv("SWIGLU_DYNAMIC_TILES", "1")      # two waves: dynamic when asked
    import oracle
    M, N, K = 2048, 2432, 128
    A, W1, W2 = workloads.random_case(M, N, K, seed=83)
    Ad = to_device_bf16(A, "cuda")
    W1d, W2d = to_device_bf16(W1, "cuda"), to_device_bf16(W2, "cuda")
    Wp = torch.empty(fi_lib.swiglu_packed_weight_bytes(N, K), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert fi_lib.swiglu_pack_weights(W1d.data_ptr(), W2d.data_ptr(), K, N, Wp.data_ptr(),
                                      stream) == 0
    ws_bytes = fi_lib.swiglu_workspace_bytes(M, N, K)
    assert ws_bytes > 0                                       # the tile counters
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")

    def run():
        Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
        assert fi_lib.swiglu_up_forward(Ad.data_ptr(), Wp.data_ptr(), Y.data_ptr(), M, N, K,
                                        ws.data_ptr(), ws_bytes, stream) == 0
        raw = ctypes.c_uint32(0)
        return Y, fi_lib.swiglu_check_device_status(stream, ctypes.byref(raw)), raw.value

    fi_lib.swiglu_test_set_fault_injection(1)
    try:
        _, status, raw = run()
    finally:
        fi_lib.swiglu_test_set_fault_injection(0)
    assert status == TIMEOUT_STATUS and raw & (MMA_TIMEOUT_BIT | PRODUCER_TIMEOUT_BIT), raw
    assert not ws.any()                                       # counters back at zero
    want = oracle.swiglu_up(A, W1, W2)["Y"]
    for _ in range(2):
        Y, status, raw = run()
        assert status == 0 and raw == 0
        r = compare(from_device_bf16(Y), want)
        assert r["mismatches"] == 0 and r["over_bound"] == 0, r
