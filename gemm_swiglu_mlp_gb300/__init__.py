"""Python binding of the GB300 fused SwiGLU up-projection C ABI (include/swiglu.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libswiglu_gb300.so. PyTorch supplies device memory and the current
stream; there is no CPU or PyTorch fallback, and the functions raise if the
library has not been built (``python -m gemm_swiglu_mlp_gb300.build``).

The names follow the C ABI:

    swiglu_packed_weight_bytes(N, K) -> int
    swiglu_pack_weights(W1, W2, Wpacked=None) -> Wpacked (uint8 tensor)
    swiglu_pack_weights_nk(W1, W2, Wpacked=None) -> Wpacked  (nn.Linear [N, K] weights)
    swiglu_workspace_bytes(M, N, K) -> int
    swiglu_up_forward(A, Wpacked, N, Y=None, workspace=None) -> Y
    swiglu_pack_weights_interleaved(W1, W2) / swiglu_up_forward_interleaved(A, Wp, N)
        (the column-interleaved packing, for comparison with the default)
    swiglu_check_device_status() -> raw status word (raises on timeout)
    swiglu_status_string(status) -> str

Y = SiLU(A x W1) (.) (A x W2) ("Tile-Level Activation Overlap for Efficient
LLM Inference", Section 1 Introduction), BF16 in and out, FP32 accumulation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

__all__ = [
    "SwigluError", "load_library", "swiglu_version", "swiglu_status_string",
    "swiglu_packed_weight_bytes", "swiglu_pack_weights", "swiglu_pack_weights_nk",
    "swiglu_workspace_bytes",
    "swiglu_up_forward", "swiglu_up_forward_noalloc", "swiglu_check_device_status",
    "swiglu_packed_weight_bytes_fp8", "swiglu_pack_weights_fp8", "swiglu_workspace_bytes_fp8",
    "swiglu_up_forward_fp8", "swiglu_down_packed_weight_bytes", "swiglu_pack_down_weights",
    "swiglu_pack_down_weights_nk", "swiglu_down_workspace_bytes", "swiglu_down_forward",
    "swiglu_mlp_workspace_bytes", "swiglu_mlp_forward", "swiglu_pack_weights_interleaved",
    "swiglu_up_forward_interleaved", "EXPORTED_SYMBOLS",
]

SWIGLU_OK = 0
SWIGLU_ERR_INVALID_ARG = 1
SWIGLU_ERR_UNSUPPORTED = 2
SWIGLU_ERR_CUDA = 3
SWIGLU_ERR_DEVICE_TIMEOUT = 4

EXPORTED_SYMBOLS = (
    "swiglu_version", "swiglu_status_string", "swiglu_packed_weight_bytes",
    "swiglu_pack_weights", "swiglu_pack_weights_nk", "swiglu_workspace_bytes",
    "swiglu_up_forward", "swiglu_up_forward_noalloc", "swiglu_check_device_status",
    "swiglu_packed_weight_bytes_fp8", "swiglu_pack_weights_fp8", "swiglu_workspace_bytes_fp8",
    "swiglu_up_forward_fp8", "swiglu_down_packed_weight_bytes", "swiglu_pack_down_weights",
    "swiglu_pack_down_weights_nk", "swiglu_down_workspace_bytes", "swiglu_down_forward",
    "swiglu_mlp_workspace_bytes", "swiglu_mlp_forward", "swiglu_pack_weights_interleaved",
    "swiglu_up_forward_interleaved",
)

_lock = threading.Lock()
_lib = None
_workspaces = {}   # (device index, stream handle) -> zero-initialised uint8 tensor
_ws_bytes = {}     # ([entry,] device index, M, N, K, kernel and schedule overrides) -> bytes


class SwigluError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, _status_name(status)))


def load_library(path: str = LIB_PATH):
    """Load libswiglu_gb300.so (no fallback: raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                "libswiglu_gb300.so is not built (%s); run "
                "`python -m gemm_swiglu_mlp_gb300.build`" % path)
        lib = ctypes.CDLL(path)
        vp, i64, sz, u32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32)
        lib.swiglu_version.argtypes = []
        lib.swiglu_version.restype = ctypes.c_int
        lib.swiglu_status_string.argtypes = [ctypes.c_int]
        lib.swiglu_status_string.restype = ctypes.c_char_p
        lib.swiglu_packed_weight_bytes.argtypes = [i64, i64]
        lib.swiglu_packed_weight_bytes.restype = sz
        lib.swiglu_pack_weights.argtypes = [vp, vp, i64, i64, vp, vp]
        lib.swiglu_pack_weights.restype = ctypes.c_int
        lib.swiglu_pack_weights_nk.argtypes = [vp, vp, i64, i64, vp, vp]
        lib.swiglu_pack_weights_nk.restype = ctypes.c_int
        lib.swiglu_workspace_bytes.argtypes = [i64, i64, i64]
        lib.swiglu_workspace_bytes.restype = sz
        lib.swiglu_up_forward.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.swiglu_up_forward.restype = ctypes.c_int
        lib.swiglu_up_forward_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        lib.swiglu_up_forward_noalloc.restype = ctypes.c_int
        lib.swiglu_packed_weight_bytes_fp8.argtypes = [i64, i64]
        lib.swiglu_packed_weight_bytes_fp8.restype = sz
        lib.swiglu_pack_weights_fp8.argtypes = [vp, vp, i64, i64, vp, vp]
        lib.swiglu_pack_weights_fp8.restype = ctypes.c_int
        lib.swiglu_workspace_bytes_fp8.argtypes = [i64, i64, i64]
        lib.swiglu_workspace_bytes_fp8.restype = sz
        f32 = ctypes.c_float
        lib.swiglu_up_forward_fp8.argtypes = [vp, vp, vp, i64, i64, i64, f32, f32, f32, vp, sz, vp]
        lib.swiglu_up_forward_fp8.restype = ctypes.c_int
        lib.swiglu_down_packed_weight_bytes.argtypes = [i64, i64]
        lib.swiglu_down_packed_weight_bytes.restype = sz
        lib.swiglu_pack_down_weights.argtypes = [vp, i64, i64, vp, vp]
        lib.swiglu_pack_down_weights.restype = ctypes.c_int
        lib.swiglu_pack_down_weights_nk.argtypes = [vp, i64, i64, vp, vp]
        lib.swiglu_pack_down_weights_nk.restype = ctypes.c_int
        lib.swiglu_down_workspace_bytes.argtypes = [i64, i64, i64]
        lib.swiglu_down_workspace_bytes.restype = sz
        lib.swiglu_down_forward.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.swiglu_down_forward.restype = ctypes.c_int
        lib.swiglu_mlp_workspace_bytes.argtypes = [i64, i64, i64]
        lib.swiglu_mlp_workspace_bytes.restype = sz
        lib.swiglu_mlp_forward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.swiglu_mlp_forward.restype = ctypes.c_int
        lib.swiglu_pack_weights_interleaved.argtypes = [vp, vp, i64, i64, vp, vp]
        lib.swiglu_pack_weights_interleaved.restype = ctypes.c_int
        lib.swiglu_up_forward_interleaved.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.swiglu_up_forward_interleaved.restype = ctypes.c_int
        lib.swiglu_check_device_status.argtypes = [vp, u32p]
        lib.swiglu_check_device_status.restype = ctypes.c_int
        _lib = lib
        return lib


def _status_name(status: int) -> str:
    try:
        return load_library().swiglu_status_string(int(status)).decode()
    except Exception:  # library missing: still give a readable message
        return "status %d" % status


def _check(status: int, what: str):
    if status != SWIGLU_OK:
        raise SwigluError(status, what)


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _require_bf16_cuda(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != torch.bfloat16:
        raise TypeError("%s must be bfloat16, got %s" % (name, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def swiglu_version() -> int:
    return load_library().swiglu_version()


def swiglu_status_string(status: int) -> str:
    return load_library().swiglu_status_string(int(status)).decode()


def swiglu_packed_weight_bytes(N: int, K: int) -> int:
    return int(load_library().swiglu_packed_weight_bytes(int(N), int(K)))


def swiglu_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().swiglu_workspace_bytes(int(M), int(N), int(K)))


def swiglu_pack_weights(W1: torch.Tensor, W2: torch.Tensor, Wpacked: torch.Tensor = None,
                        stream=None) -> torch.Tensor:
    """Pack W1, W2 ([K, N] BF16 each) into the library's fused weight operand."""
    return _pack_kn("swiglu_pack_weights", W1, W2, Wpacked, stream)


def swiglu_pack_weights_interleaved(W1: torch.Tensor, W2: torch.Tensor,
                                    Wpacked: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Pack W1, W2 ([K, N] BF16 each) column-interleaved (even packed rows
    Gate, odd rows Up), for swiglu_up_forward_interleaved."""
    return _pack_kn("swiglu_pack_weights_interleaved", W1, W2, Wpacked, stream)


def _pack_kn(entry: str, W1, W2, Wpacked, stream) -> torch.Tensor:
    lib = load_library()
    _require_bf16_cuda(W1, "W1")
    _require_bf16_cuda(W2, "W2")
    if W1.dim() != 2 or W1.shape != W2.shape:
        raise ValueError("W1 and W2 must both be [K, N]")
    K, N = W1.shape
    nbytes = swiglu_packed_weight_bytes(N, K)
    if Wpacked is None:
        Wpacked = torch.empty(nbytes, dtype=torch.uint8, device=W1.device)
    elif Wpacked.numel() * Wpacked.element_size() < nbytes or not Wpacked.is_contiguous():
        raise ValueError("Wpacked must be contiguous with at least %d bytes" % nbytes)
    with torch.cuda.device(W1.device):
        _check(getattr(lib, entry)(W1.data_ptr(), W2.data_ptr(), K, N, Wpacked.data_ptr(),
                                   _stream_handle(stream)), entry)
    return Wpacked


def swiglu_pack_weights_nk(W1: torch.Tensor, W2: torch.Tensor, Wpacked: torch.Tensor = None,
                           stream=None) -> torch.Tensor:
    """Pack nn.Linear-layout weights W1, W2 ([N, K] BF16 each, Gate = A W1^T)."""
    lib = load_library()
    _require_bf16_cuda(W1, "W1")
    _require_bf16_cuda(W2, "W2")
    if W1.dim() != 2 or W1.shape != W2.shape:
        raise ValueError("W1 and W2 must both be [N, K]")
    N, K = W1.shape
    nbytes = swiglu_packed_weight_bytes(N, K)
    if Wpacked is None:
        Wpacked = torch.empty(nbytes, dtype=torch.uint8, device=W1.device)
    elif Wpacked.numel() * Wpacked.element_size() < nbytes or not Wpacked.is_contiguous():
        raise ValueError("Wpacked must be contiguous with at least %d bytes" % nbytes)
    with torch.cuda.device(W1.device):
        _check(lib.swiglu_pack_weights_nk(W1.data_ptr(), W2.data_ptr(), N, K, Wpacked.data_ptr(),
                                          _stream_handle(stream)), "swiglu_pack_weights_nk")
    return Wpacked


def swiglu_up_forward(A: torch.Tensor, Wpacked: torch.Tensor, N: int, Y: torch.Tensor = None,
                      workspace: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Y[M, N] = SiLU(A x W1) (.) (A x W2) from A [M, K] BF16 and packed weights."""
    return _forward("swiglu_up_forward", A, Wpacked, N, Y, workspace, stream)


def swiglu_up_forward_interleaved(A: torch.Tensor, Wpacked: torch.Tensor, N: int,
                                  Y: torch.Tensor = None, workspace: torch.Tensor = None,
                                  stream=None) -> torch.Tensor:
    """swiglu_up_forward on weights from swiglu_pack_weights_interleaved."""
    return _forward("swiglu_up_forward_interleaved", A, Wpacked, N, Y, workspace, stream)


def _forward(entry: str, A, Wpacked, N, Y, workspace, stream) -> torch.Tensor:
    lib = load_library()
    _require_bf16_cuda(A, "A")
    if A.dim() != 2:
        raise ValueError("A must be [M, K]")
    M, K = A.shape
    N = int(N)
    need = swiglu_packed_weight_bytes(N, K)
    if not Wpacked.is_cuda or Wpacked.numel() * Wpacked.element_size() < need:
        raise ValueError("Wpacked must be a CUDA buffer of at least %d bytes" % need)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        _require_bf16_cuda(Y, "Y")
        if tuple(Y.shape) != (M, N):
            raise ValueError("Y must be [%d, %d]" % (M, N))
    dev = A.device.index
    switch = dev != torch.cuda.current_device()
    if switch:
        prev = torch.cuda.current_device()
        torch.cuda.set_device(dev)
    try:
        key = _plan_key(entry, dev, M, N, K)
        ws_need = _ws_bytes.get(key)
        if ws_need is None:
            ws_need = _ws_bytes[key] = swiglu_workspace_bytes(M, N, K)
        ws_ptr, ws_bytes = None, 0
        if ws_need:
            if workspace is None:
                workspace = _default_workspace(A.device, ws_need, stream)
            ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
        _check(getattr(lib, entry)(A.data_ptr(), Wpacked.data_ptr(), Y.data_ptr(), M, N, K,
                                   ws_ptr, ws_bytes, _stream_handle(stream)), entry)
    finally:
        if switch:
            torch.cuda.set_device(prev)
    return Y


def _default_workspace(device, nbytes: int, stream) -> torch.Tensor:
    """One zero-filled workspace per (device, stream), grown on demand. Calls
    on one stream run one after another, and each completed call leaves the
    workspace's counters at zero, so reuse across calls and shapes is safe.
    The zero fill is ordered on the same stream as the calls that use it."""
    dev = torch.device(device)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    key = (dev.index, int(s.cuda_stream))
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        if torch.cuda.is_current_stream_capturing():
            # an allocation made during capture belongs to the graph's pool
            raise SwigluError(SWIGLU_ERR_INVALID_ARG,
                              "this shape needs a workspace of %d bytes: allocate it before "
                              "capturing (swiglu_workspace_bytes) and pass workspace=" % nbytes)
        with torch.cuda.stream(s):
            ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def swiglu_up_forward_noalloc(A: torch.Tensor, Wpacked: torch.Tensor, N: int,
                              Y: torch.Tensor, stream=None) -> torch.Tensor:
    """The allocation-free forward: the caller passes Y; the library uses its
    own fixed device scratch instead of a workspace (include/swiglu.h)."""
    lib = load_library()
    _require_bf16_cuda(A, "A")
    _require_bf16_cuda(Y, "Y")
    M, K = A.shape
    N = int(N)
    if tuple(Y.shape) != (M, N):
        raise ValueError("Y must be [%d, %d]" % (M, N))
    with torch.cuda.device(A.device):
        _check(lib.swiglu_up_forward_noalloc(A.data_ptr(), Wpacked.data_ptr(), Y.data_ptr(),
                                             M, N, K, _stream_handle(stream)),
               "swiglu_up_forward_noalloc")
    return Y


_PLAN_SWITCHES = ("SWIGLU_FUSED_VARIANT", "SWIGLU_SCHEDULE", "SWIGLU_DYNAMIC_TILES",
                  "SWIGLU_GROUP_M", "SWIGLU_DOWN_TILE", "SWIGLU_DECODE_SPLITS",
                  "SWIGLU_SK_PAIRS")


def _plan_key(*head):
    """Cache key of a workspace size: the problem and every environment
    switch that can change the library's plan for it."""
    return tuple(head) + tuple(os.environ.get(k) for k in _PLAN_SWITCHES)


def _workspace_args(kind: str, fn, dev: int, M: int, N: int, K: int, device, workspace, stream):
    """(pointer, bytes) of the workspace for one call: the caller's, or this
    module's per-(device, stream) default, sized by the library's own query."""
    key = _plan_key(kind, dev, M, N, K)
    need = _ws_bytes.get(key)
    if need is None:
        need = _ws_bytes[key] = int(fn(M, N, K))
    if not need:
        return None, 0
    if workspace is None:
        workspace = _default_workspace(device, need, stream)
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


class _OnDevice:
    """Makes `device` current for the duration of a call."""

    def __init__(self, device):
        self.dev = device.index

    def __enter__(self):
        self.prev = torch.cuda.current_device()
        if self.dev != self.prev:
            torch.cuda.set_device(self.dev)

    def __exit__(self, *exc):
        if self.dev != self.prev:
            torch.cuda.set_device(self.prev)


def swiglu_down_packed_weight_bytes(N: int, K: int) -> int:
    return int(load_library().swiglu_down_packed_weight_bytes(int(N), int(K)))


def swiglu_down_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().swiglu_down_workspace_bytes(int(M), int(N), int(K)))


def swiglu_mlp_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().swiglu_mlp_workspace_bytes(int(M), int(N), int(K)))


def _pack_down(fn_name: str, W: torch.Tensor, N: int, K: int, W3packed, stream) -> torch.Tensor:
    lib = load_library()
    nbytes = swiglu_down_packed_weight_bytes(N, K)
    if W3packed is None:
        W3packed = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    elif W3packed.numel() * W3packed.element_size() < nbytes or not W3packed.is_contiguous():
        raise ValueError("W3packed must be contiguous with at least %d bytes" % nbytes)
    a, b = (N, K) if fn_name == "swiglu_pack_down_weights" else (K, N)
    with torch.cuda.device(W.device):
        _check(getattr(lib, fn_name)(W.data_ptr(), a, b, W3packed.data_ptr(),
                                     _stream_handle(stream)), fn_name)
    return W3packed


def swiglu_pack_down_weights(W3: torch.Tensor, W3packed: torch.Tensor = None,
                             stream=None) -> torch.Tensor:
    """Pack the down-projection weight W3 ([N, K] BF16, out = Y x W3)."""
    _require_bf16_cuda(W3, "W3")
    if W3.dim() != 2:
        raise ValueError("W3 must be [N, K]")
    N, K = W3.shape
    return _pack_down("swiglu_pack_down_weights", W3, N, K, W3packed, stream)


def swiglu_pack_down_weights_nk(W3t: torch.Tensor, W3packed: torch.Tensor = None,
                                stream=None) -> torch.Tensor:
    """Pack an nn.Linear-layout down-projection weight W3t ([K, N] BF16,
    out = Y x W3t^T): the same packed result as swiglu_pack_down_weights(W3t.T)."""
    _require_bf16_cuda(W3t, "W3t")
    if W3t.dim() != 2:
        raise ValueError("W3t must be [K, N]")
    K, N = W3t.shape
    return _pack_down("swiglu_pack_down_weights_nk", W3t, N, K, W3packed, stream)


def _out_tensor(t, shape, device, name):
    if t is None:
        return torch.empty(shape, dtype=torch.bfloat16, device=device)
    _require_bf16_cuda(t, name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must be %s" % (name, list(shape)))
    return t


def swiglu_down_forward(Y: torch.Tensor, W3packed: torch.Tensor, K: int, out: torch.Tensor = None,
                        workspace: torch.Tensor = None, stream=None) -> torch.Tensor:
    """out[M, K] = Y x W3 from Y [M, N] BF16 and packed W3 (plain product,
    FP32 accumulation, BF16 out)."""
    lib = load_library()
    _require_bf16_cuda(Y, "Y")
    if Y.dim() != 2:
        raise ValueError("Y must be [M, N]")
    M, N = Y.shape
    K = int(K)
    need = swiglu_down_packed_weight_bytes(N, K)
    if not W3packed.is_cuda or W3packed.numel() * W3packed.element_size() < need:
        raise ValueError("W3packed must be a CUDA buffer of at least %d bytes" % need)
    out = _out_tensor(out, (M, K), Y.device, "out")
    with _OnDevice(Y.device):
        ws_ptr, ws_bytes = _workspace_args("down", swiglu_down_workspace_bytes, Y.device.index,
                                           M, N, K, Y.device, workspace, stream)
        _check(lib.swiglu_down_forward(Y.data_ptr(), W3packed.data_ptr(), out.data_ptr(), M, N, K,
                                       ws_ptr, ws_bytes, _stream_handle(stream)),
               "swiglu_down_forward")
    return out


def swiglu_mlp_forward(A: torch.Tensor, Wpacked: torch.Tensor, W3packed: torch.Tensor, N: int,
                       Y: torch.Tensor = None, out: torch.Tensor = None,
                       workspace: torch.Tensor = None, stream=None) -> torch.Tensor:
    """The whole gated MLP, out[M, K] = (SiLU(A W1) (.) (A W2)) W3: the fused
    up-projection into Y [M, N] (caller's or a new buffer), then the
    down-projection. Returns out; Y holds the up-projection's output."""
    lib = load_library()
    _require_bf16_cuda(A, "A")
    if A.dim() != 2:
        raise ValueError("A must be [M, K]")
    M, K = A.shape
    N = int(N)
    for buf, nbytes, name in ((Wpacked, swiglu_packed_weight_bytes(N, K), "Wpacked"),
                              (W3packed, swiglu_down_packed_weight_bytes(N, K), "W3packed")):
        if not buf.is_cuda or buf.numel() * buf.element_size() < nbytes:
            raise ValueError("%s must be a CUDA buffer of at least %d bytes" % (name, nbytes))
    Y = _out_tensor(Y, (M, N), A.device, "Y")
    out = _out_tensor(out, (M, K), A.device, "out")
    with _OnDevice(A.device):
        ws_ptr, ws_bytes = _workspace_args("mlp", swiglu_mlp_workspace_bytes, A.device.index,
                                           M, N, K, A.device, workspace, stream)
        _check(lib.swiglu_mlp_forward(A.data_ptr(), Wpacked.data_ptr(), W3packed.data_ptr(),
                                      Y.data_ptr(), out.data_ptr(), M, N, K, ws_ptr, ws_bytes,
                                      _stream_handle(stream)), "swiglu_mlp_forward")
    return out


def _require_u8_cuda(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != torch.uint8:
        raise TypeError("%s must hold E4M3 bytes as uint8, got %s" % (name, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def swiglu_packed_weight_bytes_fp8(N: int, K: int) -> int:
    return int(load_library().swiglu_packed_weight_bytes_fp8(int(N), int(K)))


def swiglu_workspace_bytes_fp8(M: int, N: int, K: int) -> int:
    return int(load_library().swiglu_workspace_bytes_fp8(int(M), int(N), int(K)))


def swiglu_pack_weights_fp8(W1: torch.Tensor, W2: torch.Tensor, Wpacked: torch.Tensor = None,
                            stream=None) -> torch.Tensor:
    """Pack FP8 E4M3 weights W1, W2 ([K, N] uint8 bytes each)."""
    lib = load_library()
    _require_u8_cuda(W1, "W1")
    _require_u8_cuda(W2, "W2")
    if W1.dim() != 2 or W1.shape != W2.shape:
        raise ValueError("W1 and W2 must both be [K, N]")
    K, N = W1.shape
    nbytes = swiglu_packed_weight_bytes_fp8(N, K)
    if Wpacked is None:
        Wpacked = torch.empty(nbytes, dtype=torch.uint8, device=W1.device)
    with torch.cuda.device(W1.device):
        _check(lib.swiglu_pack_weights_fp8(W1.data_ptr(), W2.data_ptr(), K, N, Wpacked.data_ptr(),
                                           _stream_handle(stream)), "swiglu_pack_weights_fp8")
    return Wpacked


def swiglu_up_forward_fp8(A: torch.Tensor, Wpacked: torch.Tensor, N: int, scale_a: float,
                          scale_w1: float, scale_w2: float, Y: torch.Tensor = None,
                          workspace: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Y = SiLU(A W1) (.) (A W2) with A = scale_a*A8 ([M, K] E4M3 bytes) and
    packed FP8 weights standing for scale_w1*W1_8 and scale_w2*W2_8."""
    lib = load_library()
    _require_u8_cuda(A, "A")
    if A.dim() != 2:
        raise ValueError("A must be [M, K]")
    M, K = A.shape
    N = int(N)
    need = swiglu_packed_weight_bytes_fp8(N, K)
    if not Wpacked.is_cuda or Wpacked.numel() * Wpacked.element_size() < need:
        raise ValueError("Wpacked must be a CUDA buffer of at least %d bytes" % need)
    Y = _out_tensor(Y, (M, N), A.device, "Y")
    with torch.cuda.device(A.device):
        ws_need = swiglu_workspace_bytes_fp8(M, N, K)
        ws_ptr, ws_bytes = None, 0
        if ws_need:
            if workspace is None:
                workspace = _default_workspace(A.device, ws_need, stream)
            ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
        _check(lib.swiglu_up_forward_fp8(A.data_ptr(), Wpacked.data_ptr(), Y.data_ptr(), M, N, K,
                                         float(scale_a), float(scale_w1), float(scale_w2),
                                         ws_ptr, ws_bytes, _stream_handle(stream)),
               "swiglu_up_forward_fp8")
    return Y


def swiglu_check_device_status(stream=None) -> int:
    """Synchronize the stream and read/clear the device status word."""
    lib = load_library()
    raw = ctypes.c_uint32(0)
    st = lib.swiglu_check_device_status(_stream_handle(stream), ctypes.byref(raw))
    if st == SWIGLU_ERR_DEVICE_TIMEOUT:
        raise SwigluError(st, "device status word 0x%x" % raw.value)
    _check(st, "swiglu_check_device_status")
    return raw.value
