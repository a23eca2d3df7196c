"""Plain FP64 CPU oracle for Y = SiLU(A x W1) (.) (A x W2).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
CPU-baseline leg may import this package. The product library never calls it;
the two share no code, header, table or constant.

The arithmetic lives in ``swiglu_oracle.c`` (plain loops, binary64, one
BF16 round-to-nearest-even at the end); this module builds it with gcc and
marshals numpy arrays through ctypes. Definition followed: "Tile-Level
Activation Overlap for Efficient LLM Inference", Section 1 Introduction
(Gate = A x W1, Up = A x W2, Y = SiLU(Gate) (.) Up) and the technical
summary's problem statement; SiLU(x) = x / (1 + e^-x).

``matmul`` is the plain product C = A x B (binary64 sums, one BF16 rounding),
the down-projection out = Y x W3 that completes the gated MLP (the MLP whose
run time the paper's Figure 1 splits; the paper defines only Gate, Up and
Y); ``swiglu_mlp`` composes the two with Y rounded to BF16 in between, as
the fused kernel stores it.

Parity status: pinned (brute force with exact rationals on tiny shapes,
closed forms W1 = 0 / W2 = 0 / rank-1, SiLU identities and textbook values,
BF16 rounding on hand-built bit patterns including ties; FP8 E4M3 decoding
on hand-derived patterns and an exact field-by-field decoder, and the FP8
definition by exact-rational brute force with scales; the plain product and
the MLP composition by exact-rational brute force, column-selection and
scaling closed forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swiglu_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile swiglu_oracle.c into oracle/liboracle.so with gcc (no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
               "-pthread", "-fno-fast-math", "-ffp-contract=off",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_swiglu_up.argtypes = [u16p, u16p, u16p,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     u16p, f64p, f64p, f64p, ctypes.c_int]
    lib.oracle_swiglu_up.restype = ctypes.c_int
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_swiglu_up_fp8.argtypes = [u8p, u8p, u8p,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                         i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         u16p, f64p, f64p, f64p, ctypes.c_int]
    lib.oracle_swiglu_up_fp8.restype = ctypes.c_int
    lib.oracle_matmul.argtypes = [u16p, u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                  i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                  u16p, f64p, ctypes.c_int]
    lib.oracle_matmul.restype = ctypes.c_int
    _lib = lib
    return lib


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def double_to_bf16(x: float) -> int:
    return int(_load().oracle_double_to_bf16(float(x)))


def silu(x: float) -> float:
    return _load().oracle_silu(float(x))


def e4m3_to_double(bits: int) -> float:
    return _load().oracle_e4m3_to_double(int(bits))


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def swiglu_up(A: np.ndarray, W1: np.ndarray, W2: np.ndarray, rows=None,
              want_unrounded: bool = False, want_gate_up: bool = False,
              nthreads: int = 0, cols=None):
    """Oracle Y for BF16 bit-pattern inputs (numpy uint16).

    A is [M, K], W1 and W2 are [K, N]. ``rows`` selects output rows (default:
    all), ``cols`` = (n0, n1) a column range (default: all). Returns a dict
    with ``Y`` ([R, C] uint16 BF16 bits) and, on request, ``Yd`` (unrounded
    binary64 SiLU(g)*u), ``G`` and ``U`` (binary64 sums).
    """
    lib = _load()
    A = np.ascontiguousarray(A, dtype=np.uint16)
    W1 = np.ascontiguousarray(W1, dtype=np.uint16)
    W2 = np.ascontiguousarray(W2, dtype=np.uint16)
    M, K = A.shape
    K1, N = W1.shape
    if K1 != K or W2.shape != (K, N):
        raise ValueError("shape mismatch: A %s W1 %s W2 %s" % (A.shape, W1.shape, W2.shape))
    if rows is None:
        rows_arr = None
        R = M
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows_arr.shape[0]
    n0, n1 = (0, N) if cols is None else (int(cols[0]), int(cols[1]))
    C = max(0, n1 - n0)
    Y = np.empty((R, C), dtype=np.uint16)
    Yd = np.empty((R, C), dtype=np.float64) if want_unrounded else None
    G = np.empty((R, C), dtype=np.float64) if want_gate_up else None
    U = np.empty((R, C), dtype=np.float64) if want_gate_up else None
    rc = lib.oracle_swiglu_up(_ptr(A, ctypes.c_uint16), _ptr(W1, ctypes.c_uint16),
                              _ptr(W2, ctypes.c_uint16), M, N, K,
                              _ptr(rows_arr, ctypes.c_int64), R, n0, n1,
                              _ptr(Y, ctypes.c_uint16), _ptr(Yd, ctypes.c_double),
                              _ptr(G, ctypes.c_double), _ptr(U, ctypes.c_double),
                              int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_swiglu_up failed (status %d)" % rc)
    out = {"Y": Y}
    if want_unrounded:
        out["Yd"] = Yd
    if want_gate_up:
        out["G"] = G
        out["U"] = U
    return out


def swiglu_up_fp8(A8: np.ndarray, W18: np.ndarray, W28: np.ndarray, s_a: float, s_w1: float,
                  s_w2: float, rows=None, want_unrounded: bool = False,
                  want_gate_up: bool = False, nthreads: int = 0, cols=None):
    """Oracle Y for FP8 E4M3 inputs (numpy uint8) with per-tensor scales:
    A = s_a * A8 [M, K], W1 = s_w1 * W1_8 [K, N], W2 = s_w2 * W2_8 [K, N].
    Same outputs as swiglu_up (Y BF16 bits; G and U are the scaled sums)."""
    lib = _load()
    A8 = np.ascontiguousarray(A8, dtype=np.uint8)
    W18 = np.ascontiguousarray(W18, dtype=np.uint8)
    W28 = np.ascontiguousarray(W28, dtype=np.uint8)
    M, K = A8.shape
    K1, N = W18.shape
    if K1 != K or W28.shape != (K, N):
        raise ValueError("shape mismatch: A %s W1 %s W2 %s" % (A8.shape, W18.shape, W28.shape))
    if rows is None:
        rows_arr, R = None, M
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows_arr.shape[0]
    n0, n1 = (0, N) if cols is None else (int(cols[0]), int(cols[1]))
    C = max(0, n1 - n0)
    Y = np.empty((R, C), dtype=np.uint16)
    Yd = np.empty((R, C), dtype=np.float64) if want_unrounded else None
    G = np.empty((R, C), dtype=np.float64) if want_gate_up else None
    U = np.empty((R, C), dtype=np.float64) if want_gate_up else None
    rc = lib.oracle_swiglu_up_fp8(_ptr(A8, ctypes.c_uint8), _ptr(W18, ctypes.c_uint8),
                                  _ptr(W28, ctypes.c_uint8), M, N, K,
                                  float(s_a), float(s_w1), float(s_w2),
                                  _ptr(rows_arr, ctypes.c_int64), R, n0, n1,
                                  _ptr(Y, ctypes.c_uint16), _ptr(Yd, ctypes.c_double),
                                  _ptr(G, ctypes.c_double), _ptr(U, ctypes.c_double),
                                  int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_swiglu_up_fp8 failed (status %d)" % rc)
    out = {"Y": Y}
    if want_unrounded:
        out["Yd"] = Yd
    if want_gate_up:
        out["G"] = G
        out["U"] = U
    return out


def matmul(A: np.ndarray, B: np.ndarray, rows=None, cols=None, want_unrounded: bool = False,
           nthreads: int = 0):
    """Oracle C = A x B for BF16 bit patterns (A [M, K], B [K, N]): binary64
    sums in increasing k, one BF16 RNE rounding. Returns {"C": [R, C] uint16}
    and, on request, "Cd" (the unrounded sums). ``rows`` / ``cols`` as in
    swiglu_up."""
    lib = _load()
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    M, K = A.shape
    K1, N = B.shape
    if K1 != K:
        raise ValueError("shape mismatch: A %s B %s" % (A.shape, B.shape))
    if rows is None:
        rows_arr, R = None, M
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows_arr.shape[0]
    n0, n1 = (0, N) if cols is None else (int(cols[0]), int(cols[1]))
    C = np.empty((R, max(0, n1 - n0)), dtype=np.uint16)
    Cd = np.empty(C.shape, dtype=np.float64) if want_unrounded else None
    rc = lib.oracle_matmul(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), M, N, K,
                           _ptr(rows_arr, ctypes.c_int64), R, n0, n1,
                           _ptr(C, ctypes.c_uint16), _ptr(Cd, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_matmul failed (status %d)" % rc)
    out = {"C": C}
    if want_unrounded:
        out["Cd"] = Cd
    return out


def swiglu_mlp(A: np.ndarray, W1: np.ndarray, W2: np.ndarray, W3: np.ndarray, rows=None,
               nthreads: int = 0):
    """The whole gated MLP, out = Y x W3 with Y = SiLU(A x W1) (.) (A x W2)
    rounded to BF16 (as the fused up-projection stores it) and W3 [N, H].
    Output row m needs only row m of Y, so ``rows`` limits both products.
    Returns {"Y": [R, N], "out": [R, H]} (BF16 bits)."""
    up = swiglu_up(A, W1, W2, rows=rows, nthreads=nthreads)
    return {"Y": up["Y"], "out": matmul(up["Y"], W3, nthreads=nthreads)["C"]}
