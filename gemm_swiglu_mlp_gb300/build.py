"""Builds the in-tree C-ABI library libswiglu_gb300.so for sm_103a with nvcc.

    python -m gemm_swiglu_mlp_gb300.build [--force]

One translation unit, one -gencode (compute_103a -> sm_103a), static CUDA
runtime (the library needs no libcudart/libcuda at load time; the driver is
reached through cudaGetDriverEntryPointByVersion when a call needs it).
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libswiglu_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
SOURCES = [os.path.join(CSRC, "swiglu_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
    os.path.join(INCLUDE, "swiglu.h")]


def nvcc_path() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def nvcc_command(out_path: str, extra=()):
    return [nvcc_path(), "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3",
            "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I" + INCLUDE,
            "-Xptxas", "-v", *extra, "-o", out_path, *SOURCES]


def build_fault_injection_library(out_path: str) -> str:
    """Test-only build of the same sources with SWIGLU_TEST_FAULT_INJECTION:
    adds swiglu_test_set_fault_injection() and shortens the wait limit. Never
    used by the product binding; the failure-detection test loads it."""
    proc = subprocess.run(nvcc_command(out_path, extra=("-DSWIGLU_TEST_FAULT_INJECTION",)),
                          capture_output=True, text=True)
    if proc.returncode != 0:
        sys.stderr.write(proc.stdout + proc.stderr)
        raise RuntimeError("nvcc failed building the fault-injection test library")
    return out_path


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    proc = subprocess.run(nvcc_command(tmp), capture_output=True, text=True)
    log = proc.stdout + proc.stderr
    with open(os.path.join(PKG_DIR, "ptxas_info.txt"), "w") as f:
        f.write(log)
    if proc.returncode != 0:
        sys.stderr.write(log)
        raise RuntimeError("nvcc failed building %s" % LIB_NAME)
    if verbose:
        sys.stderr.write(log)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
