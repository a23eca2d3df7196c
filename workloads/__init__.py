"""Seeded synthetic inputs shaped like the Qwen-2.5 gated-MLP up-projections.

Shared by the oracle-side tests and the CUDA-side tests and bench: this module
only draws random numbers and rounds them to BF16 bit patterns. It holds none
of the method's arithmetic (no products, sums or activations).

Shapes ("Tile-Level Activation Overlap for Efficient LLM Inference", Section 1
Introduction and the technical summary's results: Qwen-2.5 0.5B to 72B MLPs,
BF16). The pages print no batch sizes or value distributions; the token counts
M and the distributions below are this library's workload definition:

* A  ~ N(0, 1), W1 and W2 ~ N(0, 1/K) (std K^-1/2), drawn in binary32 with
  numpy's PCG64 and rounded to BF16 (round to nearest, ties to even).
* Seeds: A = 1000 + c, W1 = 2000 + c, W2 = 3000 + c, with c the row index of
  the table below ("1s" reuses row 1's seeds).
* "stress": A multiplied by 8 (an exact power of two) so that pre-activations
  have std ~8 and SiLU saturates at both ends.
* "outlier": round(0.01 K) columns of A, chosen by a PCG64 permutation with
  seed 4000 + c, are multiplied by 20 in binary32 before rounding to BF16.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    c: str            # row label: "0", "1", "1s", "2" ... "11"
    name: str
    M: int            # tokens
    K: int            # hidden size
    N: int            # intermediate size
    variant: str = "plain"   # "plain" | "stress" | "outlier"

    @property
    def seed_index(self) -> int:
        return int(self.c.rstrip("s"))

    @property
    def flops(self) -> int:
        """4*M*N*K: two products of 2*M*N*K multiply-adds each."""
        return 4 * self.M * self.N * self.K

    @property
    def roofline_bytes(self) -> int:
        """Compulsory HBM bytes: A, W1, W2 read once and Y written once, BF16."""
        return 2 * (self.M * self.K + 2 * self.K * self.N + self.M * self.N)


WORKLOADS = [
    Workload("0", "qwen2.5-0.5b", 128, 896, 4864),
    Workload("1", "qwen2.5-1.5b", 2048, 1536, 8960),
    Workload("1s", "qwen2.5-1.5b-stress", 2048, 1536, 8960, "stress"),
    Workload("2", "qwen2.5-7b-m1", 1, 3584, 18944),
    Workload("3", "qwen2.5-7b-m16", 16, 3584, 18944),
    Workload("4", "qwen2.5-7b-m128", 128, 3584, 18944),
    Workload("5", "qwen2.5-7b-m512", 512, 3584, 18944),
    Workload("6", "qwen2.5-7b-m2048", 2048, 3584, 18944),
    Workload("7", "qwen2.5-7b-m8192", 8192, 3584, 18944),
    Workload("8", "qwen2.5-32b-m64", 64, 5120, 27648, "outlier"),
    Workload("9", "qwen2.5-32b-m4096", 4096, 5120, 27648, "outlier"),
    Workload("10", "qwen2.5-72b-m32", 32, 8192, 29568),
    Workload("11", "qwen2.5-72b-m8192", 8192, 8192, 29568),
]

BY_LABEL = {w.c: w for w in WORKLOADS}
BY_NAME = {w.name: w for w in WORKLOADS}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """binary32 array -> BF16 bit patterns (uint16), round to nearest even.

    Adds 0x7FFF plus the lowest kept bit and truncates (the usual RNE trick;
    finite inputs cannot overflow 32 bits this way). NaNs map to a quiet NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).reshape(-1)
    out = np.empty(u.shape, dtype=np.uint16)
    step = 1 << 24
    for s in range(0, u.size, step):
        v = u[s:s + step]
        r = (v >> np.uint32(16)) & np.uint32(1)
        r += np.uint32(0x7FFF)
        r += v
        r >>= np.uint32(16)
        nan = (v & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
        if nan.any():
            r[nan] = (v[nan] >> np.uint32(16)) | np.uint32(0x40)
        out[s:s + step] = r
    return out.reshape(x.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> binary32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal(seed: int, shape, scale: float) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def make_A_f32(w: Workload) -> np.ndarray:
    c = w.seed_index
    a = _normal(1000 + c, (w.M, w.K), 1.0)
    if w.variant == "stress":
        a *= np.float32(8.0)
    elif w.variant == "outlier":
        n_out = int(round(0.01 * w.K))
        perm = np.random.Generator(np.random.PCG64(4000 + c)).permutation(w.K)
        a[:, perm[:n_out]] *= np.float32(20.0)
    return a


def make_W_f32(w: Workload, which: int) -> np.ndarray:
    """which = 1 (gate weight W1) or 2 (up weight W2); [K, N] row-major."""
    assert which in (1, 2)
    c = w.seed_index
    seed = (2000 if which == 1 else 3000) + c
    return _normal(seed, (w.K, w.N), float(w.K) ** -0.5)


def make_A(w: Workload) -> np.ndarray:
    return f32_to_bf16_bits(make_A_f32(w))


def make_W(w: Workload, which: int) -> np.ndarray:
    """which = 1 (gate weight W1) or 2 (up weight W2); [K, N] row-major BF16 bits."""
    return f32_to_bf16_bits(make_W_f32(w, which))


E4M3_MAX = 448.0


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Values -> FP8 E4M3 bit patterns (uint8), round to nearest even,
    saturating at +-448 (callers scale into range first). Computed in
    binary64: the spacing is 2^(e-3) in the binade [2^e, 2^(e+1)) for
    e >= -6 and 2^-9 below 2^-6 (subnormals)."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    q = np.exp2(e - 3)
    v = np.rint(a / q) * q                      # numpy rint: ties to even
    v = np.minimum(v, E4M3_MAX)
    out = np.zeros(x.shape, dtype=np.uint8)
    sub = v < 2.0 ** -6
    out[sub] = np.rint(v[sub] / 2.0 ** -9).astype(np.uint8)
    nz = ~sub
    en = np.floor(np.log2(v[nz]))
    man = np.rint((v[nz] / np.exp2(en) - 1.0) * 8).astype(np.int64)
    out[nz] = ((en.astype(np.int64) + 7) << 3 | man).astype(np.uint8)
    out[sign] |= np.uint8(0x80)
    return out


def e4m3_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """FP8 E4M3 bit patterns -> binary64 (exact; NaN for S.1111.111)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    e = (b >> 3) & 0xF
    m = b & 0x7
    v = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7))
    v = np.where((e == 0xF) & (m == 0x7), np.nan, v)
    return np.where(b & 0x80, -v, v)


def quantize_e4m3(x: np.ndarray):
    """Per-tensor FP8: scale s = amax / 448 (binary32), patterns of x / s.
    The quantized tensor stands for s * decode(patterns)."""
    x = np.asarray(x, dtype=np.float32)
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    s = np.float32(amax / E4M3_MAX) if amax > 0 else np.float32(1.0)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    step = 1 << 20                               # elementwise: chunks only bound temporaries
    for i in range(0, flat.size, step):
        out[i:i + step] = f32_to_e4m3_bits(flat[i:i + step].astype(np.float64) / float(s))
    return out.reshape(x.shape), float(s)


def make_inputs_fp8(w: Workload):
    """FP8 E4M3 versions of the same draws: (A8, W1_8, W2_8, s_a, s_w1, s_w2)."""
    a8, sa = quantize_e4m3(make_A_f32(w))
    w18, s1 = quantize_e4m3(make_W_f32(w, 1))
    w28, s2 = quantize_e4m3(make_W_f32(w, 2))
    return a8, w18, w28, sa, s1, s2


def random_case_fp8(M: int, N: int, K: int, seed: int, a_scale: float = 1.0):
    """A small seeded FP8 case: (A8, W1_8, W2_8, s_a, s_w1, s_w2)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal(size=(M, K), dtype=np.float32) * np.float32(a_scale)
    s = np.float32(float(max(K, 1)) ** -0.5)
    w1 = rng.standard_normal(size=(K, N), dtype=np.float32) * s
    w2 = rng.standard_normal(size=(K, N), dtype=np.float32) * s
    a8, sa = quantize_e4m3(a)
    w18, s1 = quantize_e4m3(w1)
    w28, s2 = quantize_e4m3(w2)
    return a8, w18, w28, sa, s1, s2


def make_W3(w: Workload) -> np.ndarray:
    """Down-projection weight W3 [N, K] ~ N(0, 1/N), seed 5000 + c: only for
    measuring the whole gated MLP, out = Y W3, around the up-projection."""
    return f32_to_bf16_bits(_normal(5000 + w.seed_index, (w.N, w.K), float(w.N) ** -0.5))


def make_inputs(w: Workload):
    """(A [M,K], W1 [K,N], W2 [K,N]) as BF16 bit patterns (uint16)."""
    return make_A(w), make_W(w, 1), make_W(w, 2)


def random_case(M: int, N: int, K: int, seed: int, a_scale: float = 1.0):
    """A small seeded case for parity tests at arbitrary (ragged) shapes."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal(size=(M, K), dtype=np.float32) * np.float32(a_scale)
    s = np.float32(float(max(K, 1)) ** -0.5)
    w1 = rng.standard_normal(size=(K, N), dtype=np.float32) * s
    w2 = rng.standard_normal(size=(K, N), dtype=np.float32) * s
    return f32_to_bf16_bits(a), f32_to_bf16_bits(w1), f32_to_bf16_bits(w2)


def make_inputs_device(w: Workload, device, fp8: bool = False):
    """The workload's inputs drawn on the GPU with torch's seeded generator
    (Philox), same distributions and seeds as the host recipe above but not
    the same values: for timing many shapes without host-side generation.

    Returns (A, W1, W2) as BF16 device tensors, or for fp8=True
    (A8, W1_8, W2_8, s_a, s_w1, s_w2) with E4M3 bytes as uint8 tensors and
    per-tensor scales s = amax / 448."""
    import torch

    c = w.seed_index

    def normal(seed, shape, scale):
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if scale != 1.0:
            x *= scale
        return x

    a = normal(1000 + c, (w.M, w.K), 1.0)
    if w.variant == "stress":
        a *= 8.0
    elif w.variant == "outlier":
        g = torch.Generator(device=device)
        g.manual_seed(4000 + c)
        cols = torch.randperm(w.K, generator=g, device=device)[:int(round(0.01 * w.K))]
        a[:, cols] *= 20.0
    w1 = normal(2000 + c, (w.K, w.N), float(w.K) ** -0.5)
    w2 = normal(3000 + c, (w.K, w.N), float(w.K) ** -0.5)
    if not fp8:
        return a.to(torch.bfloat16), w1.to(torch.bfloat16), w2.to(torch.bfloat16)

    def quant(x):
        amax = float(x.abs().max())
        s = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
        q = (x / s).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        return q.view(torch.uint8), s

    (a8, sa), (w18, s1), (w28, s2) = quant(a), quant(w1), quant(w2)
    return a8, w18, w28, sa, s1, s2
