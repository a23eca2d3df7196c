"""Pins for the CPU oracle, checked against things other than the oracle itself.

* BF16 rounding: hand-derived bit patterns (tests/golden/bf16_rne_cases.txt)
  and an exact-rational rounder on random doubles.
* SiLU: textbook closed forms and identities.
* Gate/Up sums: brute force with exact rationals on tiny shapes.
* Y: exact rationals + 60-digit decimal SiLU + exact RNE on tiny shapes.
* Closed forms: W1 = 0, W2 = 0, rank-1 inputs.

Definition pinned: "Tile-Level Activation Overlap for Efficient LLM Inference",
Section 1 Introduction (Gate = A x W1, Up = A x W2, Y = SiLU(Gate) (.) Up);
SiLU(x) = x / (1 + e^-x).
"""
import decimal
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import workloads
from tests import exact

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden_rne_cases():
    cases = []
    with open(os.path.join(HERE, "golden", "bf16_rne_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            x, e = line.split()[:2]
            cases.append((float.fromhex(x), int(e, 16)))
    return cases


@pytest.mark.parametrize("x,expected", _golden_rne_cases())
def test_bf16_rounding_hand_derived(oracle_mod, x, expected):
    assert oracle_mod.double_to_bf16(x) == expected


def test_bf16_rounding_matches_exact_rounder(oracle_mod):
    rng = np.random.Generator(np.random.PCG64(7))
    xs = []
    # random doubles over the whole BF16 range, including subnormals
    for e in range(-140, 128, 3):
        for _ in range(8):
            xs.append(float(rng.uniform(1, 2)) * 2.0 ** e * (1 if rng.integers(2) else -1))
    # exact ties and near-ties around random BF16 values
    for _ in range(200):
        b = int(rng.integers(0x0001, 0x7F7F))
        lo = float(exact.bf16_fraction(b))
        hi = float(exact.bf16_fraction(b + 1))
        mid = (lo + hi) / 2
        xs += [mid, math.nextafter(mid, 0), math.nextafter(mid, math.inf), -mid]
    for x in xs:
        assert oracle_mod.double_to_bf16(x) == exact.round_bf16_exact(Fraction(x)), x


def test_bf16_decode_all_patterns(oracle_mod):
    for b in list(range(0, 0x7F80, 97)) + [0x0001, 0x007F, 0x0080, 0x3F80, 0x7F7F,
                                            0x8001, 0xBF80, 0xFF7F]:
        assert Fraction(oracle_mod.bf16_to_double(b)) == exact.bf16_fraction(b), hex(b)


def test_silu_closed_forms(oracle_mod):
    # SiLU(0) = 0
    assert oracle_mod.silu(0.0) == 0.0
    # SiLU(1) = 1 / (1 + 1/e) = e / (1 + e)
    ctx = decimal.Context(prec=40)
    e = ctx.exp(decimal.Decimal(1))
    want = float(ctx.divide(e, ctx.add(1, e)))
    assert abs(oracle_mod.silu(1.0) - want) <= 2e-16
    # SiLU(ln 3) = ln 3 * 3/4 (sigmoid(ln 3) = 3 / 4)
    x = math.log(3.0)
    assert abs(oracle_mod.silu(x) - 0.75 * x) <= 4e-16
    # SiLU(-ln 3) = -ln 3 / 4
    assert abs(oracle_mod.silu(-x) + 0.25 * x) <= 4e-16
    # large positive: e^-x underflows relative to 1, SiLU(x) == x
    assert oracle_mod.silu(50.0) == 50.0
    # very negative: the limit -0
    y = oracle_mod.silu(-1000.0)
    assert y == 0.0 and math.copysign(1.0, y) < 0


@pytest.mark.parametrize("x", [0.125, 0.7, 1.5, 3.0, 7.25, 12.0, 30.0])
def test_silu_reflection_identity(oracle_mod, x):
    # sigmoid(-x) = 1 - sigmoid(x)  =>  SiLU(-x) = SiLU(x) - x
    lhs = oracle_mod.silu(-x)
    rhs = oracle_mod.silu(x) - x
    assert abs(lhs - rhs) <= 4e-16 * max(1.0, x)


def _rand_bf16(rng, shape, scale=1.0):
    return workloads.f32_to_bf16_bits(
        rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale))


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 1), (3, 5, 7, 2), (8, 8, 8, 3),
                                         (2, 9, 4, 4), (7, 3, 8, 5), (5, 6, 1, 6)])
def test_bruteforce_exact_tiny(oracle_mod, M, N, K, seed):
    rng = np.random.Generator(np.random.PCG64(100 + seed))
    A = _rand_bf16(rng, (M, K), 2.0)
    W1 = _rand_bf16(rng, (K, N), 1.0)
    W2 = _rand_bf16(rng, (K, N), 1.0)
    out = oracle_mod.swiglu_up(A, W1, W2, want_gate_up=True, want_unrounded=True)
    checked = 0
    for m in range(M):
        for n in range(N):
            g = exact.exact_dot(A[m, :], W1[:, n])
            u = exact.exact_dot(A[m, :], W2[:, n])
            # sums of <= 8 products of 8-bit significands fit in 53 bits: exact
            assert Fraction(out["G"][m, n]) == g
            assert Fraction(out["U"][m, n]) == u
            y = exact.silu_decimal(exact.frac_to_decimal(g)) * exact.frac_to_decimal(u)
            assert abs(out["Yd"][m, n] - float(y)) <= 1e-14 * abs(float(y)) + 1e-300
            if exact.near_tie(y):
                continue
            assert int(out["Y"][m, n]) == exact.round_bf16_exact(y), (m, n)
            checked += 1
    assert checked >= M * N - 1


def test_zero_gate_weight_gives_zero(oracle_mod):
    A, W1, W2 = workloads.random_case(9, 17, 33, 11)
    W1[:] = 0
    Y = oracle_mod.swiglu_up(A, W1, W2)["Y"]
    assert np.all((Y == 0x0000) | (Y == 0x8000))


def test_zero_up_weight_gives_zero(oracle_mod):
    A, W1, W2 = workloads.random_case(9, 17, 33, 12)
    W2[:] = 0
    Y = oracle_mod.swiglu_up(A, W1, W2)["Y"]
    assert np.all((Y == 0x0000) | (Y == 0x8000))


def test_rank_one_closed_form(oracle_mod):
    # A has one nonzero column k0: Gate = alpha_m beta_n and Up = alpha_m gamma_n
    # exactly, so Y = BF16(SiLU(alpha beta) * alpha gamma).
    M, N, K, k0 = 6, 10, 12, 5
    rng = np.random.Generator(np.random.PCG64(13))
    A = np.zeros((M, K), np.uint16)
    W1 = _rand_bf16(rng, (K, N), 1.0)
    W2 = _rand_bf16(rng, (K, N), 1.0)
    A[:, k0] = _rand_bf16(rng, (M,), 3.0)
    Y = oracle_mod.swiglu_up(A, W1, W2)["Y"]
    for m in range(M):
        for n in range(N):
            alpha = exact.bf16_fraction(A[m, k0])
            g = alpha * exact.bf16_fraction(W1[k0, n])
            u = alpha * exact.bf16_fraction(W2[k0, n])
            y = exact.silu_decimal(exact.frac_to_decimal(g)) * exact.frac_to_decimal(u)
            if exact.near_tie(y):
                continue
            assert int(Y[m, n]) == exact.round_bf16_exact(y)


def test_power_of_two_scaling_of_up(oracle_mod):
    # Up is linear in W2; scaling W2 by 2 (exact in BF16) scales Y by 2 exactly
    A, W1, W2 = workloads.random_case(4, 24, 40, 14)
    Y1 = oracle_mod.swiglu_up(A, W1, W2, want_unrounded=True)["Yd"]
    W2x2 = W2.copy()
    nz = (W2x2 & 0x7F80) != 0                      # normal numbers: add 1 to exponent
    W2x2[nz] = W2x2[nz] + np.uint16(0x0080)
    Y2 = oracle_mod.swiglu_up(A, W1, W2x2, want_unrounded=True)["Yd"]
    assert np.array_equal(Y2, 2.0 * Y1)


def test_row_subset_and_thread_count_invariance(oracle_mod):
    A, W1, W2 = workloads.random_case(37, 50, 64, 15)
    full = oracle_mod.swiglu_up(A, W1, W2, nthreads=1)["Y"]
    many = oracle_mod.swiglu_up(A, W1, W2, nthreads=8)["Y"]
    assert np.array_equal(full, many)
    rows = [36, 0, 17, 17, 5]
    sub = oracle_mod.swiglu_up(A, W1, W2, rows=rows)["Y"]
    assert np.array_equal(sub, full[rows])


def test_bruteforce_catches_planted_mistakes(oracle_mod):
    """The brute-force pin is sensitive: feeding the oracle a mistake (swapped
    Gate/Up weights, a dropped k term, a transposed weight) changes its output."""
    M, N, K = 4, 4, 4
    rng = np.random.Generator(np.random.PCG64(16))
    A = _rand_bf16(rng, (M, K), 2.0)
    W1 = _rand_bf16(rng, (K, N))
    W2 = _rand_bf16(rng, (K, N))
    want = np.array([[exact.round_bf16_exact(
        exact.silu_decimal(exact.frac_to_decimal(exact.exact_dot(A[m], W1[:, n])))
        * exact.frac_to_decimal(exact.exact_dot(A[m], W2[:, n])))
        for n in range(N)] for m in range(M)], dtype=np.uint16)
    assert np.array_equal(oracle_mod.swiglu_up(A, W1, W2)["Y"], want)
    swapped = oracle_mod.swiglu_up(A, W2, W1)["Y"]
    dropped = oracle_mod.swiglu_up(A[:, :K - 1], W1[:K - 1], W2[:K - 1])["Y"]
    transposed = oracle_mod.swiglu_up(A, np.ascontiguousarray(W1.T), W2)["Y"]
    for bad in (swapped, dropped, transposed):
        assert not np.array_equal(bad, want)


def test_workload_generator_is_seeded_and_bf16():
    w = workloads.Workload("0", "t", 4, 64, 32)
    a1, w11, w21 = workloads.make_inputs(w)
    a2, w12, w22 = workloads.make_inputs(w)
    assert np.array_equal(a1, a2) and np.array_equal(w11, w12) and np.array_equal(w21, w22)
    assert a1.dtype == np.uint16 and a1.shape == (4, 64) and w11.shape == (64, 32)
    # W ~ N(0, 1/K): sample std close to K^-1/2
    std = workloads.bf16_bits_to_f32(workloads.make_W(workloads.Workload("0", "t", 1, 256, 512), 1)).std()
    assert abs(std - 256 ** -0.5) < 0.05 * 256 ** -0.5


def test_workload_variants():
    s = workloads.BY_LABEL["1s"]
    p = workloads.BY_LABEL["1"]
    small_s = workloads.Workload("1s", "s", 4, 64, 8, "stress")
    small_p = workloads.Workload("1", "p", 4, 64, 8)
    a_s = workloads.bf16_bits_to_f32(workloads.make_A(small_s))
    a_p = workloads.bf16_bits_to_f32(workloads.make_A(small_p))
    assert np.array_equal(a_s, 8 * a_p)            # x8 is exact in BF16
    assert s.M == p.M and s.K == p.K and s.N == p.N
    o = workloads.Workload("8", "o", 8, 500, 8, "outlier")
    a_o = workloads.bf16_bits_to_f32(workloads.make_A(o))
    big_cols = np.where(np.abs(a_o).max(axis=0) > 6.0)[0]
    assert 1 <= len(big_cols) <= 5               # round(0.01 * 500) = 5 outlier columns


def test_column_range_matches_full(oracle_mod):
    A, W1, W2 = workloads.random_case(9, 70, 33, 17)
    full = oracle_mod.swiglu_up(A, W1, W2, want_gate_up=True)
    part = oracle_mod.swiglu_up(A, W1, W2, rows=[8, 2], cols=(13, 51), want_gate_up=True)
    assert np.array_equal(part["Y"], full["Y"][[8, 2], 13:51])
    assert np.array_equal(part["G"], full["G"][[8, 2], 13:51])
    with pytest.raises(RuntimeError):
        oracle_mod.swiglu_up(A, W1, W2, cols=(10, 71))


# ----------------------------------------------------------------- FP8 E4M3
def _golden_e4m3_cases():
    cases = []
    with open(os.path.join(HERE, "golden", "e4m3_decode_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            b, v = line.split()[:2]
            cases.append((int(b, 16), float("nan") if v == "nan" else float.fromhex(v)))
    return cases


@pytest.mark.parametrize("bits,value", _golden_e4m3_cases())
def test_e4m3_decode_hand_derived(oracle_mod, bits, value):
    got = oracle_mod.e4m3_to_double(bits)
    if math.isnan(value):
        assert math.isnan(got)
    else:
        assert got == value and math.copysign(1, got) == math.copysign(1, value)


def test_e4m3_decode_matches_field_decoder(oracle_mod):
    for b in range(256):
        if (b & 0x7F) == 0x7F:
            assert math.isnan(oracle_mod.e4m3_to_double(b))
            continue
        assert Fraction(oracle_mod.e4m3_to_double(b)) == exact.e4m3_fraction(b), hex(b)


def test_e4m3_quantizer_round_trip_and_ties():
    # every finite pattern encodes back to itself; ties go to the even pattern
    pats = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)
    vals = workloads.e4m3_bits_to_f64(pats)
    back = workloads.f32_to_e4m3_bits(vals)
    assert np.array_equal(back[vals != 0], pats[vals != 0])
    # 1 + 1/16 lies halfway between 1.0 (0x38, even) and 1.125 (0x39): -> 0x38
    # 1 + 3/16 lies halfway between 1.125 (odd) and 1.25 (0x3a, even): -> 0x3a
    # 2^-10 lies halfway between 0 and the smallest subnormal: -> 0
    got = workloads.f32_to_e4m3_bits(np.array([1 + 1 / 16, 1 + 3 / 16, 2.0 ** -10, 500.0]))
    assert got.tolist() == [0x38, 0x3A, 0x00, 0x7E]


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 1), (3, 5, 7, 2), (8, 8, 8, 3), (2, 9, 4, 4)])
def test_fp8_bruteforce_exact_tiny(oracle_mod, M, N, K, seed):
    A8, W18, W28, sa, s1, s2 = workloads.random_case_fp8(M, N, K, seed=200 + seed, a_scale=2.0)
    out = oracle_mod.swiglu_up_fp8(A8, W18, W28, sa, s1, s2, want_gate_up=True,
                                   want_unrounded=True)
    for m in range(M):
        for n in range(N):
            dg = sum((exact.e4m3_fraction(A8[m, k]) * exact.e4m3_fraction(W18[k, n])
                      for k in range(K)), Fraction(0))
            du = sum((exact.e4m3_fraction(A8[m, k]) * exact.e4m3_fraction(W28[k, n])
                      for k in range(K)), Fraction(0))
            g = dg * Fraction(sa) * Fraction(s1)
            u = du * Fraction(sa) * Fraction(s2)
            # the E4M3 sums are exact; scaling rounds once in binary64
            assert out["G"][m, n] == float(g) and out["U"][m, n] == float(u)
            y = exact.silu_decimal(exact.frac_to_decimal(g)) * exact.frac_to_decimal(u)
            if exact.near_tie(y):
                continue
            assert int(out["Y"][m, n]) == exact.round_bf16_exact(y), (m, n)


def test_fp8_unit_scales_equal_bf16_definition(oracle_mod):
    # E4M3 values are exact BF16 values: with unit scales both oracle entry
    # points must agree bit for bit
    A8, W18, W28, _, _, _ = workloads.random_case_fp8(5, 12, 16, seed=31)
    to_bf16 = lambda b: workloads.f32_to_bf16_bits(workloads.e4m3_bits_to_f64(b).astype(np.float32))
    y8 = oracle_mod.swiglu_up_fp8(A8, W18, W28, 1.0, 1.0, 1.0)["Y"]
    y16 = oracle_mod.swiglu_up(to_bf16(A8), to_bf16(W18), to_bf16(W28))["Y"]
    assert np.array_equal(y8, y16)
