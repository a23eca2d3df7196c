"""Pins for the oracle's plain product (the down-projection out = Y x W3) and
its composition with the up-projection into the whole gated MLP, checked
against things other than the oracle itself.

* C = A x B: brute force with exact rationals and exact BF16 rounding on
  tiny shapes; closed forms (B = 0; B a column selection, which copies
  columns of A bit for bit; exact power-of-two scaling).
* out = (SiLU(A W1) (.) (A W2)) W3: the same brute force through both
  products, with the intermediate Y rounded to BF16 (the fused kernel's
  output), and a column selection W3 that must return Y's columns.

Definition: "Tile-Level Activation Overlap for Efficient LLM Inference",
Section 1 Introduction (Gate = A x W1, Up = A x W2, Y = SiLU(Gate) (.) Up,
the MLP whose run time Figure 1 splits); the down-projection completing that
MLP is out = Y x W3, W3 [N, H].
"""
from fractions import Fraction

import numpy as np
import pytest

import workloads
from tests import exact


def _rand_bf16(rng, shape, scale=1.0):
    return workloads.f32_to_bf16_bits(
        rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale))


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 1), (3, 5, 7, 2), (8, 8, 8, 3),
                                         (2, 9, 4, 4), (7, 3, 8, 5)])
def test_matmul_bruteforce_exact_tiny(oracle_mod, M, N, K, seed):
    rng = np.random.Generator(np.random.PCG64(300 + seed))
    A = _rand_bf16(rng, (M, K), 2.0)
    B = _rand_bf16(rng, (K, N), 1.0)
    out = oracle_mod.matmul(A, B, want_unrounded=True)
    checked = 0
    for m in range(M):
        for n in range(N):
            c = exact.exact_dot(A[m, :], B[:, n])
            # <= 8 products of 8-bit significands: the binary64 sum is exact
            assert Fraction(out["Cd"][m, n]) == c
            if exact.near_tie(exact.frac_to_decimal(c)):
                continue
            assert int(out["C"][m, n]) == exact.round_bf16_exact(c), (m, n)
            checked += 1
    assert checked >= M * N - 1


def test_matmul_zero_weight_gives_zero(oracle_mod):
    A, B, _ = workloads.random_case(6, 20, 30, 21)
    B[:] = 0
    C = oracle_mod.matmul(A, B)["C"]
    assert np.all((C == 0x0000) | (C == 0x8000))


def test_matmul_column_selection_copies_columns(oracle_mod):
    # B[sigma(h), h] = 1.0 and zero elsewhere: C[:, h] = A[:, sigma(h)] exactly
    M, K, N = 9, 40, 24
    rng = np.random.Generator(np.random.PCG64(22))
    A = _rand_bf16(rng, (M, K), 3.0)
    A[A == 0x8000] = 0x3F80                    # no -0: a sum starting at +0 gives +0
    sigma = rng.permutation(K)[:N]
    B = np.zeros((K, N), np.uint16)
    B[sigma, np.arange(N)] = 0x3F80            # 1.0
    C = oracle_mod.matmul(A, B)["C"]
    assert np.array_equal(C, A[:, sigma])


def test_matmul_power_of_two_scaling(oracle_mod):
    A, B, _ = workloads.random_case(4, 24, 40, 23)
    C1 = oracle_mod.matmul(A, B, want_unrounded=True)["Cd"]
    B2 = B.copy()
    nz = (B2 & 0x7F80) != 0
    B2[nz] = B2[nz] + np.uint16(0x0080)        # x2 on every normal value
    C2 = oracle_mod.matmul(A, B2, want_unrounded=True)["Cd"]
    assert np.array_equal(C2, 2.0 * C1)


def test_matmul_catches_planted_mistakes(oracle_mod):
    """A dropped k term or a transposed operand changes the brute-force result."""
    M = N = K = 4
    rng = np.random.Generator(np.random.PCG64(24))
    A = _rand_bf16(rng, (M, K), 2.0)
    B = _rand_bf16(rng, (K, N))
    want = np.array([[exact.round_bf16_exact(exact.exact_dot(A[m], B[:, n])) for n in range(N)]
                     for m in range(M)], dtype=np.uint16)
    assert np.array_equal(oracle_mod.matmul(A, B)["C"], want)
    dropped = oracle_mod.matmul(A[:, :K - 1], B[:K - 1])["C"]
    transposed = oracle_mod.matmul(A, np.ascontiguousarray(B.T))["C"]
    for bad in (dropped, transposed):
        assert not np.array_equal(bad, want)


def test_matmul_rows_cols_and_threads(oracle_mod):
    A, B, _ = workloads.random_case(33, 50, 64, 25)
    full = oracle_mod.matmul(A, B, nthreads=1)["C"]
    assert np.array_equal(full, oracle_mod.matmul(A, B, nthreads=7)["C"])
    rows = [32, 0, 11, 11]
    assert np.array_equal(oracle_mod.matmul(A, B, rows=rows)["C"], full[rows])
    assert np.array_equal(oracle_mod.matmul(A, B, cols=(8, 40))["C"], full[:, 8:40])


@pytest.mark.parametrize("M,N,K,H,seed", [(2, 3, 4, 5, 1), (3, 8, 8, 4, 2), (1, 6, 2, 7, 3)])
def test_mlp_bruteforce_exact_tiny(oracle_mod, M, N, K, H, seed):
    """Both products by exact rationals: Y rounded to BF16 exactly (60-digit
    SiLU), then out = Y x W3 exactly and rounded."""
    rng = np.random.Generator(np.random.PCG64(400 + seed))
    A = _rand_bf16(rng, (M, K), 2.0)
    W1 = _rand_bf16(rng, (K, N))
    W2 = _rand_bf16(rng, (K, N))
    W3 = _rand_bf16(rng, (N, H))
    got = oracle_mod.swiglu_mlp(A, W1, W2, W3)
    checked = 0
    for m in range(M):
        y_row = []
        tie = False
        for n in range(N):
            g = exact.exact_dot(A[m], W1[:, n])
            u = exact.exact_dot(A[m], W2[:, n])
            y = exact.silu_decimal(exact.frac_to_decimal(g)) * exact.frac_to_decimal(u)
            tie |= exact.near_tie(y)
            y_row.append(exact.round_bf16_exact(y))
        if tie:
            continue
        assert np.array_equal(got["Y"][m], np.array(y_row, np.uint16))
        for h in range(H):
            c = exact.exact_dot(y_row, W3[:, h])
            if exact.near_tie(exact.frac_to_decimal(c)):
                continue
            assert int(got["out"][m, h]) == exact.round_bf16_exact(c), (m, h)
            checked += 1
    assert checked >= 1


def test_mlp_selection_down_weight_returns_y_columns(oracle_mod):
    M, N, K, H = 5, 32, 48, 12
    A, W1, W2 = workloads.random_case(M, N, K, 26)
    rng = np.random.Generator(np.random.PCG64(27))
    sigma = rng.permutation(N)[:H]
    W3 = np.zeros((N, H), np.uint16)
    W3[sigma, np.arange(H)] = 0x3F80
    got = oracle_mod.swiglu_mlp(A, W1, W2, W3)
    Y = got["Y"][:, sigma].copy()
    Y[Y == 0x8000] = 0                         # -0 in Y sums to +0
    assert np.array_equal(got["out"], Y)


def test_mlp_row_subset(oracle_mod):
    A, W1, W2 = workloads.random_case(20, 40, 56, 28)
    W3 = _rand_bf16(np.random.Generator(np.random.PCG64(29)), (40, 24), 40 ** -0.5)
    full = oracle_mod.swiglu_mlp(A, W1, W2, W3)["out"]
    rows = [19, 3, 3, 0]
    assert np.array_equal(oracle_mod.swiglu_mlp(A, W1, W2, W3, rows=rows)["out"], full[rows])
