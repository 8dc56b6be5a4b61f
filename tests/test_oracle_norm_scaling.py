"""Pins for the oracle's sharper scaling rule (reading R15): scales from an
exactly computed bound on the 2-norm of each row of A and column of B,
2^s_i ||a_i||_2 <= 2^gamma, so that by Cauchy-Schwarz
sum_k |a'_ik||b'_kj| <= ||a'_i|| ||b'_j|| stays below P/2 with more bits per
operand than the largest-entry rule (reading R2) keeps.  The pages name only
"scale / exponent scan" and "exponent scaling" (the "Day 12" page,
ithelp.ithome.com.tw, sections "Profile 不能只看 Tensor Core" and
"為什麼 tile-local prologue 沒有直接贏"); its section "先定義公平比較" sets
the precision contract that a sharper scaling has to keep.

The checks tie the rule to exact arithmetic, not to a retyped formula:
Python Fraction brute force of the CRT exactness invariant
(2 max sum |a'||b'| < P, which the oracle's own CRT-vs-direct check also
enforces), the exact 2-norm against 2^gamma on both sides of the chosen
scale (it is the largest or next-largest admissible one), a closed form for
constant rows, order independence, and the method's exact invariants.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle

MODULI_ALL = [int(p) for p in oracle.moduli(20)]


def P_of(n):
    r = 1
    for p in MODULI_ALL[:n]:
        r *= p
    return r


def exact_norm2(vec):
    return sum(Fraction(float(v)) ** 2 for v in vec)


def round_even(x, s):
    return round(Fraction(float(x)) * Fraction(2) ** int(s))


def operands(M, N, K, seed, kind):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N))
    if kind == "wide":
        A *= np.ldexp(1.0, rng.integers(-30, 30, (M, K)))
        B *= np.ldexp(1.0, rng.integers(-30, 30, (K, N)))
    elif kind == "spiky":  # one dominant entry per row/column: the norm is the max
        A *= 1e-9
        B *= 1e-9
        A[np.arange(M), rng.integers(0, K, M)] = 3.0
        B[rng.integers(0, K, N), np.arange(N)] = -5.0
    elif kind == "special":
        A[0] = 0.0
        A[1 % M] = np.ldexp(rng.standard_normal(K), -1060)  # subnormal row
        B[:, 0] = np.ldexp(np.ones(K), 700)
        if K > 3:
            A[2 % M, :3] = 0.0
    return A, B


@pytest.mark.parametrize("n", [2, 3, 5, 8, 11, 14, 17, 20])
def test_gamma_keeps_the_lift_exact_at_the_norm_bound(n):
    """Two vectors of 2-norm 2^gamma plus the rounding slack sqrt(K)/2 give
    2 ||a'|| ||b'|| < P at every supported K; gamma is the largest value
    with 2^(2 gamma + 2) <= 2^floor(log2 P)."""
    P = P_of(n)
    for K in [1, 7, 64, 1000, 4096, 65536, 2**20, 2**22]:
        try:
            g = oracle.gamma(K, n)
        except oracle.OracleError:
            # unsupported only when sqrt(K) would exceed 2^(gamma - 2)
            g0 = (P.bit_length() - 1 - 2) // 2
            assert g0 < 1 or (K - 1).bit_length() > 2 * g0 - 4
            continue
        bound = Fraction(2) ** g + Fraction(math.isqrt(K) + 1, 2)
        assert 2 * bound * bound < P
        assert 2 ** (2 * g + 2) <= 2 ** (P.bit_length() - 1) < 2 ** (2 * g + 4)


@pytest.mark.parametrize("n", [8, 11, 14, 20])
@pytest.mark.parametrize("kind", ["normal", "wide", "spiky", "special"])
def test_norm_scales_keep_the_crt_invariant_and_are_near_maximal(n, kind):
    M, N, K = 6, 5, 37
    A, B = operands(M, N, K, seed=n * 7 + len(kind), kind=kind)
    g = oracle.gamma(K, n)
    s, t = oracle.scale(A, B, n, rule="norm")
    two_g = Fraction(2) ** (2 * g)
    for vecs, sc in ((list(A), s), (list(B.T), t)):
        for v, si in zip(vecs, sc):
            nrm = exact_norm2(v)
            if nrm == 0:
                assert si == 0
                continue
            # admissible: the scaled 2-norm is at most 2^gamma
            assert Fraction(2) ** (2 * int(si)) * nrm <= two_g
            # near-maximal: two more powers of two would exceed it (the bound
            # overestimates ||x||^2 by less than a factor 2 per entry plus the
            # window's slack, so the rule gives up at most one bit)
            assert Fraction(2) ** (2 * (int(si) + 2)) * nrm > two_g
    # the CRT exactness invariant on the integers themselves
    P = P_of(n)
    Ap = [[round_even(A[i, k], s[i]) for k in range(K)] for i in range(M)]
    Bp = [[round_even(B[k, j], t[j]) for j in range(N)] for k in range(K)]
    worst = max(sum(abs(Ap[i][k] * Bp[k][j]) for k in range(K)) for i in range(M) for j in range(N))
    assert 2 * worst < P
    oracle.dgemm(A, B, n, rule="norm")  # raises if the oracle's CRT ever differs from the direct sum


def test_norm_scales_give_more_bits_than_the_max_rule_on_gaussian_rows():
    """At K = 4096 the squared 2-norm of a Gaussian row is about 4096, while
    K times its largest entry squared is about 4096 x 14: the norm rule keeps
    at least one more bit on every row and column, about 1.2 on average
    (half-octave rounding of the bound gives back part of the ideal 1.9)."""
    A, B = operands(64, 48, 4096, seed=3, kind="normal")
    s_max, t_max = oracle.scale(A, B, 14)
    s_nrm, t_nrm = oracle.scale(A, B, 14, rule="norm")
    assert np.all(s_nrm >= s_max + 1) and np.all(t_nrm >= t_max + 1)
    assert np.mean(s_nrm - s_max) >= 1.1 and np.mean(t_nrm - t_max) >= 1.1


@pytest.mark.parametrize("e,m", [(0, 0), (-3, 2), (5, 5), (-1040, 3), (900, 1)])
def test_constant_rows_closed_form(e, m):
    """A row of K = 4^m entries all equal to 2^e: ||a||^2 = 4^m 4^e, every
    entry sits at the bottom of its half-octave, and the scale is
    gamma - e - m - 1 exactly (2^s ||a|| = 2^(gamma - 1))."""
    K = 4**m
    n = 14
    g = oracle.gamma(K, n)
    A = np.full((1, K), math.ldexp(1.0, e))
    B = np.ones((K, 1))
    s, _ = oracle.scale(A, B, n, rule="norm")
    assert int(s[0]) == g - e - m - 1


def test_half_octave_boundaries():
    """Single entries on both sides of sqrt(2) 2^e: the bound 2^(h+1) on x^2
    is tight to the half-octave, so the scale of a one-entry row steps
    exactly where x^2 crosses a power of two."""
    n, K = 14, 1
    g = oracle.gamma(K, n)
    r2 = math.sqrt(2.0)
    for e in [-1074 + 60, -20, -1, 0, 1, 37, 600]:
        for x in [math.ldexp(1.0, e), math.ldexp(r2, e), np.nextafter(math.ldexp(r2, e), 0.0),
                  np.nextafter(math.ldexp(r2, e), math.inf), np.nextafter(math.ldexp(2.0, e), 0.0)]:
            s, _ = oracle.scale(np.array([[x]]), np.ones((1, 1)), n, rule="norm")
            s = int(s[0])
            x2 = Fraction(float(x)) ** 2
            h = 0  # the exact floor(2 log2 |x|) from Fractions
            while Fraction(2) ** h <= x2:
                h += 1
            while Fraction(2) ** h > x2:
                h -= 1
            assert s == (2 * g - h - 1) // 2, (x, e)


def test_norm_scales_are_independent_of_the_order_of_k():
    A, B = operands(7, 9, 300, seed=11, kind="wide")
    perm = np.random.default_rng(1).permutation(300)
    s1, t1 = oracle.scale(A, B, 14, rule="norm")
    s2, t2 = oracle.scale(A[:, perm], B[perm, :], 14, rule="norm")
    assert np.array_equal(s1, s2) and np.array_equal(t1, t2)
    C1 = oracle.dgemm(A, B, 14, rule="norm")
    C2 = oracle.dgemm(A[:, perm], B[perm, :], 14, rule="norm")
    assert np.array_equal(C1.view(np.uint64), C2.view(np.uint64))


def test_norm_rule_exact_invariants():
    A, B = operands(9, 8, 50, seed=5, kind="normal")
    C = oracle.dgemm(A, B, 14, rule="norm")
    # sign
    assert np.array_equal(oracle.dgemm(-A, B, 14, rule="norm"), -C)
    # transpose: the rows of B^T are the columns of B, scaled by the same rule
    assert np.array_equal(oracle.dgemm(B.T.copy(), A.T.copy(), 14, rule="norm"), C.T)
    # a power-of-two row scaling moves the scale, not the integers
    A2 = A.copy()
    A2[3] *= 2.0**40
    C2 = oracle.dgemm(A2, B, 14, rule="norm")
    assert np.array_equal(C2[3], C[3] * 2.0**40)
    assert np.array_equal(np.delete(C2, 3, 0), np.delete(C, 3, 0))


def test_norm_rule_small_integer_matrices_are_exact():
    rng = np.random.default_rng(2)
    A = rng.integers(-1000, 1000, (11, 40)).astype(np.float64)
    B = rng.integers(-1000, 1000, (40, 13)).astype(np.float64)
    C = oracle.dgemm(A, B, 14, rule="norm")
    assert np.array_equal(C, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))


def test_norm_rule_flags_nonfinite_and_zero_rows():
    A, B = operands(4, 3, 10, seed=1, kind="normal")
    A[1, 4] = np.nan
    A[2] = 0.0
    B[7, 2] = np.inf
    s, t = oracle.scale(A, B, 14, rule="norm")
    assert s[1] == oracle.NONFINITE and t[2] == oracle.NONFINITE and s[2] == 0
    C = oracle.dgemm(A, B, 14, rule="norm")
    assert np.isnan(C[1]).all() and np.isnan(C[:, 2]).all()
    assert np.all(C[2, :2] == 0.0)
