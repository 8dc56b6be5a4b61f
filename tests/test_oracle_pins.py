"""Pins for the CPU oracle.

Every check here ties the oracle to something other than itself: exact
rational arithmetic (``fractions.Fraction``), Python big-integer brute force on
tiny inputs, the defining properties of the Chinese Remainder Theorem, closed
forms, exact invariants of the method, and the a-priori error bound that
follows from rounding each scaled operand to the nearest integer.

Method: Ozaki scheme II as described on the "Day 12" page
(ithelp.ithome.com.tw), section "Profile 不能只看 Tensor Core" (stage list) and
section "為什麼 tile-local prologue 沒有直接贏" (quantisation steps).
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle
from fp64_gemm_emulation_exponent_gb300 import workloads

MODULI_ALL = [int(p) for p in oracle.moduli(20)]


def prod(xs):
    r = 1
    for x in xs:
        r *= x
    return r


# --------------------------------------------------------------------------
# Independent brute force (Python ints and Fractions, tiny inputs only)
# --------------------------------------------------------------------------
def bf_scale(vec, beta):
    if any(not math.isfinite(v) for v in vec):
        return oracle.NONFINITE
    amax = max((abs(v) for v in vec), default=0.0)
    if amax == 0.0:
        return 0
    return beta - math.frexp(amax)[1]


def bf_round(x, s):
    if s == oracle.NONFINITE:
        return 0
    return round(Fraction(x) * Fraction(2) ** s)  # Fraction rounds half to even


def bf_unscale(X, S):
    """Correctly rounded X * 2^-S (CPython int/int true division is correctly rounded)."""
    if X == 0:
        return 0.0
    try:
        if S >= 0:
            v = X / (1 << S)
        else:
            v = float(X << (-S))
    except OverflowError:
        v = math.inf if X > 0 else -math.inf
    if v == 0.0:
        v = math.copysign(0.0, X)
    return v


def bf_method(A, B, n):
    """C, X, s, t for the whole method by brute force."""
    M, K = A.shape
    _, N = B.shape
    beta = oracle.beta(K, n)
    s = [bf_scale(list(A[i, :]), beta) for i in range(M)]
    t = [bf_scale(list(B[:, j]), beta) for j in range(N)]
    Ap = [[bf_round(float(A[i, k]), s[i]) for k in range(K)] for i in range(M)]
    Bp = [[bf_round(float(B[k, j]), t[j]) for j in range(N)] for k in range(K)]
    X = [[sum(Ap[i][k] * Bp[k][j] for k in range(K)) for j in range(N)] for i in range(M)]
    C = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            if s[i] == oracle.NONFINITE or t[j] == oracle.NONFINITE:
                C[i, j] = math.nan
            else:
                C[i, j] = bf_unscale(X[i][j], s[i] + t[j])
    return C, X, s, t, Ap, Bp


def same_bits(x, y):
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.ascontiguousarray(y, dtype=np.float64)
    return np.array_equal(x.view(np.uint64), y.view(np.uint64))


def tiny_case(rng, M, N, K, kind="normal"):
    if kind == "normal":
        return rng.standard_normal((M, K)), rng.standard_normal((K, N))
    if kind == "wide":
        e1 = rng.integers(-40, 40, (M, K))
        e2 = rng.integers(-40, 40, (K, N))
        return np.ldexp(rng.standard_normal((M, K)), e1), np.ldexp(rng.standard_normal((K, N)), e2)
    raise ValueError(kind)


# --------------------------------------------------------------------------
# Moduli and bit budget
# --------------------------------------------------------------------------
def test_moduli_pairwise_coprime_and_int8_sized():
    assert len(MODULI_ALL) == 20
    for a in range(20):
        assert 2 <= MODULI_ALL[a] <= 256
        for b in range(a):
            assert math.gcd(MODULI_ALL[a], MODULI_ALL[b]) == 1


@pytest.mark.parametrize("n", list(range(2, 21)))
def test_beta_makes_crt_exact_and_is_near_maximal(n):
    P = prod(MODULI_ALL[:n])
    for K in [1, 2, 3, 5, 64, 255, 256, 257, 1000, 1024, 4096, 8192, 65536, 131071, 10**6]:
        try:
            beta = oracle.beta(K, n)
        except oracle.OracleError:
            # refused only when beta = 2 would already break exactness
            assert 2 * K * 2 ** (2 * 2) > P
            continue
        assert beta >= 1
        # |a'|,|b'| < 2^beta  =>  |sum| < K 2^(2 beta) <= P/2: exact symmetric lift
        assert 2 * K * 2 ** (2 * beta) <= P
        # two more bits would break it: the budget wastes at most one bit
        assert 2 * K * 2 ** (2 * (beta + 2)) > P


def test_beta_values_at_the_workloads():
    # worked out by hand from log2 P = 63.58 / 87.04 / 110.16 / 132.95 / 155.37
    assert oracle.beta(256, 14) == 50
    assert oracle.beta(1024, 14) == 49 and oracle.beta(1024, 8) == 26
    assert oracle.beta(4096, 14) == 48 and oracle.beta(4096, 8) == 25
    assert oracle.beta(8192, 14) == 48
    assert [oracle.beta(512, n) for n in (8, 11, 14, 17, 20)] == [26, 38, 50, 61, 72]
    assert [oracle.beta(65536, n) for n in (8, 11, 14, 17, 20)] == [23, 35, 46, 57, 69]


# --------------------------------------------------------------------------
# Stage 1 + 2: exponent scan, scaling and rounding to integers
# --------------------------------------------------------------------------
def special_matrix(rng, rows, cols):
    X = rng.standard_normal((rows, cols))
    X[0, :] = 0.0                                  # zero row
    X[1, :] = np.ldexp(rng.standard_normal(cols), -1060)  # subnormal-ish row
    X[1, 0] = 5e-324                               # smallest subnormal
    X[2, :] = np.ldexp(rng.standard_normal(cols), 1000)
    X[3, :] = -np.ldexp(np.ones(cols), 7)          # exact powers of two
    return X


@pytest.mark.parametrize("n", [8, 14, 20])
def test_scale_matches_frexp_and_uses_the_top_bit(n):
    rng = np.random.default_rng(11 + n)
    A = special_matrix(rng, 7, 9)
    B = special_matrix(rng, 5, 9).T.copy()  # 9 x 5, special columns
    s, t = oracle.scale(A, B, n)
    beta = oracle.beta(9, n)
    assert list(s) == [bf_scale(list(A[i]), beta) for i in range(7)]
    assert list(t) == [bf_scale(list(B[:, j]), beta) for j in range(5)]
    Ap = oracle.integers(A, s, True)
    for i in range(7):
        top = max(abs(int(v)) for v in Ap[i])
        if np.any(A[i] != 0):
            # |a'| <= 2^beta, and the largest entry keeps its leading bit
            assert 2 ** (beta - 1) <= top <= 2 ** beta
        else:
            assert top == 0


def test_scale_flags_nonfinite_rows_and_columns():
    A = np.ones((4, 3))
    A[1, 2] = math.inf
    A[3, 0] = math.nan
    B = np.ones((3, 5))
    B[0, 4] = -math.inf
    s, t = oracle.scale(A, B, 14)
    assert [int(v) == oracle.NONFINITE for v in s] == [False, True, False, True]
    assert [int(v) == oracle.NONFINITE for v in t] == [False] * 4 + [True]


def test_rounding_to_nearest_integer_ties_to_even():
    rng = np.random.default_rng(5)
    X = special_matrix(rng, 6, 8)
    X[4, :] = -X[4, :]
    X[5, :] = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.25, -7.75]  # exact ties at scale 0
    # scales keep |x 2^s| below 2^73, as the exponent scan guarantees
    sc = np.array([50, 1100, -950, 3, 60, 0], dtype=np.int32)
    out = oracle.integers(X, sc, True)
    for r in range(6):
        for c in range(8):
            exact = Fraction(float(X[r, c])) * Fraction(2) ** int(sc[r])
            v = int(out[r, c])
            assert out[r, c] == v and v == bf_round(float(X[r, c]), int(sc[r]))
            assert abs(exact - v) <= Fraction(1, 2)
            if abs(exact - v) == Fraction(1, 2):
                assert v % 2 == 0
    assert list(out[5]) == [0, 2, 2, 0, -2, -2, 3, -8]
    Y = rng.standard_normal((6, 8))
    colsc = np.array([10, 20, 30, 40, 50, 1, 2, 3], dtype=np.int32)
    outc = oracle.integers(Y, colsc, False)
    for r in range(6):
        for c in range(8):
            assert int(outc[r, c]) == bf_round(float(Y[r, c]), int(colsc[c]))


# --------------------------------------------------------------------------
# Stage 3: balanced residues
# --------------------------------------------------------------------------
def test_residues_balanced_representatives():
    rng = random.Random(3)
    vals = [0, 1, -1, 127, 128, -128, -129, 255, 256, -256, 2**52, -(2**52), 2**53 - 1]
    vals += [rng.randrange(-(2**53), 2**53) for _ in range(300)]
    # exact integers above 2^53: a 53-bit significand times a power of two
    vals += [rng.randrange(2**52, 2**53) * 2 ** rng.randrange(1, 20) * rng.choice([-1, 1]) for _ in range(300)]
    xp = np.array([float(v) for v in vals])
    assert all(int(x) == v for x, v in zip(xp, vals))
    r = oracle.residues(xp, 20)
    for k, p in enumerate(MODULI_ALL):
        lo, hi = -(p // 2), (p + 1) // 2 - 1
        for e, v in enumerate(vals):
            rv = int(r[k, e])
            assert lo <= rv <= hi
            assert (v - rv) % p == 0


def test_residues_cover_each_class_once():
    for p_idx, p in enumerate(MODULI_ALL):
        xs = np.arange(-3 * p, 3 * p, dtype=np.float64)
        r = oracle.residues(xs, p_idx + 1)[p_idx]
        seen = {}
        for x, rv in zip(xs, r):
            seen.setdefault(int(x) % p, set()).add(int(rv))
        assert all(len(v) == 1 for v in seen.values()) and len(seen) == p


# --------------------------------------------------------------------------
# Stages 4-5: per-modulus integer GEMM and mod reduction
# --------------------------------------------------------------------------
def test_gemm_mod_matches_integer_matmul():
    rng = np.random.default_rng(9)
    n, M, N, K = 5, 7, 6, 33
    ra = np.stack([rng.integers(-(p // 2), (p + 1) // 2, (M, K)) for p in MODULI_ALL[:n]]).astype(np.int8)
    rb = np.stack([rng.integers(-(p // 2), (p + 1) // 2, (K, N)) for p in MODULI_ALL[:n]]).astype(np.int8)
    raw, cmod = oracle.gemm_mod(ra, rb, n)
    for k, p in enumerate(MODULI_ALL[:n]):
        ref = ra[k].astype(np.int64) @ rb[k].astype(np.int64)
        assert np.array_equal(raw[k], ref)
        assert np.array_equal(cmod[k].astype(np.int64), np.mod(ref, p))


def test_gemm_mod_worst_case_magnitude_at_k_limit():
    # every product -128 * -128: the sum reaches 2^14 K, still inside int32 for K < 2^17
    K = 2**17 - 1
    ra = np.full((1, 1, K), -128, dtype=np.int8)
    rb = np.full((1, K, 1), -128, dtype=np.int8)
    raw, cmod = oracle.gemm_mod(ra, rb, 1)
    assert int(raw[0, 0, 0]) == 2**14 * K
    assert int(cmod[0, 0, 0]) == (2**14 * K) % 256


def test_dgemm_k_beyond_the_int32_range_is_the_exact_integer_product():
    # K >= 2^17: per-modulus sums may leave int32; the residues come from the
    # exact sums (the GPU splits K into int32-exact chunks), and for small
    # integer matrices the emulated product is the exact integer product
    rng = np.random.default_rng(17)
    K = 2**17 + 3
    A = rng.integers(-7, 8, (3, K)).astype(np.float64)
    B = rng.integers(-7, 8, (K, 2)).astype(np.float64)
    A[0] = -7.0
    B[:, 0] = -7.0  # C[0, 0] = 49 K, and every residue sum of that entry is large
    ref = A.astype(np.int64) @ B.astype(np.int64)
    C = oracle.dgemm(A, B, 14)
    assert np.array_equal(C, ref.astype(np.float64))


def test_gemm_mod_raw_sums_beyond_int32_are_refused():
    K = 2**17 + 1
    ra = np.full((1, 1, K), -128, dtype=np.int8)
    rb = np.full((1, K, 1), -128, dtype=np.int8)
    with pytest.raises(oracle.OracleError):
        oracle.gemm_mod(ra, rb, 1)


# --------------------------------------------------------------------------
# Stage 6: CRT and symmetric lift
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n", [2, 3, 8, 11, 14, 17, 20])
def test_crt_satisfies_the_defining_congruences(n):
    rng = np.random.default_rng(n)
    ps = MODULI_ALL[:n]
    P = prod(ps)
    cm = np.stack([rng.integers(0, p, 64) for p in ps]).astype(np.uint8)
    cm[:, 0] = 0
    X = oracle.limbs_to_int(oracle.crt(cm, n))
    for e in range(64):
        # X = c_k (mod p_k) for all k and -P/2 <= X < P/2 fix X uniquely (CRT)
        assert -P // 2 <= X[e] < P // 2 or (P % 2 == 0 and X[e] == -P // 2)
        for k, p in enumerate(ps):
            assert X[e] % p == int(cm[k, e])
    assert X[0] == 0


@pytest.mark.parametrize("n", [2, 8, 14, 20])
def test_crt_lift_boundary_convention(n):
    """The symmetric lift keeps X in [-P/2, P/2): P/2 - 1 is positive, the
    class of P/2 lifts to -P/2, and values a little inside either end stay
    where they are (P is even: 256 is a modulus)."""
    ps = MODULI_ALL[:n]
    P = prod(ps)
    assert P % 2 == 0
    half = P // 2
    xs = [half - 1, -half, half - 2, -half + 1, half - 1 - 12345, -half + 12345, 0, -1, 1,
          half - 1 - (P >> 20), -half + (P >> 20)]
    cm = np.array([[x % p for x in xs] for p in ps], dtype=np.uint8)
    X = oracle.limbs_to_int(oracle.crt(cm, n))
    assert X == xs
    # the class of +P/2 itself
    cm_half = np.array([[half % p] for p in ps], dtype=np.uint8)
    assert oracle.limbs_to_int(oracle.crt(cm_half, n)) == [-half]


def test_crt_recovers_extreme_products():
    # values right at the edge of what beta allows: +-K 2^(2 beta)
    for n in (8, 14, 20):
        K = 512
        beta = oracle.beta(K, n)
        vals = [K * 4**beta, -K * 4**beta, K * 4**beta - 1, 1, -1, 0]
        cm = np.array([[v % p for v in vals] for p in MODULI_ALL[:n]], dtype=np.uint8)
        assert oracle.limbs_to_int(oracle.crt(cm, n)) == vals


# --------------------------------------------------------------------------
# Stage 7: undo scaling with one rounding
# --------------------------------------------------------------------------
def to_limbs(v):
    u = v % (1 << 256)
    return [(u >> (32 * l)) & 0xFFFFFFFF for l in range(oracle.LIMBS)]


def test_round_is_correctly_rounded():
    rng = random.Random(17)
    cases = [(0, 0), (1, 0), (-1, 0), (3, 1), (5, 1), (7, 2), (2**53 + 1, 0), (2**53 + 3, 0),
             (-(2**53 + 1), 0), (2**54 + 2, 1), (1, 1074), (1, 1075), (3, 1075), (1, 1076),
             (-1, 1075), (-3, 1075), (2**52 - 1, 1074), (2**53 - 1, 1075), (2**150, -870),
             (2**150, -874), (-(2**150), -900), ((2**53 - 1) << 100, -1)]
    for _ in range(2000):
        bits = rng.randrange(1, 160)
        X = rng.randrange(1 << (bits - 1), 1 << bits) * rng.choice([-1, 1])
        cases.append((X, rng.randrange(-1200, 1300)))
    # exact halfway cases, both tie directions
    for _ in range(200):
        m = rng.randrange(2**52, 2**53)
        sh = rng.randrange(1, 60)
        X = (2 * m + 1) << (sh - 1)
        cases.append((X, rng.randrange(-100, 100)))
    X = np.array([to_limbs(x) for x, _ in cases], dtype=np.uint32)
    S = np.array([s for _, s in cases], dtype=np.int32)
    out = oracle.round_scaled(X, S)
    for (x, s), got in zip(cases, out):
        want = bf_unscale(x, s)
        assert np.float64(got).view(np.uint64) == np.float64(want).view(np.uint64), (x, s, got, want)


# --------------------------------------------------------------------------
# The whole method
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n", [3, 5, 8, 11, 14, 17, 20])
@pytest.mark.parametrize("kind", ["normal", "wide"])
def test_dgemm_equals_brute_force_on_tiny_inputs(n, kind):
    rng = np.random.default_rng(100 + n)
    for (M, N, K) in [(1, 1, 1), (3, 4, 5), (5, 2, 7), (2, 3, 16)]:
        try:
            oracle.beta(K, n)
        except oracle.OracleError:
            continue
        A, B = tiny_case(rng, M, N, K, kind)
        C = oracle.dgemm(A, B, n)
        Cb, Xb, s, t, Ap, Bp = bf_method(A, B, n)
        assert same_bits(C, Cb)
        # stage values
        so, to = oracle.scale(A, B, n)
        assert list(so) == s and list(to) == t
        Xd = oracle.limbs_to_int(oracle.direct(np.array(Ap, dtype=np.float64), np.array(Bp, dtype=np.float64)))
        assert Xd == [x for row in Xb for x in row]
        ra = oracle.residues(np.array(Ap, dtype=np.float64), n)
        rb = oracle.residues(np.array(Bp, dtype=np.float64), n)
        raw, cm = oracle.gemm_mod(ra, rb, n)
        assert oracle.limbs_to_int(oracle.crt(cm, n)) == Xd
        # the sampled entry point agrees with the full one
        ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        Cs, raws, cms, Xs = oracle.sample(A, B, n, ii.ravel(), jj.ravel())
        assert same_bits(Cs, C.ravel())
        assert np.array_equal(raws, raw.reshape(n, -1).T)
        assert oracle.limbs_to_int(Xs) == Xd


def exact_product(A, B):
    M, K = A.shape
    _, N = B.shape
    FA = [[Fraction(float(A[i, k])) for k in range(K)] for i in range(M)]
    FB = [[Fraction(float(B[k, j])) for j in range(N)] for k in range(K)]
    return [[sum(FA[i][k] * FB[k][j] for k in range(K)) for j in range(N)] for i in range(M)]


@pytest.mark.parametrize("n", [6, 8, 11, 14, 20])
def test_dgemm_within_the_rounding_error_bound(n):
    # a' = a 2^s - da, |da| <= 1/2: |C - AB| <= 2^-(t+1) sum|a| + 2^-(s+1) sum|b|
    # + K 2^-(s+t+2), plus half an ulp of C
    rng = np.random.default_rng(7 * n)
    M, N, K = 6, 5, 40
    A, B = tiny_case(rng, M, N, K, "wide")
    C = oracle.dgemm(A, B, n)
    s, t = oracle.scale(A, B, n)
    ex = exact_product(A, B)
    for i in range(M):
        for j in range(N):
            sa = sum(Fraction(abs(float(A[i, k]))) for k in range(K))
            sb = sum(Fraction(abs(float(B[k, j]))) for k in range(K))
            two = Fraction(2)
            bound = (two ** -(int(t[j]) + 1) * sa + two ** -(int(s[i]) + 1) * sb
                     + K * two ** -(int(s[i]) + int(t[j]) + 2))
            half_ulp = Fraction(math.ulp(float(C[i, j]))) / 2
            assert abs(Fraction(float(C[i, j])) - ex[i][j]) <= bound + half_ulp


def test_dgemm_exact_invariants():
    rng = np.random.default_rng(21)
    M, N, K = 9, 7, 50
    A, B = tiny_case(rng, M, N, K, "wide")
    for n in (8, 14):
        C = oracle.dgemm(A, B, n)
        perm = rng.permutation(K)
        assert same_bits(oracle.dgemm(A[:, perm], B[perm, :], n), C)       # order of k
        assert same_bits(oracle.dgemm(-A, B, n), -C)                         # sign
        assert same_bits(oracle.dgemm(B.T.copy(), A.T.copy(), n), C.T)      # transpose
        A2 = A.copy()
        A2[3] *= 2.0**40
        A2[5] *= 2.0**-33
        C2 = oracle.dgemm(A2, B, n)
        assert same_bits(C2[3], C[3] * 2.0**40) and same_bits(C2[5], C[5] * 2.0**-33)
        A3 = A.copy()
        A3[2] = 0.0
        B3 = B.copy()
        B3[:, 4] = 0.0
        C3 = oracle.dgemm(A3, B3, n)
        assert np.all(C3[2] == 0) and np.all(C3[:, 4] == 0)


def test_small_integer_matrices_are_exact():
    rng = np.random.default_rng(4)
    A = rng.integers(-(2**20), 2**20, (12, 16)).astype(np.float64)
    B = rng.integers(-(2**20), 2**20, (16, 10)).astype(np.float64)
    C = oracle.dgemm(A, B, 14)
    assert np.array_equal(C, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))


def test_k1_is_the_correctly_rounded_outer_product():
    rng = np.random.default_rng(8)
    a = rng.standard_normal((13, 1)) * 2.0 ** rng.integers(-30, 30, (13, 1))
    b = rng.standard_normal((1, 11)) * 2.0 ** rng.integers(-30, 30, (1, 11))
    # beta(1, 14) = 54 >= 53: no bit is rounded away, and a*b is one IEEE product
    assert same_bits(oracle.dgemm(a, b, 14), a * b)


def test_twenty_moduli_without_lost_bits_round_the_exact_product():
    # beta = 72 at K = 512: rows/columns spanning <= 2^19 lose no bit, so C is
    # the correctly rounded exact product
    rng = np.random.default_rng(31)
    M, N, K = 5, 4, 512
    A = np.ldexp(rng.uniform(0.5, 1, (M, K)) * rng.choice([-1, 1], (M, K)), rng.integers(-9, 10, (M, K)))
    B = np.ldexp(rng.uniform(0.5, 1, (K, N)) * rng.choice([-1, 1], (K, N)), rng.integers(-9, 10, (K, N)))
    assert oracle.beta(K, 20) == 72
    C = oracle.dgemm(A, B, 20)
    ex = exact_product(A, B)
    want = np.array([[float(ex[i][j]) for j in range(N)] for i in range(M)])  # Fraction -> float rounds correctly
    assert same_bits(C, want)


def test_nonfinite_rows_and_columns_give_nan():
    rng = np.random.default_rng(2)
    A, B = rng.standard_normal((4, 6)), rng.standard_normal((6, 5))
    A[1, 3] = math.inf
    B[2, 4] = math.nan
    C = oracle.dgemm(A, B, 14)
    assert np.all(np.isnan(C[1])) and np.all(np.isnan(C[:, 4]))
    mask = np.ones_like(C, dtype=bool)
    mask[1] = False
    mask[:, 4] = False
    assert np.all(np.isfinite(C[mask]))


def test_empty_and_k0():
    A = np.zeros((3, 0))
    B = np.zeros((0, 4))
    assert np.array_equal(oracle.dgemm(A, B, 14), np.zeros((3, 4)))
    assert oracle.dgemm(np.zeros((0, 5)), np.zeros((5, 2)), 14).shape == (0, 2)


# --------------------------------------------------------------------------
# Compensated reference and the tolerances
# --------------------------------------------------------------------------
def test_dot2_is_twice_working_precision():
    rng = np.random.default_rng(12)
    M, N, K = 4, 3, 64
    A = rng.standard_normal((M, K)) * 2.0 ** rng.integers(-20, 20, (M, K))
    B = rng.standard_normal((K, N))
    B[:, 0] = -B[:, 1]  # heavy cancellation against column 1 is fine too
    R = oracle.dot2(A, B)
    ex = exact_product(A, B)
    u = Fraction(1, 2**53)
    g = K * u / (1 - K * u)
    for i in range(M):
        for j in range(N):
            absdot = sum(abs(Fraction(float(A[i, k])) * Fraction(float(B[k, j]))) for k in range(K))
            assert abs(Fraction(float(R[i, j])) - ex[i][j]) <= u * abs(ex[i][j]) + g * g * absdot


def eta(C, R, absAB):
    return float(np.max(np.abs(C - R) / absAB))


def test_tolerances_of_the_moduli_counts():
    A, B = workloads.operands(48, 40, 512, "normal", 0)
    R = oracle.dot2(A, B)
    absAB = np.abs(A) @ np.abs(B)
    assert eta(oracle.dgemm(A, B, 14), R, absAB) <= 1e-14
    assert eta(oracle.dgemm(A, B, 11), R, absAB) <= 2.0**-30
    # 8 moduli give beta = 26 at K = 512: check the a-priori bound instead
    C8 = oracle.dgemm(A, B, 8)
    s, t = oracle.scale(A, B, 8)
    bound = (np.abs(A).sum(1)[:, None] * np.ldexp(1.0, -t - 1)[None, :]
             + np.ldexp(1.0, -s - 1)[:, None] * np.abs(B).sum(0)[None, :]
             + 512 * np.ldexp(1.0, -(s[:, None] + t[None, :] + 2)))
    assert np.all(np.abs(C8 - R) <= bound * (1 + 1e-12) + np.spacing(np.abs(C8)))
