"""GPU parity at the edges the kernels' exactness rests on, against the oracle.

1. The residue GEMM runs on fp16 tensor cores with fp32 accumulators in TMEM.
   It is exact only because every fp32 partial sum of a 1024-term chunk is
   an integer that fp32 holds exactly (at most 1024 * 2^14 = 2^24 in
   magnitude).  A K split of several chunks converts each with cvt.rni and
   adds them in int32; a split of at most 1024 terms is one chunk, reduced
   mod p in fp32 (q = round(x/p) estimated by an fma, r = x - q p exact).
   Residues drawn from data keep chunk sums near 2^17, so these tests feed
   crafted slices that drive every chunk to the bound (all products
   (-128)(-128) = 2^14: a chunk sum of exactly K 2^14, up to 2^24), one odd
   small term short of it (products of 2^14 and one of +-1, +-3, 127, ...),
   and the negative side (products of -16256), plus one-chunk sums spread
   over the whole range and every residue class, where the fp32 estimate of
   round(x/p) can go either way.  The int32 sums (out_kind 1), the residues
   mod p (out_kind 0) and the pair residues (out_kind 2) must equal the
   oracle's exact sums bit for bit, on the single-CTA kernel (K < 2048: one
   chunk up to K = 1024, several from there) and on the CTA-pair kernel
   (K >= 2048).

2. The combine's unscale rounds X 2^-(s+t) to nearest, ties to even, from
   integer bits (a funnel-shift path for normal results, a general one for
   subnormals and overflow).  Random residues give X with ~100 significant
   bits, so an exact halfway case never occurs by chance.  These tests feed
   residues of X = +-(odd 54-bit integer) 2^k (halfway between two doubles at
   any normal scale), of X = +-odd 2^k with S = k + 1075 (halfway between two
   subnormals), and the ties at the subnormal/normal boundary and at the
   overflow threshold, through all three input kinds and both combine kernels
   (runtime moduli count for narrow outputs, compile-time count for wide
   ones), against the oracle's Garner CRT and correctly rounded unscale.

3. The combine's quotient estimate q = round(S/P) may be off by one within
   P 2^-19 of the lift boundary +-P/2, where an exact lift decides; random
   residues land there about once in 2^18 outputs.  These tests put every
   output there (X = P/2 - 1 - d or -P/2 + d, from d = 0 up to the edge of
   that window), through all input kinds, both kernels and the limb output.

4. The quantiser rounds a 2^s to the nearest integer, ties to even; data
   rarely scale to exact halves.  These tests build rows and columns whose
   entries mostly do, at every integer width of the quantiser and through
   the fused row scan of ozk_dgemm.

Method: Ozaki scheme II on the "Day 12" page (ithelp.ithome.com.tw), sections
"Profile 不能只看 Tensor Core" (the integer GEMM per modulus, mod reduction,
CRT reconstruction, undo scaling) and "先定義公平比較" (the precision
contract: the integer stage is exact, the FP64 output one correct rounding).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from fp64_gemm_emulation_exponent_gb300 import ozk
from gpu_helpers import dev, f16_to_int, run_combine, run_gemm, run_lift, run_quantize, run_scale, same_bits

pytestmark = pytest.mark.gpu


# --------------------------------------------------------------------------
# 1. fp32 chunk sums at their bounds
# --------------------------------------------------------------------------
def f16_slices(r: np.ndarray, kpad: int) -> torch.Tensor:
    """int8 residues n x rows x K -> fp16 bit patterns n x rows x kpad (zero padded)."""
    n, rows, K = r.shape
    out = np.zeros((n, rows, kpad), dtype=np.float16)
    out[:, :, :K] = r.astype(np.float16)
    return dev(out.view(np.int16))


def crafted_operands(M, N, K, seed):
    """Two moduli's residues: modulus 0 with products (-128)(-128) = 2^14,
    modulus 1 with products (-128)(127) = -16256, each row of A and column of
    B holding at most one entry that breaks the pattern (a small or extreme
    value at the start, the end or a chunk edge of K).  Rows/columns whose
    special value is -128 (resp. 127 in B of modulus 1) keep the pattern, so
    their chunk sums sit exactly on the bound."""
    rng = np.random.default_rng(seed)
    ra = np.full((2, M, K), -128, dtype=np.int8)
    rb = np.empty((2, K, N), dtype=np.int8)
    rb[0] = -128
    rb[1] = 127
    spots = sorted({0, K - 1, min(K - 1, 255), min(K - 1, 256), min(K - 1, 1023), min(K - 1, 1024), K // 2})
    vals = np.array([-128, 1, -1, 3, -3, 127, 0, 2, -127, 64], dtype=np.int8)
    for i in range(M):
        v = vals[i % len(vals)]
        ra[:, i, spots[(i // len(vals)) % len(spots)]] = v
    for j in range(N):
        v = vals[(j * 7) % len(vals)]
        k = spots[(j // 3) % len(spots)]
        rb[0, k, j] = v
        rb[1, k, j] = v if v != -128 else 127
    # a few rows and columns with the pattern everywhere, whatever the table gave them
    ra[:, rng.integers(0, M, 4)] = -128
    for j in rng.integers(0, N, 4):
        rb[0, :, j] = -128
        rb[1, :, j] = 127
    return ra, rb


@pytest.mark.parametrize("K", [1024, 1088, 2048, 3072, 4096, 9000, 20000])
def test_gemm_chunk_sums_at_two_to_the_24(K):
    """1024-term chunks (single CTA at K = 1024, one chunk, and 1088, two;
    CTA pairs from 2048, up to 20 chunks, whose fp32 cuts add up before the
    one reduction): chunk sums of exactly 2^24, 2^24 - 2^14 + small odd
    terms, and their negative counterparts, bit-exact."""
    M, N, n = 300, 260, 2
    ra, rb = crafted_operands(M, N, K, seed=K)
    raw, cmod = oracle.gemm_mod(ra, rb, n)
    # the crafted sums really reach the bound: some chunk of modulus 0 is 2^24 exactly
    assert int(raw[0].max()) == K * 2**14  # every 1024-term chunk of a full row/column is 2^24
    kpad = ozk.ozk_kpad(K)
    a_sl = f16_slices(ra, kpad)
    b_sl = f16_slices(rb.transpose(0, 2, 1), kpad)
    out32, _ = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=1)
    assert np.array_equal(out32.cpu().numpy()[0, :, :, :N], raw)
    out8, _ = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=0)
    assert np.array_equal(out8.cpu().numpy()[:, :, :N], cmod)
    assert ozk.ozk_stream_status() == 0


@pytest.mark.parametrize("K", [255, 256, 512, 768, 960])
def test_gemm_one_chunk_sums_at_the_bound(K):
    """K below 1024, one chunk reduced in fp32: sums of exactly K 2^14 and
    just below, and their negative counterparts, bit-exact."""
    M, N, n = 300, 260, 2
    ra, rb = crafted_operands(M, N, K, seed=K)
    raw, cmod = oracle.gemm_mod(ra, rb, n)
    assert int(raw[0].max()) == K * 2**14  # a full row/column of (-128)(-128)
    kpad = ozk.ozk_kpad(K)
    a_sl = f16_slices(ra, kpad)
    b_sl = f16_slices(rb.transpose(0, 2, 1), kpad)
    out32, _ = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=1)
    assert np.array_equal(out32.cpu().numpy()[0, :, :, :N], raw)
    out8, _ = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=0)
    assert np.array_equal(out8.cpu().numpy()[:, :, :N], cmod)
    assert ozk.ozk_stream_status() == 0


def wide_sum_operands(n, M, N, K, seed):
    """Residues whose sums spread over the whole exact range: each row of A
    and column of B of one sign, magnitudes 88 to 128 (sums near +-K 2^13.5,
    about +-2^23.5 at K = 1024), every seventh row of A small (|r| <= 3,
    sums near zero, either sign) and one row of zeros."""
    rng = np.random.default_rng(seed)
    sa = rng.choice([-1, 1], size=(n, M, 1))
    sb = rng.choice([-1, 1], size=(n, 1, N))
    ra = np.where(sa > 0, 127 - rng.integers(0, 40, (n, M, K)), -128 + rng.integers(0, 40, (n, M, K)))
    rb = np.where(sb > 0, 127 - rng.integers(0, 40, (n, K, N)), -128 + rng.integers(0, 40, (n, K, N)))
    ra[:, ::7] = rng.integers(-3, 4, ra[:, ::7].shape)
    ra[:, 3] = 0
    return ra.astype(np.int8), rb.astype(np.int8)


@pytest.mark.parametrize("K", [1024, 333, 64])
def test_gemm_one_chunk_residues_over_the_whole_range(K):
    """One-chunk sums over [-2^24, 2^24] and every residue class of all 20
    moduli, among them sums within 2^-7 p of a half-integer multiple of p
    (x/p = j + 1/2 +- 1/(2p)), where at K = 1024 the fp32 estimate of
    round(x/p) is off by one for several hundred: residues (out_kind 0), int32 sums (1) and pair residues
    (2) bit-exact against the oracle."""
    M, N, n = 300, 260, 20
    ra, rb = wide_sum_operands(n, M, N, K, seed=K + 11)
    raw, cmod = oracle.gemm_mod(ra, rb, n)
    ps = [int(p) for p in oracle.moduli(n)]
    x = raw.astype(np.int64)
    assert np.abs(x).max() > K * 2**13
    near_half = [np.count_nonzero(np.isin(x[k] % p, [(p - 1) // 2, (p + 1) // 2, p // 2]) & (np.abs(x[k]) > K * 2**13))
                 for k, p in enumerate(ps)]
    assert min(near_half) > 20
    kpad = ozk.ozk_kpad(K)
    a_sl = f16_slices(ra, kpad)
    b_sl = f16_slices(rb.transpose(0, 2, 1), kpad)
    out8, _ = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=0)
    assert np.array_equal(out8.cpu().numpy()[:, :, :N], cmod)
    out32, _ = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=1)
    assert np.array_equal(out32.cpu().numpy()[0, :, :, :N], raw)
    out16, _ = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=2)
    g16 = out16.cpu().numpy()[:, :, :N].view(np.uint16).astype(np.int64)
    for j in range(n // 2):
        assert np.all(g16[j] < ps[2 * j] * ps[2 * j + 1])
        assert np.array_equal(g16[j] % ps[2 * j], cmod[2 * j].astype(np.int64))
        assert np.array_equal(g16[j] % ps[2 * j + 1], cmod[2 * j + 1].astype(np.int64))
    assert ozk.ozk_stream_status() == 0


def test_gemm_one_chunk_residue_planes_by_tma_store():
    """The one-chunk epilogue writes the residue planes by TMA stores of
    128 x 32 boxes, clipped at M and ldo: bit-exact against the oracle with
    ragged M and N, at two base offsets, and nothing written outside the
    planes; a base off the 16-byte grid is refused before any launch."""
    M, N, K, n = 333, 200, 500, 14
    ra, rb = wide_sum_operands(n, M, N, K, seed=3)
    _, cmod = oracle.gemm_mod(ra, rb, n)
    kpad = ozk.ozk_kpad(K)
    a_sl = f16_slices(ra, kpad)
    b_sl = f16_slices(rb.transpose(0, 2, 1), kpad)
    ldo = (N + 15) // 16 * 16
    for offset in (0, 16):
        buf = torch.full((offset + n * M * ldo + 64,), 0xEE, dtype=torch.uint8, device="cuda")
        out = buf[offset:offset + n * M * ldo].view(n, M, ldo)
        ozk.ozk_residue_gemm(M, N, K, a_sl, b_sl, n, 0, out, ldo, 1)
        got = buf.cpu().numpy()
        assert np.all(got[:offset] == 0xEE) and np.all(got[offset + n * M * ldo:] == 0xEE)
        assert np.array_equal(out.cpu().numpy()[:, :, :N], cmod)
    buf = torch.full((8 + n * M * ldo,), 0xEE, dtype=torch.uint8, device="cuda")
    with pytest.raises(ozk.OzkError) as e:
        ozk.ozk_residue_gemm(M, N, K, a_sl, b_sl, n, 0, buf[8:].view(n, M, ldo), ldo, 1)
    assert e.value.status == ozk.OZK_ERR_INVALID_ARG
    assert np.all(buf.cpu().numpy() == 0xEE)
    assert ozk.ozk_stream_status() == 0


def test_gemm_chunk_bound_split_k():
    """Split-K shares of the CTA-pair kernel, each share's chunks at 2^24."""
    M, N, n, K, splits = 260, 300, 2, 6144, 3
    ra, rb = crafted_operands(M, N, K, seed=5)
    raw, _ = oracle.gemm_mod(ra, rb, n)
    kpad = ozk.ozk_kpad(K)
    out32, _ = run_gemm(f16_slices(ra, kpad), f16_slices(rb.transpose(0, 2, 1), kpad), M, N, K, n,
                        out_kind=1, splits=splits)
    got = out32.cpu().numpy()[:, :, :, :N].astype(np.int64).sum(axis=0)
    assert np.array_equal(got, raw.astype(np.int64))
    assert ozk.ozk_stream_status() == 0


# --------------------------------------------------------------------------
# 2. round-to-even ties in the unscale
# --------------------------------------------------------------------------
def tie_problem(n, M, N, seed):
    """Exact halfway cases X 2^-S, S = s_i (t_j = 0).  Returns the byte
    residues (n x M x N), the pair residues ((n+1)/2 x M x N), s, t and the
    constructed X as Python ints for a spot check."""
    rng = np.random.default_rng(seed)
    ps = [int(p) for p in oracle.moduli(n)]
    P = 1
    for p in ps:
        P *= p
    kmax = (P // 2).bit_length() - 1 - 54  # odd54 2^k < 2^(54 + k) <= P/2
    assert kmax >= 0
    odd = np.zeros((M, N), dtype=np.int64)
    k = np.zeros((M, N), dtype=np.int64)
    s = np.zeros(M, dtype=np.int64)
    kind = rng.integers(0, 8, M)
    kind[:4] = [0, 1, 2, 3]
    for i in range(M):
        if kind[i] in (0, 4, 5, 6, 7):  # normal result: odd 54-bit significand, any k
            odd[i] = (1 << 53) | (rng.integers(0, 1 << 52, N) << 1) | 1
            k[i] = rng.integers(0, kmax + 1, N)
            s[i] = rng.integers(-850, 900)  # 53 + k - S stays in the normal exponent range
        elif kind[i] == 1:  # halfway between two subnormals: value = odd 2^-1075, odd < 2^53
            kr = int(rng.integers(0, kmax + 1))
            bits = rng.integers(2, 53, N)
            odd[i] = (np.int64(1) << (bits - 1)) | (rng.integers(0, 1 << 50, N) % (np.int64(1) << (bits - 1))) | 1
            k[i] = kr
            s[i] = kr + 1075
        elif kind[i] == 2:  # the largest subnormal tie: rounds up to the smallest normal
            kr = int(rng.integers(0, kmax + 1))
            odd[i] = (1 << 53) - 1
            k[i] = kr
            s[i] = kr + 1075
        else:  # (2^54 - 1) 2^970: halfway between the largest double and 2^1024 -> Inf
            kr = int(rng.integers(0, kmax + 1))
            odd[i] = (1 << 54) - 1
            k[i] = kr
            s[i] = kr - 970
    sign = rng.choice(np.array([-1, 1], dtype=np.int64), size=(M, N))

    def residues_mod(m):
        pk = np.array([pow(2, int(e), m) for e in range(int(k.max()) + 1)], dtype=np.int64)
        r = (odd % m) * pk[k] % m
        return np.where(sign < 0, (m - r) % m, r)

    cmod = np.stack([residues_mod(p) for p in ps]).astype(np.uint8)
    pairs = [residues_mod(ps[2 * j] * ps[2 * j + 1]) if 2 * j + 1 < n else residues_mod(ps[2 * j])
             for j in range((n + 1) // 2)]
    pair = np.stack(pairs).astype(np.uint16)
    spot = [(int(i), int(j)) for i, j in zip(rng.integers(0, M, 40), rng.integers(0, N, 40))]
    X = {(i, j): int(sign[i, j]) * int(odd[i, j]) * 2 ** int(k[i, j]) for i, j in spot}
    return cmod, pair, s.astype(np.int32), np.zeros(N, dtype=np.int32), X


def is_tie(x: int, S: int, got: float) -> bool:
    """x 2^-S lies exactly halfway between `got` and a neighbouring double."""
    exact = Fraction(x, 1) / Fraction(2) ** S if S >= 0 else Fraction(x * 2 ** (-S))
    if np.isinf(got):
        return exact == Fraction((2**54 - 1) * (1 if x > 0 else -1)) * Fraction(2) ** 970
    g = Fraction(got)
    other = Fraction(float(np.nextafter(got, np.inf if exact > g else -np.inf)))
    return exact == (g + other) / 2


@pytest.mark.parametrize("n", [8, 14, 20])
@pytest.mark.parametrize("M,N", [(96, 200), (1024, 1248)])
def test_crt_round_to_even_ties(n, M, N):
    """All outputs halfway cases, both parities of the kept bit, both signs;
    byte residues (in_kind 0), pair residues (2) and split int32 sums (1);
    the runtime-count kernel at 96 x 200, the compile-time-count kernel at
    1024 x 1248 (in_kind 0 and 2)."""
    cmod, pair, s, t, Xspot = tie_problem(n, M, N, seed=1000 * n + M)
    Xo = oracle.crt(cmod, n)
    for (i, j), x in Xspot.items():  # the oracle's CRT recovers the constructed X
        assert oracle.limbs_to_int(Xo[i, j]) == x
    S = np.broadcast_to(s[:, None].astype(np.int64) + t[None, :], (M, N)).astype(np.int32)
    want = oracle.round_scaled(Xo.reshape(-1, oracle.LIMBS), S.ravel().copy()).reshape(M, N)
    for (i, j), x in Xspot.items():  # and they are exact ties
        assert is_tie(x, int(S[i, j]), float(want[i, j]))
    ds, dt = dev(s), dev(t)
    ld8 = (N + 15) // 16 * 16
    planes8 = np.zeros((n, M, ld8), dtype=np.uint8)
    planes8[:, :, :N] = cmod
    C8 = run_combine(dev(planes8), 0, ld8, 1, ds, dt, M, N, n).cpu().numpy()
    assert same_bits(C8, want)
    ld16 = (N + 7) // 8 * 8
    planes16 = np.zeros((pair.shape[0], M, ld16), dtype=np.uint16)
    planes16[:, :, :N] = pair
    C16 = run_combine(dev(planes16.view(np.int16)), 2, ld16, 1, ds, dt, M, N, n).cpu().numpy()
    assert same_bits(C16, want)
    # int32 partial sums of two K shares whose residues add up to c mod p
    rng = np.random.default_rng(n + M)
    ps = oracle.moduli(n).astype(np.int64)[:, None, None]
    ld32 = (N + 3) // 4 * 4
    part0 = rng.integers(-(2**29), 2**29, (n, M, N))
    part1 = (cmod.astype(np.int64) - part0) % ps + ps * rng.integers(-(2**20), 2**20, (n, M, N))
    planes32 = np.zeros((2, n, M, ld32), dtype=np.int32)
    planes32[0, :, :, :N] = part0
    planes32[1, :, :, :N] = part1
    C32 = run_combine(dev(planes32), 1, ld32, 2, ds, dt, M, N, n).cpu().numpy()
    assert same_bits(C32, want)
    # the lifted integers themselves
    X8 = run_lift(dev(planes8), 0, ld8, 1, M, N, n).cpu().numpy().view(np.uint32)
    assert np.array_equal(X8, Xo)
    assert ozk.ozk_stream_status() == 0


# --------------------------------------------------------------------------
# 3. the symmetric lift at its boundary
# --------------------------------------------------------------------------
def lift_boundary_problem(n, M, N, seed):
    """X within P 2^-19 of the lift boundary, X in [-P/2, P/2): P/2 - 1 - d or
    -P/2 + d.  There the combine's quotient estimate q = round(S/P) may be
    off by one and the exact lift decides.  Per row a size for d: zero (the
    two boundary values themselves), small, about P 2^-21, and about P 2^-19
    (the edge of the window the kernels check).  Returns byte residues,
    pair residues, s, t and a dict of spot-checked X."""
    rng = np.random.default_rng(seed)
    ps = [int(p) for p in oracle.moduli(n)]
    P = 1
    for p in ps:
        P *= p
    half = P // 2  # P is even (256 is a modulus): -P/2 <= X < P/2
    bits_p = P.bit_length()
    limbs = (bits_p + 31) // 32
    dbits = np.select([np.arange(M) % 4 == 0, np.arange(M) % 4 == 1, np.arange(M) % 4 == 2],
                      [0, 12, bits_p - 21], bits_p - 19)
    d = rng.integers(0, 2**32, (M, N, limbs), dtype=np.uint64)
    keep = np.clip(dbits[:, None] - 32 * np.arange(limbs)[None, :], 0, 32)  # bits of limb l kept in row i
    d &= ((np.uint64(1) << keep.astype(np.uint64)) - np.uint64(1))[:, None, :]
    neg = rng.integers(0, 2, (M, N)).astype(bool)

    def residues_mod(m):
        pw = np.array([pow(2, 32 * l, m) for l in range(limbs)], dtype=np.uint64)
        dm = (d % np.uint64(m) * pw).sum(axis=2).astype(np.int64) % m
        return np.where(neg, (dm - half % m) % m, ((half - 1) % m - dm) % m)

    cmod = np.stack([residues_mod(p) for p in ps]).astype(np.uint8)
    pair = np.stack([residues_mod(ps[2 * j] * ps[2 * j + 1]) if 2 * j + 1 < n else residues_mod(ps[2 * j])
                     for j in range((n + 1) // 2)]).astype(np.uint16)
    s = rng.integers(-800, 900, M).astype(np.int32)
    spot = [(int(i), int(j)) for i, j in zip(rng.integers(0, M, 60), rng.integers(0, N, 60))]
    spot += [(0, 0), (0, N - 1), (M - 1, 0)]

    def xval(i, j):
        dv = sum(int(d[i, j, l]) << (32 * l) for l in range(limbs))
        return -half + dv if neg[i, j] else half - 1 - dv

    return cmod, pair, s, np.zeros(N, dtype=np.int32), {(i, j): xval(i, j) for i, j in spot}


@pytest.mark.parametrize("n", [8, 14, 20])
@pytest.mark.parametrize("M,N", [(96, 200), (1024, 1248)])
def test_crt_lift_at_the_boundary(n, M, N):
    """Every output within P 2^-19 of +-P/2 (the two boundary values
    included): the lifted integers (from byte and pair residues) and C (byte,
    pair and split int32 inputs; the runtime-count kernel at 96 x 200, the
    compile-time-count kernel at 1024 x 1248) against the oracle."""
    cmod, pair, s, t, Xspot = lift_boundary_problem(n, M, N, seed=7000 + 100 * n + M)
    Xo = oracle.crt(cmod, n)
    for (i, j), x in Xspot.items():  # the oracle lifts to the constructed X
        assert oracle.limbs_to_int(Xo[i, j]) == x
    S = np.broadcast_to(s[:, None].astype(np.int64) + t[None, :], (M, N)).astype(np.int32)
    want = oracle.round_scaled(Xo.reshape(-1, oracle.LIMBS), S.ravel().copy()).reshape(M, N)
    ds, dt = dev(s), dev(t)
    ld8 = (N + 15) // 16 * 16
    planes8 = np.zeros((n, M, ld8), dtype=np.uint8)
    planes8[:, :, :N] = cmod
    assert np.array_equal(run_lift(dev(planes8), 0, ld8, 1, M, N, n).cpu().numpy().view(np.uint32), Xo)
    assert same_bits(run_combine(dev(planes8), 0, ld8, 1, ds, dt, M, N, n).cpu().numpy(), want)
    ld16 = (N + 7) // 8 * 8
    planes16 = np.zeros((pair.shape[0], M, ld16), dtype=np.uint16)
    planes16[:, :, :N] = pair
    p16 = dev(planes16.view(np.int16))
    assert np.array_equal(run_lift(p16, 2, ld16, 1, M, N, n).cpu().numpy().view(np.uint32), Xo)
    assert same_bits(run_combine(p16, 2, ld16, 1, ds, dt, M, N, n).cpu().numpy(), want)
    rng = np.random.default_rng(n * 31 + M)
    ps = oracle.moduli(n).astype(np.int64)[:, None, None]
    ld32 = (N + 3) // 4 * 4
    part0 = rng.integers(-(2**29), 2**29, (n, M, N))
    part1 = (cmod.astype(np.int64) - part0) % ps + ps * rng.integers(-(2**20), 2**20, (n, M, N))
    planes32 = np.zeros((2, n, M, ld32), dtype=np.int32)
    planes32[0, :, :, :N] = part0
    planes32[1, :, :, :N] = part1
    assert same_bits(run_combine(dev(planes32), 1, ld32, 2, ds, dt, M, N, n).cpu().numpy(), want)
    assert ozk.ozk_stream_status() == 0


# --------------------------------------------------------------------------
# 4. round-to-nearest-even ties in the quantiser
# --------------------------------------------------------------------------
def quantize_tie_operands(M, N, K, n, seed):
    """A and B whose scaled entries are mostly exact halves.  With the
    largest-entry rule a row (column) whose largest entry is 0.75 2^E (frexp
    exponent E) gets the scale beta - E, so an entry (2k+1) 2^(E - beta - 1)
    scales to (2k+1)/2: a tie, which rounds to the even neighbour.  About
    three entries in four are ties of either sign, the rest random below the
    largest; E varies from row to row."""
    rng = np.random.default_rng(seed)
    beta = oracle.beta(K, n)
    top = min(beta, 52)  # |2k+1| < 2^top stays exact in a double

    def lines(count, length):
        E = rng.integers(-60, 60, count)
        odd = (rng.integers(0, 2**(top - 1), (count, length)) * 2 + 1) * rng.choice([-1, 1], (count, length))
        x = np.ldexp(odd.astype(np.float64), (E - beta - 1)[:, None])
        plain = rng.random((count, length)) < 0.25
        x = np.where(plain, np.ldexp(rng.uniform(-0.7, 0.7, (count, length)), E[:, None]), x)
        x[np.arange(count), rng.integers(0, length, count)] = np.ldexp(0.75, E)  # the largest entry
        return x

    return lines(M, K), np.ascontiguousarray(lines(N, K).T)


@pytest.mark.parametrize("n,K", [(8, 300), (14, 1000), (17, 100), (17, 16), (18, 1000), (20, 700), (20, 64)])
def test_quantize_round_half_to_even(n, K):
    """Scales and every residue slice bit-exact against the oracle when most
    scaled entries are exact halves: beta 26, 49 and 62 (the two-word
    integer path of the quantiser), 63, 64, 72 and 74 (three words)."""
    M, N = 70, 90
    A, B = quantize_tie_operands(M, N, K, n, seed=n * 100 + K)
    s, t = run_scale(dev(A), dev(B), n)
    so, to = oracle.scale(A, B, n)
    assert np.array_equal(s.cpu().numpy(), so) and np.array_equal(t.cpu().numpy(), to)
    beta = oracle.beta(K, n)
    assert np.all(so == beta - np.frexp(np.abs(A).max(axis=1))[1])  # the construction's scale
    Ap = oracle.integers(A, so, True)
    ties = np.abs(np.ldexp(A, so[:, None]) - np.trunc(np.ldexp(A, so[:, None]))) == 0.5
    assert ties.mean() > 0.6 and np.all(Ap[ties] % 2 == 0)  # ties went to the even neighbour
    a_sl, b_sl = run_quantize(dev(A), dev(B), s, t, n)
    Bp = oracle.integers(B, to, False)
    ga = a_sl.cpu().numpy().view(np.uint16)
    gb = b_sl.cpu().numpy().view(np.uint16)
    assert np.array_equal(f16_to_int(ga[:, :, :K]), oracle.residues(Ap, n).astype(np.int64))
    assert np.array_equal(f16_to_int(gb[:, :, :K]), oracle.residues(Bp, n).transpose(0, 2, 1).astype(np.int64))
    assert ozk.ozk_stream_status() == 0


@pytest.mark.parametrize("n", [14, 20])
def test_dgemm_round_half_to_even_fused_row_scan(n):
    """The same ties through ozk_dgemm where the rows of A are scanned and
    quantised in one block each (M kpad >= 2^22, K <= 4096): sampled outputs
    bit-exact against the oracle."""
    M, N, K = 1100, 200, 4000
    A, B = quantize_tie_operands(M, N, K, n, seed=n)
    C = ozk.dgemm(dev(A), dev(B), n)
    torch.cuda.synchronize()
    assert ozk.ozk_stream_status() == 0
    rng = np.random.default_rng(n)
    ii = np.concatenate([rng.integers(0, M, 300), [0, M - 1]])
    jj = np.concatenate([rng.integers(0, N, 300), [N - 1, 0]])
    Cg = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    assert same_bits(Cg, oracle.sample(A, B, n, ii, jj)[0])
