"""GPU parity: the CUDA path through the C-ABI against the CPU oracle.

Integer stages (scales, residue slices, per-modulus int32 sums, reduced
residues, lifted integers) must match bit for bit.  The final FP64 C is the
correctly rounded value of an exact integer, so it must match bit for bit as
well; the error against the compensated reference is checked on top (the
tolerances of the precision contract: 1e-14 at 14+ moduli, 2^-30 at 11).

Method: Ozaki scheme II on the "Day 12" page (ithelp.ithome.com.tw), section
"Profile 不能只看 Tensor Core" (stage list).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from fp64_gemm_emulation_exponent_gb300 import ozk, workloads
from gpu_helpers import (f16_to_int, dev, dgemm, ld_of, run_combine, run_gemm, run_lift,
                         run_quantize, run_scale, same_bits, strided)

pytestmark = pytest.mark.gpu


def inputs(M, N, K, seed, kind="normal"):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N))
    if kind == "special":
        if M > 3:
            A[0] = 0.0
            A[1] = np.ldexp(rng.standard_normal(K), -1040)   # subnormal row
            A[2] = np.ldexp(rng.standard_normal(K), 900)     # huge row
            A[3] = np.ldexp(rng.standard_normal(K), rng.integers(-60, 60, K))  # wide row
        if N > 2:
            B[:, 0] = 0.0
            B[:, 1] = np.ldexp(rng.standard_normal(K), -300)
            B[:, 2] = -np.ldexp(np.ones(K), 5)
    return A, B


def check_stages(A, B, n, splits=1):
    M, K = A.shape
    _, N = B.shape
    dA, dB = dev(A), dev(B)
    # 1. exponent scan
    s, t = run_scale(dA, dB, n)
    so, to = oracle.scale(A, B, n)
    assert np.array_equal(s.cpu().numpy(), so)
    assert np.array_equal(t.cpu().numpy(), to)
    # 2. residue slices
    a_sl, b_sl = run_quantize(dA, dB, s, t, n)
    Ap = oracle.integers(A, so, True)
    Bp = oracle.integers(B, to, False)
    ra = oracle.residues(Ap, n)  # n x M x K
    rb = oracle.residues(Bp, n)  # n x K x N
    ga = a_sl.cpu().numpy().view(np.uint16)
    gb = b_sl.cpu().numpy().view(np.uint16)
    assert np.array_equal(f16_to_int(ga[:, :, :K]), ra.astype(np.int64))
    assert np.array_equal(f16_to_int(gb[:, :, :K]), rb.transpose(0, 2, 1).astype(np.int64))
    assert np.all(ga[:, :, K:] == 0) and np.all(gb[:, :, K:] == 0)
    # 3. per-modulus exact int32 sums, and their reduction mod p
    raw, cmod = oracle.gemm_mod(ra, rb, n)
    out32, ld32 = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=1, splits=splits)
    g32 = out32.cpu().numpy()[:, :, :, :N].astype(np.int64).sum(axis=0)
    assert np.array_equal(g32, raw.astype(np.int64))
    out8, ld8 = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=0)
    assert np.array_equal(out8.cpu().numpy()[:, :, :N], cmod)
    # 3b. residues of the moduli pairs (2j, 2j+1) as uint16: the unique r < p_2j p_2j+1
    #     with r = c_2j mod p_2j and r = c_2j+1 mod p_2j+1; an odd last plane holds c_n-1
    out16, ld16 = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=2)
    g16 = out16.cpu().numpy()[:, :, :N].view(np.uint16).astype(np.int64)
    ps = oracle.moduli(n)
    for j in range((n + 1) // 2):
        if 2 * j + 1 < n:
            assert np.all(g16[j] < ps[2 * j] * ps[2 * j + 1])
            assert np.array_equal(g16[j] % ps[2 * j], cmod[2 * j].astype(np.int64))
            assert np.array_equal(g16[j] % ps[2 * j + 1], cmod[2 * j + 1].astype(np.int64))
        else:
            assert np.array_equal(g16[j], cmod[2 * j].astype(np.int64))
    # 4. lifted integers, from either representation
    Xo = oracle.crt(cmod, n)
    X8 = run_lift(out8, 0, ld8, 1, M, N, n).cpu().numpy().view(np.uint32)
    assert np.array_equal(X8, Xo)
    X32 = run_lift(out32, 1, ld32, splits, M, N, n).cpu().numpy().view(np.uint32)
    assert np.array_equal(X32, Xo)
    X16 = run_lift(out16, 2, ld16, 1, M, N, n).cpu().numpy().view(np.uint32)
    assert np.array_equal(X16, Xo)
    # 5. undo scaling, write double
    Co = oracle.dgemm(A, B, n)
    C8 = run_combine(out8, 0, ld8, 1, s, t, M, N, n).cpu().numpy()
    assert same_bits(C8, Co)
    C32 = run_combine(out32, 1, ld32, splits, s, t, M, N, n).cpu().numpy()
    assert same_bits(C32, Co)
    C16 = run_combine(out16, 2, ld16, 1, s, t, M, N, n).cpu().numpy()
    assert same_bits(C16, Co)
    return Co


STAGE_SHAPES = [(1, 1, 1), (7, 5, 3), (128, 256, 64), (129, 257, 65), (256, 256, 256),
                (300, 200, 1000), (33, 17, 2000), (64, 600, 129)]


@pytest.mark.parametrize("M,N,K", STAGE_SHAPES)
@pytest.mark.parametrize("n", [8, 14, 20])
def test_stages_bit_exact(M, N, K, n):
    A, B = inputs(M, N, K, seed=M * 7 + N * 3 + K + n, kind="special")
    check_stages(A, B, n)


@pytest.mark.parametrize("n", [2, 3, 5, 11, 17])
def test_stages_other_moduli_counts(n):
    K = 40 if n <= 3 else 300
    if ozk.ozk_beta(K, n) < 1:
        pytest.skip("too few moduli for K")
    A, B = inputs(130, 270, K, seed=n, kind="special")
    check_stages(A, B, n)


@pytest.mark.parametrize("n,K", [(17, 100), (17, 16), (17, 5), (18, 300), (18, 1000), (16, 1), (20, 700), (20, 2),
                                 (20, 1)])
def test_stages_across_the_integer_widths(n, K):
    """beta 62 (two 32-bit words per scaled element), 63, 64, 65, 72, 76 and
    77, the largest budget of any moduli count (three words; the integer
    crosses 2^64 from beta 64): every stage bit-exact."""
    A, B = inputs(70, 90, K, seed=n * 1000 + K, kind="special")
    check_stages(A, B, n)


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_split_k_partials_sum_to_the_exact_product(splits):
    A, B = inputs(70, 300, 4000, seed=splits)
    check_stages(A, B, 14, splits=splits)


@pytest.mark.parametrize("n", list(range(2, 21)))
def test_crt_wide_outputs_every_moduli_count(n):
    """Outputs wide enough for the kernels compiled per moduli count (uint16
    residues of moduli pairs): random residues (any residue vector is a valid
    CRT input), scales that give
    normal, subnormal, underflowing, overflowing and NaN results; sampled
    outputs against the oracle's CRT and rounding."""
    M, N = 2048, 640
    rng = np.random.default_rng(100 + n)
    ps = [int(p) for p in oracle.moduli(n)]
    # random residues of the moduli pairs; the byte residues follow from them
    pair = np.stack([rng.integers(0, ps[2 * j] * ps[2 * j + 1] if 2 * j + 1 < n else ps[2 * j], size=(M, N))
                     for j in range((n + 1) // 2)]).astype(np.int64)
    res = np.stack([pair[k // 2] % p for k, p in enumerate(ps)]).astype(np.uint8)
    s = rng.integers(-200, 200, M).astype(np.int32)
    t = rng.integers(-200, 200, N).astype(np.int32)
    s[10:20] = 1050 - 8 * n   # |X| 2^-(s+t) near the subnormal range
    s[20:30] = -1000 + 8 * n  # near overflow
    s[3] = oracle.NONFINITE
    t[5] = oracle.NONFINITE
    C = run_combine(dev(pair.astype(np.uint16).view(np.int16)), 2, N, 1, dev(s), dev(t), M, N, n).cpu().numpy()
    C8 = run_combine(dev(res), 0, N, 1, dev(s), dev(t), M, N, n).cpu().numpy()
    assert same_bits(C8, C)  # byte residues through the runtime-count kernel
    ii = np.concatenate([rng.integers(0, M, 3000), np.arange(10, 30).repeat(20), np.full(50, 3)])
    jj = np.concatenate([rng.integers(0, N, 3000), rng.integers(0, N, 400), rng.integers(0, N, 50)])
    ii = np.concatenate([ii, rng.integers(0, M, 50)])
    jj = np.concatenate([jj, np.full(50, 5)])
    X = oracle.crt(res[:, ii, jj], n)
    nonfinite = (s[ii] == oracle.NONFINITE) | (t[jj] == oracle.NONFINITE)
    S = np.where(nonfinite, 0, s[ii].astype(np.int64) + t[jj]).astype(np.int32)
    want = np.where(nonfinite, np.nan, oracle.round_scaled(X, S))
    assert same_bits(C[ii, jj], want)
    assert np.isnan(C[3]).all() and np.isnan(C[:, 5]).all()


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 700, 3), (513, 1, 77), (256, 256, 256), (129, 257, 1025)])
@pytest.mark.parametrize("n", [8, 11, 14, 17, 20])
def test_dgemm_bit_exact(M, N, K, n):
    A, B = inputs(M, N, K, seed=1 + n, kind="special")
    assert same_bits(dgemm(A, B, n), oracle.dgemm(A, B, n))


@pytest.mark.parametrize("M,N,K,n", [(65, 300, 32800, 13), (130, 90, 32768, 14), (65, 300, 8200, 13)])
def test_dgemm_bit_exact_long_k(M, N, K, n):
    """Long K in one split: byte planes whose 33, 32 or 9 chunks are each cut
    in fp32 and added before the one reduction, against the oracle."""
    A, B = inputs(M, N, K, seed=M + N + K + n)
    assert same_bits(dgemm(A, B, n), oracle.dgemm(A, B, n))


@pytest.mark.parametrize("M,N,K,n", [(2048, 96, 2000, 14), (1024, 64, 4033, 14), (2048, 40, 2100, 18),
                                     (4096, 40, 1030, 20)])
def test_dgemm_bit_exact_fused_row_scan(M, N, K, n):
    """Enough rows of at most 4096 entries: each row of A is scanned inside its
    own quantisation (one block per row).  Special rows (zero, subnormal,
    2^900, wide range, Inf, NaN) and ragged K against the oracle, all outputs,
    for each integer width (beta 48: two 32-bit words; 63 and 71: three)."""
    A, B = inputs(M, N, K, seed=M + N + K, kind="special")
    A[5, K // 3] = np.inf
    A[9, K - 1] = np.nan
    C = dgemm(A, B, n)
    assert same_bits(C, oracle.dgemm(A, B, n))
    assert np.isnan(C[5]).all() and np.isnan(C[9]).all()


@pytest.mark.parametrize("M,N,K", [(129, 257, 2100), (1, 700, 4096), (300, 1, 2049), (257, 520, 6000)])
def test_dgemm_bit_exact_cta_pairs(M, N, K):
    """K of 2048 or more runs the residue GEMM on CTA pairs (256-row tiles,
    1024-term chunks): ragged rows, columns and K against the oracle."""
    A, B = inputs(M, N, K, seed=M + N + K)
    assert same_bits(dgemm(A, B, 14), oracle.dgemm(A, B, 14))


@pytest.mark.parametrize("M,N,K,n", [(5, 9, 2**17 + 3, 14), (3, 5, 2**20 + 7, 14), (17, 3, 300000, 20),
                                     (2, 3, ozk.OZK_MAX_K, 14)])
def test_dgemm_k_beyond_one_int32_sum(M, N, K, n):
    """K >= 2^17: the residue GEMM splits K into int32-exact shares (at most
    OZK_SPLIT_MAX_K terms) and the combine reduces each share mod p; up to the
    largest K the library takes (OZK_MAX_K, 33 shares)."""
    A, B = inputs(M, N, K, seed=K % 1000)
    assert same_bits(dgemm(A, B, n), oracle.dgemm(A, B, n))


@pytest.mark.parametrize("target", [30, 40, 48])
def test_dgemm_bits_picks_the_count_and_keeps_its_bound(target):
    """ozk_dgemm_bits = ozk_dgemm with the smallest count whose beta reaches the
    target; the result keeps the a-priori bound of its beta."""
    A, B = inputs(96, 80, 3000, seed=target)
    n = ozk.ozk_moduli_for_bits(3000, target)
    assert 2 <= n <= 20 and oracle.beta(3000, n) >= target
    Cb = ozk.dgemm(dev(A), dev(B), target_bits=target).cpu().numpy()
    assert same_bits(Cb, dgemm(A, B, n))
    R = oracle.dot2(A, B)
    beta = oracle.beta(3000, n)
    so, to = oracle.scale(A, B, n)
    bound = (np.ldexp(1.0, -so.astype(np.int64))[:, None] * np.abs(B).sum(0)[None, :]
             + np.ldexp(1.0, -to.astype(np.int64))[None, :] * np.abs(A).sum(1)[:, None]
             + 3000 * np.ldexp(1.0, -(so[:, None].astype(np.int64) + to[None, :])) + np.spacing(np.abs(R)))
    assert np.all(np.abs(Cb - R) <= bound)
    assert beta >= target


def test_dgemm_square256_normal_n14():
    w = workloads.WORKLOADS["square256_normal"]
    A, B = workloads.workload_operands(w)
    C = dgemm(A, B, 14)
    assert same_bits(C, oracle.dgemm(A, B, 14))
    R = oracle.dot2(A, B)
    eta = np.max(np.abs(C - R) / (np.abs(A) @ np.abs(B)))
    assert eta <= 1e-14


@pytest.mark.parametrize("n", [14, 8, 11])
def test_dgemm_square1024_wide(n):
    w = workloads.WORKLOADS["square1024_wide"]
    A, B = workloads.workload_operands(w)
    C = dgemm(A, B, n)
    assert same_bits(C, oracle.dgemm(A, B, n))
    R = oracle.dot2(A, B)
    eta = np.max(np.abs(C - R) / (np.abs(A) @ np.abs(B)))
    if n >= 14:
        assert eta <= 1e-14
    elif n == 11:
        assert eta <= 2.0**-30
    else:  # 8 moduli: the a-priori rounding bound
        s, t = oracle.scale(A, B, n)
        bound = (np.abs(A).sum(1)[:, None] * np.ldexp(1.0, -t - 1)[None, :]
                 + np.ldexp(1.0, -s - 1)[:, None] * np.abs(B).sum(0)[None, :]
                 + w.K * np.ldexp(1.0, -(s[:, None] + t[None, :] + 2)))
        assert np.all(np.abs(C - R) <= bound * (1 + 1e-12) + np.spacing(np.abs(C)))


def sample_pairs(M, N, count, seed):
    rng = np.random.default_rng(seed)
    ii = list(rng.integers(0, M, count))
    jj = list(rng.integers(0, N, count))
    for i in {0, 127, 128, M - 1}:
        for j in {0, 255, 256, N - 1}:
            if i < M and j < N:
                ii.append(i)
                jj.append(j)
    return np.array(ii, dtype=np.int64), np.array(jj, dtype=np.int64)


def check_sampled(name, n, count):
    w = workloads.WORKLOADS[name]
    A, B = workloads.workload_operands(w)
    dA, dB = dev(A), dev(B)
    C = ozk.dgemm(dA, dB, n)
    torch.cuda.synchronize()
    assert ozk.ozk_stream_status() == 0
    ii, jj = sample_pairs(w.M, w.N, count, seed=n)
    Cg = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    Co, _, _, _ = oracle.sample(A, B, n, ii, jj)
    assert same_bits(Cg, Co)
    R, absAB = oracle.dot2_sample(A, B, ii, jj)
    eta = float(np.max(np.abs(Cg - R) / absAB))
    if n >= 14:
        assert eta <= 1e-14
    elif n == 11:
        assert eta <= 2.0**-30
    del dA, dB, C
    torch.cuda.empty_cache()
    return eta


@pytest.mark.parametrize("n", [14, 8])
def test_square4096_sampled(n):
    check_sampled("square4096_normal", n, 384)


def test_square8192_sampled():
    check_sampled("square8192_uniform", 14, 192)


@pytest.mark.parametrize("n", [8, 11, 14, 17, 20])
def test_wide8192_k512_sampled(n):
    check_sampled("wide8192_k512", n, 384)


@pytest.mark.parametrize("n", [8, 11, 14, 17, 20])
def test_tall512_k65536_sampled(n):
    check_sampled("tall512_k65536", n, 96)


# ----------------------------------------------------------------- edge cases
def test_empty_and_k0():
    for (M, N) in [(0, 5), (5, 0), (0, 0)]:
        A = torch.zeros((M, 3), dtype=torch.float64, device="cuda")
        B = torch.zeros((3, N), dtype=torch.float64, device="cuda")
        C = ozk.dgemm(A, B, 14)
        assert C.shape == (M, N)
    A = torch.zeros((4, 0), dtype=torch.float64, device="cuda")
    B = torch.zeros((0, 6), dtype=torch.float64, device="cuda")
    C = torch.full((4, 6), 5.0, dtype=torch.float64, device="cuda")
    ozk.ozk_dgemm(4, 6, 0, A, 1, B, 6, C, 6, 14)
    torch.cuda.synchronize()
    assert torch.all(C == 0)


def test_rejected_arguments():
    A = torch.ones((4, 8), dtype=torch.float64, device="cuda")
    B = torch.ones((8, 5), dtype=torch.float64, device="cuda")
    C = torch.empty((4, 5), dtype=torch.float64, device="cuda")
    L = ozk.lib()
    s = ozk._stream(None)
    p = ctypes.c_void_p
    call = lambda M, N, K, a, lda, b, ldb, c, ldc, n: L.ozk_dgemm(M, N, K, p(a), lda, p(b), ldb, p(c), ldc, n, s)
    a, b, c = A.data_ptr(), B.data_ptr(), C.data_ptr()
    assert call(4, 5, 8, a, 8, b, 5, c, 5, 1) == ozk.OZK_ERR_UNSUPPORTED
    assert call(4, 5, 8, a, 8, b, 5, c, 5, 21) == ozk.OZK_ERR_UNSUPPORTED
    big = ozk.OZK_MAX_K + 1
    assert call(4, 5, big, a, big, b, 5, c, 5, 14) == ozk.OZK_ERR_UNSUPPORTED
    assert call(4, 5, 8, a, 7, b, 5, c, 5, 14) == ozk.OZK_ERR_INVALID_ARG      # lda < K
    assert call(4, 5, 8, a, 8, b, 5, c, 4, 14) == ozk.OZK_ERR_INVALID_ARG      # ldc < N
    assert call(4, 5, 8, a, 8, b, 5, a, 5, 14) == ozk.OZK_ERR_INVALID_ARG      # C overlaps A
    assert call(-1, 5, 8, a, 8, b, 5, c, 5, 14) == ozk.OZK_ERR_INVALID_ARG
    assert call(4, 5, 8, 0, 8, b, 5, c, 5, 14) == ozk.OZK_ERR_INVALID_ARG      # null A
    assert call(4, 5, 60000, a, 60000, b, 5, c, 5, 2) == ozk.OZK_ERR_UNSUPPORTED  # beta < 1
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    rc = L.ozk_dgemm_ws(4, 5, 8, p(a), 8, p(b), 5, p(c), 5, 14, p(ws.data_ptr()), 16, s)
    assert rc == ozk.OZK_ERR_WORKSPACE
    # residue GEMM stage: one int32-exact sum needs K < 2^17; splits of at most OZK_SPLIT_MAX_K
    sl = torch.zeros(2 * 4 * 262144, dtype=torch.int16, device="cuda")
    out = torch.zeros(2 * 4 * 16 * 4, dtype=torch.int32, device="cuda")
    gemm = lambda K, kind, ldo, splits: L.ozk_residue_gemm(4, 4, K, p(sl.data_ptr()), p(sl.data_ptr()), 2, kind,
                                                          p(out.data_ptr()), ldo, splits, s)
    assert gemm(2**17, 0, 16, 1) == ozk.OZK_ERR_INVALID_ARG
    assert gemm(2**17, 1, 4, 1) == ozk.OZK_ERR_INVALID_ARG
    assert gemm(262144, 1, 4, 2) == ozk.OZK_ERR_INVALID_ARG   # 131072 terms per split
    assert ozk.ozk_stream_status() == 0


def test_nonfinite_rows_and_columns():
    A, B = inputs(40, 50, 70, seed=3)
    A[5, 9] = np.inf
    A[17, 0] = np.nan
    B[3, 44] = -np.inf
    C = dgemm(A, B, 14)
    Co = oracle.dgemm(A, B, 14)
    assert same_bits(C, Co)
    assert np.all(np.isnan(C[5])) and np.all(np.isnan(C[17])) and np.all(np.isnan(C[:, 44]))


def test_subnormal_and_overflowing_results():
    rng = np.random.default_rng(5)
    A = rng.standard_normal((9, 33))
    B = rng.standard_normal((33, 11))
    A[0:3] *= 2.0**-560
    B[:, 0:4] *= 2.0**-560        # products near 2^-1120: subnormal and underflow
    A[4:6] *= 2.0**520
    B[:, 6:8] *= 2.0**510         # products near 2^1030: overflow to inf
    for n in (8, 14, 20):
        assert same_bits(dgemm(A, B, n), oracle.dgemm(A, B, n))


@pytest.mark.parametrize("pad,offset", [(3, 1), (1, 0), (0, 1)])
def test_strided_and_unaligned_operands(pad, offset):
    A, B = inputs(65, 130, 97, seed=pad + offset, kind="special")
    dA, _ba = strided(A, pad, offset)
    dB, _bb = strided(B, pad + 1, offset)
    C = torch.empty((65, 130), dtype=torch.float64, device="cuda")
    ozk.ozk_dgemm(65, 130, 97, dA, ld_of(dA), dB, ld_of(dB), C, 130, 14)
    torch.cuda.synchronize()
    assert same_bits(C.cpu().numpy(), oracle.dgemm(A, B, 14))


def test_caller_workspace_and_host_buffers_agree():
    A, B = inputs(200, 300, 500, seed=9)
    C0 = dgemm(A, B, 14)
    dA, dB = dev(A), dev(B)
    need = ozk.ozk_workspace_size(200, 300, 500, 14)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    C1 = torch.empty((200, 300), dtype=torch.float64, device="cuda")
    ozk.ozk_dgemm_ws(200, 300, 500, dA, 500, dB, 300, C1, 300, 14, ws, need)
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.empty((200, 300), dtype=torch.float64).pin_memory()
    ozk.ozk_dgemm_host(200, 300, 500, hA, 500, hB, 300, hC, 300, 14)
    torch.cuda.synchronize()
    assert same_bits(C1.cpu().numpy(), C0)
    assert same_bits(hC.numpy(), C0)
    assert ozk.ozk_stream_status() == 0


@pytest.mark.parametrize("M,N,K", [(2100, 300, 700), (2100, 2300, 700), (3000, 2048, 300), (2048, 72, 32800)])
def test_host_buffers_in_blocks(M, N, K):
    """ozk_dgemm_host on row and column blocks (a dimension >= 2048 goes in
    four blocks of whole 256-row or 256-column tiles, copies overlapping the
    stages; ragged last blocks here) with padded host leading dimensions:
    equal to the device path bit for bit, and to the oracle on sampled
    outputs, block edges included (one chunk per tile at K <= 700, 33 at
    K = 32800)."""
    A, B = inputs(M, N, K, seed=M + N + K)
    hA = torch.zeros((M, K + 3), dtype=torch.float64).pin_memory()
    hB = torch.zeros((K, N + 5), dtype=torch.float64).pin_memory()
    hC = torch.full((M, N + 2), np.nan, dtype=torch.float64).pin_memory()
    hA[:, :K] = torch.from_numpy(A)
    hB[:, :N] = torch.from_numpy(B)
    ozk.ozk_dgemm_host(M, N, K, hA, K + 3, hB, N + 5, hC, N + 2, 14)
    C = hC.numpy()[:, :N]
    assert same_bits(C, dgemm(A, B, 14))
    assert np.isnan(hC.numpy()[:, N:]).all()  # padding untouched
    rng = np.random.default_rng(M)
    edges_i = [e for e in [0, 767, 768, 1535, 1536, 2303, 2304, M - 1] if e < M]
    edges_j = [e for e in [0, 511, 512, 767, 768, 1023, 1024, 1535, 1536, 2303, N - 1] if e < N]
    ei, ej = np.meshgrid(edges_i, edges_j, indexing="ij")
    ii = np.concatenate([rng.integers(0, M, 200), ei.ravel()])
    jj = np.concatenate([rng.integers(0, N, 200), ej.ravel()])
    assert same_bits(C[ii, jj], oracle.sample(A, B, 14, ii, jj)[0])
    assert ozk.ozk_stream_status() == 0


def test_host_async_calls_in_flight():
    """Four ozk_dgemm_host_async calls in flight on one stream, more than the
    library's two sets of device buffers, each with its own host operands and
    output (the last of another shape): after one synchronisation every C
    equals the device path bit for bit."""
    shapes = [(2100, 2300, 700), (2100, 2300, 700), (2100, 2300, 700), (300, 260, 2100)]
    st = torch.cuda.Stream()
    calls = []
    for idx, (M, N, K) in enumerate(shapes):
        A, B = inputs(M, N, K, seed=200 + idx)
        hA = torch.from_numpy(A).pin_memory()
        hB = torch.from_numpy(B).pin_memory()
        hC = torch.full((M, N), np.nan, dtype=torch.float64).pin_memory()
        ozk.ozk_dgemm_host_async(M, N, K, hA, K, hB, N, hC, N, 14, stream=st)
        calls.append((A, B, hA, hB, hC))
    st.synchronize()
    assert ozk.ozk_stream_status(st) == 0
    for A, B, _, _, hC in calls:
        assert same_bits(hC.numpy(), dgemm(A, B, 14))


def test_host_async_long_k_and_split_k_outputs():
    """Back-to-back ozk_dgemm_host_async calls whose later ones find an earlier
    call still computing (the whole-product schedule), with K = 32800 (byte
    planes over 33 chunks) and K >= 2^17 (int32 split-K partials): every C
    equals the device path bit for bit."""
    shapes = [(768, 768, 32800), (768, 392, 32800), (96, 40, 140000), (96, 40, 140000)]
    st = torch.cuda.Stream()
    calls = []
    for idx, (M, N, K) in enumerate(shapes):
        A, B = inputs(M, N, K, seed=300 + idx)
        hA = torch.from_numpy(A).pin_memory()
        hB = torch.from_numpy(B).pin_memory()
        hC = torch.full((M, N), np.nan, dtype=torch.float64).pin_memory()
        ozk.ozk_dgemm_host_async(M, N, K, hA, K, hB, N, hC, N, 14, stream=st)
        calls.append((A, B, hA, hB, hC))
    st.synchronize()
    assert ozk.ozk_stream_status(st) == 0
    for A, B, _, _, hC in calls:
        assert same_bits(hC.numpy(), dgemm(A, B, 14))


def test_host_async_from_two_threads():
    """Two host threads, each with its own stream, enqueue three
    ozk_dgemm_host_async calls apiece (the library serialises the enqueueing
    and shares its two buffer sets among them): every C is right."""
    import threading

    results, errors = {}, []

    def worker(tid):
        try:
            st = torch.cuda.Stream()
            mine = []
            for c in range(3):
                M, N, K = 640 + 64 * tid, 2100, 300 + 100 * c
                A, B = inputs(M, N, K, seed=1000 * tid + c)
                hA = torch.from_numpy(A).pin_memory()
                hB = torch.from_numpy(B).pin_memory()
                hC = torch.full((M, N), np.nan, dtype=torch.float64).pin_memory()
                ozk.ozk_dgemm_host_async(M, N, K, hA, K, hB, N, hC, N, 14, stream=st)
                mine.append((A, B, hA, hB, hC))
            st.synchronize()
            results[tid] = (mine, ozk.ozk_stream_status(st))
        except Exception as e:  # reported in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(tid,)) for tid in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors
    for tid in range(2):
        mine, status = results[tid]
        assert status == 0
        for A, B, _, _, hC in mine:
            assert same_bits(hC.numpy(), dgemm(A, B, 14))


def test_release_cached_and_reuse():
    """ozk_release_cached frees the cached workspaces, the host-path buffers,
    streams and events; the next calls set them up again and agree with the
    results from before the release bit for bit."""
    M, N, K = 2100, 300, 700
    A, B = inputs(M, N, K, seed=501)
    before = dgemm(A, B, 14)
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float64).pin_memory()
    ozk.ozk_dgemm_host(M, N, K, hA, K, hB, N, hC, N, 14)
    assert same_bits(hC.numpy(), before)
    ozk.ozk_release_cached()
    assert same_bits(dgemm(A, B, 14), before)
    hC.zero_()
    st = torch.cuda.Stream()
    ozk.ozk_dgemm_host_async(M, N, K, hA, K, hB, N, hC, N, 14, stream=st)
    st.synchronize()
    assert same_bits(hC.numpy(), before)
    ozk.ozk_release_cached()
    hC.zero_()
    ozk.ozk_dgemm_host(M, N, K, hA, K, hB, N, hC, N, 14)
    assert same_bits(hC.numpy(), before)
    assert ozk.ozk_stream_status() == 0


def test_caller_workspace_call_captures_into_a_cuda_graph():
    """ozk_dgemm_ws only enqueues work (no synchronisation, no allocation), so
    a warmed-up call can be captured into a CUDA graph (here one large enough
    for the fused row kernel, whose side stream joins the capture); replays
    reproduce it bit for bit and follow new input values in the same buffers."""
    M, N, K, n = 2048, 72, 2100, 14
    A, B = inputs(M, N, K, seed=77)
    dA, dB = dev(A), dev(B)
    C = torch.empty((M, N), dtype=torch.float64, device="cuda")
    need = ozk.ozk_workspace_size(M, N, K, n)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        ozk.ozk_dgemm_ws(M, N, K, dA, K, dB, N, C, N, n, ws, need, stream=st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        ozk.ozk_dgemm_ws(M, N, K, dA, K, dB, N, C, N, n, ws, need, stream=st)
    C.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert same_bits(C.cpu().numpy(), oracle.dgemm(A, B, n))
    A2, B2 = inputs(M, N, K, seed=78, kind="special")
    dA.copy_(torch.from_numpy(A2))
    dB.copy_(torch.from_numpy(B2))
    g.replay()
    torch.cuda.synchronize()
    assert same_bits(C.cpu().numpy(), oracle.dgemm(A2, B2, n))
    assert ozk.ozk_stream_status() == 0


def test_deterministic_and_stream_ordered():
    A, B = inputs(300, 700, 900, seed=4)
    dA, dB = dev(A), dev(B)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        C1 = ozk.dgemm(dA, dB, 14, stream=st)
        C2 = ozk.dgemm(dA, dB, 14, stream=st)
    st.synchronize()
    assert torch.equal(C1.view(torch.int64), C2.view(torch.int64))
    assert ozk.ozk_stream_status(st) == 0


def test_back_to_back_calls_on_one_workspace():
    """Kernels launch while the one before them finishes (dependent launches):
    calls issued back to back on one stream and one caller workspace, with
    other inputs, shapes and moduli counts (a split-K one among them) and the
    caller's own work in between, must each see only their own data.  Each
    result is checked against the oracle at sampled outputs after one final
    synchronisation."""
    cases = [(600, 520, 2100, 14, 1), (600, 520, 2100, 14, 2), (256, 300, 40000, 11, 3), (700, 90, 900, 20, 4),
             (600, 520, 2100, 8, 5)]
    ops = [inputs(M, N, K, seed=seed) for (M, N, K, n, seed) in cases]
    need = max(ozk.ozk_workspace_size(M, N, K, n) for (M, N, K, n, _) in cases)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    outs, snaps = [], []
    with torch.cuda.stream(st):
        devs = [(dev(A), dev(B)) for (A, B) in ops]
        st.synchronize()
        for (M, N, K, n, _), (dA, dB) in zip(cases, devs):
            C = torch.full((M, N), float("nan"), dtype=torch.float64, device="cuda")
            ozk.ozk_dgemm_ws(M, N, K, dA, K, dB, N, C, N, n, ws, need, st)
            snaps.append(C.clone())  # the caller's kernel right behind the call
            dA.mul_(3.0)  # and one that overwrites an input the call has read
            outs.append(C)
    st.synchronize()
    assert ozk.ozk_stream_status(st) == 0
    for (M, N, K, n, seed), (A, B), C, S in zip(cases, ops, outs, snaps):
        ii, jj = sample_pairs(M, N, 160, seed=seed)
        Co, _, _, _ = oracle.sample(A, B, n, ii, jj)
        assert same_bits(C.cpu().numpy()[ii, jj], Co), (M, N, K, n)
        assert torch.equal(C.view(torch.int64), S.view(torch.int64))
