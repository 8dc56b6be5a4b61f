"""ozk_scale_noalloc: the exponent scan for callers that cannot hand the
library device memory (an application whose allocator owns every device byte,
or a loop that must not call cudaMalloc).  Its scratch is a fixed array inside
the library, so these tests check that, called through the C-ABI, it gives
exactly the scales of ozk_scale (which takes caller scratch) and of the CPU
oracle on two calls in a row with different inputs, that the second call is
not disturbed by what the first left in the shared array, that the largest
accepted size (M + N equal to the array's length) is right to its last
element, and that sizes beyond the fixed array are refused before anything
runs.

This file is collected last on purpose: a failure here comes after every other
test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from fp64_gemm_emulation_exponent_gb300 import ozk

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K)) * np.ldexp(1.0, rng.integers(-40, 40, (M, 1)))
    B = rng.standard_normal((K, N)) * np.ldexp(1.0, rng.integers(-40, 40, (1, N)))
    A[0] = 0.0
    A[1, 3 % K] = np.inf
    B[:, 1] = np.ldexp(rng.standard_normal(K), -1060)
    return A, B


def _with_caller_scratch(A, B, n):
    M, K = A.shape
    N = B.shape[1]
    s = torch.empty(M, dtype=torch.int32, device="cuda")
    t = torch.empty(N, dtype=torch.int32, device="cuda")
    scratch = torch.empty(M + N, dtype=torch.int64, device="cuda")
    ozk.ozk_scale(M, N, K, A, K, B, N, n, s, t, scratch)
    return s, t


def _without_scratch(A, B, n):
    M, K = A.shape
    N = B.shape[1]
    s = torch.full((M,), 7, dtype=torch.int32, device="cuda")
    t = torch.full((N,), 7, dtype=torch.int32, device="cuda")
    ozk.ozk_scale_noalloc(M, N, K, A, K, B, N, n, s, t)
    return s, t


def test_noalloc_scan_matches_ozk_scale_on_two_calls_in_a_row():
    # the first call leaves larger maxima in the shared array than the second needs
    cases = [(300, 700, 500, 14, 1), (64, 90, 77, 8, 2)]
    for M, N, K, n, seed in cases:
        A, B = _inputs(M, N, K, seed)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        s_ref, t_ref = _with_caller_scratch(dA, dB, n)
        s, t = _without_scratch(dA, dB, n)
        torch.cuda.synchronize()
        assert ozk.ozk_stream_status() == 0
        assert torch.equal(s, s_ref)
        assert torch.equal(t, t_ref)
        so, to = oracle.scale(A, B, n)
        assert np.array_equal(s.cpu().numpy(), so)
        assert np.array_equal(t.cpu().numpy(), to)


def test_noalloc_scan_at_its_largest_size():
    """M + N exactly OZK_SCALE_NOALLOC_MAX: the last column's maximum lands in
    the array's last element."""
    M, K, n = 8, 4, 14
    N = ozk.OZK_SCALE_NOALLOC_MAX - M
    rng = np.random.default_rng(3)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N)) * np.ldexp(1.0, rng.integers(-30, 30, (1, N)))
    B[:, N - 1] = np.ldexp(1.0, 77)  # the last element: a distinctive scale
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    s, t = _without_scratch(dA, dB, n)
    s_ref, t_ref = _with_caller_scratch(dA, dB, n)
    torch.cuda.synchronize()
    assert ozk.ozk_stream_status() == 0
    assert torch.equal(s, s_ref) and torch.equal(t, t_ref)
    so, to = oracle.scale(A, B, n)
    assert np.array_equal(s.cpu().numpy(), so)
    assert np.array_equal(t.cpu().numpy(), to)
    assert int(t[N - 1]) == ozk.ozk_beta(K, n) - 78


def test_noalloc_scan_refuses_sizes_beyond_its_fixed_scratch():
    L = ozk.lib()
    p = ctypes.c_void_p
    s = torch.empty(8, dtype=torch.int32, device="cuda")
    A = torch.ones((8, 4), dtype=torch.float64, device="cuda")
    too_many = ozk.OZK_SCALE_NOALLOC_MAX  # M + N = limit + 8
    rc = L.ozk_scale_noalloc(8, too_many, 4, p(A.data_ptr()), 4, p(A.data_ptr()), too_many, 14,
                             p(s.data_ptr()), p(s.data_ptr()), ozk._stream(None))
    assert rc == ozk.OZK_ERR_WORKSPACE
    huge = 2**62  # M + N would overflow int64: refused all the same
    rc = L.ozk_scale_noalloc(huge, huge, 4, p(A.data_ptr()), 4, p(A.data_ptr()), huge, 14,
                             p(s.data_ptr()), p(s.data_ptr()), ozk._stream(None))
    assert rc == ozk.OZK_ERR_WORKSPACE
