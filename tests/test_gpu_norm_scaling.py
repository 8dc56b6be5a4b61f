"""GPU parity of the sharper scaling rule (scales from an exactly computed
2-norm bound per row of A and column of B; the oracle's reading R15) against
the CPU oracle: the scales bit for bit (ozk_scale_norm, and inside
ozk_dgemm_norm on both scan paths: rows of A scanned separately, or inside
their quantisation when a row holds at most 4096 entries), and C bit for bit
on ragged shapes, every integer width of the quantiser, the CTA-pair GEMM
and split K; sampled outputs at the workload sizes.

Method: Ozaki scheme II, the "Day 12" page (ithelp.ithome.com.tw), sections
"Profile 不能只看 Tensor Core" (scale / exponent scan, then the integer
stages) and "先定義公平比較" (the precision contract a sharper scaling must
keep: the same exactness, more bits per operand).
"""
import numpy as np
import pytest
import torch

import oracle
from fp64_gemm_emulation_exponent_gb300 import ozk, workloads
from gpu_helpers import dev, same_bits

pytestmark = pytest.mark.gpu


def inputs(M, N, K, seed, kind="normal"):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N))
    if kind == "special":
        if M > 5:
            A[0] = 0.0
            A[1] = np.ldexp(rng.standard_normal(K), -1060)                   # subnormal row
            A[2] = np.ldexp(rng.standard_normal(K), 900)                     # huge row
            A[3] = np.ldexp(rng.standard_normal(K), rng.integers(-60, 60, K))  # wide row
            A[4] = 1e-12
            A[4, K // 2] = 7.0                                               # one dominant entry
            A[5, K // 3] = np.inf
        if N > 3:
            B[:, 0] = 0.0
            B[:, 1] = np.ldexp(rng.standard_normal(K), -300)
            B[:, 2] = -np.ldexp(np.ones(K), 5)                              # constant column
            B[K - 1, 3] = np.nan
    return A, B


def run_norm(A, B, n):
    C = ozk.dgemm(dev(A), dev(B), n, scaling="norm")
    torch.cuda.synchronize()
    assert ozk.ozk_stream_status() == 0
    return C.cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 5, 3), (129, 257, 65), (300, 200, 1000), (33, 17, 5000)])
@pytest.mark.parametrize("n", [8, 14, 17, 20])
def test_scale_norm_matches_the_oracle(M, N, K, n):
    A, B = inputs(M, N, K, seed=M + N + K + n, kind="special")
    s = torch.empty(M, dtype=torch.int32, device="cuda")
    t = torch.empty(N, dtype=torch.int32, device="cuda")
    scratch = torch.empty(2 * (M + N), dtype=torch.int64, device="cuda")
    ozk.ozk_scale_norm(M, N, K, dev(A), K, dev(B), N, n, s, t, scratch)
    so, to = oracle.scale(A, B, n, rule="norm")
    assert np.array_equal(s.cpu().numpy(), so)
    assert np.array_equal(t.cpu().numpy(), to)
    assert ozk.ozk_gamma(K, n) == oracle.gamma(K, n)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 257, 65), (300, 200, 1000), (129, 257, 2100),
                                   (2048, 96, 2000), (1024, 64, 4033)])
@pytest.mark.parametrize("n", [8, 13, 14, 16, 17, 20])
def test_dgemm_norm_bit_exact(M, N, K, n):
    """Small shapes scan A's rows separately; 2048 x 2000 and 1024 x 4033 scan
    and quantise each row in one block; K >= 2048 runs the CTA-pair GEMM.
    gamma 54 (14 moduli) and 61 (16) take the 64-bit integer path of the
    quantiser, 65 and 77 (17, 20) the four-limb one."""
    A, B = inputs(M, N, K, seed=3 * M + N + K + n, kind="special")
    C = run_norm(A, B, n)
    assert same_bits(C, oracle.dgemm(A, B, n, rule="norm"))


def test_dgemm_norm_split_k():
    A, B = inputs(5, 9, 2**17 + 3, seed=4)
    assert same_bits(run_norm(A, B, 14), oracle.dgemm(A, B, 14, rule="norm"))


def test_dgemm_norm_caller_workspace_and_two_calls():
    A, B = inputs(300, 400, 900, seed=6, kind="special")
    A2, B2 = inputs(300, 400, 900, seed=7)
    need = ozk.ozk_workspace_size(300, 400, 900, 14)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    C = torch.empty((300, 400), dtype=torch.float64, device="cuda")
    for a, b in ((A, B), (A2, B2)):
        ozk.ozk_dgemm_norm_ws(300, 400, 900, dev(a), 900, dev(b), 400, C, 400, 14, ws, need)
        torch.cuda.synchronize()
        assert same_bits(C.cpu().numpy(), oracle.dgemm(a, b, 14, rule="norm"))
    assert ozk.ozk_stream_status() == 0


@pytest.mark.parametrize("name,n", [("square4096_normal", 13), ("wide8192_k512", 13), ("tall512_k65536", 13)])
def test_workloads_norm_rule_sampled(name, n):
    w = workloads.WORKLOADS[name]
    A, B = workloads.workload_operands(w)
    C = ozk.dgemm(dev(A), dev(B), n, scaling="norm")
    torch.cuda.synchronize()
    assert ozk.ozk_stream_status() == 0
    rng = np.random.default_rng(n)
    ii = np.concatenate([rng.integers(0, w.M, 96), [0, 255, 256, w.M - 1]])
    jj = np.concatenate([rng.integers(0, w.N, 96), [0, w.N - 1, 255, 256]])
    Cg = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    del C
    torch.cuda.empty_cache()
    assert same_bits(Cg, oracle.sample(A, B, n, ii, jj, rule="norm")[0])
