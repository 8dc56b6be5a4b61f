"""The bounded-wait failure path of the residue GEMM, exercised without a
fault.  Every mbarrier wait of the GEMM kernels has a time limit; when one
runs out the kernel latches OZK_ERR_TIMEOUT, every role of the CTA stops, the
copies and MMAs in flight drain, TMEM is freed and the kernel returns.
ozk_residue_gemm_withheld runs the single-CTA kernel with a short limit and
one tile copy never issued, so that the MMA issuer's wait runs out.  The
tests check that the host reads the status, that the other CTAs' tiles are
right, and that the next normal calls are bit-exact against the oracle (which
they could not be, or would not even run, if the aborted CTA had kept its
TMEM or left the context broken).

Why every wait is bounded: a wrong mbarrier phase or arrive count leaves a
wait hanging (the async Tensor Core article on yfxerp.com, section 6.1).
"""
import numpy as np
import pytest
import torch

import oracle
from fp64_gemm_emulation_exponent_gb300 import ozk
from gpu_helpers import dev, run_gemm

pytestmark = pytest.mark.gpu


def slices(M, N, K, n, seed):
    rng = np.random.default_rng(seed)
    ps = oracle.moduli(n)
    ra = np.stack([rng.integers(-(p // 2), (p + 1) // 2, (M, K)) for p in ps]).astype(np.int8)
    rb = np.stack([rng.integers(-(p // 2), (p + 1) // 2, (K, N)) for p in ps]).astype(np.int8)
    kpad = ozk.ozk_kpad(K)
    fa = np.zeros((n, M, kpad), dtype=np.float16)
    fb = np.zeros((n, N, kpad), dtype=np.float16)
    fa[:, :, :K] = ra
    fb[:, :, :K] = rb.transpose(0, 2, 1)
    return ra, rb, dev(fa.view(np.int16)), dev(fb.view(np.int16))


@pytest.mark.parametrize("K,withhold_kb", [(512, 1), (512, 0), (1100, 7)])
def test_withheld_copy_times_out_and_the_next_calls_are_exact(K, withhold_kb):
    M, N, n = 300, 260, 2
    ra, rb, a_sl, b_sl = slices(M, N, K, n, seed=K + withhold_kb)
    _, cmod = oracle.gemm_mod(ra, rb, n)
    ldo = (N + 15) // 16 * 16
    out = torch.full((n, M, ldo), 0xEE, dtype=torch.uint8, device="cuda")
    ozk.ozk_residue_gemm_withheld(M, N, K, a_sl, b_sl, n, out, ldo, withhold_kb, 2000)
    assert ozk.ozk_stream_status() == ozk.OZK_ERR_TIMEOUT
    assert ozk.ozk_stream_status() == ozk.OZK_OK  # reading the status clears it
    got = out.cpu().numpy()[:, :, :N]
    # CTA 0's first unit is modulus 0's tile of rows 0..127, columns 0..255: never
    # written; every other tile was computed by the other CTAs
    mask = np.ones_like(got, dtype=bool)
    mask[0, :128, :256] = False
    assert np.array_equal(got[mask], cmod[mask])
    assert np.all(got[0, :128, :256] == 0xEE)
    # the same launch configuration right after, and again: bit-exact
    for _ in range(2):
        out8, _ = run_gemm(a_sl, b_sl, M, N, K, n, out_kind=0)
        torch.cuda.synchronize()
        assert ozk.ozk_stream_status() == ozk.OZK_OK
        assert np.array_equal(out8.cpu().numpy()[:, :, :N], cmod)


def test_withheld_copy_rejects_the_pair_kernel_and_bad_limits():
    M, N, n = 64, 64, 2
    _, _, a_sl, b_sl = slices(M, N, 2048, n, seed=1)
    out = torch.zeros((n, M, 64), dtype=torch.uint8, device="cuda")
    L = ozk.lib()
    p = lambda t: ozk._ptr(t)
    s = ozk._stream(None)
    assert L.ozk_residue_gemm_withheld(M, N, 2048, p(a_sl), p(b_sl), n, p(out), 64, 0, 1000, s) == \
        ozk.OZK_ERR_INVALID_ARG  # K of the CTA-pair kernel
    assert L.ozk_residue_gemm_withheld(M, N, 512, p(a_sl), p(b_sl), n, p(out), 64, 8, 1000, s) == \
        ozk.OZK_ERR_INVALID_ARG  # k-block beyond kpad / 64
    assert L.ozk_residue_gemm_withheld(M, N, 512, p(a_sl), p(b_sl), n, p(out), 64, 0, 0, s) == \
        ozk.OZK_ERR_INVALID_ARG  # no time limit
    assert ozk.ozk_stream_status() == ozk.OZK_OK
