"""The intermediate buffers of one real ozk_dgemm_ws call, read back from its
workspace (ozk_workspace_layout) and compared with the oracle: the scales,
sampled rows of A's residue slices and columns of B's, the residue GEMM's
planes at sampled outputs (byte residues, or int32 split-K sums for
K >= 2^17) and C.  The stage entry points run each
kernel alone; this checks every stage in the launch configuration of the
whole call (fused row scan, CTA-pair GEMM, split-K, the combine kernel
compiled per moduli count).

Method: Ozaki scheme II, the "Day 12" page (ithelp.ithome.com.tw), section
"Profile 不能只看 Tensor Core" (scale, residue quantization, integer GEMM per
modulus, mod reduction, CRT reconstruction, undo scaling, write double).
"""
import numpy as np
import pytest
import torch

import oracle
from fp64_gemm_emulation_exponent_gb300 import ozk
from gpu_helpers import dev, f16_to_int, same_bits

pytestmark = pytest.mark.gpu


def region(ws, offset, count, dtype):
    nbytes = count * np.dtype(dtype).itemsize
    return ws[offset: offset + nbytes].cpu().numpy().view(dtype)


@pytest.mark.parametrize("M,N,K,n,kind", [(2048, 1024, 2100, 14, 0), (600, 520, 9000, 13, 0),
                                          (600, 520, 33000, 13, 1),
                                          (96, 80, 140000, 14, 1), (513, 300, 700, 20, 0)])
def test_stage_buffers_of_one_call(M, N, K, n, kind):
    rng = np.random.default_rng(M + K)
    A = rng.standard_normal((M, K)) * np.ldexp(1.0, rng.integers(-20, 20, (M, 1)))
    B = rng.standard_normal((K, N))
    A[3] = 0.0
    B[:, 5] = np.ldexp(B[:, 5], -600)
    info = ozk.ozk_workspace_layout(M, N, K, n)
    assert info.total_bytes == ozk.ozk_workspace_size(M, N, K, n)
    assert info.planes_kind == kind and info.kpad == ozk.ozk_kpad(K)
    ws = torch.empty(info.total_bytes, dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), dtype=torch.float64, device="cuda")
    ozk.ozk_dgemm_ws(M, N, K, dev(A), K, dev(B), N, C, N, n, ws, info.total_bytes)
    torch.cuda.synchronize()
    assert ozk.ozk_stream_status() == 0
    # 1. scales
    s = region(ws, info.s_offset, M, np.int32)
    t = region(ws, info.t_offset, N, np.int32)
    so, to = oracle.scale(A, B, n)
    assert np.array_equal(s, so) and np.array_equal(t, to)
    # 2. residue slices: sampled rows of A, sampled columns of B
    kp = info.kpad
    rows = np.unique(np.concatenate([rng.integers(0, M, 6), [0, 3, M - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, N, 6), [0, 5, N - 1]]))
    a_all = region(ws, info.a_slices_offset, (n - 1) * info.a_plane + M * kp, np.uint16)
    b_all = region(ws, info.b_slices_offset, (n - 1) * info.b_plane + N * kp, np.uint16)
    ra = oracle.residues(oracle.integers(A[rows], so[rows], True), n)            # n x rows x K
    rb = oracle.residues(oracle.integers(B[:, cols], to[cols], False), n)        # n x K x cols
    for p in range(n):
        ga = a_all[p * info.a_plane:p * info.a_plane + M * kp].reshape(M, kp)[rows]
        gb = b_all[p * info.b_plane:p * info.b_plane + N * kp].reshape(N, kp)[cols]
        assert np.array_equal(f16_to_int(ga[:, :K]), ra[p].astype(np.int64))
        assert np.array_equal(f16_to_int(gb[:, :K]), rb[p].T.astype(np.int64))
        assert np.all(ga[:, K:] == 0) and np.all(gb[:, K:] == 0)
    # 3. the residue GEMM's planes at sampled outputs, and C
    ii = np.concatenate([rng.integers(0, M, 200), [0, M - 1, 255 % M, 256 % M]])
    jj = np.concatenate([rng.integers(0, N, 200), [N - 1, 0, 255 % N, 256 % N]])
    Co, _, cmod, _ = oracle.sample(A, B, n, ii, jj)
    ld, pl = info.planes_ld, info.planes_plane
    ps = oracle.moduli(n).astype(np.int64)
    if kind == 0:
        planes = region(ws, info.planes_offset, (n - 1) * pl + M * ld, np.uint8)
        got = np.stack([planes[p * pl + ii * ld + jj] for p in range(n)], axis=1)
        assert np.array_equal(got, cmod)
    else:
        sp = info.splits
        assert sp >= 2
        planes = region(ws, info.planes_offset, (sp * n - 1) * pl + M * ld, np.int32).astype(np.int64)
        for p in range(n):
            tot = sum(planes[(q * n + p) * pl + ii * ld + jj] for q in range(sp))
            assert np.array_equal(tot % ps[p], cmod[:, p])
    assert same_bits(C.cpu().numpy()[ii, jj], Co)
