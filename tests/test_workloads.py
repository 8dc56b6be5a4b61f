"""The seeded synthetic inputs (the recipe every test, the oracle baseline and
the benchmark draw from): shapes, moduli counts and seeds of the six
workloads, the three value distributions, and determinism.  CPU only."""
import numpy as np
import pytest

from fp64_gemm_emulation_exponent_gb300 import workloads


def test_the_six_workloads():
    want = {
        "square256_normal": (256, 256, 256, "normal", (14,), 0),
        "square1024_wide": (1024, 1024, 1024, "wide", (14, 8, 11), 1),
        "square4096_normal": (4096, 4096, 4096, "normal", (14, 8, 11), 2),
        "square8192_uniform": (8192, 8192, 8192, "uniform", (14,), 3),
        "wide8192_k512": (8192, 8192, 512, "normal", (8, 11, 14, 17, 20), 4),
        "tall512_k65536": (512, 512, 65536, "normal", (8, 11, 14, 17, 20), 5),
    }
    assert set(workloads.WORKLOADS) == set(want)
    for name, (M, N, K, dist, moduli, seed) in want.items():
        w = workloads.WORKLOADS[name]
        assert (w.M, w.N, w.K, w.dist, w.moduli, w.seed) == (M, N, K, dist, moduli, seed)
        assert w.flops == 2 * M * N * K


def test_operands_are_seeded_and_reproducible():
    A1, B1 = workloads.operands(33, 17, 65, "normal", seed=2)
    A2, B2 = workloads.operands(33, 17, 65, "normal", seed=2)
    assert A1.shape == (33, 65) and B1.shape == (65, 17)
    assert A1.dtype == np.float64 and A1.flags.c_contiguous and B1.flags.c_contiguous
    assert np.array_equal(A1, A2) and np.array_equal(B1, B2)
    # A and B come from different streams (seeds 1000 + c and 2000 + c)
    assert np.array_equal(A1, workloads.draw((33, 65), "normal", 1002))
    assert np.array_equal(B1, workloads.draw((65, 17), "normal", 2002))
    assert not np.array_equal(workloads.draw((8, 8), "normal", 1002), workloads.draw((8, 8), "normal", 2002))


def test_distributions():
    n = 200_000
    x = workloads.draw((n,), "normal", 5)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    u = workloads.draw((n,), "uniform", 5)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    w = workloads.draw((n,), "wide", 5)
    mant, ex = np.frexp(np.abs(w))  # |w| = mant 2^ex, mant in [0.5, 1)
    assert np.all((mant >= 0.5) & (mant < 1.0))
    assert ex.min() == -10 and ex.max() == 10  # sign U(0.5, 1) 2^e, e uniform on -10..10
    counts = np.bincount(ex + 10, minlength=21)
    assert counts.min() > 0.8 * n / 21
    assert abs(np.mean(w > 0) - 0.5) < 0.01
    with pytest.raises(ValueError):
        workloads.draw((2,), "cauchy", 0)
