"""CPU oracle for Ozaki-scheme-II FP64 GEMM emulation: TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It is a ctypes view of ``ozk_oracle.c`` (plain C,
compiled by ``oracle/build.py``) and shares nothing with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

LIMBS = 8
NONFINITE = -(2**31)

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        sigs = {
            "ozk_ref_moduli": [i32, vp],
            "ozk_ref_beta": [i64, i32],
            "ozk_ref_scale": [i64, i64, i64, vp, i64, vp, i64, i32, vp, vp],
            "ozk_ref_integers": [i64, i64, vp, i64, vp, i32, vp],
            "ozk_ref_residues": [i64, vp, i32, vp],
            "ozk_ref_gemm_mod": [i64, i64, i64, vp, vp, i32, vp, vp],
            "ozk_ref_crt": [i64, i32, vp, vp],
            "ozk_ref_direct": [i64, i64, i64, vp, vp, vp],
            "ozk_ref_round": [i64, vp, vp, vp],
            "ozk_ref_dgemm": [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32],
            "ozk_ref_sample": [i64, i64, i64, vp, i64, vp, i64, i32, i64, vp, vp, vp, vp, vp, vp],
            "ozk_ref_dot2": [i64, i64, i64, vp, i64, vp, i64, vp],
            "ozk_ref_dot2_sample": [i64, vp, i64, vp, i64, i64, vp, vp, vp, vp],
            "ozk_ref_threads": [],
            "ozk_ref_gamma": [i64, i32],
            "ozk_ref_scale_norm": [i64, i64, i64, vp, i64, vp, i64, i32, vp, vp],
            "ozk_ref_dgemm_norm": [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32],
            "ozk_ref_sample_norm": [i64, i64, i64, vp, i64, vp, i64, i32, i64, vp, vp, vp, vp, vp, vp],
        }
        for name, args in sigs.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc < 0:
        raise OracleError(f"{what} failed with code {rc}")
    return rc


def _f64(x):
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 2 or x.strides[1] != 8:
        x = np.ascontiguousarray(x)
    return x


def moduli(n):
    out = np.zeros(n, dtype=np.int32)
    _check(lib().ozk_ref_moduli(n, _p(out)), "moduli")
    return out


def beta(K, n):
    """Bit budget per operand; raises OracleError when n is too small for K."""
    return _check(lib().ozk_ref_beta(K, n), "beta")


def scale(A, B, n, rule="max"):
    """Row and column scales: rule "max" (the largest entry, reading R2) or
    "norm" (the computed 2-norm bound, reading R15)."""
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    s = np.zeros(M, dtype=np.int32)
    t = np.zeros(N, dtype=np.int32)
    f = lib().ozk_ref_scale_norm if rule == "norm" else lib().ozk_ref_scale
    _check(f(M, N, K, _p(A), A.strides[0] // 8, _p(B), B.strides[0] // 8, n, _p(s), _p(t)), "scale")
    return s, t


def gamma(K, n):
    """Norm budget per operand of the "norm" rule; raises OracleError when unsupported."""
    return _check(lib().ozk_ref_gamma(K, n), "gamma")


def integers(X, sc, by_row):
    """X * 2^scale rounded to nearest integers (ties to even), as exact float64."""
    X = _f64(X)
    rows, cols = X.shape
    sc = np.ascontiguousarray(sc, dtype=np.int32)
    out = np.zeros((rows, cols), dtype=np.float64)
    _check(lib().ozk_ref_integers(rows, cols, _p(X), X.strides[0] // 8, _p(sc), 1 if by_row else 0, _p(out)),
           "integers")
    return out


def residues(xp, n):
    """n x shape residues (int8) of exact integers held in float64."""
    xp = np.ascontiguousarray(xp, dtype=np.float64)
    out = np.zeros((n,) + xp.shape, dtype=np.int8)
    _check(lib().ozk_ref_residues(xp.size, _p(xp), n, _p(out)), "residues")
    return out


def gemm_mod(ra, rb, n):
    """ra: n x M x K, rb: n x K x N int8 -> (raw int32 n x M x N, cmod uint8 n x M x N)."""
    ra = np.ascontiguousarray(ra, dtype=np.int8)
    rb = np.ascontiguousarray(rb, dtype=np.int8)
    _, M, K = ra.shape
    _, _, N = rb.shape
    raw = np.zeros((n, M, N), dtype=np.int32)
    cmod = np.zeros((n, M, N), dtype=np.uint8)
    _check(lib().ozk_ref_gemm_mod(M, N, K, _p(ra), _p(rb), n, _p(raw), _p(cmod)), "gemm_mod")
    return raw, cmod


def crt(cmod, n):
    """cmod: n x ... canonical residues -> signed wide integers, shape (...) x LIMBS uint32."""
    cmod = np.ascontiguousarray(cmod, dtype=np.uint8)
    count = cmod[0].size
    X = np.zeros(cmod.shape[1:] + (LIMBS,), dtype=np.uint32)
    _check(lib().ozk_ref_crt(count, n, _p(cmod), _p(X)), "crt")
    return X


def direct(Ap, Bp):
    Ap = np.ascontiguousarray(Ap, dtype=np.float64)
    Bp = np.ascontiguousarray(Bp, dtype=np.float64)
    M, K = Ap.shape
    _, N = Bp.shape
    X = np.zeros((M, N, LIMBS), dtype=np.uint32)
    _check(lib().ozk_ref_direct(M, N, K, _p(Ap), _p(Bp), _p(X)), "direct")
    return X


def round_scaled(X, S):
    X = np.ascontiguousarray(X, dtype=np.uint32)
    S = np.ascontiguousarray(S, dtype=np.int32)
    out = np.zeros(S.shape, dtype=np.float64)
    _check(lib().ozk_ref_round(S.size, _p(X), _p(S), _p(out)), "round")
    return out


def dgemm(A, B, n, rule="max"):
    """The whole method on the CPU.  Raises if the CRT check fails anywhere."""
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    _, N = B.shape
    C = np.zeros((M, N), dtype=np.float64)
    f = lib().ozk_ref_dgemm_norm if rule == "norm" else lib().ozk_ref_dgemm
    _check(f(M, N, K, _p(A), A.strides[0] // 8, _p(B), B.strides[0] // 8, _p(C), N, n), "dgemm")
    return C


def sample(A, B, n, ii, jj, rule="max"):
    """Method at chosen outputs: returns (C, raw n-per-pair, cmod n-per-pair, X limbs)."""
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    _, N = B.shape
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    q = ii.size
    C = np.zeros(q, dtype=np.float64)
    raw = np.zeros((q, n), dtype=np.int32)
    cmod = np.zeros((q, n), dtype=np.uint8)
    X = np.zeros((q, LIMBS), dtype=np.uint32)
    f = lib().ozk_ref_sample_norm if rule == "norm" else lib().ozk_ref_sample
    _check(f(M, N, K, _p(A), A.strides[0] // 8, _p(B), B.strides[0] // 8, n, q,
             _p(ii), _p(jj), _p(C), _p(raw), _p(cmod), _p(X)), "sample")
    return C, raw, cmod, X


def dot2(A, B):
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    _, N = B.shape
    R = np.zeros((M, N), dtype=np.float64)
    _check(lib().ozk_ref_dot2(M, N, K, _p(A), A.strides[0] // 8, _p(B), B.strides[0] // 8, _p(R)), "dot2")
    return R


def dot2_sample(A, B, ii, jj):
    """Compensated reference and sum_k |a_ik||b_kj| at chosen outputs."""
    A, B = _f64(A), _f64(B)
    _, K = A.shape
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    R = np.zeros(ii.size, dtype=np.float64)
    ab = np.zeros(ii.size, dtype=np.float64)
    _check(lib().ozk_ref_dot2_sample(K, _p(A), A.strides[0] // 8, _p(B), B.strides[0] // 8, ii.size,
                                     _p(ii), _p(jj), _p(R), _p(ab)), "dot2_sample")
    return R, ab


def threads():
    return lib().ozk_ref_threads()


def limbs_to_int(X):
    """Signed Python int(s) from LIMBS x uint32 two's-complement limbs."""
    X = np.asarray(X, dtype=np.uint32)
    if X.ndim == 1:
        v = 0
        for l in range(LIMBS - 1, -1, -1):
            v = (v << 32) | int(X[l])
        if v >> (32 * LIMBS - 1):
            v -= 1 << (32 * LIMBS)
        return v
    flat = X.reshape(-1, LIMBS)
    return [limbs_to_int(r) for r in flat]
