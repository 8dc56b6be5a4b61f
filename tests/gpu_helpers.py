"""Helpers for the GPU tests: run the library's stages through the C-ABI and
bring the results back as numpy arrays."""
from __future__ import annotations

import numpy as np
import torch

from fp64_gemm_emulation_exponent_gb300 import ozk


def dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def strided(x: np.ndarray, pad: int, offset: int = 0) -> tuple[torch.Tensor, torch.Tensor]:
    """Device copy of x inside a wider buffer: leading dimension cols + pad, first
    element at `offset` doubles from an allocation boundary.  Returns (view, buffer)."""
    rows, cols = x.shape
    ld = cols + pad
    buf = torch.zeros(offset + rows * ld + 1, dtype=torch.float64, device="cuda")
    view = buf[offset: offset + rows * ld].view(rows, ld)[:, :cols]
    view.copy_(torch.from_numpy(x))
    return view, buf


def ld_of(t: torch.Tensor) -> int:
    return max(t.stride(0), t.size(1), 1)


def f16_to_int(bits: np.ndarray) -> np.ndarray:
    """Integers held in IEEE binary16 bit patterns (exact for |v| <= 2048)."""
    f = np.ascontiguousarray(bits).astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.all(f == np.round(f))
    return f.astype(np.int64)


def run_scale(A: torch.Tensor, B: torch.Tensor, n: int):
    M, K = A.shape
    _, N = B.shape
    s = torch.empty(M, dtype=torch.int32, device="cuda")
    t = torch.empty(N, dtype=torch.int32, device="cuda")
    scratch = torch.empty(M + N, dtype=torch.int64, device="cuda")
    ozk.ozk_scale(M, N, K, A, ld_of(A), B, ld_of(B), n, s, t, scratch)
    return s, t


def run_quantize(A: torch.Tensor, B: torch.Tensor, s, t, n: int):
    M, K = A.shape
    _, N = B.shape
    kpad = ozk.ozk_kpad(K)
    a_sl = torch.full((n, M, kpad), 0x7FFF, dtype=torch.int16, device="cuda")  # poison padding
    b_sl = torch.full((n, N, kpad), 0x7FFF, dtype=torch.int16, device="cuda")
    ozk.ozk_quantize_a(M, K, A, ld_of(A), s, n, a_sl)
    ozk.ozk_quantize_b(K, N, B, ld_of(B), t, n, b_sl)
    return a_sl, b_sl


def run_gemm(a_sl, b_sl, M, N, K, n, out_kind=0, splits=1):
    if out_kind == 0:
        ldo = (N + 15) // 16 * 16
        out = torch.full((n, M, ldo), 0xEE, dtype=torch.uint8, device="cuda")
    elif out_kind == 2:
        ldo = (N + 7) // 8 * 8
        out = torch.full(((n + 1) // 2, M, ldo), -1, dtype=torch.int16, device="cuda")
    else:
        ldo = (N + 3) // 4 * 4
        out = torch.full((splits, n, M, ldo), -7, dtype=torch.int32, device="cuda")
    ozk.ozk_residue_gemm(M, N, K, a_sl, b_sl, n, out_kind, out, ldo, splits)
    return out, ldo


def run_lift(out, in_kind, ldo, splits, M, N, n):
    X = torch.zeros((M, N, ozk.OZK_LIMBS), dtype=torch.int32, device="cuda")
    ozk.ozk_crt_lift(M, N, n, out, in_kind, ldo, splits, X)
    return X


def run_combine(out, in_kind, ldo, splits, s, t, M, N, n):
    C = torch.full((M, N), np.nan, dtype=torch.float64, device="cuda")
    ozk.ozk_crt_combine(M, N, n, out, in_kind, ldo, splits, s, t, C, N)
    return C


def dgemm(A: np.ndarray, B: np.ndarray, n: int) -> np.ndarray:
    C = ozk.dgemm(dev(A), dev(B), n)
    torch.cuda.synchronize()
    assert ozk.ozk_stream_status() == 0
    return C.cpu().numpy()


def same_bits(x, y) -> bool:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.ascontiguousarray(y, dtype=np.float64)
    xb, yb = x.view(np.uint64), y.view(np.uint64)
    nan = np.isnan(x) & np.isnan(y)
    return bool(np.all((xb == yb) | nan))
