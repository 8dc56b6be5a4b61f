"""Python binding of libozk (ctypes): argument marshalling only.

Every function here forwards to the C-ABI entry point of the same name in
``include/ozk.h``; all computation runs in the library's CUDA kernels.  The
library must have been built (``fp64_gemm_emulation_exponent_gb300.build``);
loading fails loudly otherwise, and there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libozk.so")

OZK_OK = 0
OZK_ERR_INVALID_ARG = 1
OZK_ERR_UNSUPPORTED = 2
OZK_ERR_WORKSPACE = 3
OZK_ERR_CUDA = 4
OZK_ERR_TIMEOUT = 5
OZK_ERR_DEVICE = 6
OZK_MAX_MODULI = 20
OZK_MAX_K = 4194304
OZK_SPLIT_MAX_K = 131008
OZK_SCALE_NONFINITE = -(2**31)
OZK_LIMBS = 8
OZK_SCALE_NOALLOC_MAX = 262144

_i64, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t

# name -> (restype, argtypes), mirroring include/ozk.h
SIGNATURES = {
    "ozk_status_string": (ctypes.c_char_p, [_i32]),
    "ozk_moduli": (_i32, [_i32, _vp]),
    "ozk_beta": (_i32, [_i64, _i32]),
    "ozk_kpad": (_i64, [_i64]),
    "ozk_gamma": (_i32, [_i64, _i32]),
    "ozk_dgemm_norm": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp]),
    "ozk_dgemm_norm_ws": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _sz, _vp]),
    "ozk_dgemm_norm_ws_timed": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _sz, _vp, _vp]),
    "ozk_scale_norm": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _vp, _vp]),
    "ozk_moduli_for_bits": (_i32, [_i64, _i32]),
    "ozk_dgemm_bits": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp]),
    "ozk_workspace_size": (_sz, [_i64, _i64, _i64, _i32]),
    "ozk_workspace_layout": (_i32, [_i64, _i64, _i64, _i32, _vp]),
    "ozk_dgemm": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp]),
    "ozk_dgemm_ws": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _sz, _vp]),
    "ozk_dgemm_ws_timed": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _sz, _vp, _vp]),
    "ozk_dgemm_host": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp]),
    "ozk_dgemm_host_async": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp]),
    "ozk_stream_status": (_i32, [_vp]),
    "ozk_release_cached": (_i32, []),
    "ozk_scale": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _vp, _vp]),
    "ozk_scale_noalloc": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _vp]),
    "ozk_quantize_a": (_i32, [_i64, _i64, _vp, _i64, _vp, _i32, _vp, _vp]),
    "ozk_quantize_b": (_i32, [_i64, _i64, _vp, _i64, _vp, _i32, _vp, _vp]),
    "ozk_residue_gemm": (_i32, [_i64, _i64, _i64, _vp, _vp, _i32, _i32, _vp, _i64, _i32, _vp]),
    "ozk_residue_gemm_withheld": (_i32, [_i64, _i64, _i64, _vp, _vp, _i32, _vp, _i64, _i32, ctypes.c_uint32, _vp]),
    "ozk_crt_combine": (_i32, [_i64, _i64, _i32, _vp, _i32, _i64, _i32, _vp, _vp, _vp, _i64, _vp]),
    "ozk_crt_lift": (_i32, [_i64, _i64, _i32, _vp, _i32, _i64, _i32, _vp, _vp]),
    "ozk_event_create": (_i32, [_vp]),
    "ozk_event_destroy": (_i32, [_vp]),
    "ozk_event_record": (_i32, [_vp, _vp]),
    "ozk_event_elapsed": (_i32, [_vp, _vp, _vp]),
    "ozk_device_sm_count": (_i32, []),
}

class WorkspaceInfo(ctypes.Structure):
    """ozk_workspace_info of include/ozk.h."""
    _fields_ = [("total_bytes", ctypes.c_size_t), ("maxima_offset", ctypes.c_size_t),
                ("s_offset", ctypes.c_size_t), ("t_offset", ctypes.c_size_t),
                ("a_slices_offset", ctypes.c_size_t), ("b_slices_offset", ctypes.c_size_t),
                ("planes_offset", ctypes.c_size_t), ("kpad", ctypes.c_int64), ("a_plane", ctypes.c_int64),
                ("b_plane", ctypes.c_int64), ("planes_kind", ctypes.c_int), ("planes_ld", ctypes.c_int64),
                ("planes_plane", ctypes.c_int64), ("splits", ctypes.c_int)]


_lib = None


class OzkError(RuntimeError):
    def __init__(self, name, status):
        self.status = status
        super().__init__(f"{name} returned {status}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """The loaded libozk.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
            )
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().ozk_status_string(status).decode()


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != OZK_OK:
        raise OzkError(name, rc)
    return rc


# ---------------------------------------------------------------- host helpers
def ozk_moduli(n_moduli: int):
    out = (ctypes.c_int32 * n_moduli)()
    _call("ozk_moduli", n_moduli, ctypes.cast(out, _vp))
    return list(out)


def ozk_beta(K: int, n_moduli: int) -> int:
    return lib().ozk_beta(K, n_moduli)


def ozk_kpad(K: int) -> int:
    return lib().ozk_kpad(K)


def ozk_moduli_for_bits(K: int, target_bits: int) -> int:
    return lib().ozk_moduli_for_bits(K, target_bits)


def ozk_workspace_size(M: int, N: int, K: int, n_moduli: int) -> int:
    return lib().ozk_workspace_size(M, N, K, n_moduli)


# ---------------------------------------------------------------- torch helpers
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ld(t):
    """Leading dimension (elements) of a row-major 2-D tensor with unit column stride."""
    if t.dim() != 2 or (t.stride(1) != 1 and t.size(1) > 1):
        raise ValueError("expected a 2-D row-major tensor with unit column stride")
    return max(t.stride(0), t.size(1), 1)


# ---------------------------------------------------------------- the GEMM
def ozk_dgemm(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, stream=None):
    """C-ABI ozk_dgemm on device tensors (A, B, C are torch.float64 CUDA tensors)."""
    return _call("ozk_dgemm", M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n_moduli, _stream(stream))


def ozk_dgemm_ws(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, workspace, workspace_bytes, stream=None):
    return _call("ozk_dgemm_ws", M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n_moduli,
                 _ptr(workspace), workspace_bytes, _stream(stream))


def ozk_dgemm_ws_timed(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, workspace, workspace_bytes, events,
                       stream=None):
    ev = (ctypes.c_void_p * 5)(*[e.value for e in events]) if events is not None else None
    return _call("ozk_dgemm_ws_timed", M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n_moduli,
                 _ptr(workspace), workspace_bytes, _stream(stream), ctypes.cast(ev, _vp) if ev else None)


def ozk_dgemm_norm_ws_timed(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, workspace, workspace_bytes, events,
                            stream=None):
    ev = (ctypes.c_void_p * 5)(*[e.value for e in events]) if events is not None else None
    return _call("ozk_dgemm_norm_ws_timed", M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n_moduli,
                 _ptr(workspace), workspace_bytes, _stream(stream), ctypes.cast(ev, _vp) if ev else None)


def ozk_dgemm_host(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, stream=None):
    """Host (CPU, ideally pinned) float64 tensors in and out; synchronous."""
    return _call("ozk_dgemm_host", M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n_moduli, _stream(stream))


def ozk_dgemm_host_async(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, stream=None):
    """Host (pinned) float64 tensors; returns once enqueued, C is complete when the stream gets there."""
    return _call("ozk_dgemm_host_async", M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n_moduli,
                 _stream(stream))


def ozk_stream_status(stream=None):
    return lib().ozk_stream_status(_stream(stream))


def ozk_release_cached():
    return _call("ozk_release_cached")


def dgemm(A, B, n_moduli: int = 14, out=None, stream=None, target_bits=None, scaling="max"):
    """C = A @ B for float64 CUDA tensors through ozk_dgemm (or ozk_dgemm_bits
    when target_bits is given: the moduli count then follows from K; or
    ozk_dgemm_norm with scaling="norm": scales from the rows' 2-norms)."""
    import torch

    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float64, device=A.device)
    if scaling == "norm":
        if target_bits is not None:
            raise ValueError("target_bits picks the count of the largest-entry rule")
        ozk_dgemm_norm(M, N, K, A, _ld(A), B, _ld(B), out, _ld(out), n_moduli, stream)
    elif scaling != "max":
        raise ValueError(f"unknown scaling {scaling!r}")
    elif target_bits is None:
        ozk_dgemm(M, N, K, A, _ld(A), B, _ld(B), out, _ld(out), n_moduli, stream)
    else:
        _call("ozk_dgemm_bits", M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(out), _ld(out), target_bits,
              _stream(stream))
    return out


# ---------------------------------------------------------------- stages
def ozk_scale(M, N, K, A, lda, B, ldb, n_moduli, s, t, scratch, stream=None):
    return _call("ozk_scale", M, N, K, _ptr(A), lda, _ptr(B), ldb, n_moduli, _ptr(s), _ptr(t), _ptr(scratch),
                 _stream(stream))


def ozk_workspace_layout(M: int, N: int, K: int, n_moduli: int) -> WorkspaceInfo:
    info = WorkspaceInfo()
    _call("ozk_workspace_layout", M, N, K, n_moduli, ctypes.cast(ctypes.pointer(info), _vp))
    return info


def ozk_gamma(K: int, n_moduli: int) -> int:
    return lib().ozk_gamma(K, n_moduli)


def ozk_dgemm_norm(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, stream=None):
    return _call("ozk_dgemm_norm", M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n_moduli, _stream(stream))


def ozk_dgemm_norm_ws(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, workspace, workspace_bytes, stream=None):
    return _call("ozk_dgemm_norm_ws", M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n_moduli, _ptr(workspace),
                 workspace_bytes, _stream(stream))


def ozk_scale_norm(M, N, K, A, lda, B, ldb, n_moduli, s, t, scratch, stream=None):
    return _call("ozk_scale_norm", M, N, K, _ptr(A), lda, _ptr(B), ldb, n_moduli, _ptr(s), _ptr(t), _ptr(scratch),
                 _stream(stream))


def ozk_scale_noalloc(M, N, K, A, lda, B, ldb, n_moduli, s, t, stream=None):
    return _call("ozk_scale_noalloc", M, N, K, _ptr(A), lda, _ptr(B), ldb, n_moduli, _ptr(s), _ptr(t),
                 _stream(stream))


def ozk_quantize_a(M, K, A, lda, s, n_moduli, a_slices, stream=None):
    return _call("ozk_quantize_a", M, K, _ptr(A), lda, _ptr(s), n_moduli, _ptr(a_slices), _stream(stream))


def ozk_quantize_b(K, N, B, ldb, t, n_moduli, b_slices, stream=None):
    return _call("ozk_quantize_b", K, N, _ptr(B), ldb, _ptr(t), n_moduli, _ptr(b_slices), _stream(stream))


def ozk_residue_gemm(M, N, K, a_slices, b_slices, n_moduli, out_kind, out, ldo, splits, stream=None):
    return _call("ozk_residue_gemm", M, N, K, _ptr(a_slices), _ptr(b_slices), n_moduli, out_kind, _ptr(out), ldo,
                 splits, _stream(stream))


def ozk_residue_gemm_withheld(M, N, K, a_slices, b_slices, n_moduli, out, ldo, withhold_kb, timeout_us,
                              stream=None):
    return _call("ozk_residue_gemm_withheld", M, N, K, _ptr(a_slices), _ptr(b_slices), n_moduli, _ptr(out), ldo,
                 withhold_kb, timeout_us, _stream(stream))


def ozk_crt_combine(M, N, n_moduli, inp, in_kind, ldi, splits, s, t, C, ldc, stream=None):
    return _call("ozk_crt_combine", M, N, n_moduli, _ptr(inp), in_kind, ldi, splits, _ptr(s), _ptr(t), _ptr(C), ldc,
                 _stream(stream))


def ozk_crt_lift(M, N, n_moduli, inp, in_kind, ldi, splits, X, stream=None):
    return _call("ozk_crt_lift", M, N, n_moduli, _ptr(inp), in_kind, ldi, splits, _ptr(X), _stream(stream))


# ---------------------------------------------------------------- events
class Event:
    """A CUDA event created by the library (for stage timing)."""

    def __init__(self):
        self.handle = ctypes.c_void_p()
        _call("ozk_event_create", ctypes.byref(self.handle))

    @property
    def value(self):
        return self.handle.value

    def record(self, stream=None):
        _call("ozk_event_record", self.handle, _stream(stream))

    def elapsed_ms(self, end: "Event") -> float:
        ms = ctypes.c_float()
        _call("ozk_event_elapsed", self.handle, end.handle, ctypes.byref(ms))
        return ms.value

    def __del__(self):
        try:
            if self.handle and _lib is not None:
                _lib.ozk_event_destroy(self.handle)
        except Exception:
            pass


def sm_count() -> int:
    return lib().ozk_device_sm_count()
