"""FP64 GEMM emulated with exact integer residue GEMMs on GB300 tensor cores
and Chinese-Remainder reconstruction (Ozaki scheme II).

The computation lives in ``libozk.so`` (CUDA kernels for sm_103a behind the
C-ABI of ``include/ozk.h``); ``ozk`` is its ctypes binding.
"""
from .ozk import dgemm  # noqa: F401
