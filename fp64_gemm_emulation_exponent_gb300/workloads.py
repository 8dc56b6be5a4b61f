"""Seeded synthetic inputs for the FP64 GEMM workloads.

This module holds no arithmetic of the method: it only draws matrices.  Both
the CUDA path's tests/benchmark and the CPU oracle take their inputs from here.

Workloads (all row-major float64, A is M x K, B is K x N):

* ``normal``   i.i.d. N(0, 1)
* ``uniform``  i.i.d. U(-1, 1)
* ``wide``     sign * U(0.5, 1) * 2^e with e uniform on the integers -10..10,
               independently per element (stresses per-row/column scaling)

Seeds: A uses ``1000 + c`` and B uses ``2000 + c`` for workload number ``c``.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str
    moduli: tuple
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five GEMM shapes the method is measured on; index = seed offset.
WORKLOADS = {
    "square256_normal": Workload("square256_normal", 256, 256, 256, "normal", (14,), 0),
    "square1024_wide": Workload("square1024_wide", 1024, 1024, 1024, "wide", (14, 8, 11), 1),
    "square4096_normal": Workload("square4096_normal", 4096, 4096, 4096, "normal", (14, 8, 11), 2),
    "square8192_uniform": Workload("square8192_uniform", 8192, 8192, 8192, "uniform", (14,), 3),
    "wide8192_k512": Workload("wide8192_k512", 8192, 8192, 512, "normal", (8, 11, 14, 17, 20), 4),
    "tall512_k65536": Workload("tall512_k65536", 512, 512, 65536, "normal", (8, 11, 14, 17, 20), 5),
}


def draw(shape, dist: str, seed: int) -> np.ndarray:
    """A float64 array of ``shape`` from distribution ``dist``, seeded."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if dist == "normal":
        x = rng.standard_normal(shape)
    elif dist == "uniform":
        x = rng.uniform(-1.0, 1.0, shape)
    elif dist == "wide":
        sign = np.where(rng.integers(0, 2, shape) == 0, -1.0, 1.0)
        mag = rng.uniform(0.5, 1.0, shape)
        e = rng.integers(-10, 11, shape)
        x = sign * np.ldexp(mag, e)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return np.ascontiguousarray(x, dtype=np.float64)


def operands(M: int, N: int, K: int, dist: str = "normal", seed: int = 0):
    """(A, B) for one GEMM: A is M x K with seed 1000+seed, B is K x N with 2000+seed."""
    return draw((M, K), dist, 1000 + seed), draw((K, N), dist, 2000 + seed)


def workload_operands(w: Workload):
    return operands(w.M, w.N, w.K, w.dist, w.seed)
