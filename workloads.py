"""Seeded synthetic inputs for the Ozaki-II FP64 GEMM workloads.

This module only draws random matrices and names the workloads. It holds none
of the method's arithmetic, so both the CUDA path (tests, bench) and the CPU
oracle may be fed from it without sharing any code of the method.

Input recipe (the profiling study, "Profiling Ozaki II: The Cost Behind Fast
INT8 GEMMs", §4, names the generator's parameters phi and seed, and says A and
B use the same seed): every entry is (U(0,1) - 0.5) * exp(phi * N(0,1)).
Reading taken here: one seeded stream is drawn in the order
U for A, N for A, U for B, N for B; reseeding for B would make A == B in the
square workloads, a structure the study does not intend.  Matrices are FP64,
column-major (Fortran order), A is p x q and B is q x r.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    p: int
    q: int
    r: int
    s: int
    mode: str  # "fast" or "accu"
    phi: float
    seed: int

    @property
    def flops(self) -> float:
        """Effective FP64 work 2pqr (the study's effective-TFLOPS numerator)."""
        return 2.0 * self.p * self.q * self.r


# The five workloads: a small one the oracle finishes in seconds, the n=1024
# study size, an accu case with wider dynamic range, the n=8192 headline case
# (s in {14, 18}, both bound modes) and a rectangular wide-range accu case.
WORKLOADS = {
    "n128_s8_fast": Workload("n128_s8_fast", 128, 128, 128, 8, "fast", 0.5, 1),
    "n1024_s14_fast": Workload("n1024_s14_fast", 1024, 1024, 1024, 14, "fast", 0.5, 123456),
    # a mid size whose planes (235 MB) still exceed L2: used for detailed kernel profiles
    "n2048_s14_fast": Workload("n2048_s14_fast", 2048, 2048, 2048, 14, "fast", 0.5, 123456),
    # the headline's inner dimension at a few GB on the device: kernel profiles of the
    # preprocessing (B's one-read kernel on 2048-column parts, A's residues at q = 8192)
    "p2048_q8192_r4096_s14_fast": Workload("p2048_q8192_r4096_s14_fast", 2048, 8192, 4096, 14, "fast", 0.5, 123456),
    "n4096_s14_accu": Workload("n4096_s14_accu", 4096, 4096, 4096, 14, "accu", 1.0, 7),
    # the pages' mid size for fast mode (paper Table 3 column n = 4096)
    "n4096_s14_fast": Workload("n4096_s14_fast", 4096, 4096, 4096, 14, "fast", 0.5, 123456),
    "n8192_s14_fast": Workload("n8192_s14_fast", 8192, 8192, 8192, 14, "fast", 0.5, 123456),
    "n8192_s14_accu": Workload("n8192_s14_accu", 8192, 8192, 8192, 14, "accu", 0.5, 123456),
    "n8192_s18_fast": Workload("n8192_s18_fast", 8192, 8192, 8192, 18, "fast", 0.5, 123456),
    "n8192_s18_accu": Workload("n8192_s18_accu", 8192, 8192, 8192, 18, "accu", 0.5, 123456),
    "p16384_q8192_r16384_s18_accu": Workload(
        "p16384_q8192_r16384_s18_accu", 16384, 8192, 16384, 18, "accu", 2.0, 99),
}

HEADLINE = "n8192_s14_fast"


def make_matrices(p: int, q: int, r: int, phi: float, seed: int):
    """Return (A, B): A is p x q, B is q x r, FP64, Fortran (column-major) order."""
    rng = np.random.default_rng(seed)
    ua = rng.random(p * q)
    na = rng.standard_normal(p * q)
    a = (ua - 0.5) * np.exp(phi * na)
    ub = rng.random(q * r)
    nb = rng.standard_normal(q * r)
    b = (ub - 0.5) * np.exp(phi * nb)
    A = np.asfortranarray(a.reshape((p, q), order="F"))
    B = np.asfortranarray(b.reshape((q, r), order="F"))
    return A, B


def make_workload(w: Workload):
    return make_matrices(w.p, w.q, w.r, w.phi, w.seed)
