"""ctypes binding of the native CPU oracle (oz2_oracle.c).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests, the smoke
check and the benchmark's CPU-baseline and reference legs use it; the library
never does.  This module builds the C oracle with the host C compiler (no
architecture flags, so it builds the same on x86-64 and aarch64) and passes
numpy arrays to it.  Every step of the method runs in the C code, except that
the integer products P_t = A_t B_t may instead be taken as an exact float64
BLAS product of the residue planes (a library matmul serving as that step).

Layouts match the checking outputs of the CUDA library's debug entry point:
alpha [p], beta [r] int32; Ares [s, p, q], Bres [s, r, q] int8; R [s, r, p]
uint8; X [r, p, 3] uint64 (192-bit two's complement, little-endian limbs);
C (p, r) float64, column-major.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "oz2_oracle.c")
_LIB = os.path.join(_DIR, "liboz2oracle.so")
_lib = None

OUTPUTS = ("alpha", "beta", "Ares", "Bres", "R", "X", "C")


def build(force: bool = False) -> str:
    """Compile liboz2oracle.so next to its source (when missing or stale)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB + ".tmp"
    cmd = [cc, "-O3", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"building the native oracle failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oz2o_moduli.argtypes = [i32, vp]
    lib.oz2o_moduli.restype = i32
    lib.oz2o_dgemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, i64]
    lib.oz2o_dgemm.restype = i32
    lib.oz2o_residues.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, i32, i32, vp, vp, vp, vp]
    lib.oz2o_residues.restype = i32
    lib.oz2o_products.argtypes = [i64, i64, i64, i32, i32, vp, vp, vp]
    lib.oz2o_products.restype = i32
    lib.oz2o_crt.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp, i64]
    lib.oz2o_crt.restype = i32
    lib.oz2o_exponents.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, i32, i32, vp, vp]
    lib.oz2o_exponents.restype = i32
    lib.oz2o_entries.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, vp, vp, i64, vp, vp, i32, vp, vp, vp]
    lib.oz2o_entries.restype = i32
    lib.oz2o_exact_entries.argtypes = [i64, i64, i64, vp, i64, vp, i64, i64, vp, vp, i32, vp, vp, vp, vp, i32]
    lib.oz2o_exact_entries.restype = i32
    _lib = lib
    return lib


def threads() -> int:
    """Host threads the native oracle uses: every core this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _colmajor(X):
    X = np.asarray(X, dtype=np.float64)
    if not X.flags.f_contiguous:
        X = np.asfortranarray(X)
    return X


def _ptr(a):
    return None if a is None else a.ctypes.data


def moduli(s: int) -> list[int]:
    out = np.zeros(20, dtype=np.int32)
    n = _load().oz2o_moduli(int(s), out.ctypes.data)
    if n < 0:
        raise ValueError("s out of range")
    return [int(v) for v in out[:n]]


def products_blas(Ares, Bres, moduli):
    """R_t = (A_t B_t) mod m_t through a float64 BLAS product of the residue planes.

    Exact: every entry is an integer of magnitude <= 128, so each partial sum is
    an integer of magnitude <= q 2**14 < 2**53 whatever order the BLAS takes
    (q < 2**39).  Returns uint8 [s, r, p]."""
    s, p, q = Ares.shape
    r = Bres.shape[1]
    if q * 2**14 >= 2**53:
        raise ValueError("inner dimension too long for an exact float64 product")
    R = np.empty((s, r, p), dtype=np.uint8)
    for t, m in enumerate(moduli):
        # P^T = B_t A_t^T (r x p), so that R_t comes out in its [r][p] layout
        Pt = Bres[t].astype(np.float64) @ Ares[t].astype(np.float64).T
        R[t] = np.mod(Pt.astype(np.int64), m).astype(np.uint8)
    return R


def dgemm(A, B, s: int, mode: str, want=OUTPUTS, nthreads: int | None = None, products: str = "c") -> dict:
    """Every stage of Ozaki-II in the native oracle; returns the requested outputs.

    products: "c" (the C oracle's own exact integer products) or "blas" (an
    exact float64 BLAS product of the residue planes, products_blas)."""
    A = _colmajor(A)
    B = _colmajor(B)
    p, q = A.shape
    q2, r = B.shape
    if q != q2:
        raise ValueError("inner dimensions differ")
    md = {"fast": 0, "accu": 1}[mode]
    nt = nthreads or threads()
    lib = _load()
    alpha = np.empty(p, dtype=np.int32)
    beta = np.empty(r, dtype=np.int32)
    Ares = np.empty((s, p, q), dtype=np.int8)
    Bres = np.empty((s, r, q), dtype=np.int8)
    rc = lib.oz2o_residues(p, q, r, A.ctypes.data, p, B.ctypes.data, q, int(s), md, nt, alpha.ctypes.data,
                           beta.ctypes.data, Ares.ctypes.data, Bres.ctypes.data)
    if rc != 0:
        raise ValueError(f"native oracle refused the problem (code {rc})")
    if products == "blas":
        R = products_blas(Ares, Bres, moduli(s))
    elif products == "c":
        R = np.empty((s, r, p), dtype=np.uint8)
        rc = lib.oz2o_products(p, q, r, int(s), nt, Ares.ctypes.data, Bres.ctypes.data, R.ctypes.data)
        if rc != 0:
            raise ValueError(f"native oracle products failed (code {rc})")
    else:
        raise ValueError(products)
    X = np.empty((r, p, 3), dtype=np.uint64) if "X" in want else None
    C = np.empty((p, r), dtype=np.float64, order="F") if "C" in want else None
    if X is not None or C is not None:
        rc = lib.oz2o_crt(p, r, int(s), nt, R.ctypes.data, alpha.ctypes.data, beta.ctypes.data, _ptr(X), _ptr(C), p)
        if rc != 0:
            raise ValueError(f"native oracle CRT failed (code {rc})")
    o = {"alpha": alpha, "beta": beta, "Ares": Ares, "Bres": Bres, "R": R, "X": X, "C": C}
    return {k: o[k] for k in want if o.get(k) is not None}


def dgemm_all_in_c(A, B, s: int, mode: str, nthreads: int | None = None) -> dict:
    """The same stages through the C oracle's single entry point (every output)."""
    A = _colmajor(A)
    B = _colmajor(B)
    p, q = A.shape
    r = B.shape[1]
    o = {"alpha": np.empty(p, dtype=np.int32), "beta": np.empty(r, dtype=np.int32),
         "Ares": np.empty((s, p, q), dtype=np.int8), "Bres": np.empty((s, r, q), dtype=np.int8),
         "R": np.empty((s, r, p), dtype=np.uint8), "X": np.empty((r, p, 3), dtype=np.uint64),
         "C": np.empty((p, r), dtype=np.float64, order="F")}
    rc = _load().oz2o_dgemm(p, q, r, A.ctypes.data, p, B.ctypes.data, q, int(s), {"fast": 0, "accu": 1}[mode],
                            nthreads or threads(), *[o[k].ctypes.data for k in OUTPUTS], p)
    if rc != 0:
        raise ValueError(f"native oracle refused the problem (code {rc})")
    return o


def exponents(A, B, s: int, mode: str, nthreads: int | None = None):
    """(alpha, beta): the row and column exponents of the native oracle."""
    A = _colmajor(A)
    B = _colmajor(B)
    p, q = A.shape
    r = B.shape[1]
    alpha = np.empty(p, dtype=np.int32)
    beta = np.empty(r, dtype=np.int32)
    rc = _load().oz2o_exponents(p, q, r, A.ctypes.data, p, B.ctypes.data, q, int(s), {"fast": 0, "accu": 1}[mode],
                                nthreads or threads(), alpha.ctypes.data, beta.ctypes.data)
    if rc != 0:
        raise ValueError(f"native oracle refused the problem (code {rc})")
    return alpha, beta


def entries(A, B, s: int, alpha, beta, ii, jj, nthreads: int | None = None) -> dict:
    """The pipeline at sampled outputs (ii[k], jj[k]) only, given the exponents.

    Returns R [n, s] uint8, X [n, 3] uint64 (192-bit two's complement) and C [n]."""
    A = _colmajor(A)
    B = _colmajor(B)
    p, q = A.shape
    r = B.shape[1]
    alpha = np.ascontiguousarray(alpha, dtype=np.int32)
    beta = np.ascontiguousarray(beta, dtype=np.int32)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    n = ii.shape[0]
    R = np.empty((n, s), dtype=np.uint8)
    X = np.empty((n, 3), dtype=np.uint64)
    C = np.empty(n, dtype=np.float64)
    rc = _load().oz2o_entries(p, q, r, A.ctypes.data, p, B.ctypes.data, q, int(s), alpha.ctypes.data,
                              beta.ctypes.data, n, ii.ctypes.data, jj.ctypes.data, nthreads or threads(),
                              R.ctypes.data, X.ctypes.data, C.ctypes.data)
    if rc != 0:
        raise ValueError(f"native oracle refused the entries (code {rc})")
    return {"R": R, "X": X, "C": C}


def exact_entries(A, B, ii, jj, Chats=(), nthreads: int | None = None):
    """Exact dot products at the sampled outputs (ii[k], jj[k]), each rounded once.

    Returns (exact, absprod, err): RN((AB)_ij), RN((|A||B|)_ij) and, for each
    array in Chats (values at the same entries), RN(C_hat_ij - (AB)_ij)."""
    A = _colmajor(A)
    B = _colmajor(B)
    p, q = A.shape
    r = B.shape[1]
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    n = ii.shape[0]
    nc = len(Chats)
    Ch = np.ascontiguousarray(np.stack([np.asarray(c, dtype=np.float64) for c in Chats])) if nc else None
    exact = np.empty(n, dtype=np.float64)
    absprod = np.empty(n, dtype=np.float64)
    err = np.empty((nc, n), dtype=np.float64) if nc else None
    rc = _load().oz2o_exact_entries(p, q, r, A.ctypes.data, p, B.ctypes.data, q, n, ii.ctypes.data,
                                    jj.ctypes.data, nc, _ptr(Ch), exact.ctypes.data, absprod.ctypes.data,
                                    _ptr(err), nthreads or threads())
    if rc != 0:
        raise ValueError(f"native oracle refused the entries (code {rc})")
    return exact, absprod, (list(err) if nc else [])


def _norm2(x):
    """Euclidean norm without overflow or underflow of the squares."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    m = float(x.max()) if x.size else 0.0
    if m == 0.0 or not np.isfinite(m):
        return m
    return m * float(np.sqrt(np.sum((x / m) ** 2)))


def accuracy_at(A, B, ii, jj, values: dict) -> dict:
    """Errors against the exact AB at the entries (ii[k], jj[k]).

    values: name -> the product's values at those entries.  For each name:
    normwise      = ||C_hat - AB|| / ||AB||   (2-norms over the entries),
    componentwise = max |C_hat - AB|_ij / (|A||B|)_ij over entries with (|A||B|)_ij > 0
                    (inf if C_hat is nonzero where |A||B| is zero),
    max_abs_err   = max |C_hat - AB|_ij."""
    names = list(values)
    exact, absprod, errs = exact_entries(A, B, ii, jj, [values[k] for k in names])
    out = {"entries": int(len(exact))}
    den = _norm2(exact)
    pos = absprod > 0
    for k, e in zip(names, errs):
        comp = float(np.max(np.abs(e[pos]) / absprod[pos])) if np.any(pos) else 0.0
        if np.any(e[~pos] != 0):
            comp = float("inf")
        out[k] = {"normwise": _norm2(e) / den if den > 0 else _norm2(e),
                  "componentwise": comp, "max_abs_err": float(np.max(np.abs(e))) if e.size else 0.0}
    return out


def accuracy(A, B, Cs: dict) -> dict:
    """accuracy_at over every entry of the full (p, r) products in Cs."""
    p, r = np.shape(A)[0], np.shape(B)[1]
    jj_g, ii_g = np.meshgrid(np.arange(r), np.arange(p))
    ii, jj = ii_g.ravel(), jj_g.ravel()
    return accuracy_at(A, B, ii, jj, {k: np.asarray(v)[ii, jj] for k, v in Cs.items()})
