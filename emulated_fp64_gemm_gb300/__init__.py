"""Ozaki Scheme II FP64 GEMM for GB300 (sm_103a): Python binding of libozaki2.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libozaki2.so`` behind the C ABI declared in ``include/ozaki2.h``.
PyTorch supplies device memory and streams.  There is no CPU fallback: if
the library is not built, loading it raises.

Matrices follow the library's column-major convention: a (p, q) tensor with
strides (1, ld), ld >= p, is passed as is.  Any other layout (row-major,
or a non-unit row stride) is first copied into a column-major tensor on the
same device, so the library always sees column-major operands.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "FAST", "ACCU", "Ozaki2Error", "load_library", "library_path", "moduli", "dgemm",
    "dgemm_debug", "dgemm_stages", "dgemm_host", "last_error", "workspace_release",
    "selftest_wait_timeout", "STAGE_NAMES", "profile_begin", "profile_end", "launch_count",
]

FAST = 0
ACCU = 1
S_MIN, S_MAX = 2, 20
# exclusive inner-dimension limits: fast mode, accu mode, debug output P (int32)
Q_LIMIT_FAST, Q_LIMIT_ACCU, Q_LIMIT_P = 1 << 24, 133145, 131072
STAGE_NAMES = ["scale", "bound_gemm", "residues", "gemm_mod", "crt", "total"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libozaki2.so"
_lib = None

STATUS = {
    0: "OZ2_OK", 1: "OZ2_ERR_INVALID_ARG", 2: "OZ2_ERR_Q_TOO_LARGE", 3: "OZ2_ERR_NO_MEMORY",
    4: "OZ2_ERR_CUDA", 5: "OZ2_ERR_DEVICE_TIMEOUT", 6: "OZ2_ERR_UNSUPPORTED_DEVICE",
    7: "OZ2_ERR_SCRATCH_TOO_SMALL",
}


class Ozaki2Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


def library_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


def load_library():
    """Load libozaki2.so (in-tree).  Raises OSError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
    common = [i64, i64, i64, dp, i64, dp, i64, dp, i64, i32, i32, vp]
    lib.ozaki2_dgemm.argtypes = common
    lib.ozaki2_dgemm.restype = i32
    lib.ozaki2_dgemm_debug.argtypes = common + [vp] * 7
    lib.ozaki2_dgemm_debug.restype = i32
    lib.ozaki2_dgemm_stages.argtypes = common + [ctypes.POINTER(ctypes.c_float)]
    lib.ozaki2_dgemm_stages.restype = i32
    lib.ozaki2_dgemm_host.argtypes = common
    lib.ozaki2_dgemm_host.restype = i32
    lib.ozaki2_moduli.argtypes = [i32, ctypes.POINTER(ctypes.c_int32)]
    lib.ozaki2_moduli.restype = i32
    lib.ozaki2_last_error.argtypes = []
    lib.ozaki2_last_error.restype = i32
    lib.ozaki2_workspace_release.argtypes = []
    lib.ozaki2_workspace_release.restype = None
    lib.ozaki2_status_string.argtypes = [i32]
    lib.ozaki2_status_string.restype = ctypes.c_char_p
    lib.ozaki2_profile_begin.argtypes = [i32]
    lib.ozaki2_profile_begin.restype = i32
    lib.ozaki2_profile_end.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]
    lib.ozaki2_profile_end.restype = i32
    lib.ozaki2_launch_count.argtypes = []
    lib.ozaki2_launch_count.restype = ctypes.c_uint64
    lib.ozaki2_selftest_wait_timeout.argtypes = [i32]
    lib.ozaki2_selftest_wait_timeout.restype = i32
    _lib = lib
    return lib


def _check(code: int, what: str):
    if code != 0:
        raise Ozaki2Error(code, what)


def _mode(mode) -> int:
    if mode in ("fast", FAST):
        return FAST
    if mode in ("accu", ACCU):
        return ACCU
    raise ValueError(f"mode must be 'fast' or 'accu', got {mode!r}")


def moduli(s: int) -> list[int]:
    """The s moduli the library uses (host-side; needs no GPU)."""
    lib = load_library()
    buf = (ctypes.c_int32 * S_MAX)()
    n = lib.ozaki2_moduli(int(s), buf)
    if n < 0:
        raise ValueError(f"s must be in [{S_MIN}, {S_MAX}]")
    return list(buf[:n])


def _colmajor(T):
    """(ptr, ld) if T (2-D) is column-major with ld >= rows, else None.

    The stride of a dimension of size 1 is never used to address an element,
    so it is not checked: a 1 x q row with any row stride and a p x 1 column
    with any column stride are column-major."""
    p, q = T.shape
    s0, s1 = T.stride()
    if p > 1 and s0 != 1:
        return None
    if q <= 1:
        return T.data_ptr(), max(p, 1)
    if s1 < max(p, 1):
        return None
    return T.data_ptr(), s1


def _as_colmajor(T):
    """T itself if column-major, else a column-major copy."""
    import torch

    if _colmajor(T) is not None:
        return T
    C = torch.empty((T.shape[1], T.shape[0]), dtype=T.dtype, device=T.device).t()
    C.copy_(T)
    return C


def _stream_handle(stream):
    import torch

    st = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(st.cuda_stream)


def _prepare(A, B):
    import torch

    if A.dtype != torch.float64 or B.dtype != torch.float64:
        raise TypeError("A and B must be float64")
    if not (A.is_cuda and B.is_cuda) or A.device != B.device:
        raise ValueError("A and B must be CUDA tensors on the same device")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)}")
    A, B = _as_colmajor(A), _as_colmajor(B)
    return A, B, _colmajor(A), _colmajor(B)


def dgemm(A, B, s: int = 14, mode="fast", out=None, stream=None):
    """C = A @ B by Ozaki Scheme II (CUDA float64 tensors).  Asynchronous on `stream`."""
    import torch

    A, B, (pa, lda), (pb, ldb) = _prepare(A, B)
    p, q = A.shape
    r = B.shape[1]
    if out is None:
        out = torch.empty((r, p), dtype=torch.float64, device=A.device).t()
    c = _colmajor(out)
    if c is None or tuple(out.shape) != (p, r):
        raise ValueError("out must be a column-major (p, r) float64 tensor")
    lib = load_library()
    _check(lib.ozaki2_dgemm(p, q, r, pa, lda, pb, ldb, c[0], c[1], int(s), _mode(mode),
                            _stream_handle(stream)), "ozaki2_dgemm")
    return out


def dgemm_debug(A, B, s: int = 14, mode="fast", want_p: bool = True, stream=None) -> dict:
    """Run the pipeline and return every stage's output (for checking).

    alpha [p], beta [r] int32; Ares [s, p, q], Bres [s, r, q] int8; P [s, r, p]
    int32 (if want_p); R [s, r, p] uint8; X [r, p, 3] int64 (two's complement
    192-bit limbs, as unsigned bit patterns); C (p, r) column-major float64.
    """
    import torch

    A, B, (pa, lda), (pb, ldb) = _prepare(A, B)
    p, q = A.shape
    r = B.shape[1]
    dev = A.device
    o = {
        "C": torch.empty((r, p), dtype=torch.float64, device=dev).t(),
        "alpha": torch.empty(p, dtype=torch.int32, device=dev),
        "beta": torch.empty(r, dtype=torch.int32, device=dev),
        "Ares": torch.empty((s, p, q), dtype=torch.int8, device=dev),
        "Bres": torch.empty((s, r, q), dtype=torch.int8, device=dev),
        "P": torch.empty((s, r, p), dtype=torch.int32, device=dev) if want_p else None,
        "R": torch.empty((s, r, p), dtype=torch.uint8, device=dev),
        "X": torch.empty((r, p, 3), dtype=torch.int64, device=dev),
    }
    lib = load_library()
    ptr = lambda t: None if t is None else t.data_ptr()
    _check(lib.ozaki2_dgemm_debug(
        p, q, r, pa, lda, pb, ldb, o["C"].data_ptr(), p, int(s), _mode(mode), _stream_handle(stream),
        ptr(o["alpha"]), ptr(o["beta"]), ptr(o["Ares"]), ptr(o["Bres"]), ptr(o["P"]), ptr(o["R"]),
        ptr(o["X"])), "ozaki2_dgemm_debug")
    return o


def dgemm_stages(A, B, s: int = 14, mode="fast", out=None, stream=None):
    """(C, {stage: ms}) — one call with CUDA events between the stages."""
    import torch

    A, B, (pa, lda), (pb, ldb) = _prepare(A, B)
    p, q = A.shape
    r = B.shape[1]
    if out is None:
        out = torch.empty((r, p), dtype=torch.float64, device=A.device).t()
    c = _colmajor(out)
    ms = (ctypes.c_float * 6)()
    lib = load_library()
    _check(lib.ozaki2_dgemm_stages(p, q, r, pa, lda, pb, ldb, c[0], c[1], int(s), _mode(mode),
                                   _stream_handle(stream), ms), "ozaki2_dgemm_stages")
    return out, dict(zip(STAGE_NAMES, [float(x) for x in ms]))


def dgemm_host(A, B, s: int = 14, mode="fast", out=None, stream=None):
    """C = A @ B for HOST tensors (CPU float64; pinned memory copies fastest).

    The library copies A and B to the device, runs the pipeline and copies C
    back; the call returns when C is on the host.
    """
    import torch

    if A.is_cuda or B.is_cuda:
        raise ValueError("dgemm_host takes host (CPU) tensors")
    if A.dtype != torch.float64 or B.dtype != torch.float64:
        raise TypeError("A and B must be float64")
    A, B = _as_colmajor(A), _as_colmajor(B)
    a, b = _colmajor(A), _colmajor(B)
    p, q = A.shape
    r = B.shape[1]
    if out is None:
        out = torch.empty((r, p), dtype=torch.float64).t()
    c = _colmajor(out)
    lib = load_library()
    _check(lib.ozaki2_dgemm_host(p, q, r, a[0], a[1], b[0], b[1], c[0], c[1], int(s), _mode(mode),
                                 _stream_handle(stream)), "ozaki2_dgemm_host")
    return out


def profile_begin(max_calls: int) -> None:
    """Record stage events in the next max_calls dgemm calls (no synchronisation)."""
    _check(load_library().ozaki2_profile_begin(int(max_calls)), "ozaki2_profile_begin")


def profile_end():
    """(calls, {stage: summed ms}) of the calls recorded since profile_begin."""
    ms = (ctypes.c_float * 6)()
    n = ctypes.c_int(0)
    _check(load_library().ozaki2_profile_end(ms, ctypes.byref(n)), "ozaki2_profile_end")
    return n.value, dict(zip(STAGE_NAMES, [float(x) for x in ms]))


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load_library().ozaki2_launch_count())


def last_error() -> int:
    return load_library().ozaki2_last_error()


def workspace_release() -> None:
    load_library().ozaki2_workspace_release()


def selftest_wait_timeout(limit_us: int = 2000) -> int:
    return load_library().ozaki2_selftest_wait_timeout(int(limit_us))
