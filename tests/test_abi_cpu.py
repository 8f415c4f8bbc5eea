"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every declared entry point; host logic (moduli, argument checks)
behaves as documented; without a GPU the product path fails loudly."""
import ctypes

import pytest

import emulated_fp64_gemm_gb300 as oz2
from emulated_fp64_gemm_gb300 import _build
from oracle import ozaki2_oracle as oracle
from tests._util import header_functions


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return oz2.load_library()


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_moduli_match_oracle(lib):
    for s in range(oz2.S_MIN, oz2.S_MAX + 1):
        assert oz2.moduli(s) == oracle.greedy_moduli(s)
    with pytest.raises(ValueError):
        oz2.moduli(1)
    with pytest.raises(ValueError):
        oz2.moduli(21)


def test_status_strings(lib):
    # every code of oz2_status (include/ozaki2.h) has its own text, and the binding names it
    texts = [lib.ozaki2_status_string(code) for code in range(8)]
    assert all(texts) and len(set(texts)) == 8
    assert lib.ozaki2_status_string(8) == b"unknown status"
    assert sorted(oz2.STATUS) == list(range(8))
    import re
    header = open(oz2.library_path().replace("emulated_fp64_gemm_gb300/libozaki2.so", "include/ozaki2.h")).read()
    enum = dict((int(v), k) for k, v in re.findall(r"\b(OZ2_(?:OK|ERR_\w+))\s*=\s*(\d+)", header))
    assert enum == oz2.STATUS


def _call(lib, p=4, q=4, r=4, A=1, lda=4, B=1, ldb=4, C=1, ldc=4, s=8, mode=0):
    vp = ctypes.c_void_p
    return lib.ozaki2_dgemm(p, q, r, vp(A), lda, vp(B), ldb, vp(C), ldc, s, mode, vp(0))


def test_argument_errors_are_returned_before_any_device_work(lib):
    assert _call(lib, p=0) == 1
    assert _call(lib, q=-1) == 1
    assert _call(lib, r=0) == 1
    assert _call(lib, lda=3) == 1
    assert _call(lib, ldb=3) == 1
    assert _call(lib, ldc=3) == 1
    assert _call(lib, A=0) == 1
    assert _call(lib, B=0) == 1
    assert _call(lib, C=0) == 1
    assert _call(lib, s=1) == 1
    assert _call(lib, s=21) == 1
    assert _call(lib, mode=2) == 1
    # inner-dimension limits per mode: the K-blocked modular GEMMs lift the
    # single-accumulation INT32 condition q < 2^17; what remains is the 64-bit
    # fast statistic (q < 2^24) and the INT32 accu bound product (q 127^2 < 2^31)
    assert _call(lib, q=1 << 24, ldb=1 << 24, mode=0) == 2
    assert _call(lib, q=(1 << 24) - 1, ldb=1 << 24, mode=0) != 2
    assert _call(lib, q=131072, ldb=131072, mode=0) != 2
    assert _call(lib, q=133145, ldb=133145, mode=1) == 2
    assert _call(lib, q=133144, ldb=133144, mode=1) != 2
    assert oz2.Q_LIMIT_ACCU == oracle.ACCU_Q_LIMIT and oz2.Q_LIMIT_FAST == oracle.FAST_Q_LIMIT
    assert (oz2.Q_LIMIT_ACCU - 1) * 127**2 < 2**31 <= oz2.Q_LIMIT_ACCU * 127**2


def test_no_gpu_means_a_loud_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call(lib) == 4  # OZ2_ERR_CUDA: there is no CPU fallback


def test_column_major_views_pass_through_and_others_are_copied():
    """The binding hands the library (pointer, leading dimension) of a
    column-major view as it is and copies anything else into one."""
    torch = pytest.importorskip("torch")
    base = torch.arange(60, dtype=torch.float64).reshape(6, 10)  # row-major
    cases = [
        base.t(),                       # 10 x 6 column-major, ld 10
        base.t()[2:7, 1:4],             # a block of it, ld 10
        base[2:3, :],                   # 1 x 10 row, row stride 10
        base.t()[:, 4:5],               # 10 x 1 column, column stride 10
        torch.ones(1, 7, dtype=torch.float64).as_strided((1, 7), (7, 1)),
        torch.ones(7, 1, dtype=torch.float64).as_strided((7, 1), (1, 1)),
        torch.ones(1, 1, dtype=torch.float64),
    ]
    for T in cases:
        ptr, ld = oz2._colmajor(T)
        assert ptr == T.data_ptr() and ld >= T.shape[0]
        assert oz2._as_colmajor(T) is T
        # every element sits at ptr + 8 (i + j ld)
        flat = T.untyped_storage()
        for i in range(T.shape[0]):
            for j in range(T.shape[1]):
                off = (ptr - T.untyped_storage().data_ptr()) // 8 + i + j * ld
                assert torch.tensor([], dtype=torch.float64).set_(flat)[off] == T[i, j]
    for T in [base, base[:, 1:3], base[:, 4:5], torch.ones(3, 4, dtype=torch.float64).expand(3, 4)[:, :],
              torch.ones(1, 4, dtype=torch.float64).expand(3, 4)]:
        assert oz2._colmajor(T) is None
        C = oz2._as_colmajor(T)
        assert oz2._colmajor(C) is not None and torch.equal(C, T)
