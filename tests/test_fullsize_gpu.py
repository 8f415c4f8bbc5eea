"""Full-size parity and the accuracy report, through the C ABI on the GPU.

* Every stage at the full n = 8192, s = 14 fast workload and the full
  16384 x 8192 x 16384, s = 18 accu workload (phi = 2) against the native
  CPU oracle, element by element: exponents, residue planes, output residues
  and the CRT integer bit for bit, C within 2 ulp, in the launch
  configuration the benchmark times (the production entry point's C must
  equal the checking entry point's).
* The accuracy report ("Ozaki II supplement: INT8 range conditions and paper
  performance results" §1.1; "Profiling Ozaki II: The Cost Behind Fast INT8
  GEMMs" §1: X = A'B' exactly, so the only error is the truncation of DA and
  BE plus the final rounding): the normwise error ||C_hat - C||_F / ||C||_F and
  the componentwise error max |C_hat - C| / (|A||B|) against the exact
  product, over every entry up to n = 1024 and 4096 sampled entries above,
  for every workload; the GPU's errors must not exceed the oracle's.
* Host-side fault injection: a failed workspace allocation is reported and
  the next call recovers.
"""
import os

import numpy as np
import pytest

from oracle import native
from tests._util import ulp_distance
from workloads import WORKLOADS, make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ULP_TOL = 2
# the oracle's exact integer products: the C loops or an exact float64 BLAS product
ORACLE_PRODUCTS = "blas"


@pytest.fixture(scope="module")
def oz2():
    import __graft_entry__ as g

    g.build()
    import emulated_fp64_gemm_gb300 as m

    assert torch.cuda.is_available()
    return m


def _dev(x):
    return torch.from_numpy(np.asfortranarray(x)).cuda()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["n8192_s14_fast", "p16384_q8192_r16384_s18_accu"])
def test_full_size_every_stage_elementwise(oz2, name):
    w = WORKLOADS[name]
    A, B = make_workload(w)
    dA, dB = _dev(A), _dev(B)
    C = oz2.dgemm(dA, dB, w.s, w.mode).cpu().numpy()  # the benchmark's launch configuration
    got = oz2.dgemm_debug(dA, dB, w.s, w.mode, want_p=False)
    torch.cuda.synchronize()
    del dA, dB
    g = {k: v.cpu().numpy() for k, v in got.items() if v is not None}
    del got
    torch.cuda.empty_cache()
    ref = native.dgemm(A, B, w.s, w.mode, products=ORACLE_PRODUCTS)
    np.testing.assert_array_equal(g["alpha"], ref["alpha"], err_msg="alpha")
    np.testing.assert_array_equal(g["beta"], ref["beta"], err_msg="beta")
    np.testing.assert_array_equal(g["Ares"], ref["Ares"], err_msg="A residue planes")
    np.testing.assert_array_equal(g["Bres"], ref["Bres"], err_msg="B residue planes")
    np.testing.assert_array_equal(g["R"], ref["R"], err_msg="output residues")
    np.testing.assert_array_equal(g["X"].view(np.uint64), ref["X"], err_msg="CRT integer X")
    assert ulp_distance(g["C"], ref["C"]) <= ULP_TOL
    np.testing.assert_array_equal(C, g["C"])
    assert oz2.last_error() == 0


ACCURACY_WORKLOADS = ["n128_s8_fast", "n1024_s14_fast", "n4096_s14_accu", "n8192_s14_fast", "n8192_s14_accu",
                      "n8192_s18_fast", "n8192_s18_accu", "p16384_q8192_r16384_s18_accu"]


def accuracy_of(oz2, name, nsamp=4096):
    """The accuracy report of one workload: the GPU's and the oracle's errors."""
    w = WORKLOADS[name]
    A, B = make_workload(w)
    C = oz2.dgemm(_dev(A), _dev(B), w.s, w.mode).cpu().numpy()
    if w.p * w.r <= 1024 * 1024:
        Co = native.dgemm(A, B, w.s, w.mode, want=("C",), products=ORACLE_PRODUCTS)["C"]
        return native.accuracy(A, B, {"gpu": C, "oracle": Co})
    rng = np.random.default_rng(2024)
    ii = rng.integers(0, w.p, nsamp)
    jj = rng.integers(0, w.r, nsamp)
    al, be = native.exponents(A, B, w.s, w.mode)
    Co = native.entries(A, B, w.s, al, be, ii, jj)["C"]
    return native.accuracy_at(A, B, ii, jj, {"gpu": C[ii, jj], "oracle": Co})


@pytest.mark.slow
@pytest.mark.parametrize("name", ACCURACY_WORKLOADS)
def test_accuracy_not_worse_than_the_oracle(oz2, name):
    rep = accuracy_of(oz2, name)
    print(f"\naccuracy {name}: {rep}")
    g, o = rep["gpu"], rep["oracle"]
    assert g["normwise"] <= o["normwise"]
    assert g["componentwise"] <= o["componentwise"]
    # with 14 or more moduli (110+ range bits, "Ozaki II supplement" §1.4) every
    # scaled operand keeps more than 53 bits, so the result is at FP64 level;
    # 8 moduli (63.6 bits) leave about 31 bits per operand
    if WORKLOADS[name].s >= 14:
        assert g["normwise"] < 1e-13
    else:
        assert g["normwise"] < 1e-7


def test_failed_workspace_allocation_reports_and_recovers(oz2, monkeypatch):
    """Host-side fault injection: OZ2_FAIL_ALLOC makes the first workspace
    allocation of a fresh stream fail (OZ2_ERR_NO_MEMORY, status 3, before any
    launch); once it is unset, the same call on the same stream succeeds."""
    from workloads import make_matrices
    from oracle import ozaki2_oracle as oracle

    A, B = make_matrices(300, 200, 100, 0.5, 12)
    dA, dB = _dev(A), _dev(B)
    st = torch.cuda.Stream()  # a stream the library has no workspace for yet
    monkeypatch.setenv("OZ2_FAIL_ALLOC", "1")
    with pytest.raises(oz2.Ozaki2Error) as ex:
        oz2.dgemm(dA, dB, 14, "fast", stream=st)
    assert ex.value.code == 3
    monkeypatch.delenv("OZ2_FAIL_ALLOC")
    C = oz2.dgemm(dA, dB, 14, "fast", stream=st)
    st.synchronize()
    ref = oracle.oracle_dgemm(A, B, 14, "fast")
    assert ulp_distance(C.cpu().numpy(), ref["C"]) <= ULP_TOL
    assert oz2.last_error() == 0
    assert os.environ.get("OZ2_FAIL_ALLOC") is None
