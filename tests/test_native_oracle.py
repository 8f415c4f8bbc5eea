"""Pins for the native CPU oracle (oracle/oz2_oracle.c), on the CPU.

The native oracle is tied to things other than itself: the Python oracle
(itself pinned in test_oracle_pins.py) bit for bit on every stage, X = A'B'
by big-integer brute force, and its exact dot products to Python Fractions.
Sources: "Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" §1-§2 and
"Ozaki II supplement: INT8 range conditions and paper performance results"
§1.1-§1.3.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import native
from oracle import ozaki2_oracle as oz
from tests._util import decode_x
from workloads import make_matrices


def _compare_with_python_oracle(A, B, s, mode):
    got = native.dgemm(A, B, s, mode, nthreads=4)
    ref = oz.oracle_dgemm(A, B, s, mode)
    np.testing.assert_array_equal(got["alpha"], ref["alpha"])
    np.testing.assert_array_equal(got["beta"], ref["beta"])
    np.testing.assert_array_equal(got["Ares"], ref["Ares"])
    np.testing.assert_array_equal(got["Bres"], np.transpose(ref["Bres"], (0, 2, 1)))
    np.testing.assert_array_equal(got["R"], np.transpose(ref["R"], (0, 2, 1)))
    p, r = ref["X"].shape
    X = got["X"]
    for i in range(p):
        for j in range(r):
            assert decode_x(X[j, i]) == ref["X"][i, j], (i, j)
    # one correct rounding on both sides: identical bits (+0 and -0 compare equal)
    np.testing.assert_array_equal(got["C"], ref["C"])
    return got, ref


def test_moduli_match():
    for s in range(1, 21):
        assert native.moduli(s) == oz.greedy_moduli(s)


@pytest.mark.parametrize("mode", ["fast", "accu"])
@pytest.mark.parametrize("p,q,r,s,phi", [
    (1, 1, 1, 2, 0.5), (7, 13, 5, 8, 1.0), (33, 70, 65, 14, 0.5), (64, 129, 30, 18, 2.0),
    (20, 300, 17, 20, 3.0), (50, 5000, 3, 11, 0.5), (3, 64, 70, 15, 1.0)])
def test_every_stage_matches_the_python_oracle(mode, p, q, r, s, phi):
    A, B = make_matrices(p, q, r, phi, 1000 * p + q + r + s)
    _compare_with_python_oracle(A, B, s, mode)


@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_special_values_match(mode):
    A, B = make_matrices(24, 40, 20, 2.0, 5)
    A[3, :] = 0.0
    B[:, 4] = 0.0
    A[5, :] *= 1e-310
    A[6, 7] = 1e300
    A[7, :] = -A[7, :] * 2.0**600
    B[11, :] = 5e-324
    B[:, 9] *= 2.0**-1000
    A[8, ::2] = -0.0
    _compare_with_python_oracle(A, B, 14, mode)


def test_wide_range_accu_general_residues():
    A = np.array([[1e300, 0.0, 0.0], [-2.0, 1e-300, 1e-310]], order="F")
    B = np.array([[0.0, 0.0], [1.0, -1e-5], [0.0, 7.0]], order="F")
    got, ref = _compare_with_python_oracle(A, B, 14, "accu")
    assert got["alpha"][0] == 0


def test_x_equals_aprime_bprime_brute_force():
    """[P] §1: X = A'B' exactly, with A' = trunc(2^alpha A) formed from Fractions."""
    for mode in ("fast", "accu"):
        A, B = make_matrices(6, 9, 5, 1.5, 77)
        got = native.dgemm(A, B, 14, mode, nthreads=2)
        for i in range(6):
            for j in range(5):
                x = sum(int(Fraction(float(A[i, l])) * Fraction(2) ** int(got["alpha"][i])) *
                        int(Fraction(float(B[l, j])) * Fraction(2) ** int(got["beta"][j])) for l in range(9))
                assert decode_x(got["X"][j, i]) == x


def test_bound_condition_refusals():
    with pytest.raises(ValueError):
        native.dgemm(np.ones((1, oz.ACCU_Q_LIMIT)), np.ones((oz.ACCU_Q_LIMIT, 1)), 8, "accu")


def _rn(f: Fraction) -> float:
    """One correct rounding of a rational (Python's int/int division rounds to
    nearest even), overflowing to +-inf."""
    if f == 0:
        return 0.0
    try:
        return f.numerator / f.denominator
    except OverflowError:
        return math.inf if f > 0 else -math.inf


def _exact(A, B, i, j):
    return sum(Fraction(float(A[i, l])) * Fraction(float(B[l, j])) for l in range(A.shape[1]))


def test_exact_dot_products_against_fractions():
    rng = np.random.default_rng(8)
    A, B = make_matrices(9, 40, 8, 6.0, 3)  # wide exponent range
    A[0, :] = [1e300, -1e300] * 20          # total cancellation
    B[:, 1] = 1.0
    A[1, :5] = 5e-324
    B[:5, 2] = 5e-324                        # products below the smallest subnormal
    A[2, :] = 2.0**1000
    B[:, 3] = 2.0**23                        # near the top of the range
    ii = np.repeat(np.arange(9), 8)
    jj = np.tile(np.arange(8), 9)
    Chat = rng.standard_normal(len(ii))
    exact, absprod, (err,) = native.exact_entries(A, B, ii, jj, [Chat])
    for k in range(len(ii)):
        i, j = int(ii[k]), int(jj[k])
        ex = _exact(A, B, i, j)
        ab = sum(abs(Fraction(float(A[i, l])) * Fraction(float(B[l, j]))) for l in range(40))
        assert exact[k] == _rn(ex), (i, j)
        assert absprod[k] == _rn(ab), (i, j)
        assert err[k] == _rn(Fraction(float(Chat[k])) - ex), (i, j)
    assert exact[0 * 8 + 1] == 0.0 and absprod[0 * 8 + 1] == _rn(Fraction(40) * Fraction(1e300))
    assert np.any(np.isinf(absprod))  # some |A||B| entries of row 0 pass the largest double


def test_exact_dot_rounding_ties_and_subnormal_results():
    # sum of two products exactly half an ulp apart from representable values
    A = np.array([[1.0, 2.0**-53], [2.0**-1074, 2.0**-1074], [1.0, 2.0**-53 + 2.0**-105]], order="F")
    B = np.array([[1.0], [1.0]], order="F")
    exact, absprod, _ = native.exact_entries(A, B, [0, 1, 2], [0, 0, 0])
    assert exact[0] == 1.0                      # 1 + 2^-53: tie, rounds to even
    assert exact[1] == 2.0**-1073
    assert exact[2] == 1.0 + 2.0**-52           # just above the tie
    A2 = np.array([[2.0**-600, 0.0], [2.0**-600, 2.0**-600], [2.0**-600, 2.0**-700]], order="F")
    B2 = np.array([[2.0**-475], [2.0**-475]], order="F")
    e2, _, _ = native.exact_entries(A2, B2, [0, 1, 2], [0, 0, 0])
    assert e2[0] == 0.0                         # 2^-1075: half the smallest subnormal, ties to 0
    assert e2[1] == 2.0**-1074                  # two halves
    assert e2[2] == 2.0**-1074                  # just above the half


def test_accuracy_report_on_exact_and_perturbed_products():
    rng = np.random.default_rng(2)
    A = np.asfortranarray(rng.integers(-8, 9, size=(12, 30)).astype(np.float64))
    B = np.asfortranarray(rng.integers(-8, 9, size=(30, 10)).astype(np.float64))
    C = A @ B  # small integers: exact
    bad = C.copy()
    bad[3, 4] += 1.0
    rep = native.accuracy(A, B, {"exact": C, "bad": bad})
    assert rep["entries"] == 120
    assert rep["exact"]["normwise"] == 0.0 and rep["exact"]["componentwise"] == 0.0
    absAB = np.abs(A) @ np.abs(B)
    assert rep["bad"]["componentwise"] == pytest.approx(1.0 / absAB[3, 4], rel=1e-15)
    assert rep["bad"]["normwise"] == pytest.approx(1.0 / np.linalg.norm(C), rel=1e-12)
    # sampled entries
    rep2 = native.accuracy_at(A, B, np.array([3, 0]), np.array([4, 0]), {"bad": bad[[3, 0], [4, 0]]})
    assert rep2["entries"] == 2 and rep2["bad"]["max_abs_err"] == 1.0


def test_oracle_error_within_the_truncation_bound():
    """The Ozaki-II result's error on a wide-range product stays within the
    a-posteriori truncation bound of [P] §1 (each truncation loses < 1 unit)."""
    A, B = make_matrices(16, 64, 12, 2.0, 19)
    got = native.dgemm(A, B, 14, "fast", nthreads=2)
    rep = native.accuracy(A, B, {"oz2": got["C"]})
    assert 0 < rep["oz2"]["normwise"] < 1e-12
    assert math.isfinite(rep["oz2"]["componentwise"])


@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_product_paths_and_entry_points_agree(mode):
    """The C oracle's integer products and the exact float64 BLAS product of the
    same residue planes give the same R, X and C; so does the single C entry point."""
    A, B = make_matrices(150, 700, 90, 1.0, 61)
    a = native.dgemm(A, B, 18, mode, products="c")
    b = native.dgemm(A, B, 18, mode, products="blas")
    c = native.dgemm_all_in_c(A, B, 18, mode)
    for k in native.OUTPUTS:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
        np.testing.assert_array_equal(a[k], c[k], err_msg=k)


@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_sampled_entries_and_exponents_match_the_full_path(mode):
    A, B = make_matrices(70, 300, 50, 2.0, 71)
    A[5, :] *= 1e-310
    A[6, 3] = 1e300
    B[:, 7] = 0.0
    full = native.dgemm(A, B, 18, mode)
    al, be = native.exponents(A, B, 18, mode)
    np.testing.assert_array_equal(al, full["alpha"])
    np.testing.assert_array_equal(be, full["beta"])
    rng = np.random.default_rng(1)
    ii = np.concatenate([rng.integers(0, 70, 200), [0, 69, 5, 6]])
    jj = np.concatenate([rng.integers(0, 50, 200), [49, 0, 7, 7]])
    e = native.entries(A, B, 18, al, be, ii, jj)
    np.testing.assert_array_equal(e["R"], full["R"][:, jj, ii].T)
    np.testing.assert_array_equal(e["X"], full["X"][jj, ii])
    np.testing.assert_array_equal(e["C"], full["C"][ii, jj])
