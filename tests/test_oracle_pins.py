"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources: "Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" (cited [P]) and
"Ozaki II supplement: INT8 range conditions and paper performance results"
(cited [S]).  The checks are brute force on tiny inputs, closed forms the pages
print, textbook special cases and exact rational arithmetic; none of them
re-types the oracle's own formulas.
"""
import json
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest

from oracle import ozaki2_oracle as oz
from workloads import make_matrices

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))


# --------------------------------------------------------------------------- moduli
def test_moduli_pairwise_coprime_and_greedy():
    for s in range(1, 21):
        ms = oz.greedy_moduli(s)
        assert len(ms) == s and all(2 <= m <= 256 for m in ms)
        for a in range(s):
            for b in range(a + 1, s):
                assert math.gcd(ms[a], ms[b]) == 1
        # greedy from the top: every skipped integer shares a factor with a larger kept one
        for k in range(ms[-1] + 1, 257):
            if k not in ms:
                assert any(math.gcd(k, m) > 1 for m in ms if m > k)


def test_range_bits_about_125_for_16_moduli():
    g = GOLDEN["range_bits_s16"]
    bits = sum(math.log2(m) for m in oz.greedy_moduli(g["s"]))
    assert abs(bits - g["about"]) < 0.5


def test_constants_against_definition():
    for s in (2, 8, 14, 18, 20):
        c = oz.modulus_constants(oz.greedy_moduli(s))
        assert c["M"] == math.prod(c["moduli"])
        for t, m in enumerate(c["moduli"]):
            # the CRT basis element e_t = inv_t * M/m_t is 1 mod m_t and 0 mod the others
            e = c["inv"][t] * c["Mt"][t]
            for u, mu in enumerate(c["moduli"]):
                assert e % mu == (1 if u == t else 0)


# --------------------------------------------------------------------------- residues
def test_centered_residue_brute_force():
    for m in range(2, 257):
        lo, hi = -(m // 2), (m + 1) // 2 - 1
        seen = set()
        for x in range(-3 * m, 3 * m + 1):
            r = oz.centered_residue(x, m)
            assert lo <= r <= hi and (x - r) % m == 0
            seen.add(r)
        assert seen == set(range(lo, hi + 1))  # a complete residue system


def test_centered_residue_page_values():
    g = GOLDEN["centered_residue_256"]
    vals = [oz.centered_residue(x, 256) for x in range(-1000, 1000)]
    assert [min(vals), max(vals)] == g["range"]
    for x, want in g["maps"]:
        assert oz.centered_residue(x, 256) == want
    # numpy arrays follow the same rule as Python ints
    xs = np.arange(-70000, 70000, 37, dtype=np.int64)
    for m in (173, 255, 256):
        np.testing.assert_array_equal(oz.centered_residue(xs, m),
                                      [oz.centered_residue(int(x), m) for x in xs])


def test_residue_planes_match_bigint_definition():
    """rho_m(trunc(2**k x)) formed with exact Python integers, including huge shifts."""
    rng = np.random.default_rng(5)
    xs = np.concatenate([(rng.random(40) - 0.5) * np.exp(3 * rng.standard_normal(40)),
                         [0.0, -0.0, 5e-324, -2.5e-310, 1e300, -1.7e308, 1.0, -1.0, 0.75]])
    X = xs.reshape(7, 7)
    moduli = oz.greedy_moduli(20)
    for exps in (np.arange(7) * 3 - 10, np.array([0, 60, 200, 1100, -1074, 2000, 5])):
        planes = oz.residue_planes(X, exps, axis=1, moduli=moduli)
        for i in range(7):
            for l in range(7):
                fx = Fraction(float(X[i, l])) * Fraction(2) ** int(exps[i])
                a = int(fx)  # int(Fraction) truncates toward zero
                for t, m in enumerate(moduli):
                    r = int(planes[t, i, l])
                    assert -(m // 2) <= r <= (m + 1) // 2 - 1
                    assert (a - r) % m == 0


# --------------------------------------------------------------------------- CRT
@pytest.mark.parametrize("s", [2, 8, 14, 18, 20])
def test_crt_round_trip(s):
    c = oz.modulus_constants(oz.greedy_moduli(s))
    M = c["M"]
    rnd = random.Random(s)
    xs = [-M // 2, M // 2 - 1, 0, 1, -1, M // 4, -(M // 4) - 1]
    xs += [rnd.randrange(-M // 2, M // 2) for _ in range(300)]
    for x in xs:
        res = [x % m for m in c["moduli"]]
        assert oz.crt(res, c) == x
    R = np.array([[x % m for x in xs] for m in c["moduli"]], dtype=np.int64)[:, None, :]
    assert list(oz.crt_matrix(R, c)[0]) == xs


# --------------------------------------------------------------------------- final rounding
def test_round_scaled_closed_forms():
    rs = oz.round_scaled
    assert rs(2**53 + 1, 0) == 2.0**53  # tie -> even
    assert rs(2**53 + 3, 0) == 2.0**53 + 4  # tie -> even (upwards)
    assert rs(-(2**53 + 1), 0) == -(2.0**53)
    assert rs(3, 1075) == 2.0**-1073  # 1.5 * 2**-1074 -> 2 * 2**-1074
    assert rs(1, 1075) == 0.0  # 0.5 * 2**-1074 -> 0 (even)
    assert rs(3, 1076) == 2.0**-1074  # 0.75 ulp -> 1 ulp
    assert rs(1, 1074) == 5e-324
    assert rs(2**1024, 0) == math.inf and rs(-(2**1024), 0) == -math.inf
    top = (2**53 - 1) * 2**971
    assert rs(top, 0) == 1.7976931348623157e308
    assert rs(top + 2**970, 0) == math.inf  # halfway to 2**1024 (ulp 2**971) rounds to even -> overflow
    assert rs(top + 2**970 - 1, 0) == 1.7976931348623157e308
    assert rs(5, -3) == 40.0 and rs(0, 7) == 0.0


# --------------------------------------------------------------------------- whole pipeline
def _bigint_scaled(X, exps, axis):
    """trunc(2**exp * x) with Fractions, independent of the oracle's residue path."""
    out = [[0] * X.shape[1] for _ in range(X.shape[0])]
    for i in range(X.shape[0]):
        for j in range(X.shape[1]):
            k = int(exps[i] if axis == 1 else exps[j])
            out[i][j] = int(Fraction(float(X[i, j])) * Fraction(2) ** k)
    return out


def _check_x_equals_aprime_bprime(A, B, s, mode):
    o = oz.oracle_dgemm(A, B, s, mode)
    Ap = _bigint_scaled(A, o["alpha"], axis=1)
    Bp = _bigint_scaled(B, o["beta"], axis=0)
    p, q = A.shape
    r = B.shape[1]
    L = o["consts"]["L"]
    for i in range(p):
        for j in range(r):
            x = sum(Ap[i][l] * Bp[l][j] for l in range(q))
            assert o["X"][i, j] == x, (i, j)
            # [P] §1: scaling keeps every |(A'B')_ij| < M/2; here within L = M/2 - 1
            assert sum(abs(Ap[i][l] * Bp[l][j]) for l in range(q)) <= L
    return o


@pytest.mark.parametrize("mode", ["fast", "accu"])
@pytest.mark.parametrize("s,phi,seed", [(2, 0.5, 1), (8, 0.5, 2), (14, 1.0, 3), (18, 2.0, 4), (20, 3.0, 5)])
def test_x_equals_aprime_bprime(mode, s, phi, seed):
    """[P] §1 / [S] §1.1: exact reconstruction gives X = A'B'."""
    A, B = make_matrices(5, 7, 4, phi, seed)
    _check_x_equals_aprime_bprime(A, B, s, mode)


def test_x_equals_aprime_bprime_wide_range_accu():
    """A huge entry that meets only a zero of B: trunc(2**alpha a) is thousands of bits."""
    A = np.array([[1e300, 0.0, 0.0], [-2.0, 1e-300, 1e-310]], order="F")
    B = np.array([[0.0, 0.0], [1.0, -1e-5], [0.0, 7.0]], order="F")
    o = _check_x_equals_aprime_bprime(A, B, 14, "accu")
    # row 0 of the bound product is zero, so alpha_0 = 0 and a'_00 = 1e300 exactly
    assert o["alpha"][0] == 0 and abs(_bigint_scaled(A, o["alpha"], 1)[0][0]) > 2**900
    _check_x_equals_aprime_bprime(A, B, 14, "fast")


def test_zero_rows_and_columns():
    A, B = make_matrices(4, 6, 3, 0.5, 9)
    A[1, :] = 0.0
    B[:, 2] = 0.0
    for mode in ("fast", "accu"):
        o = _check_x_equals_aprime_bprime(A, B, 8, mode)
        assert o["alpha"][1] == 0 and o["beta"][2] == 0
        assert np.all(o["C"][1, :] == 0) and np.all(o["C"][:, 2] == 0)


def test_worst_case_products_reach_the_int32_bound():
    """[P] §1 / [S] §1.3: |P_t| <= q 2**14; all -128 residues reach it."""
    g = GOLDEN["int32_inner_dim_limit"]
    assert g["value"] == oz.Q_LIMIT
    assert GOLDEN["max_product_magnitude"]["value"] == 128 * 128
    assert (g["value"] - 1) * 2**14 < 2**31 <= g["value"] * 2**14
    q = 4096
    Ares = np.full((1, 3, q), -128, dtype=np.int64)
    Bres = np.full((1, q, 2), -128, dtype=np.int64)
    P = oz.products(Ares, Bres)
    assert np.all(P == q * 2**14)


def test_inner_dimension_beyond_the_int32_condition():
    """[S] §1.3, last paragraph: past q = 2**17 the inner dimension is blocked
    and each block reduced modulo m_t; the residues combine to P_t mod m_t of
    the exact product.  Pins: worst-case residues at q = 2**17 + 64 (|P_t| >
    2**31) give R_t = (q 2**14) mod m_t; all-ones operands give C = q exactly;
    the remaining limits are the 64-bit fast statistic and the INT32 accu bound."""
    q = oz.Q_LIMIT + 64
    moduli = oz.greedy_moduli(8)
    Ares = np.full((8, 1, q), -128, dtype=np.int64)
    Bres = np.full((8, q, 1), -128, dtype=np.int64)
    R = oz.output_residues(oz.products(Ares, Bres), moduli)
    assert [int(R[t, 0, 0]) for t in range(8)] == [(q * 2**14) % m for m in moduli]
    o = oz.oracle_dgemm(np.ones((2, q)), np.ones((q, 3)), 8, "fast")
    assert np.all(o["C"] == float(q))
    assert (oz.FAST_Q_LIMIT - 1) * 2**(2 * oz.F_FAST) < 2**64
    assert (oz.ACCU_Q_LIMIT - 1) * oz.BOUND_QMAX**2 < 2**31 <= oz.ACCU_Q_LIMIT * oz.BOUND_QMAX**2
    with pytest.raises(ValueError):
        oz.oracle_dgemm(np.ones((1, oz.ACCU_Q_LIMIT)), np.ones((oz.ACCU_Q_LIMIT, 1)), 8, "accu")


def test_residue_count_closed_form():
    g = GOLDEN["residue_count_n8192_s14"]
    n, s = g["n"], g["s"]
    assert s * (n * n + n * n) == g["value"]
    assert GOLDEN["gemm_to_residue_work_ratio"]["value"] == (s * n**3) // g["value"]


# --------------------------------------------------------------------------- exponents
def _eq18_k(s, q):
    """Eq. (18) of [S] §2 in the expanded log form, evaluated in floating point."""
    ms = oz.greedy_moduli(s)
    M = math.prod(ms)
    return math.floor(0.5 * (sum(math.log2(m) for m in ms) - math.log2(q) - 1 + math.log2(1 - 2 / M)))


@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_eq18_on_unit_matrices(mode):
    """For +-1 inputs every bound is exact (U = q), so each exponent is Eq. (18)'s k."""
    rng = np.random.default_rng(0)
    for s in (2, 5, 8, 11, 14, 16, 18, 20):
        for q in (1, 3, 7, 128, 1000, 8192):
            A = np.asfortranarray(np.where(rng.random((2, q)) < 0.5, -1.0, 1.0))
            B = np.asfortranarray(np.where(rng.random((q, 3)) < 0.5, -1.0, 1.0))
            al, be, _ = oz.exponents(A, B, s, mode)
            k = _eq18_k(s, q)
            ms = oz.greedy_moduli(s)
            exact = Fraction(math.prod(ms) // 2 - 1, q)
            if abs(math.log2(exact) / 2 - round(math.log2(exact) / 2)) < 1e-9:
                continue  # float floor ambiguous at an exact power of 4
            assert set(al.tolist()) == {k} and set(be.tolist()) == {k}, (s, q)


def test_exponents_scale_equivariant():
    """Both modes: scaling row i of A by 2**c lowers alpha_i by c and scaling
    column j of B by 2**c lowers beta_j by c, leaving every other exponent
    alone (accu: u_i shifts by c while Abar and Wbar stay the same, so each
    row and column keeps its own scale)."""
    A, B = make_matrices(6, 9, 5, 1.0, 11)
    al, be, _ = oz.exponents(A, B, 14, "fast")
    A2 = A.copy()
    A2[2, :] *= 2.0**7
    A2[4, :] *= 2.0**-33
    B2 = B.copy()
    B2[:, 1] *= 2.0**12
    al2, be2, _ = oz.exponents(A2, B2, 14, "fast")
    want_a = al.copy()
    want_a[2] -= 7
    want_a[4] += 33
    want_b = be.copy()
    want_b[1] -= 12
    np.testing.assert_array_equal(al2, want_a)
    np.testing.assert_array_equal(be2, want_b)
    al, be, _ = oz.exponents(A, B, 14, "accu")
    al2, be2, _ = oz.exponents(A2, B2, 14, "accu")
    want_a = al.copy()
    want_a[2] -= 7
    want_a[4] += 33
    want_b = be.copy()
    want_b[1] -= 12
    np.testing.assert_array_equal(al2, want_a)
    np.testing.assert_array_equal(be2, want_b)


def test_fast_statistic_sandwich_and_near_maximality():
    """||x||^2 <= U <= (||x|| + sqrt(q) 2**(e-F))^2 and the exponent is the largest safe one."""
    A, B = make_matrices(5, 33, 4, 2.0, 21)
    c = oz.modulus_constants(oz.greedy_moduli(14))
    L = c["L"]
    al = oz.fast_exponents(A, axis=1, L=L)
    for i in range(5):
        row = [Fraction(float(v)) for v in A[i]]
        n2 = sum(v * v for v in row)
        e = math.frexp(max(abs(float(v)) for v in A[i]))[1]
        slack = Fraction(2) ** (e - oz.F_FAST)
        hi = sum((abs(v) + slack) ** 2 for v in row)
        a = int(al[i])
        assert Fraction(4) ** a * n2 <= L  # sound
        assert Fraction(4) ** (a + 1) * hi > L  # no larger exponent is provably safe


def _max_pow4_brute(U: Fraction, L: int) -> int:
    """max { a : 4**a U <= L } by stepping from a = 0 (U > 0), independent of the oracle."""
    a = 0
    if Fraction(4) ** a * U <= L:
        while Fraction(4) ** (a + 1) * U <= L:
            a += 1
    else:
        while Fraction(4) ** a * U > L:
            a -= 1
    return a


@pytest.mark.parametrize("q", [1 << 23, (1 << 23) + 1])
def test_fast_statistic_past_two_to_the_63(q):
    """[P] §5.1 (sum of squares rounded up) at the top of its range.

    Every entry is 1 - 2**-53, the largest double below 1: e = 0 and every
    rounded-up term is ceil((1 - 2**-53) 2**20) = 2**20, so S = q 2**40 >= 2**63
    (a signed 64-bit sum wraps here) and U = S 4**-20 = q exactly."""
    x = 1.0 - 2.0**-53
    row = np.full((1, q), x)
    for s in (8, 14, 20):
        L = oz.modulus_constants(oz.greedy_moduli(s))["L"]
        got = int(oz.fast_exponents(row, axis=1, L=L)[0])
        assert got == _max_pow4_brute(Fraction(q), L)
        # sound against the exact squared norm, and the next exponent is not
        n2 = q * Fraction(x) ** 2
        assert Fraction(4) ** got * n2 <= L < Fraction(4) ** (got + 1) * Fraction(q)
    col = np.full((q, 1), x)
    L = oz.modulus_constants(oz.greedy_moduli(14))["L"]
    assert int(oz.fast_exponents(col, axis=0, L=L)[0]) == _max_pow4_brute(Fraction(q), L)


def test_accu_exponents_subnormal_row_and_huge_column():
    """accu mode with a row of |a| ~ 1e-310 (u_i ~ 1030) and a column of B near
    1e300 (v_j ~ -990): alpha_i = u_i + max {a : 4**a R_i <= L} with R_i the
    brute-force row maximum of Wbar, beta_j likewise, and the scaled bound
    2**(alpha_i + beta_j) (|A||B|)_ij <= L on exact values."""
    A, B = make_matrices(5, 12, 4, 1.0, 44)
    A[1, :] *= 1e-310
    B[:, 2] *= 1e300
    L = oz.modulus_constants(oz.greedy_moduli(14))["L"]
    al, be, Abar, Bbar, u, v, W = oz.accu_exponents(A, B, L)
    assert u[1] > 1000 and v[2] < -900
    for i in range(5):
        Ri = max(int(W[i, j]) for j in range(4))
        assert int(al[i]) == (int(u[i]) + _max_pow4_brute(Fraction(Ri), L) if Ri else 0)
    for j in range(4):
        Kj = max(int(W[i, j]) for i in range(5))
        assert int(be[j]) == (int(v[j]) + _max_pow4_brute(Fraction(Kj), L) if Kj else 0)
    for i in range(5):
        for j in range(4):
            exact = sum(abs(Fraction(float(A[i, l])) * Fraction(float(B[l, j]))) for l in range(12))
            assert Fraction(2) ** (int(al[i]) + int(be[j])) * exact <= L


def test_accu_rows_and_columns_keep_their_own_scale():
    """Rows of A at 2**+-1000 and columns of B at 2**30 .. 2**-100: no row's or
    column's exponent is set by another's magnitude, so every output keeps
    its significant bits.  The oracle's C at every entry against the exact
    product (Fractions): relative error below 2**-40, exact zeros where the
    product is zero, and +-inf exactly where the product passes the double
    range."""
    A, B = make_matrices(8, 24, 7, 0.5, 12)
    A[0, :] *= 2.0**1000
    A[1, :] *= -(2.0**1000)
    A[2, :] *= 2.0**-1000
    B[:, 0] *= 2.0**30
    B[:, 1] *= 2.0**-70
    B[:, 2] *= 2.0**-100
    C = oz.oracle_dgemm(A, B, 14, "accu")["C"]
    big = Fraction(2) ** 1024
    for i in range(8):
        for j in range(7):
            ex = sum(Fraction(float(A[i, l])) * Fraction(float(B[l, j])) for l in range(24))
            if abs(ex) >= big:
                assert np.isinf(C[i, j]) and (C[i, j] > 0) == (ex > 0)
            elif ex == 0:
                assert C[i, j] == 0
            elif abs(ex) >= Fraction(2) ** -1022:  # normal results: relative error
                assert abs(Fraction(float(C[i, j])) - ex) <= abs(ex) * Fraction(2) ** -40, (i, j)
            else:  # subnormal range: within a few units of 2**-1074
                assert abs(Fraction(float(C[i, j])) - ex) <= Fraction(2) ** -1070, (i, j)


def test_accu_bound_dominates_abs_product():
    A, B = make_matrices(4, 10, 5, 2.0, 31)
    c = oz.modulus_constants(oz.greedy_moduli(14))
    al, be, Abar, Bbar, u, v, W = oz.accu_exponents(A, B, c["L"])
    assert Abar.max() <= 127 and Bbar.max() <= 127 and Abar.min() >= 0
    for i in range(4):
        assert math.ceil(Fraction(float(np.abs(A[i]).max())) * Fraction(2) ** int(u[i])) <= 127
        assert math.ceil(Fraction(float(np.abs(A[i]).max())) * Fraction(2) ** int(u[i] + 1)) > 127
        for j in range(5):
            exact = sum(abs(Fraction(float(A[i, l])) * Fraction(float(B[l, j]))) for l in range(10))
            w = Fraction(int(W[i, j])) * Fraction(2) ** (-int(u[i]) - int(v[j]))
            assert exact <= w
            assert Fraction(2) ** (int(al[i]) + int(be[j])) * w <= c["L"]


# --------------------------------------------------------------------------- textbook special cases
@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_small_integer_inputs_reproduce_integer_product(mode):
    rng = np.random.default_rng(3)
    A = np.asfortranarray(rng.integers(-8, 9, size=(12, 64)).astype(np.float64))
    B = np.asfortranarray(rng.integers(-8, 9, size=(64, 10)).astype(np.float64))
    o = oz.oracle_dgemm(A, B, 8, mode)
    want = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64)
    np.testing.assert_array_equal(o["C"], want)


def test_dyadic_inputs_reproduce_exact_product():
    rng = np.random.default_rng(4)
    A = np.asfortranarray(rng.integers(-2**10, 2**10, size=(9, 16)) * 2.0**-12)
    B = np.asfortranarray(rng.integers(-2**10, 2**10, size=(16, 7)) * 2.0**5)
    for mode in ("fast", "accu"):
        o = oz.oracle_dgemm(A, B, 14, mode)
        want = [[float(sum(Fraction(float(A[i, l])) * Fraction(float(B[l, j])) for l in range(16)))
                 for j in range(7)] for i in range(9)]
        np.testing.assert_array_equal(o["C"], np.array(want))


def test_identity_right_factor_returns_truncated_left():
    A, _ = make_matrices(6, 6, 6, 1.0, 8)
    B = np.asfortranarray(np.eye(6))
    o = oz.oracle_dgemm(A, B, 14, "fast")
    for i in range(6):
        for j in range(6):
            # C_ij = trunc(2**alpha_i a_ij) * 2**beta_j / 2**(alpha_i + beta_j): error < 2**-alpha_i
            assert abs(Fraction(float(o["C"][i, j])) - Fraction(float(A[i, j]))) < Fraction(2) ** -int(o["alpha"][i])


@pytest.mark.parametrize("mode", ["fast", "accu"])
@pytest.mark.parametrize("s,phi", [(8, 0.5), (14, 0.5), (14, 2.0), (18, 1.0)])
def test_error_bound_against_exact_product(mode, s, phi):
    """|C_hat - AB| <= 2**-(a+b) (sum|b'| + sum|2**a a|) + ulp/2, against exact Fractions."""
    A, B = make_matrices(6, 24, 5, phi, 17 + s)
    o = oz.oracle_dgemm(A, B, s, mode)
    Bp = _bigint_scaled(B, o["beta"], axis=0)
    for i in range(6):
        ai = int(o["alpha"][i])
        for j in range(5):
            bj = int(o["beta"][j])
            exact = sum(Fraction(float(A[i, l])) * Fraction(float(B[l, j])) for l in range(24))
            err_int = sum(abs(Bp[l][j]) for l in range(24)) + sum(
                abs(Fraction(float(A[i, l])) * Fraction(2) ** ai) for l in range(24))
            c = float(o["C"][i, j])
            half_ulp = Fraction(math.ulp(c)) / 2
            assert abs(Fraction(c) - exact) <= err_int * Fraction(2) ** (-ai - bj) + half_ulp


def test_sampled_entries_agree_with_full_pipeline():
    A, B = make_matrices(20, 30, 17, 1.0, 13)
    for mode in ("fast", "accu"):
        full = oz.oracle_dgemm(A, B, 14, mode)
        ii = np.array([0, 19, 7, 7, 3])
        jj = np.array([16, 0, 7, 8, 3])
        part = oz.oracle_entries(A, B, 14, mode, ii, jj)
        for k in range(5):
            assert part["X"][k] == full["X"][ii[k], jj[k]]
            assert part["C"][k] == full["C"][ii[k], jj[k]]
            np.testing.assert_array_equal(part["P"][:, k], full["P"][:, ii[k], jj[k]])


# --------------------------------------------------------------------------- planted mistakes
def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check a pin fails."""
    A, B = make_matrices(4, 6, 3, 1.0, 2)

    def fails(fn):
        try:
            fn()
        except (AssertionError, ValueError):
            return True
        return False

    run = lambda: _check_x_equals_aprime_bprime(A, B, 8, "fast")
    assert not fails(run)
    orig_planes = oz.residue_planes

    def wrong_sign_a(X, exps, axis, moduli):
        out = orig_planes(X, exps, axis, moduli)
        return -out if axis == 1 else out  # sign error on the A side only

    monkeypatch.setattr(oz, "residue_planes", wrong_sign_a)
    assert fails(run)
    monkeypatch.setattr(oz, "residue_planes", orig_planes)
    orig_res = oz.centered_residue
    monkeypatch.setattr(oz, "centered_residue", lambda x, m: orig_res(x, m) + 1)  # off by one
    assert fails(test_centered_residue_brute_force)
    monkeypatch.setattr(oz, "centered_residue", orig_res)

    orig_crt = oz.crt_matrix

    def dropped_term(R, c):
        c2 = dict(c)
        c2["inv"] = [0] + list(c["inv"][1:])  # drops the first channel's term
        return orig_crt(R, c2)

    monkeypatch.setattr(oz, "crt_matrix", dropped_term)
    assert fails(run)
    monkeypatch.setattr(oz, "crt_matrix", orig_crt)

    orig_prod = oz.products
    monkeypatch.setattr(oz, "products", lambda Ar, Br: orig_prod(Ar[:, ::-1, :].copy(), Br))  # wrong row index
    assert fails(run)
    monkeypatch.setattr(oz, "products", orig_prod)

    orig_fast = oz.fast_exponents
    monkeypatch.setattr(oz, "fast_exponents", lambda X, axis, L: orig_fast(X, axis, L) + 1)  # too large
    assert fails(run)
    monkeypatch.setattr(oz, "fast_exponents", orig_fast)
    assert not fails(run)

    # the fast statistic summed in signed 64 bits wraps at q = 2**23
    class Int64Sum:
        def __getattr__(self, name):
            return getattr(np, name)

        @staticmethod
        def sum(a, axis=None, dtype=None):
            return np.sum(np.asarray(a).astype(np.int64), axis=axis, dtype=np.int64)

    big = lambda: test_fast_statistic_past_two_to_the_63(1 << 23)
    assert not fails(big)
    monkeypatch.setattr(oz, "np", Int64Sum())
    assert fails(big)
    monkeypatch.setattr(oz, "np", np)

    # accu exponents from the bound's maxima in the original scale, split
    # evenly between the row and the column (an earlier reading): a huge row
    # then sets every column's beta and the other rows lose their bits
    orig_accu = oz.accu_exponents

    def original_scale_split(A, B, L):
        al, be, Abar, Bbar, u, v, W = orig_accu(A, B, L)
        Wf = [[Fraction(int(W[i, j])) * Fraction(2) ** (-int(u[i]) - int(v[j])) for j in range(W.shape[1])]
              for i in range(W.shape[0])]
        al2 = np.array([oz.max_pow4_exponent(max(row), L) if max(row) else 0 for row in Wf])
        be2 = np.array([oz.max_pow4_exponent(max(col), L) if max(col) else 0 for col in zip(*Wf)])
        return al2, be2, Abar, Bbar, u, v, W

    monkeypatch.setattr(oz, "accu_exponents", original_scale_split)
    assert fails(test_accu_rows_and_columns_keep_their_own_scale)
    assert fails(test_exponents_scale_equivariant)
    monkeypatch.setattr(oz, "accu_exponents", orig_accu)
    assert not fails(test_accu_rows_and_columns_keep_their_own_scale)
