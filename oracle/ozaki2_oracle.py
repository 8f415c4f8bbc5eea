"""Ozaki Scheme II: a plain, slow CPU oracle of the emulated FP64 GEMM.

TEST INFRASTRUCTURE ONLY.  This module is the independent reference that the
CUDA library is checked against.  Only the tests, the package's smoke check and
the benchmark's CPU-baseline / reference legs may import it; the library never
does, and this module imports nothing from the library.

It restates the method step by step, in exact integer arithmetic (numpy int64
where the values provably fit, Python integers and Fractions elsewhere).  The
one library primitive used as a step is a float64 matrix product of integer
matrices, used only where every partial sum is an integer below 2**53, so the
product is exact under any summation order the BLAS picks.

Sources (web pages; cited by title and section):
  [P]  "Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" (kevinhyj.github.io)
       §1 pipeline table, §2 the two bounds, §5.1 statistics, §6 cost model,
       §10.1 integer residue proposal.
  [S]  "Ozaki II supplement: INT8 range conditions and paper performance
       results" (edgep.me) §1.1 pipeline, §1.2 centered residues, §1.3 INT32
       condition, §1.4 range bits, §2 Eq. (18).

The pages leave several rules open; the readings taken here are numbered
R1..R14 in the docstrings below and collected in the design notes.

Parity pins (tests/test_oracle_pins.py) tie every function here to something
other than itself: brute force on tiny inputs (X == A'B' with Python big
integers), CRT round trips, closed forms (Eq. (18) on +-1 matrices, the INT32
limit 131072, the residue count 2 s n^2), textbook special cases (small-integer
and dyadic inputs reproduce the exact product) and exact Fraction products.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

# Fractional bits kept per element in the fast-mode sum-of-squares statistic
# (each |x| is rounded up to a multiple of 2**(e - F)).  Each rounded-up term is <= 2**F and its square <= 2**(2F),
# so for q < 2**24 the sum of squares is < 2**64 and fits an unsigned 64-bit
# integer (FAST_Q_LIMIT); it is summed in uint64, since from q = 2**23 on it
# can pass 2**63.
F_FAST = 20
# Largest magnitude of an upward-quantised bound entry: signed INT8.
BOUND_QMAX = 127
# [S] §1.3: q * 2**14 < 2**31  <=>  q < 131072, the bound for one unblocked
# INT32 accumulation of a residue product.  For longer inner dimensions the
# same section splits K into blocks, reduces each block's product modulo the
# modulus and combines the residues; the result R_t = P_t mod m_t is the same
# number, so the oracle computes P_t exactly (int64: |P_t| <= q 2**14) and
# reduces it, for any q.
Q_LIMIT = 131072
# Limits that remain: the 64-bit fast statistic (above) and the accu bound
# product Wbar = Abar Bbar, an exact INT32 accumulation (q 127**2 < 2**31).
FAST_Q_LIMIT = 1 << 24
ACCU_Q_LIMIT = 133145


# ----------------------------------------------------------------------------
# O0  moduli and CRT constants
# ----------------------------------------------------------------------------
def greedy_moduli(s: int) -> list[int]:
    """Walk down from 256, keep each integer coprime to every one kept.

    [S] §1.2 asks only for pairwise-coprime m_t <= 256, with larger moduli
    giving more range bits; taking them greedily from the top is the plainest
    set that meets both.
    """
    if s < 1:
        raise ValueError("s must be >= 1")
    out: list[int] = []
    m = 256
    while len(out) < s:
        if m < 2:
            raise ValueError("not enough coprime moduli <= 256")
        if all(math.gcd(m, k) == 1 for k in out):
            out.append(m)
        m -= 1
    return out


def modulus_constants(moduli: list[int]) -> dict:
    """M = prod m_t, the CRT weights M/m_t and their inverses mod m_t.

    The reconstruction bound is L = M/2 - 1 (Eq. (18)'s numerator in [S] §2;
    [P] §1 asks max |(A'B')_ij| < M/2).
    """
    M = 1
    for m in moduli:
        M *= m
    Mt = [M // m for m in moduli]
    inv = [pow(Mt[t] % m, -1, m) for t, m in enumerate(moduli)]
    return {"moduli": list(moduli), "M": M, "L": M // 2 - 1, "Mt": Mt, "inv": inv}


# ----------------------------------------------------------------------------
# helpers: exact decomposition of doubles
# ----------------------------------------------------------------------------
def decompose(x: np.ndarray):
    """|x| = mant * 2**E exactly, mant an integer < 2**53 (0 for x == 0)."""
    x = np.asarray(x, dtype=np.float64)
    f, e = np.frexp(np.abs(x))  # f in [0.5, 1), exact
    mant = (f * 2.0**53).astype(np.int64)  # exact: f has <= 53 significant bits
    E = e.astype(np.int64) - 53
    sign = np.where(np.signbit(x), -1, 1).astype(np.int64)
    return sign, mant, E


def floor_log2_plus1(amax: np.ndarray) -> np.ndarray:
    """e with 2**(e-1) <= amax < 2**e (the frexp exponent); 0 where amax == 0."""
    return np.frexp(np.asarray(amax, dtype=np.float64))[1].astype(np.int64)


def _shift_right_ceil(mant: np.ndarray, d: np.ndarray) -> np.ndarray:
    """ceil(mant / 2**d) for mant >= 0, d >= 0 (int64, elementwise)."""
    dd = np.minimum(d, 62)
    q = (mant + (np.int64(1) << dd) - 1) >> dd
    # d >= 62 with 0 < mant < 2**53: the quotient is in (0, 1), so its ceiling is 1.
    return np.where(d >= 62, (mant > 0).astype(np.int64), q)


def ceil_scaled(mant: np.ndarray, E: np.ndarray, k) -> np.ndarray:
    """ceil(mant * 2**(E + k)) as int64; the caller guarantees the result fits."""
    sh = E + k
    up = np.where(sh > 0, sh, 0)
    left = mant << np.minimum(up, 62)
    right = _shift_right_ceil(mant, np.where(sh < 0, -sh, 0))
    return np.where(sh >= 0, left, right)


def max_pow4_exponent(U: Fraction, L: int) -> int:
    """max { a in Z : 4**a * U <= L }, and 0 when U == 0 (an all-zero vector leaves a free)."""
    if U < 0:
        raise ValueError("a bound on a sum of squares or of |A||B| cannot be negative")
    if U == 0:
        return 0
    # start near the answer from bit lengths, then step to the exact maximum
    est = (L.bit_length() - (U.numerator.bit_length() - U.denominator.bit_length())) // 2

    def ok(a: int) -> bool:
        return (Fraction(4) ** a) * U <= L

    a = est
    while not ok(a):
        a -= 1
    while ok(a + 1):
        a += 1
    return a


# ----------------------------------------------------------------------------
# O2  scaling exponents
# ----------------------------------------------------------------------------
def fast_exponents(X: np.ndarray, axis: int, L: int) -> np.ndarray:
    """fast bound, [P] §2 and §5.1 (row max-abs and sum of squares, rounded up).

    For each vector x (a row of A: axis=1; a column of B: axis=0):
      e   = floor(log2 max|x|) + 1,
      S   = sum_l ceil(|x_l| * 2**(F - e))**2   (an exact integer),
      U   = S * 2**(2(e - F))  >=  ||x||_2**2,
      exp = max { a : 4**a * U <= L }.
    By Cauchy-Schwarz (|A||B|)_ij <= ||A(i,:)|| ||B(:,j)||, so the scaled
    integers satisfy |(A'B')_ij| <= sqrt(L) * sqrt(L) = L < M/2.
    """
    X = np.asarray(X, dtype=np.float64)
    sign, mant, E = decompose(X)
    amax = np.max(np.abs(X), axis=axis) if X.shape[axis] > 0 else np.zeros(X.shape[1 - axis])
    e = floor_log2_plus1(amax)
    e_b = np.expand_dims(e, axis)
    terms = ceil_scaled(mant, E, F_FAST - e_b)
    # each term is <= 2**F, its square <= 2**(2F) = 2**40, so a sum of q < 2**24
    # squares is < 2**64: exact in uint64 (int64 would wrap from q >= 2**23)
    if X.shape[axis] >= FAST_Q_LIMIT:
        raise ValueError("q >= 2**24: the sum of squares may leave 64 bits")
    sq = (terms * terms).astype(np.uint64)
    S = np.sum(sq, axis=axis, dtype=np.uint64)
    out = np.zeros(S.shape, dtype=np.int64)
    for i in range(S.shape[0]):
        Si = int(S[i])
        if Si == 0:
            out[i] = 0
            continue
        U = Fraction(Si) * Fraction(2) ** (2 * (int(e[i]) - F_FAST))
        out[i] = max_pow4_exponent(U, L)
    return out


def bound_quant_exponents(amax: np.ndarray) -> np.ndarray:
    """u = max { u : ceil(amax * 2**u) <= 127 } (0 for a zero vector)."""
    out = np.zeros(amax.shape, dtype=np.int64)
    for i, a in enumerate(np.asarray(amax, dtype=np.float64)):
        if a == 0.0:
            continue
        fa = Fraction(float(a))
        u = 6 - math.frexp(a)[1]  # 2**(e-1) <= a < 2**e  =>  a * 2**(6-e) in [32, 64)
        while math.ceil(fa * Fraction(2) ** (u + 1)) <= BOUND_QMAX:
            u += 1
        while math.ceil(fa * Fraction(2) ** u) > BOUND_QMAX:
            u -= 1
        out[i] = u
    return out


def bound_inputs(X: np.ndarray, axis: int):
    """accu, [P] §2: upward quantisation of |X| into [0, 127] per row / column.

    Returns (Xbar, u) with Xbar = ceil(|X| * 2**u) elementwise, u per vector.
    """
    X = np.asarray(X, dtype=np.float64)
    amax = np.max(np.abs(X), axis=axis) if X.shape[axis] > 0 else np.zeros(X.shape[1 - axis])
    u = bound_quant_exponents(amax)
    _, mant, E = decompose(X)
    Xbar = ceil_scaled(mant, E, np.expand_dims(u, axis))
    return Xbar, u


def _exact_int_matmul(Ai: np.ndarray, Bi: np.ndarray) -> np.ndarray:
    """Product of integer matrices, exact when every |partial sum| < 2**53.

    The callers guarantee q * max|a| * max|b| < 2**53 (checked here), so the
    float64 BLAS product is exact under any summation order.
    """
    q = Ai.shape[1]
    amax = int(np.max(np.abs(Ai))) if Ai.size else 0
    bmax = int(np.max(np.abs(Bi))) if Bi.size else 0
    if q * amax * bmax >= 2**53:
        raise ValueError("integer product would not be exact in float64")
    P = np.asarray(Ai, dtype=np.float64) @ np.asarray(Bi, dtype=np.float64)
    return P.astype(np.int64)


def accu_exponents(A: np.ndarray, B: np.ndarray, L: int):
    """accu bound, [P] §2 and §5.1: one extra integer GEMM on |A|, |B|.

    Abar = ceil(|A| * 2**u_i) (rows), Bbar = ceil(|B| * 2**v_j) (columns),
    Wbar = Abar Bbar (exact), so (|A||B|)_ij * 2**(u_i + v_j) <= Wbar_ij.
    Reading of "row/column maxima of the bound output -> final scale
    exponents": the maxima are taken in the quantised scale,
      R_i = max_j Wbar_ij,  K_j = max_i Wbar_ij,
      alpha_i = u_i + max { a : 4**a R_i <= L },  beta_j = v_j + max { b : 4**b K_j <= L }
    (0 for a zero row or column of Wbar).  Then
      2**(alpha_i + beta_j) (|A||B|)_ij <= 2**(a_i + b_j) Wbar_ij
                                        <= sqrt(4**a_i R_i * 4**b_j K_j) <= L,
    and each row and column keeps its own scale u_i, v_j.
    Returns (alpha, beta, Abar, Bbar, u, v, Wbar).
    """
    Abar, u = bound_inputs(A, axis=1)
    Bbar, v = bound_inputs(B, axis=0)
    Wbar = _exact_int_matmul(Abar, Bbar)
    p, r = Wbar.shape
    R = Wbar.max(axis=1) if r else np.zeros(p, dtype=np.int64)
    K = Wbar.max(axis=0) if p else np.zeros(r, dtype=np.int64)
    alpha = np.zeros(p, dtype=np.int64)
    beta = np.zeros(r, dtype=np.int64)
    for i in range(p):
        if R[i] > 0:
            alpha[i] = int(u[i]) + max_pow4_exponent(Fraction(int(R[i])), L)
    for j in range(r):
        if K[j] > 0:
            beta[j] = int(v[j]) + max_pow4_exponent(Fraction(int(K[j])), L)
    return alpha, beta, Abar, Bbar, u, v, Wbar


# ----------------------------------------------------------------------------
# O3/O4  integerise and centered residues
# ----------------------------------------------------------------------------
def centered_residue(x, m: int):
    """rho_m(x) = ((x + floor(m/2)) mod m) - floor(m/2) in [-floor(m/2), ceil(m/2)-1].

    [S] §1.2; for m = 256 the range is [-128, 127] and 128 maps to -128.
    Works on Python ints and numpy int64 arrays.
    """
    h = m // 2
    return ((x + h) % m) - h


def scaled_trunc_bigint(x: float, k: int) -> int:
    """trunc(2**k * x) as a Python integer (truncation toward zero, [P] §1)."""
    if x == 0.0:
        return 0
    fx = Fraction(float(x)) * Fraction(2) ** k
    n = abs(fx.numerator) // fx.denominator
    return -n if fx < 0 else n


def residue_planes(X: np.ndarray, exps: np.ndarray, axis: int, moduli: list[int]) -> np.ndarray:
    """rho_{m_t}(trunc(2**exp * x)) for every entry and every modulus.

    axis=1: exps[i] scales row i (A' = trunc(DA)); axis=0: exps[j] scales
    column j (B' = trunc(BE)).  Returns int64 [s, *X.shape].
    The magnitude |x'| = floor(mant * 2**sh) with sh = E + exp.  For sh <= 0
    it is an int64 below 2**53; for sh > 0 its residue is taken through
    (mant mod m) * (2**sh mod m) mod m, which is the same residue without
    forming the (possibly thousands of bits long) integer.
    """
    X = np.asarray(X, dtype=np.float64)
    sign, mant, E = decompose(X)
    sh = E + np.expand_dims(np.asarray(exps, dtype=np.int64), axis)
    neg_sh = np.where(sh < 0, -sh, 0)
    small = mant >> np.minimum(neg_sh, 62)  # floor(mant / 2**-sh) for sh <= 0
    small = np.where(neg_sh >= 62, 0, small)
    pos = sh > 0
    out = np.empty((len(moduli),) + X.shape, dtype=np.int64)
    max_sh = int(sh.max()) if sh.size else 0
    for t, m in enumerate(moduli):
        if pos.any():
            table = np.array([pow(2, k, m) for k in range(max(max_sh, 0) + 1)], dtype=np.int64)
            big = ((mant % m) * table[np.where(pos, sh, 0)]) % m
            mag_mod = np.where(pos, big, small % m)
        else:
            mag_mod = small % m
        out[t] = centered_residue(sign * mag_mod, m)
    return out


# ----------------------------------------------------------------------------
# O5..O8  products, output residues, CRT, inverse scaling
# ----------------------------------------------------------------------------
def products(Ares: np.ndarray, Bres: np.ndarray) -> np.ndarray:
    """P_t = A_t B_t, exact ([P] §1 yellow stage; [S] §1.3 bound q * 2**14)."""
    s = Ares.shape[0]
    q = Ares.shape[2]
    P = np.empty((s, Ares.shape[1], Bres.shape[2]), dtype=np.int64)
    for t in range(s):
        P[t] = _exact_int_matmul(Ares[t], Bres[t])
    if P.size:
        assert int(np.max(np.abs(P))) <= q * 2**14
    return P


def output_residues(P: np.ndarray, moduli: list[int]) -> np.ndarray:
    """R_t = P_t mod m_t, nonnegative ([P] §1 blue stage; the nonnegative remainder)."""
    R = np.empty(P.shape, dtype=np.int64)
    for t, m in enumerate(moduli):
        R[t] = np.mod(P[t], m)
    return R


def crt(residues, consts: dict) -> int:
    """CRT_M: the unique X in [-M/2, M/2) with X = R_t (mod m_t) for all t.

    [P] §1 red stage.  w_t = R_t * inv_t mod m_t, Y = sum_t w_t M/m_t mod M,
    X = Y - M if Y >= M/2 else Y (-M/2 included, M/2 excluded).
    """
    M = consts["M"]
    Y = 0
    for t, m in enumerate(consts["moduli"]):
        w = (int(residues[t]) * consts["inv"][t]) % m
        Y += w * consts["Mt"][t]
    Y %= M
    return Y - M if 2 * Y >= M else Y


def crt_matrix(R: np.ndarray, consts: dict) -> np.ndarray:
    """crt() for every entry; returns an object array of Python integers."""
    M = consts["M"]
    Y = np.zeros(R.shape[1:], dtype=object)
    for t, m in enumerate(consts["moduli"]):
        w = (R[t] * consts["inv"][t]) % m
        Y = Y + w.astype(object) * consts["Mt"][t]
    Y = Y % M
    return np.where(2 * Y >= M, Y - M, Y)


def round_scaled(X: int, k: int) -> float:
    """RN_even(X * 2**-k): one correct rounding to double, with overflow to +-inf.

    Python's int true division and int-to-float conversion are correctly
    rounded (ties to even), subnormal range included.
    """
    X = int(X)
    if X == 0:
        return 0.0
    try:
        if k >= 0:
            return X / (1 << k)
        return float(X << (-k))
    except OverflowError:
        return math.inf if X > 0 else -math.inf


def inverse_scaling(X: np.ndarray, alpha: np.ndarray, beta: np.ndarray) -> np.ndarray:
    """C_hat = D^-1 X E^-1 with D = diag(2**alpha), E = diag(2**beta)."""
    p, r = X.shape
    C = np.empty((p, r), dtype=np.float64, order="F")
    for j in range(r):
        bj = int(beta[j])
        for i in range(p):
            C[i, j] = round_scaled(X[i, j], int(alpha[i]) + bj)
    return C


# ----------------------------------------------------------------------------
# the whole pipeline
# ----------------------------------------------------------------------------
def exponents(A: np.ndarray, B: np.ndarray, s: int, mode: str):
    consts = modulus_constants(greedy_moduli(s))
    L = consts["L"]
    if mode == "fast":
        alpha = fast_exponents(A, axis=1, L=L)
        beta = fast_exponents(B, axis=0, L=L)
    elif mode == "accu":
        alpha, beta = accu_exponents(A, B, L)[:2]
    else:
        raise ValueError(mode)
    return alpha, beta, consts


def oracle_dgemm(A: np.ndarray, B: np.ndarray, s: int, mode: str) -> dict:
    """Every stage of Ozaki-II on the CPU ([P] §1 table; [S] §1.1).

    Returns alpha, beta, Ares [s,p,q], Bres [s,q,r], P [s,p,r], R [s,p,r],
    X (object array of ints, p x r), C (float64, p x r).
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    if A.shape[1] != B.shape[0]:
        raise ValueError("inner dimensions differ")
    q = A.shape[1]
    if mode == "fast" and q >= FAST_Q_LIMIT:
        raise ValueError("q >= 2**24: the fast sum-of-squares statistic leaves 64 bits")
    if mode == "accu" and q >= ACCU_Q_LIMIT:
        raise ValueError("q * 127**2 >= 2**31: the bound product leaves INT32")
    alpha, beta, consts = exponents(A, B, s, mode)
    moduli = consts["moduli"]
    Ares = residue_planes(A, alpha, axis=1, moduli=moduli)
    Bres = residue_planes(B, beta, axis=0, moduli=moduli)
    P = products(Ares, Bres)
    R = output_residues(P, moduli)
    X = crt_matrix(R, consts)
    C = inverse_scaling(X, alpha, beta)
    return {"alpha": alpha, "beta": beta, "Ares": Ares, "Bres": Bres, "P": P, "R": R,
            "X": X, "C": C, "consts": consts}


def oracle_entries(A: np.ndarray, B: np.ndarray, s: int, mode: str, ii, jj,
                   alpha=None, beta=None) -> dict:
    """The same pipeline evaluated only at the sampled outputs (ii[k], jj[k]).

    The exponents need whole rows / columns (and, in accu mode, the whole bound
    product); pass alpha/beta to reuse them.  Per sampled entry it forms the
    residue rows and columns it needs, P_t[i,j] as a dot product, R_t, X, C.
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    if alpha is None or beta is None:
        alpha, beta, consts = exponents(A, B, s, mode)
    else:
        consts = modulus_constants(greedy_moduli(s))
    moduli = consts["moduli"]
    ii = np.asarray(ii, dtype=np.int64)
    jj = np.asarray(jj, dtype=np.int64)
    ui, inv_i = np.unique(ii, return_inverse=True)
    uj, inv_j = np.unique(jj, return_inverse=True)
    Arows = residue_planes(A[ui, :], alpha[ui], axis=1, moduli=moduli)  # [s, ni, q]
    Bcols = residue_planes(B[:, uj], beta[uj], axis=0, moduli=moduli)  # [s, q, nj]
    n = ii.shape[0]
    P = np.empty((len(moduli), n), dtype=np.int64)
    for t in range(len(moduli)):
        P[t] = np.einsum("kq,qk->k", Arows[t][inv_i, :], Bcols[t][:, inv_j])
    R = np.stack([np.mod(P[t], m) for t, m in enumerate(moduli)])
    X = [crt(R[:, k], consts) for k in range(n)]
    C = np.array([round_scaled(X[k], int(alpha[ii[k]]) + int(beta[jj[k]])) for k in range(n)])
    return {"alpha": alpha, "beta": beta, "P": P, "R": R, "X": X, "C": C,
            "Arows": Arows, "Bcols": Bcols, "rows": ui, "cols": uj, "consts": consts}
