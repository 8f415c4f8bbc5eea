"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Integer stages (exponents, residue planes, products, output residues, CRT
integer) must match bit for bit; C within 2 ulp (|ord(a) - ord(b)| <= 2 on
the sign-magnitude order of the bit patterns).  Small and medium cases are
compared element by element; the full-size workloads are compared on their
exponents and on sampled outputs computed one by one by the oracle.
"""
import numpy as np
import pytest

from oracle import ozaki2_oracle as oracle
from tests._util import decode_x, ulp_distance
from workloads import WORKLOADS, make_matrices, make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ULP_TOL = 2


@pytest.fixture(scope="module")
def oz2():
    import __graft_entry__ as g

    g.build()
    import emulated_fp64_gemm_gb300 as m

    assert torch.cuda.is_available()
    return m


def _dev(x):
    return torch.from_numpy(np.asfortranarray(x)).cuda()


def _full_check(oz2, A, B, s, mode, check_p=True):
    got = oz2.dgemm_debug(_dev(A), _dev(B), s, mode, want_p=check_p)
    torch.cuda.synchronize()
    ref = oracle.oracle_dgemm(A, B, s, mode)
    np.testing.assert_array_equal(got["alpha"].cpu().numpy(), ref["alpha"], err_msg="alpha")
    np.testing.assert_array_equal(got["beta"].cpu().numpy(), ref["beta"], err_msg="beta")
    np.testing.assert_array_equal(got["Ares"].cpu().numpy(), ref["Ares"], err_msg="A residues")
    np.testing.assert_array_equal(got["Bres"].cpu().numpy(), np.transpose(ref["Bres"], (0, 2, 1)),
                                  err_msg="B residues")
    if check_p:
        np.testing.assert_array_equal(got["P"].cpu().numpy(), np.transpose(ref["P"], (0, 2, 1)),
                                      err_msg="products")
    np.testing.assert_array_equal(got["R"].cpu().numpy(), np.transpose(ref["R"], (0, 2, 1)),
                                  err_msg="output residues")
    X = got["X"].cpu().numpy()
    p, r = ref["X"].shape
    for i in range(p):
        for j in range(r):
            assert decode_x(X[j, i]) == ref["X"][i, j], ("X", i, j)
    C = got["C"].cpu().numpy()
    assert ulp_distance(C, ref["C"]) <= ULP_TOL
    # the production entry point gives the same C as the checking one
    C2 = oz2.dgemm(_dev(A), _dev(B), s, mode).cpu().numpy()
    np.testing.assert_array_equal(C2, C)
    assert oz2.last_error() == 0
    return got, ref


def test_bounded_wait_gives_up_and_reports(oz2):
    # a barrier that nothing completes: the wait must end with a timeout status
    assert oz2.selftest_wait_timeout(2000) == 5
    assert oz2.selftest_wait_timeout(50) == 5


def test_small_workload_every_stage(oz2):
    w = WORKLOADS["n128_s8_fast"]
    A, B = make_workload(w)
    _full_check(oz2, A, B, w.s, w.mode)


@pytest.mark.parametrize("mode", ["fast", "accu"])
@pytest.mark.parametrize("p,q,r,s", [
    (1, 1, 1, 2), (7, 13, 5, 8), (129, 1000, 257, 14), (1000, 129, 7, 18),
    (300, 70, 513, 20), (64, 961, 40, 14), (130, 1921, 260, 16), (257, 64, 1, 3),
    # the largest channel count of each CRT limb bucket other than 20 (their
    # M/m_t use every coefficient byte the bucket's kernel reads)
    (150, 333, 90, 15), (77, 250, 130, 11),
])
def test_ragged_shapes(oz2, p, q, r, s, mode):
    A, B = make_matrices(p, q, r, 1.0, p * 1000 + q + r + s)
    _full_check(oz2, A, B, s, mode)


@pytest.mark.parametrize("q", [2048, 3000, 8192, 8200])
def test_fast_b_side_register_chunks_and_fallback(oz2, q):
    # fast mode makes B's statistics and residue planes in one read of B for
    # q <= 8192 (one, two or four 2048-element chunks per thread); q = 8200
    # takes the separate statistics and residue kernels
    A, B = make_matrices(40, q, 24, 0.5, q)
    _full_check(oz2, A, B, 14, "fast")


@pytest.mark.parametrize("mode", ["fast", "accu"])
@pytest.mark.parametrize("q", [777, 3001, 8191])
def test_b_side_unaligned_columns(oz2, q, mode):
    """odd q and odd ldb = q + 4: the odd columns of B start 8 bytes past a
    16-byte boundary.  q = 777: the one-read kernels' scalar loads; q = 3001
    and 8191: the bulk-copy kernels (fast: statistics; accu: maximum and
    quantised bound row), whose copy covers each column's aligned middle,
    with the element before it (odd columns) or the one after it (even
    columns) read separately."""
    A, B = make_matrices(48, q, 33, 2.0, 11)
    bigB = torch.zeros((33, q + 4), dtype=torch.float64).t()  # (q + 4, 33), strides (1, q + 4)
    bigB[:q] = torch.from_numpy(B)
    dB = bigB.cuda()[:q]
    assert dB.stride() == (1, q + 4)
    got = oz2.dgemm_debug(_dev(A), dB, 14, mode, want_p=False)
    ref = oracle.oracle_dgemm(A, B, 14, mode)
    np.testing.assert_array_equal(got["beta"].cpu().numpy(), ref["beta"])
    np.testing.assert_array_equal(got["Bres"].cpu().numpy(), np.transpose(ref["Bres"], (0, 2, 1)))
    assert ulp_distance(got["C"].cpu().numpy(), ref["C"]) <= ULP_TOL
    C2 = oz2.dgemm(_dev(A), dB, 14, mode).cpu().numpy()
    np.testing.assert_array_equal(C2, got["C"].cpu().numpy())


def test_fast_inner_dimension_past_the_int32_condition(oz2):
    """q = 140000 > 2^17: the modular GEMMs reduce every K-block modulo m_t
    (supplement §1.3, blocked form), so every stage still matches the oracle
    (P itself is int32 and is not requested past 2^17)."""
    A, B = make_matrices(24, 140000, 16, 0.5, 17)
    _full_check(oz2, A, B, 14, "fast", check_p=False)
    with pytest.raises(oz2.Ozaki2Error):
        oz2.dgemm_debug(_dev(A), _dev(B), 14, "fast", want_p=True)


def test_accu_bound_product_at_its_int32_limit(oz2):
    """q = 133144 with every quantised bound entry 127 (|a| = |b| = 127/128):
    Wbar = q 127^2 = 2147479576, the largest INT32-exact bound product."""
    q = oz2.Q_LIMIT_ACCU - 1
    rng = np.random.default_rng(9)
    A = np.where(rng.random((8, q)) < 0.5, -1.0, 1.0) * (127 / 128)
    B = np.where(rng.random((q, 8)) < 0.5, -1.0, 1.0) * (127 / 128)
    got = oz2.dgemm_debug(_dev(A), _dev(B), 14, "accu", want_p=False)
    ref = oracle.oracle_dgemm(A, B, 14, "accu")
    np.testing.assert_array_equal(got["alpha"].cpu().numpy(), ref["alpha"])
    np.testing.assert_array_equal(got["beta"].cpu().numpy(), ref["beta"])
    assert ulp_distance(got["C"].cpu().numpy(), ref["C"]) <= ULP_TOL
    assert oz2.last_error() == 0


def test_leading_dimensions_larger_than_rows(oz2):
    A, B = make_matrices(150, 90, 70, 0.5, 3)
    bigA = torch.zeros((200, 90), dtype=torch.float64).t().contiguous().t()  # strides (1, 200)
    bigA[:150] = torch.from_numpy(A)
    bigB = torch.zeros((100, 70), dtype=torch.float64).t().contiguous().t()
    bigB[:90] = torch.from_numpy(B)
    dA = bigA.cuda()[:150]
    dB = bigB.cuda()[:90]
    assert dA.stride() == (1, 200) and dB.stride() == (1, 100)
    C = oz2.dgemm(dA, dB, 14, "fast").cpu().numpy()
    ref = oracle.oracle_dgemm(A, B, 14, "fast")
    assert ulp_distance(C, ref["C"]) <= ULP_TOL
    Cbig = torch.full((160, 70), 7.0, dtype=torch.float64).t().contiguous().t().cuda()  # ldc = 160
    oz2.dgemm(dA, dB, 14, "fast", out=Cbig[:150])
    Cb = Cbig.cpu().numpy()
    assert ulp_distance(Cb[:150], ref["C"]) <= ULP_TOL
    assert np.all(Cb[150:] == 7.0)  # rows past p untouched


@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_special_values(oz2, mode):
    A, B = make_matrices(96, 200, 80, 2.0, 5)
    A[3, :] = 0.0                      # zero row
    B[:, 4] = 0.0                      # zero column
    A[5, :] *= 1e-310                  # subnormal row
    A[6, 7] = 1e300                    # one huge entry
    A[7, :] = -A[7, :] * 2.0**600
    B[11, :] = 5e-324                  # smallest subnormals
    B[:, 9] *= 2.0**-1000
    A[8, ::2] = -0.0
    _full_check(oz2, A, B, 14, mode)


@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_outputs_past_the_double_range(oz2, mode):
    """Outputs that overflow to +-inf, that sit next to the overflow threshold,
    that are subnormal and that underflow: the CRT's exact rounding path
    (results outside the normal range) against the oracle's one correct
    rounding with overflow to +-inf and gradual underflow."""
    A, B = make_matrices(64, 100, 40, 0.5, 12)
    A[0, :] *= 2.0**1000
    A[1, :] *= -(2.0**1000)
    A[2, :] *= 2.0**-1000
    A[3, :] *= -(2.0**-1000)
    B[:, 0] *= 2.0**30    # rows 0, 1: far past the largest double
    B[:, 1] *= 2.0**20    # next to it
    B[:, 2] *= 2.0**22
    B[:, 3] *= 2.0**-70   # rows 2, 3: subnormal
    B[:, 4] *= 2.0**-100  # underflow toward zero
    B[:, 5] *= 2.0**-52
    got, ref = _full_check(oz2, A, B, 14, mode)
    C = ref["C"]  # (the GPU's C equals it within 2 ulp, checked above)
    assert C[0, 0] == np.inf and C[1, 0] == -np.inf
    assert np.isfinite(C[0, 2]) and abs(C[0, 2]) > 1e307  # next to the largest double
    sub = np.abs(C[2:4, 3:6])
    assert np.any((sub > 0) & (sub < np.finfo(np.float64).tiny))


def test_wide_range_accu_general_residue_path(oz2):
    """A huge entry meeting only zeros of B: trunc(2^alpha a) needs the general residue path."""
    A, B = make_matrices(40, 64, 30, 1.0, 8)
    A[2, :] = 0.0
    A[2, 0] = 1e300
    B[0, :] = 0.0
    got, ref = _full_check(oz2, A, B, 14, "accu")
    assert ref["alpha"][2] == 0


def test_small_integer_inputs_exact(oz2):
    rng = np.random.default_rng(3)
    A = rng.integers(-8, 9, size=(200, 300)).astype(np.float64)
    B = rng.integers(-8, 9, size=(300, 100)).astype(np.float64)
    C = oz2.dgemm(_dev(A), _dev(B), 8, "fast").cpu().numpy()
    np.testing.assert_array_equal(C, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))


def test_row_major_operands(oz2):
    A, B = make_matrices(70, 50, 60, 0.5, 4)
    dA = torch.from_numpy(np.ascontiguousarray(A)).cuda()  # row-major
    dB = torch.from_numpy(np.ascontiguousarray(B)).cuda()
    C = oz2.dgemm(dA, dB, 14, "fast").cpu().numpy()
    ref = oracle.oracle_dgemm(A, B, 14, "fast")
    assert ulp_distance(C, ref["C"]) <= ULP_TOL


def test_host_entry_point(oz2):
    A, B = make_matrices(300, 200, 100, 0.5, 6)
    hA = torch.from_numpy(np.asfortranarray(A)).pin_memory()
    hB = torch.from_numpy(np.asfortranarray(B)).pin_memory()
    C = oz2.dgemm_host(hA, hB, 14, "fast").numpy()
    ref = oracle.oracle_dgemm(A, B, 14, "fast")
    assert ulp_distance(C, ref["C"]) <= ULP_TOL


def test_host_entry_point_staged_uploads(oz2):
    """The host entry point uploads A by row blocks and B by column parts as the
    schedule needs them: strided host operands (lda > p, ldb > q), two column
    parts (r = 2600) and two calls in a row through the same staging copies must
    each give the device entry point's C bit for bit."""
    for seed in (81, 82):
        A, B = make_matrices(2500, 300, 2600, 0.5, seed)
        hAbig = torch.zeros((300, 2504), dtype=torch.float64)  # column-major 2504 x 300
        hAbig.t()[:2500] = torch.from_numpy(A)
        hBbig = torch.zeros((2600, 304), dtype=torch.float64)  # column-major 304 x 2600
        hBbig.t()[:300] = torch.from_numpy(B)
        hA = hAbig.pin_memory().t()[:2500]
        hB = hBbig.pin_memory().t()[:300]
        assert hA.stride() == (1, 2504) and hB.stride() == (1, 304)
        Ch = oz2.dgemm_host(hA, hB, 14, "fast").numpy()
        Cd = oz2.dgemm(_dev(A), _dev(B), 14, "fast").cpu().numpy()
        np.testing.assert_array_equal(Ch, Cd)
    rng = np.random.default_rng(3)
    ii, jj = rng.integers(0, 2500, 64), rng.integers(0, 2600, 64)
    ref = oracle.oracle_entries(A, B, 14, "fast", ii, jj)
    assert ulp_distance(Ch[ii, jj], ref["C"]) <= ULP_TOL


def test_host_entry_point_four_column_parts(oz2):
    """r = 6000: the host entry point uploads B in four column parts (0, 1536,
    3072, 4608) and splits the first and last row blocks' GEMMs the same way,
    each part's CRT and download running beside the next part's GEMM."""
    A, B = make_matrices(2500, 300, 6000, 0.5, 83)
    hA = torch.from_numpy(np.asfortranarray(A)).pin_memory()
    hB = torch.from_numpy(np.asfortranarray(B)).pin_memory()
    Ch = oz2.dgemm_host(hA, hB, 14, "fast").numpy()
    Cd = oz2.dgemm(_dev(A), _dev(B), 14, "fast").cpu().numpy()
    np.testing.assert_array_equal(Ch, Cd)
    rng = np.random.default_rng(4)
    ii = np.concatenate([rng.integers(0, 2500, 100), [0, 1023, 1024, 2047, 2048, 2499]])
    jj = np.concatenate([rng.integers(0, 6000, 100), [1535, 1536, 3071, 3072, 4607, 4608]])
    ref = oracle.oracle_entries(A, B, 14, "fast", ii, jj)
    assert ulp_distance(Ch[ii, jj], ref["C"]) <= ULP_TOL


@pytest.mark.parametrize("p,q,r", [(5000, 700, 6100), (2049, 3000, 9000), (4100, 2100, 2048)])
def test_host_entry_point_large_strided(oz2, p, q, r):
    """Fast mode with p, r >= 2048 and ragged sizes: the host entry point's
    staged uploads, overlapped row blocks and split first and last blocks
    (A's one-read kernel for q <= 2048, its three kernels above; B's bulk-copy
    statistics).  Strided host A, B and C (lda > p, ldb > q, ldc > p); C must
    equal the device entry point's bit for bit, and sampled entries the
    oracle's, and nothing outside C may be written."""
    A, B = make_matrices(p, q, r, 0.5, 90 + q % 7)
    hAbig = torch.zeros((q, p + 8), dtype=torch.float64)
    hAbig.t()[:p] = torch.from_numpy(A)
    hBbig = torch.zeros((r, q + 4), dtype=torch.float64)
    hBbig.t()[:q] = torch.from_numpy(B)
    hA = hAbig.pin_memory().t()[:p]
    hB = hBbig.pin_memory().t()[:q]
    big = torch.full((r, p + 16), 7.0, dtype=torch.float64).pin_memory()
    hC = big.t()[:p]
    oz2.dgemm_host(hA, hB, 14, "fast", out=hC)
    Cd = oz2.dgemm(_dev(A), _dev(B), 14, "fast").cpu().numpy()
    np.testing.assert_array_equal(hC.numpy(), Cd)
    assert np.all(big.t()[p:].numpy() == 7.0)
    rng = np.random.default_rng(p + r)
    ii = np.concatenate([rng.integers(0, p, 60), [0, 1023, 1024, p - 1]])
    jj = np.concatenate([rng.integers(0, r, 60), [0, 1023, 1024, r - 1]])
    ref = oracle.oracle_entries(A, B, 14, "fast", ii, jj)
    assert ulp_distance(hC.numpy()[ii, jj], ref["C"]) <= ULP_TOL
    assert oz2.last_error() == 0


@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_single_cta_gemm_selection_matches(oz2, mode, monkeypatch):
    """OZ2_GEMM_1SM=1 selects the single-CTA tcgen05 kernel for the modular and
    bound GEMMs (read per call); it must give the CTA-pair kernel's C bit for bit."""
    A, B = make_matrices(700, 600, 530, 1.0, 91)
    dA, dB = _dev(A), _dev(B)
    C2 = oz2.dgemm(dA, dB, 14, mode).cpu().numpy()
    monkeypatch.setenv("OZ2_GEMM_1SM", "1")
    C1 = oz2.dgemm(dA, dB, 14, mode).cpu().numpy()
    monkeypatch.delenv("OZ2_GEMM_1SM")
    np.testing.assert_array_equal(C1, C2)
    assert oz2.last_error() == 0


def test_stage_timing_entry_point(oz2):
    A, B = make_matrices(256, 256, 256, 0.5, 2)
    for mode in ("fast", "accu"):
        C, ms = oz2.dgemm_stages(_dev(A), _dev(B), 14, mode)
        ref = oracle.oracle_dgemm(A, B, 14, mode)
        assert ulp_distance(C.cpu().numpy(), ref["C"]) <= ULP_TOL
        assert ms["total"] > 0 and all(v >= 0 for v in ms.values())


def test_n1024_workload_every_stage(oz2):
    w = WORKLOADS["n1024_s14_fast"]
    A, B = make_workload(w)
    _full_check(oz2, A, B, w.s, w.mode)


def _sampled_check(oz2, name, nsamp=384):
    w = WORKLOADS[name]
    A, B = make_workload(w)
    dA, dB = _dev(A), _dev(B)
    # the launch configuration the benchmark times: the production entry point
    C = oz2.dgemm(dA, dB, w.s, w.mode)
    got = oz2.dgemm_debug(dA, dB, w.s, w.mode, want_p=False)
    torch.cuda.synchronize()
    alpha, beta, _ = oracle.exponents(A, B, w.s, w.mode)
    np.testing.assert_array_equal(got["alpha"].cpu().numpy(), alpha, err_msg="alpha")
    np.testing.assert_array_equal(got["beta"].cpu().numpy(), beta, err_msg="beta")
    rng = np.random.default_rng(99)
    ii = rng.integers(0, w.p, nsamp)
    jj = rng.integers(0, w.r, nsamp)
    ii[:4] = [0, w.p - 1, 0, w.p - 1]
    jj[:4] = [0, 0, w.r - 1, w.r - 1]
    ref = oracle.oracle_entries(A, B, w.s, w.mode, ii, jj, alpha=alpha, beta=beta)
    ti = torch.from_numpy(ii).cuda()
    tj = torch.from_numpy(jj).cuda()
    Cs = C[ti, tj].cpu().numpy()
    assert ulp_distance(Cs, ref["C"]) <= ULP_TOL
    Rs = got["R"][:, tj, ti].cpu().numpy()
    np.testing.assert_array_equal(Rs, ref["R"])
    Xs = got["X"][tj, ti].cpu().numpy()
    for k in range(nsamp):
        assert decode_x(Xs[k]) == ref["X"][k], k
    # residue planes on the sampled rows / columns
    rows = torch.from_numpy(ref["rows"]).cuda()
    cols = torch.from_numpy(ref["cols"]).cuda()
    np.testing.assert_array_equal(got["Ares"][:, rows, :].cpu().numpy(), ref["Arows"])
    np.testing.assert_array_equal(got["Bres"][:, cols, :].cpu().numpy(), np.transpose(ref["Bcols"], (0, 2, 1)))
    assert oz2.last_error() == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["n4096_s14_accu", "n8192_s14_fast", "n8192_s14_accu",
                                  "n8192_s18_fast", "n8192_s18_accu", "p16384_q8192_r16384_s18_accu"])
def test_full_size_workloads_sampled(oz2, name):
    _sampled_check(oz2, name)


# Products below 2^35 multiply-adds in fast mode (2^32 in accu mode) run as one
# row block; these shapes sit above those sizes so that the overlapped
# schedule runs.
OVERLAP_SHAPES = {"fast": (2500, 5600, 2500), "accu": (2500, 900, 2000)}


def _sampled_entries(p, r, seed, extra_i=(), extra_j=()):
    rng = np.random.default_rng(seed)
    ii = np.concatenate([rng.integers(0, p, 200), [0, p - 1, *extra_i]])
    jj = np.concatenate([rng.integers(0, r, 200), [r - 1, 0, *extra_j]])
    return ii.astype(np.int64), jj.astype(np.int64)


@pytest.mark.parametrize("mode", ["fast", "accu"])
def test_overlapped_row_blocks_match_sequential(oz2, mode):
    """p = 2500 gives three row blocks (1024, 1024, 452) in the overlapped schedule."""
    p, q, r = OVERLAP_SHAPES[mode]
    assert p * q * r >= (2**35 if mode == "fast" else 2**32)
    A, B = make_matrices(p, q, r, 1.0, 77)
    dA, dB = _dev(A), _dev(B)
    got = oz2.dgemm_debug(dA, dB, 14, mode, want_p=False)  # stages one after another
    C = oz2.dgemm(dA, dB, 14, mode)                          # overlapped row blocks
    torch.cuda.synchronize()
    Cn = C.cpu().numpy()
    np.testing.assert_array_equal(Cn, got["C"].cpu().numpy())
    ref_a, ref_b, _ = oracle.exponents(A, B, 14, mode)
    np.testing.assert_array_equal(got["alpha"].cpu().numpy(), ref_a)
    np.testing.assert_array_equal(got["beta"].cpu().numpy(), ref_b)
    ii, jj = _sampled_entries(p, r, 6, [1023, 1024, 2047, 2048], [1, 2, 3, 4])
    ref = oracle.oracle_entries(A, B, 14, mode, ii, jj, alpha=ref_a, beta=ref_b)
    assert ulp_distance(Cn[ii, jj], ref["C"]) <= ULP_TOL
    Rn = got["R"].cpu().numpy()  # [s][r][p]
    np.testing.assert_array_equal(Rn[:, jj, ii], ref["R"])


def test_overlapped_first_block_column_parts(oz2):
    """r = 2500: the first row block's GEMM runs as two column parts (0..1535,
    1536..2499), the first starting once B's first columns are ready."""
    p, q, r = OVERLAP_SHAPES["fast"]
    A, B = make_matrices(p, q, r, 0.5, 78)
    dA, dB = _dev(A), _dev(B)
    got = oz2.dgemm_debug(dA, dB, 14, "fast", want_p=False)  # stages one after another
    C = oz2.dgemm(dA, dB, 14, "fast")                          # overlapped schedule
    torch.cuda.synchronize()
    Cn = C.cpu().numpy()
    np.testing.assert_array_equal(Cn, got["C"].cpu().numpy())
    alpha, beta = got["alpha"].cpu().numpy(), got["beta"].cpu().numpy()
    ref_a, ref_b, _ = oracle.exponents(A, B, 14, "fast")
    np.testing.assert_array_equal(alpha, ref_a)
    np.testing.assert_array_equal(beta, ref_b)
    ii, jj = _sampled_entries(p, r, 5, [1023, 1024], [1535, 1536])
    ref = oracle.oracle_entries(A, B, 14, "fast", ii, jj, alpha=ref_a, beta=ref_b)
    assert ulp_distance(Cn[ii, jj], ref["C"]) <= ULP_TOL


def test_host_entry_point_overlapped_blocks(oz2):
    """p = 2500: row blocks overlap, C returns block by block into a host C with ldc > p."""
    A, B = make_matrices(2500, 200, 150, 0.5, 66)
    hA = torch.from_numpy(np.asfortranarray(A)).pin_memory()
    hB = torch.from_numpy(np.asfortranarray(B)).pin_memory()
    big = torch.full((150, 2600), 3.0, dtype=torch.float64).pin_memory()  # column-major (2600 x 150), ldc 2600
    hC = big.t()[:2500]
    assert hC.stride() == (1, 2600)
    oz2.dgemm_host(hA, hB, 14, "fast", out=hC)
    ref = oracle.oracle_dgemm(A, B, 14, "fast")
    assert ulp_distance(hC.numpy(), ref["C"]) <= ULP_TOL
    assert np.all(big.t()[2500:].numpy() == 3.0)
    dev = oz2.dgemm(_dev(A), _dev(B), 14, "fast").cpu().numpy()
    np.testing.assert_array_equal(hC.numpy(), dev)


@pytest.mark.parametrize("p,q,r,mode", [(1024, 1024, 1024, "fast"), (2500, 5600, 2500, "fast"),
                                        (2500, 900, 2000, "accu")])
def test_cuda_graph_capture_replays_the_call(oz2, p, q, r, mode):
    """One ozaki2_dgemm call captured into a CUDA graph on a stream whose
    workspace exists already (a first call grows it; capture allocates
    nothing).  The overlapped schedule forks onto the library's second and
    GEMM streams through events, which the capture follows; replays must give
    the direct call's C bit for bit."""
    A, B = make_matrices(p, q, r, 0.5, 31)
    dA, dB = _dev(A), _dev(B)
    ref = oz2.dgemm(dA, dB, 14, mode).cpu().numpy()
    st = torch.cuda.Stream()
    C = torch.full((r, p), float("nan"), dtype=torch.float64, device="cuda").t()
    with torch.cuda.stream(st):
        oz2.dgemm(dA, dB, 14, mode, out=C)  # sizes this stream's workspace, creates its streams
    st.synchronize()
    C.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        oz2.dgemm(dA, dB, 14, mode, out=C)
    for _ in range(2):
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(C.cpu().numpy(), ref)
    assert oz2.last_error() == 0


def test_workspace_release_and_recreate(oz2):
    """ozaki2_workspace_release frees the workspaces and destroys the library's
    streams and events; the next call builds them again and gives the same C."""
    A, B = make_matrices(2500, 900, 2000, 0.5, 41)  # accu: above the one-block size, overlapped
    dA, dB = _dev(A), _dev(B)
    C0 = oz2.dgemm(dA, dB, 14, "accu").cpu().numpy()
    oz2.workspace_release()
    C1 = oz2.dgemm(dA, dB, 14, "accu").cpu().numpy()
    np.testing.assert_array_equal(C1, C0)
    oz2.workspace_release()
    C2 = oz2.dgemm(dA, dB, 14, "fast").cpu().numpy()
    ref = oracle.oracle_entries(A, B, 14, "fast", np.arange(0, 2500, 97), np.arange(0, 2000, 79)[:26])
    assert ulp_distance(C2[np.arange(0, 2500, 97), np.arange(0, 2000, 79)[:26]], ref["C"]) <= ULP_TOL
    assert oz2.last_error() == 0


@pytest.mark.parametrize("s", list(range(2, 21)))
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_crt_at_the_edge_of_its_range(oz2, s, sign):
    """X next to +-M/2, where the CRT's quotient estimate can round to the
    wrong side and the exact comparison with M/2 must correct it.

    A is a row of q ones and B a column of q (+-)ones.  The fast bound of
    "Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" §5.1 sees e = 1 and
    q terms ceil(1 * 2^19)^2, so U = q and alpha = beta = a with
    a = max {a : 4^a q <= L}.  With q = floor(L / 4^a0) the product
    X = A'B' = +-q 4^a (§1) lies within 4^a of L = M/2 - 1, about M/(2q)
    below M/2, closer than the float estimate of X/M resolves; C = +-q."""
    ms = oracle.greedy_moduli(s)
    M = 1
    for m in ms:
        M *= m
    L = M // 2 - 1
    a0 = 0
    while L // 4 ** (a0 + 1) >= 1 and L // 4 ** a0 >= 2**23:
        a0 += 1
    q = L // 4**a0
    a = 0
    while 4 ** (a + 1) * q <= L:
        a += 1
    assert a == a0 and 0 <= L - q * 4**a < 4**a
    A = np.ones((1, q))
    B = np.full((q, 1), sign)
    got = oz2.dgemm_debug(_dev(A), _dev(B), s, "fast", want_p=False)
    torch.cuda.synchronize()
    assert got["alpha"].cpu().numpy()[0] == a and got["beta"].cpu().numpy()[0] == a
    x = decode_x(got["X"].cpu().numpy()[0, 0])
    assert x == int(sign) * q * 4**a
    assert got["C"].cpu().numpy()[0, 0] == sign * q
    C = oz2.dgemm(_dev(A), _dev(B), s, "fast").cpu().numpy()
    assert C[0, 0] == sign * q
    assert oz2.last_error() == 0
