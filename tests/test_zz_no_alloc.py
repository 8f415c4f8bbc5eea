"""The entry point that allocates no device memory.

Frameworks that hand out all device memory from their own pool, loops that
must not block on cudaMalloc and plug-ins barred from the allocator call
ozaki2_fast_exponents_noalloc instead of letting the library allocate a
workspace.  It must give exactly the fast-mode exponents that ozaki2_dgemm
itself uses (reported by ozaki2_dgemm_debug), call after call, although every
call reuses the same fixed scratch array.
"""
import ctypes

import numpy as np
import pytest

from workloads import make_matrices

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OZ2_ERR_SCRATCH_TOO_SMALL = 7
MAX_VECTORS = 1 << 20


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g

    g.build()
    import emulated_fp64_gemm_gb300 as oz2

    lib = oz2.load_library()
    f = lib.ozaki2_fast_exponents_noalloc
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    f.argtypes = [i64, i64, i64, vp, i64, vp, i64, ctypes.c_int, vp, vp, vp]
    f.restype = ctypes.c_int
    return lib


def _dev(x):
    return torch.from_numpy(np.asfortranarray(x)).cuda()


def _noalloc(lib, dA, dB, s):
    p, q = dA.shape
    r = dB.shape[1]
    alpha = torch.full((p,), -7, dtype=torch.int32, device="cuda")
    beta = torch.full((r,), -7, dtype=torch.int32, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.ozaki2_fast_exponents_noalloc(p, q, r, dA.data_ptr(), dA.stride(1), dB.data_ptr(),
                                           dB.stride(1), s, alpha.data_ptr(), beta.data_ptr(), st)
    assert rc == 0
    torch.cuda.synchronize()
    return alpha.cpu().numpy(), beta.cpu().numpy()


def test_noalloc_exponents_match_the_pipeline_on_consecutive_calls(lib):
    import emulated_fp64_gemm_gb300 as oz2

    # a larger call first, then a smaller one: stale scratch must not leak into the second
    cases = [(make_matrices(700, 900, 500, 2.0, 11), 14), (make_matrices(300, 257, 129, 0.5, 12), 18)]
    for (A, B), s in cases:
        dA, dB = _dev(A), _dev(B)
        got_a, got_b = _noalloc(lib, dA, dB, s)
        ref = oz2.dgemm_debug(dA, dB, s, "fast", want_p=False)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got_a, ref["alpha"].cpu().numpy())
        np.testing.assert_array_equal(got_b, ref["beta"].cpu().numpy())


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    dA = torch.zeros((4, 4), dtype=torch.float64, device="cuda")
    st = ctypes.c_void_p(0)
    out = torch.zeros(8, dtype=torch.int32, device="cuda")
    rc = lib.ozaki2_fast_exponents_noalloc(MAX_VECTORS, 1, 1, dA.data_ptr(), MAX_VECTORS,
                                           dA.data_ptr(), 1, 14, out.data_ptr(), out.data_ptr(), st)
    assert rc == OZ2_ERR_SCRATCH_TOO_SMALL


def test_noalloc_call_leaves_free_device_memory_unchanged(lib):
    """After a first call (which looks up the scratch array and loads the
    kernels), a further call must not change the device's free memory: it
    allocates nothing, neither through the CUDA runtime nor through torch."""
    A, B = make_matrices(640, 512, 384, 1.0, 13)
    dA, dB = _dev(A), _dev(B)
    alpha = torch.empty(640, dtype=torch.int32, device="cuda")
    beta = torch.empty(384, dtype=torch.int32, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        rc = lib.ozaki2_fast_exponents_noalloc(640, 512, 384, dA.data_ptr(), dA.stride(1), dB.data_ptr(),
                                               dB.stride(1), 14, alpha.data_ptr(), beta.data_ptr(), st)
        assert rc == 0
        torch.cuda.synchronize()

    call()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(3):
        call()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0


def test_noalloc_at_its_scratch_limit(lib):
    """p + r equal to the limit is accepted and gives the pipeline's exponents."""
    import emulated_fp64_gemm_gb300 as oz2

    r = 8
    p = MAX_VECTORS - r
    rng = np.random.default_rng(14)
    A = (rng.random((p, 3)) - 0.5) * np.exp(rng.standard_normal((p, 3)))
    B = (rng.random((3, r)) - 0.5) * np.exp(rng.standard_normal((3, r)))
    dA, dB = _dev(A), _dev(B)
    got_a, got_b = _noalloc(lib, dA, dB, 14)
    ref = oz2.dgemm_debug(dA, dB, 14, "fast", want_p=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got_a, ref["alpha"].cpu().numpy())
    np.testing.assert_array_equal(got_b, ref["beta"].cpu().numpy())
    # one more vector is refused before anything is enqueued
    out = torch.zeros(8, dtype=torch.int32, device="cuda")
    rc = lib.ozaki2_fast_exponents_noalloc(p + 1, 3, r, dA.data_ptr(), p + 1, dB.data_ptr(), 3, 14,
                                           out.data_ptr(), out.data_ptr(), ctypes.c_void_p(0))
    assert rc == OZ2_ERR_SCRATCH_TOO_SMALL
