"""The allocation-free DGEMM entry point against the allocating one.

ozemu_dgemm_noalloc serves callers that cannot allocate device memory (a
framework that reserves the GPU's memory up front, or code where an
allocation's implicit device synchronisation or failure is not acceptable).
It keeps all its scratch in one fixed static device array.  These checks call
it through the C ABI twice in a row on different inputs, so a second call
cannot lean on what the first left in the shared array, and compare each
result bit for bit with ozemu_dgemm, the tolerance every fp64 parity test here
uses; the first result is also compared with the CPU oracle directly.  The
status word the call keeps in its array is read with ozemu_get_status_noalloc
(which allocates nothing either): a non-finite input sets it, and the next
clean call starts from a cleared word.  The file is named to be collected
last.
"""

import numpy as np
import pytest

import oracle
from workloads import make_pair

NULL = None
FAKE = 0x10000  # non-null, never dereferenced (rejected before any device work)


def test_noalloc_rejects_problems_beyond_its_scratch():
    import ozaki_ii_fp64_gb300 as oz
    oz.load()
    st = oz.ozemu_dgemm_noalloc(2048, 2048, 2048, FAKE, 2048, FAKE, 2048, FAKE, 2048, 13, NULL)
    assert st == oz.OZEMU_ERR_SCRATCH_TOO_SMALL
    assert oz.ozemu_dgemm_noalloc(4, 4, 4, FAKE, 3, FAKE, 4, FAKE, 4, 13, NULL) == oz.OZEMU_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_dgemm_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ozaki_ii_fp64_gb300 as oz
    oz.load()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    cases = [(300, 170, 1000, 13, "wide", 1), (1024, 1024, 1024, 13, "uniform", 2)]
    for m, n, k, r, dist, seed in cases:
        A_h, B_h = make_pair(m, n, k, seed=seed, dist=dist)
        A = torch.from_numpy(A_h).to(dev)
        B = torch.from_numpy(B_h).to(dev)
        C_ref = torch.empty((m, n), dtype=torch.float64, device=dev)
        C_new = torch.full((m, n), np.nan, dtype=torch.float64, device=dev)
        assert oz.ozemu_dgemm(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C_ref.data_ptr(), n, r, stream) == 0
        assert oz.ozemu_dgemm_noalloc(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C_new.data_ptr(), n, r,
                                      stream) == 0
        torch.cuda.synchronize(dev)
        assert oz.ozemu_get_status(stream) == 0          # the allocating call's flags
        assert oz.ozemu_get_status_noalloc(stream) == 0  # the allocation-free call's word
        assert torch.equal(C_new.view(torch.int64), C_ref.view(torch.int64))
        if seed == 1:
            want = oracle.dgemm(A_h, B_h, r)
            assert (C_new.cpu().numpy().view(np.int64) == want.view(np.int64)).all()


@pytest.mark.gpu
def test_noalloc_status_word_reports_nonfinite_and_is_cleared():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ozaki_ii_fp64_gb300 as oz
    oz.load()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    m, n, k, r = 200, 150, 300, 13
    A_h, B_h = make_pair(m, n, k, seed=5, dist="normal")
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    C = torch.empty((m, n), dtype=torch.float64, device=dev)
    A_bad = A.clone()
    A_bad[17, 33] = float("inf")
    assert oz.ozemu_dgemm_noalloc(m, n, k, A_bad.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, r, stream) == 0
    assert oz.ozemu_get_status_noalloc(stream) == oz.OZEMU_ERR_NONFINITE
    # the allocating path's flags are untouched by the noalloc call
    assert oz.ozemu_get_status(stream) == 0
    # reading the word cleared it, and the next call clears it again first:
    # a clean call after a non-finite one reports OK and the right product
    assert oz.ozemu_dgemm_noalloc(m, n, k, A_bad.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, r, stream) == 0
    assert oz.ozemu_dgemm_noalloc(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, r, stream) == 0
    assert oz.ozemu_get_status_noalloc(stream) == 0
    C_ref = oz.dgemm(A, B, r)
    assert oz.ozemu_get_status(stream) == 0
    assert torch.equal(C.view(torch.int64), C_ref.view(torch.int64))
