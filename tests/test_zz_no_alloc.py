"""The allocation-free DGEMM entry point against the allocating one.

ozemu_dgemm_noalloc serves callers that cannot allocate device memory (a
framework that reserves the GPU's memory up front, or code where an
allocation's implicit device synchronisation or failure is not acceptable).
It keeps all its scratch in one fixed static device array.  These checks call
it through the C ABI twice in a row on different inputs, so a second call
cannot lean on what the first left in the shared array, and compare each
result bit for bit with ozemu_dgemm, the tolerance every fp64 parity test here
uses.  The file is named to be collected last.
"""

import numpy as np
import pytest

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
        assert oz.ozemu_get_status(stream) == 0
        assert torch.equal(C_new.view(torch.int64), C_ref.view(torch.int64))
