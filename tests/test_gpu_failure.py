"""Failure detection on the device, without a GPU fault.

* The bounded pipeline wait: ozemu_probe_wait_timeout makes one thread wait,
  with a short limit, on an mbarrier phase that nothing completes (no copy or
  tensor operation in flight).  The wait must give up, the next
  ozemu_get_status must report OZEMU_ERR_TIMEOUT and clear it, and the
  context must stay usable: a product afterwards is bit-exact.
* A forced allocation failure: with a workspace cap below what a product
  needs, the call returns OZEMU_ERR_ALLOC before enqueueing anything; with
  the cap removed the same call succeeds.
"""

import time

import numpy as np
import pytest

import oracle
from workloads import make_pair

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def oz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ozaki_ii_fp64_gb300 as oz
    oz.load()
    return oz


def _product_ok(oz, seed):
    A_h, B_h = make_pair(130, 90, 257, seed=seed, dist="wide")
    C = oz.dgemm(torch.from_numpy(A_h).to(DEV), torch.from_numpy(B_h).to(DEV), 13)
    assert oz.get_status() == oz.OZEMU_OK
    return (C.cpu().numpy().view(np.int64) == oracle.dgemm(A_h, B_h, 13).view(np.int64)).all()


def test_bounded_wait_gives_up_and_reports_timeout(oz):
    assert _product_ok(oz, 1)
    s = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    assert oz.ozemu_probe_wait_timeout(2_000_000, s) == oz.OZEMU_OK  # 2 ms limit
    assert oz.ozemu_get_status(s) == oz.OZEMU_ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    assert oz.ozemu_get_status(s) == oz.OZEMU_OK  # cleared by the read
    assert _product_ok(oz, 2)                        # the context is still usable


def test_probe_rejects_out_of_range_limits(oz):
    s = torch.cuda.current_stream().cuda_stream
    assert oz.ozemu_probe_wait_timeout(0, s) == oz.OZEMU_ERR_INVALID_ARG
    assert oz.ozemu_probe_wait_timeout(2_000_000_000, s) == oz.OZEMU_ERR_INVALID_ARG


def test_workspace_cap_forces_alloc_failure(oz):
    s = torch.cuda.current_stream().cuda_stream
    m = n = k = 512
    A_h, B_h = make_pair(m, n, k, seed=3, dist="uniform")
    A = torch.from_numpy(A_h).to(DEV)
    B = torch.from_numpy(B_h).to(DEV)
    C = torch.full((m, n), np.nan, dtype=torch.float64, device=DEV)
    try:
        assert oz.ozemu_set_workspace_limit(1 << 20) == oz.OZEMU_OK  # 1 MiB: far below what 512^3 needs
        assert oz.ozemu_workspace_limit() == 1 << 20
        st = oz.ozemu_dgemm(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, 13, s)
        assert st == oz.OZEMU_ERR_ALLOC
        torch.cuda.synchronize()
        assert torch.isnan(C).all()  # nothing was enqueued
    finally:
        assert oz.ozemu_set_workspace_limit(0) == oz.OZEMU_OK
    assert oz.ozemu_dgemm(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, 13, s) == oz.OZEMU_OK
    assert oz.ozemu_get_status(s) == oz.OZEMU_OK
    assert (C.cpu().numpy().view(np.int64) == oracle.dgemm(A_h, B_h, 13).view(np.int64)).all()
