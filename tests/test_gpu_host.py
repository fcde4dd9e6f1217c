"""ozemu_dgemm_host: the product with host buffers, against the oracle.

The result must equal the oracle's bit for bit (and ozemu_dgemm's) for
pinned and pageable buffers, padded leading dimensions, row counts that
split into ragged chunks, B wide enough to come over in column blocks,
narrow B (the fused path), k = 0, and two calls in a row on one stream (the
second must not overwrite the first's workspace while it is in use).
"""

import numpy as np
import pytest

import oracle
from workloads import make_pair

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def oz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ozaki_ii_fp64_gb300 as oz
    oz.load()
    return oz


def host(x, pinned, pad=0):
    t = torch.zeros((x.shape[0], x.shape[1] + pad), dtype=torch.float64)
    t[:, :x.shape[1]] = torch.from_numpy(np.ascontiguousarray(x))
    t = t.pin_memory() if pinned else t
    return t[:, :x.shape[1]]


def same_bits(x, y):
    return (np.ascontiguousarray(x).view(np.int64) == np.ascontiguousarray(y).view(np.int64)).all()


@pytest.mark.parametrize("m,n,k,r,pinned", [
    (2300, 130, 700, 13, True),   # four ragged row chunks
    (2048, 300, 257, 12, False),  # pageable buffers
    (300, 250, 1000, 13, True),   # one chunk
    (700, 2, 900, 12, True),      # narrow B: the fused path
    (3000, 70, 9000, 12, True),   # chunked K inside each row chunk
    (2100, 4500, 300, 13, True),  # B in two column blocks (ragged second block)
    (4100, 4200, 200, 12, False), # eight row chunks x two column blocks, pageable
])
def test_dgemm_host_matches_oracle(oz, m, n, k, r, pinned):
    A, B = make_pair(m, n, k, seed=m + 3 * n + k, dist="wide")
    Ah, Bh = host(A, pinned, pad=3), host(B, pinned, pad=1)
    Ch = host(np.full((m, n), 7.0), pinned, pad=2)
    oz.dgemm_host(Ah, Bh, r, out=Ch)
    assert oz.get_status() == oz.OZEMU_OK
    rows = np.arange(m) if m * n * k <= 300 * 250 * 1000 else np.unique(np.r_[0:5, m // 2, m - 5:m])
    Cref = oracle.dgemm_block(A, B, r, rows=rows)
    assert same_bits(Ch.numpy()[rows], Cref)
    Cd = oz.dgemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), r)
    assert same_bits(Ch.numpy(), Cd.cpu().numpy())


def test_dgemm_host_k0_and_repeated_calls(oz):
    A = host(np.zeros((5, 0)), True)
    B = host(np.zeros((0, 4)), True)
    C = oz.dgemm_host(A, B, 13)
    assert (C.numpy() == 0).all()
    A1, B1 = make_pair(2100, 90, 300, seed=1, dist="normal")
    A2, B2 = make_pair(2100, 90, 300, seed=2, dist="normal")
    C1 = host(np.zeros((2100, 90)), True)
    C2 = host(np.zeros((2100, 90)), True)
    s = torch.cuda.current_stream()
    for (A_, B_, C_) in ((A1, B1, C1), (A2, B2, C2)):
        Ah, Bh = host(A_, True), host(B_, True)
        assert oz.ozemu_dgemm_host(2100, 90, 300, Ah.data_ptr(), 300, Bh.data_ptr(), 90, C_.data_ptr(), 90, 13,
                                   s.cuda_stream) == oz.OZEMU_OK
    s.synchronize()
    for (A_, B_, C_) in ((A1, B1, C1), (A2, B2, C2)):
        rows = np.array([0, 1, 1000, 2099])
        assert same_bits(C_.numpy()[rows], oracle.dgemm_block(A_, B_, 13, rows=rows))


@pytest.mark.parametrize("m,n,k,r", [(2300, 130, 700, 13), (4100, 257, 300, 12)])
def test_dgemm_device_chunked(oz, m, n, k, r):
    # ozemu_dgemm pipelines row chunks of A on helper streams when m >= 2048;
    # padded leading dimensions of A and C, rows checked against the oracle.
    A, B = make_pair(m, n, k, seed=5 * m + n, dist="wide")
    Ad = torch.zeros((m, k + 5), dtype=torch.float64, device="cuda")
    Ad[:, :k] = torch.from_numpy(A).cuda()
    Cd = torch.full((m, n + 3), 7.0, dtype=torch.float64, device="cuda")
    oz.dgemm(Ad[:, :k], torch.from_numpy(B).cuda(), r, out=Cd[:, :n])
    assert oz.get_status() == oz.OZEMU_OK
    C = Cd.cpu().numpy()
    assert (C[:, n:] == 7.0).all()
    rows = np.unique(np.r_[0:3, m // 4 - 1: m // 4 + 2, m // 2, 3 * m // 4, m - 3:m])
    assert same_bits(C[rows, :n], oracle.dgemm_block(A, B, r, rows=rows))
