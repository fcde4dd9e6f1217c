"""Parity of the fused narrow-N path (n <= 2 columns) with the oracle.

For n <= 2, ``ozemu_dgemm`` deconstructs the rows of A in registers and
dots them with B's residues directly (no limb planes); the residues it hands
to the CRT and the fp64 result must equal the oracle's bit for bit, and equal
the limb-plane path's (``OZEMU_NARROW=0``).  Cases cover both integer widths
of the kernel (p_A <= 40: two 21-bit chunks; up to 52: three), ragged K (not a
multiple of 8 or 16), padded leading dimensions of A, B and C, special and
subnormal values, overflow, and the non-finite flag from either operand.
"""

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


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def run(oz, A, B, r, pads=(0, 0, 0)):
    """C = A B through ozemu_dgemm with padded leading dimensions."""
    m, k = A.shape
    n = B.shape[1]
    pa, pb, pc = pads
    Ad = torch.zeros((m, k + pa), dtype=torch.float64, device=DEV)
    Ad[:, :k] = to_dev(A)
    Bd = torch.zeros((k, n + pb), dtype=torch.float64, device=DEV)
    Bd[:, :n] = to_dev(B)
    Cd = torch.full((m, n + pc), 7.0, dtype=torch.float64, device=DEV)
    oz.dgemm(Ad[:, :k], Bd[:, :n], r, out=Cd[:, :n])
    st = oz.get_status()
    C = Cd.cpu().numpy()
    if pc:
        assert (C[:, n:] == 7.0).all()
    return st, C[:, :n].copy()


def same_bits(x, y):
    return (np.ascontiguousarray(x).view(np.int64) == np.ascontiguousarray(y).view(np.int64)).all()


# bound: whether r leaves enough bits for the per-entry bound on these inputs
# (the oracle's own ratio; with too few moduli, or wide-range rows at tiny K,
# the scaling error exceeds it while the integer stages stay exact).
@pytest.mark.parametrize("m,n,k,r,dist,bound", [
    (300, 1, 1000, 11, "normal", False),   # p_A = 38: two chunks
    (300, 1, 1000, 13, "normal", True),    # p_A = 46: three chunks
    (257, 2, 777, 12, "wide", False),
    (129, 2, 1000, 11, "uniform", False),
    (1, 1, 1, 16, "uniform", True),        # p_A = 62: ozemu_dgemm takes the limb planes
    (33, 2, 5, 16, "wide", False),         # p_A = 61: likewise
    (40, 2, 40, 14, "wide", False),        # p_A = 52: the fused path's widest budget
    (40, 1, 30, 14, "normal", True),       # p_A = 52
    (40, 1, 10, 14, "normal", False),      # p_A = 53: ozemu_dgemm takes the limb planes
    (64, 1, 999, 13, "wide", True),
    (70, 1, 20000, 12, "normal", False),   # longer than one FP4 K chunk
    (1000, 1, 3001, 12, "normal", False),
])
def test_narrow_dgemm_parity(oz, m, n, k, r, dist, bound):
    A, B = make_pair(m, n, k, seed=7 * m + n + k, dist=dist)
    st, C = run(oz, A, B, r, pads=(3, 1, 2))
    assert st == oz.OZEMU_OK
    Cref = oracle.dgemm(A, B, r)
    assert same_bits(C, Cref)
    if bound:
        assert oracle.error_bound_ratio(A, B, C) <= 1.0


@pytest.mark.parametrize("m,n,k,r", [(300, 1, 1000, 11), (130, 2, 2001, 13)])
def test_narrow_stage_call_residues(oz, m, n, k, r):
    A, B = make_pair(m, n, k, seed=m + k, dist="wide")
    res, sa, sb = oz.residues_narrow_f64(to_dev(A), to_dev(B), r)
    assert oz.get_status() == oz.OZEMU_OK
    Cref, st = oracle.dgemm(A, B, r, stages=True)
    _, pA, pB = oracle.bit_budget(k, r)
    assert (sa.cpu().numpy() == oracle.row_shifts(A, pA)).all()
    assert (sb.cpu().numpy() == oracle.row_shifts(B.T, pB)).all()
    assert (res.cpu().numpy()[:, :, :n].astype(np.int64) == st["res"]).all()
    C = oz.crt_f64(m, n, r, res, sa, sb)
    assert oz.get_status() == oz.OZEMU_OK
    assert same_bits(C.cpu().numpy(), Cref)


@pytest.mark.parametrize("n", [1, 2])
def test_narrow_matches_limb_plane_path(oz, n, monkeypatch):
    A, B = make_pair(400, n, 2500, seed=40 + n, dist="wide")
    st, C_narrow = run(oz, A, B, 13)
    assert st == oz.OZEMU_OK
    monkeypatch.setenv("OZEMU_NARROW", "0")
    st, C_planes = run(oz, A, B, 13)
    assert st == oz.OZEMU_OK
    assert same_bits(C_narrow, C_planes)


def test_narrow_special_values(oz):
    A, _ = make_pair(40, 1, 64, seed=11, dist="wide")
    A[0, :8] = [0.5, 1.5, 2.5, -2.5, 3.5, 2.0 ** -1074, -1e-310, 0.0]
    A[2] = 0.0
    A[3] = 2.0 ** -1060 * np.arange(1, 65)
    A[4] = 1e300 * np.sign(A[4])
    B = np.zeros((64, 2))
    B[:, 0] = np.linspace(-3.0, 5.0, 64)
    B[:, 1] = 2.0 ** -1000 * np.arange(64)     # a column at subnormal scale
    B[5, 1] = 0.0
    for r in (13, 16):
        st, C = run(oz, A, B, r)
        assert st == oz.OZEMU_OK
        assert same_bits(C, oracle.dgemm(A, B, r))


def test_narrow_zero_column_and_rows(oz):
    A, B = make_pair(20, 2, 100, seed=3, dist="normal")
    B[:, 1] = 0.0
    A[7] = 0.0
    st, C = run(oz, A, B, 12)
    assert st == oz.OZEMU_OK
    assert same_bits(C, oracle.dgemm(A, B, 12))
    assert (C[:, 1] == 0).all() and (C[7] == 0).all()


def test_narrow_subnormal_results_and_overflow(oz):
    A = np.full((4, 4), 2.0 ** -540)
    B = (np.full((4, 1), 2.0 ** -540).T * np.array([1.0, 3.0, 0.75, -1.25])).T
    st, C = run(oz, A, B, 16)
    assert st == oz.OZEMU_OK
    assert same_bits(C, oracle.dgemm(A, B, 16))
    A = np.full((2, 2), 1.5e154)
    B = np.full((2, 1), -1.5e154)
    st, C = run(oz, A, B, 16)
    assert st == oz.OZEMU_OK
    assert np.isneginf(C).all()
    assert same_bits(C, oracle.dgemm(A, B, 16))


@pytest.mark.parametrize("where", ["A", "B"])
def test_narrow_nonfinite_flag(oz, where):
    A, B = make_pair(8, 1, 16, seed=1, dist="normal")
    if where == "A":
        A[3, 5] = np.nan
    else:
        B[9, 0] = -np.inf
    st, _ = run(oz, A, B, 13)
    assert st == oz.OZEMU_ERR_NONFINITE
    assert oz.get_status() == oz.OZEMU_OK
