"""Parity of the two-limb CUDA path (moduli up to 113, 4 FP4 products per
modulus) with the oracle run at the same modulus ceiling.

Digits, shifts and residues must match bit for bit; the fp64 product must
equal the oracle's single correct rounding of C' 2^-(s_i + t_j) bit for bit.
"""

import numpy as np
import pytest

import oracle
from planes import decode_planes
from workloads import make_pair, sample_indices

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CEIL = oracle.MODULUS_CEILING_2LIMB


@pytest.fixture(scope="module")
def oz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ozaki_ii_fp64_gb300 as oz
    oz.load()
    return oz


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def status_ok(oz):
    assert oz.get_status() == oz.OZEMU_OK


def special_matrix(rows, k, seed):
    A, _ = make_pair(rows, 1, k, seed=seed, dist="wide")
    vals = [0.5, 1.5, 2.5, -2.5, 3.5, 2.0 ** -1074, -1e-310, 0.0]
    A[0, :min(8, k)] = vals[:min(8, k)]
    if rows > 2:
        A[2] = 0.0
    if rows > 3:
        A[3, :] = 2.0 ** -1060 * np.arange(1, k + 1)
    if rows > 4:
        A[4, :] = 1e300 * np.sign(A[4])
    return A


def oracle_dgemm(A, B, r, stages=False):
    return oracle.dgemm(A, B, r, stages=stages, ceiling=CEIL)


# ---------------------------------------------------------------- splits

@pytest.mark.parametrize("rows,k,p,r,pad", [(300, 1000, 40, 16, 0), (1, 1, 62, 16, 0), (129, 257, 30, 5, 0),
                                           (77, 1000, 40, 16, 2), (50, 3000, 36, 12, 1)])
def test_split_rows_two_limb_parity(oz, rows, k, p, r, pad):
    A = special_matrix(rows, k, seed=rows + k + 1)
    Ad = torch.zeros((rows, k + pad), dtype=torch.float64, device=DEV)
    Ad[:, :k] = to_dev(A)
    planes, shifts = oz.split_rows_f64_2limb(Ad[:, :k], p, r)
    status_ok(oz)
    assert planes.numel() == oz.ozemu_plane_bytes_2limb(rows, k, r)
    ref = oracle.deconstruct(A, p, r, CEIL)
    assert (ref["digits"][:, 2] == 0).all()
    assert (shifts.cpu().numpy() == ref["shift"]).all()
    digits, codes = decode_planes(planes.cpu().numpy(), rows, k, r, limbs=2)
    assert (digits[:, :, :rows, :k] == ref["digits"][:, :2]).all()
    assert (codes[:, :, rows:, :] == 0).all() and (codes[:, :, :, k:] == 0).all()


@pytest.mark.parametrize("k,cols,p,r", [(777, 200, 36, 16), (5, 3, 20, 4)])
def test_split_cols_two_limb_parity(oz, k, cols, p, r):
    B = special_matrix(cols, k, seed=cols * 5 + k).T.copy()
    planes, shifts = oz.split_cols_f64_2limb(to_dev(B), p, r)
    status_ok(oz)
    ref = oracle.deconstruct(B.T, p, r, CEIL)
    assert (shifts.cpu().numpy() == ref["shift"]).all()
    digits, codes = decode_planes(planes.cpu().numpy(), cols, k, r, limbs=2)
    assert (digits[:, :, :cols, :k] == ref["digits"][:, :2]).all()
    assert (codes[:, :, cols:, :] == 0).all() and (codes[:, :, :, k:] == 0).all()


# ---------------------------------------------------------- residues, CRT

@pytest.mark.parametrize("m,n,k,r,dist", [(200, 150, 300, 16, "uniform"), (130, 20, 1000, 14, "wide"),
                                          (64, 64, 9000, 12, "normal"), (257, 230, 2000, 16, "wide")])
def test_residue_gemm_two_limb_parity(oz, m, n, k, r, dist):
    A, B = make_pair(m, n, k, seed=m + n + k + 3, dist=dist)
    pA, pB = oz.ozemu_bit_budget_2limb(k, r)
    ap, sa = oz.split_rows_f64_2limb(to_dev(A), pA, r)
    bp, sb = oz.split_cols_f64_2limb(to_dev(B), pB, r)
    res = oz.residue_gemm_2limb(m, n, k, r, ap, bp)
    C = oz.crt_f64_2limb(m, n, r, res, sa, sb)
    status_ok(oz)
    Cref, st = oracle_dgemm(A, B, r, stages=True)
    got = res.cpu().numpy()[:, :, :n].astype(np.int64)
    assert (got == st["res"]).all()
    assert (C.cpu().numpy().view(np.int64) == Cref.view(np.int64)).all()


@pytest.mark.parametrize("m,n,k,r", [(200, 150, 300, 16), (513, 257, 4000, 15), (256, 230, 4097, 16),
                                     (130, 250, 20000, 12)])
def test_two_limb_pair_and_single_cta_gemm_agree(oz, m, n, k, r, monkeypatch):
    # CTA-pair and single-CTA kernels, each with the 4-product schedule; for
    # k > 8192 both accumulate exact chunks and add their residues.
    A, B = make_pair(m, n, k, seed=m + n + 5 * k, dist="wide")
    pA, pB = oz.ozemu_bit_budget_2limb(k, r)
    ap, _ = oz.split_rows_f64_2limb(to_dev(A), pA, r)
    bp, _ = oz.split_cols_f64_2limb(to_dev(B), pB, r)
    monkeypatch.setenv("OZEMU_GEMM_PAIR", "1")
    res_pair = oz.residue_gemm_2limb(m, n, k, r, ap, bp)
    monkeypatch.setenv("OZEMU_GEMM_PAIR", "0")
    res_one = oz.residue_gemm_2limb(m, n, k, r, ap, bp)
    status_ok(oz)
    assert torch.equal(res_pair[:, :, :n], res_one[:, :, :n])
    _, st = oracle_dgemm(A, B, r, stages=True)
    assert (res_pair.cpu().numpy()[:, :, :n].astype(np.int64) == st["res"]).all()


# ------------------------------------------------------------ full dgemm

def check_dgemm(oz, A, B, r, lda_pad=0, ldc_pad=0):
    m, k = A.shape
    n = B.shape[1]
    Ad = torch.zeros((m, k + lda_pad), dtype=torch.float64, device=DEV)
    Ad[:, :k] = to_dev(A)
    Cd = torch.full((m, n + ldc_pad), 7.0, dtype=torch.float64, device=DEV)
    oz.dgemm_2limb(Ad[:, :k], to_dev(B), r, out=Cd[:, :n])
    status_ok(oz)
    C = Cd.cpu().numpy()
    Cref = oracle_dgemm(A, B, r)
    assert (C[:, :n].view(np.int64) == Cref.view(np.int64)).all()
    if ldc_pad:
        assert (C[:, n:] == 7.0).all()
    return C[:, :n]


@pytest.mark.parametrize("m,n,k,r,dist", [(200, 77, 300, 16, "wide"), (1, 1, 1, 16, "uniform"),
                                          (300, 1, 1000, 16, "normal"), (300, 8, 1000, 16, "normal"),
                                          (129, 129, 129, 16, "uniform"), (64, 64, 20000, 14, "normal")])
def test_dgemm_two_limb_shapes(oz, m, n, k, r, dist):
    A, B = make_pair(m, n, k, seed=m * n + k + 9, dist=dist)
    C = check_dgemm(oz, A, B, r, lda_pad=3, ldc_pad=5)
    # r = 16 two-limb moduli give 92-102 bits of budget here: enough for the
    # 2 K 2^-53 |A||B| bound on narrow-range data, not on the wide range or
    # at k = 1 (51-bit operands), so the bound is asserted on those only.
    if dist != "wide" and k > 1 and m * n * k <= 200 * 77 * 300:
        assert oracle.error_bound_ratio(A, B, C) <= 1.0


@pytest.mark.parametrize("m,n,k,r", [(20, 30, 40, 1), (33, 70, 100, 2), (65, 17, 300, 3), (40, 90, 500, 5),
                                     (130, 80, 1000, 8), (50, 66, 700, 11)])
def test_dgemm_two_limb_few_moduli(oz, m, n, k, r):
    # Small r: the CRT's word counts (bytes of W_l, 16-bit positions, limbs of
    # C') change with the bit length of M; every instance against the oracle.
    A, B = make_pair(m, n, k, seed=m + n + k + r, dist="normal")
    check_dgemm(oz, A, B, r)


def test_dgemm_two_limb_k1_correctly_rounded(oz):
    # r = 16 two-limb moduli leave p_A = p_B = 51 bits at k = 1, so operands
    # with at most 51 significant bits pass exactly and C = fl(A B).
    rng = np.random.default_rng(6)
    A = rng.integers(-2 ** 50, 2 ** 50, size=(50, 1)) * 2.0 ** rng.integers(-300, 300, size=(50, 1))
    B = rng.integers(-2 ** 50, 2 ** 50, size=(1, 40)) * 2.0 ** rng.integers(-300, 300, size=(1, 40))
    C = check_dgemm(oz, A, B, 16)
    assert (C == A * B).all()


def test_dgemm_two_limb_special_values(oz):
    A = special_matrix(40, 64, seed=21)
    B = special_matrix(30, 64, seed=22).T.copy()
    check_dgemm(oz, A, B, 16)


def test_dgemm_two_limb_subnormal_and_overflow(oz):
    A = np.full((4, 4), 2.0 ** -540)
    B = np.full((4, 4), 2.0 ** -540) * np.array([1.0, 3.0, 0.75, -1.25])
    check_dgemm(oz, A, B, 16)
    C = check_dgemm(oz, np.full((2, 2), 1.5e154), np.full((2, 2), 1.5e154), 16)
    assert np.isinf(C).all()


def test_dgemm_two_limb_empty_k0_and_nonfinite(oz):
    C = oz.dgemm_2limb(to_dev(np.zeros((3, 0))), to_dev(np.zeros((0, 4))), 16)
    status_ok(oz)
    assert (C.cpu().numpy() == 0).all()
    A, B = make_pair(8, 8, 16, seed=2, dist="normal")
    B[3, 5] = np.nan
    oz.dgemm_2limb(to_dev(A), to_dev(B), 16)
    assert oz.get_status() == oz.OZEMU_ERR_NONFINITE
    assert oz.get_status() == oz.OZEMU_OK


@pytest.mark.parametrize("m,n,k,r,dist", [(2100, 300, 500, 16, "wide"), (4100, 70, 300, 15, "normal")])
def test_dgemm_two_limb_row_chunked(oz, m, n, k, r, dist):
    # m >= 2048 takes the path pipelined over row chunks; the oracle is
    # evaluated on sampled rows (each row's exponent sees its full row) and
    # all columns, including the rows at the chunk edges and the last row.
    A, B = make_pair(m, n, k, seed=m + 11 * n + k, dist=dist)
    C = oz.dgemm_2limb(to_dev(A), to_dev(B), r)
    status_ok(oz)
    rows = np.unique(np.concatenate([sample_indices(m, 40, seed=m), [0, m // 8 - 1, m // 8, m // 4, m - 1]]))
    Cref = oracle.dgemm_block(A, B, r, rows=rows, ceiling=CEIL)
    got = C.cpu().numpy()[rows]
    assert (got.view(np.int64) == Cref.view(np.int64)).all()


def test_two_limb_and_three_limb_agree_within_bound(oz):
    # Both families round the same exact product at comparable budgets
    # (r = 16 two-limb vs r = 13 three-limb), so both meet the bound.
    A, B = make_pair(150, 120, 700, seed=33, dist="normal")
    C2 = oz.dgemm_2limb(to_dev(A), to_dev(B), 16).cpu().numpy()
    C3 = oz.dgemm(to_dev(A), to_dev(B), 13).cpu().numpy()
    status_ok(oz)
    assert oracle.error_bound_ratio(A, B, C2) <= 1.0
    assert oracle.error_bound_ratio(A, B, C3) <= 1.0


@pytest.mark.parametrize("m,n,k,r", [(300, 200, 500, 16), (4100, 4200, 200, 16), (3, 5, 0, 16)])
def test_dgemm_host_two_limb_matches_device(oz, m, n, k, r):
    # Host buffers through the pipelined copies (B in two column blocks and
    # uneven row chunks for the larger shape): the same bits as the device
    # entry point, and the oracle's on sampled rows.
    A, B = make_pair(m, n, k, seed=m + n + k, dist="wide")
    A_pin = torch.from_numpy(A).pin_memory()
    B_pin = torch.from_numpy(B).pin_memory()
    C = oz.dgemm_host_2limb(A_pin, B_pin, r).numpy()
    status_ok(oz)
    Cd = oz.dgemm_2limb(to_dev(A), to_dev(B), r).cpu().numpy()
    status_ok(oz)
    assert (C.view(np.int64) == Cd.view(np.int64)).all()
    if k == 0:
        assert (C == 0).all()
        return
    rows = np.unique(np.concatenate([sample_indices(m, 12, seed=k), [m - 1]]))
    Cref = oracle.dgemm_block(A, B, r, rows=rows, ceiling=CEIL)
    assert (C[rows].view(np.int64) == Cref.view(np.int64)).all()
