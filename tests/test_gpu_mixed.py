"""Parity of the mixed-digit CUDA path (single-digit moduli 8 13 11 9 7 5 at
one FP4 product each, then two-digit moduli at four) with the oracle run on
the same list.

Digits, shifts and residues must match bit for bit; the fp64 product must
equal the oracle's single correct rounding of C' 2^-(s_i + t_j) bit for bit.
"""

import numpy as np
import pytest

import oracle
from planes import decode_planes_mixed
from workloads import make_pair, sample_indices

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
MIX = oracle.MIXED


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


def test_library_lists_the_oracle_moduli(oz):
    assert oz.ozemu_max_moduli_mixed() == 20 and oz.ozemu_single_digit_moduli_mixed() == 6
    assert oz.ozemu_moduli_mixed(20) == oracle.moduli(20, MIX)
    for r in (1, 6, 7, 19, 20):
        assert oz.ozemu_products_mixed(r) == sum(oracle.products_per_modulus(l, MIX) for l in range(r))
    for k, r in ((1, 20), (8192, 19), (65536, 17), (300, 3)):
        assert sum(oz.ozemu_bit_budget_mixed(k, r)) == oracle.bit_budget(k, r, MIX)[0]


# ---------------------------------------------------------------- splits

@pytest.mark.parametrize("rows,k,p,r,pad", [(300, 1000, 40, 20, 0), (1, 1, 50, 19, 0), (129, 257, 30, 6, 0),
                                           (77, 1000, 40, 4, 2), (50, 3000, 36, 9, 1), (140, 200, 20, 1, 0)])
def test_split_rows_mixed_parity(oz, rows, k, p, r, pad):
    A = special_matrix(rows, k, seed=rows + k + 7)
    Ad = torch.zeros((rows, k + pad), dtype=torch.float64, device=DEV)
    Ad[:, :k] = to_dev(A)
    planes, shifts = oz.split_rows_f64_mixed(Ad[:, :k], p, r)
    status_ok(oz)
    assert planes.numel() == oz.ozemu_plane_bytes_mixed(rows, k, r)
    ref = oracle.deconstruct(A, p, r, MIX)
    assert (shifts.cpu().numpy() == ref["shift"]).all()
    digits, codes = decode_planes_mixed(planes.cpu().numpy(), rows, k, r)
    assert (digits[:, :, :rows, :k] == ref["digits"][:, :2]).all()
    assert (codes[:, :, rows:, :] == 0).all() and (codes[:, :, :, k:] == 0).all()


@pytest.mark.parametrize("k,cols,p,r", [(777, 200, 36, 19), (5, 3, 20, 7)])
def test_split_cols_mixed_parity(oz, k, cols, p, r):
    B = special_matrix(cols, k, seed=cols * 3 + k).T.copy()
    planes, shifts = oz.split_cols_f64_mixed(to_dev(B), p, r)
    status_ok(oz)
    ref = oracle.deconstruct(B.T, p, r, MIX)
    assert (shifts.cpu().numpy() == ref["shift"]).all()
    digits, codes = decode_planes_mixed(planes.cpu().numpy(), cols, k, r)
    assert (digits[:, :, :cols, :k] == ref["digits"][:, :2]).all()
    assert (codes[:, :, cols:, :] == 0).all() and (codes[:, :, :, k:] == 0).all()


# ---------------------------------------------------------- residues, CRT

@pytest.mark.parametrize("m,n,k,r,dist", [(200, 150, 300, 19, "uniform"), (130, 20, 1000, 14, "wide"),
                                          (64, 64, 9000, 12, "normal"), (257, 230, 2000, 20, "wide"),
                                          (150, 100, 700, 6, "normal"), (90, 300, 500, 3, "uniform")])
def test_residue_gemm_mixed_parity(oz, m, n, k, r, dist):
    A, B = make_pair(m, n, k, seed=m + n + k + 13, dist=dist)
    pA, pB = oz.ozemu_bit_budget_mixed(k, r)
    ap, sa = oz.split_rows_f64_mixed(to_dev(A), pA, r)
    bp, sb = oz.split_cols_f64_mixed(to_dev(B), pB, r)
    res = oz.residue_gemm_mixed(m, n, k, r, ap, bp)
    C = oz.crt_f64_mixed(m, n, r, res, sa, sb)
    status_ok(oz)
    Cref, st = oracle.dgemm(A, B, r, stages=True, ceiling=MIX)
    got = res.cpu().numpy()[:, :, :n].astype(np.int64)
    assert (got == st["res"]).all()
    assert (C.cpu().numpy().view(np.int64) == Cref.view(np.int64)).all()


@pytest.mark.parametrize("m,n,k,r", [(200, 150, 300, 19), (513, 257, 4000, 15), (256, 230, 4097, 20),
                                     (130, 250, 20000, 12), (130, 96, 270000, 8)])
def test_mixed_pair_and_single_cta_gemm_agree(oz, m, n, k, r, monkeypatch):
    # CTA-pair and single-CTA kernels; single-digit moduli accumulate exact
    # chunks of 2^18 (k = 270000 takes two), two-digit ones chunks of 4096.
    A, B = make_pair(m, n, k, seed=m + n + 3 * k, dist="wide")
    pA, pB = oz.ozemu_bit_budget_mixed(k, r)
    ap, _ = oz.split_rows_f64_mixed(to_dev(A), pA, r)
    bp, _ = oz.split_cols_f64_mixed(to_dev(B), pB, r)
    monkeypatch.setenv("OZEMU_GEMM_PAIR", "1")
    res_pair = oz.residue_gemm_mixed(m, n, k, r, ap, bp)
    monkeypatch.setenv("OZEMU_GEMM_PAIR", "0")
    res_one = oz.residue_gemm_mixed(m, n, k, r, ap, bp)
    status_ok(oz)
    assert torch.equal(res_pair[:, :, :n], res_one[:, :, :n])
    rows = sample_indices(m, 24, seed=k)
    _, st = oracle.dgemm_block(A, B, r, rows=rows, stages=True, ceiling=MIX)
    assert (res_pair.cpu().numpy()[:, rows, :n].astype(np.int64) == st["res"]).all()


def test_single_digit_worst_case_accumulation_is_exact(oz):
    # Every digit at -8 (FP4 code 0xE) over k = 2^18, one exact chunk: the
    # fp32 accumulator reaches 64 k = 2^24, the largest exact integer of its
    # range.  Moduli 8 and 13: 2^24 = 0 (mod 8) and 1 (mod 13); a sum off by
    # one product (64) would give 2 mod 13.
    k = 1 << 18
    m, n, r = 256, 224, 2
    plane = lambda rows: r * ((rows + 127) // 128 * 128) * (k // 2)
    ap = torch.full((plane(m),), 0xEE, dtype=torch.uint8, device=DEV)
    bp = torch.full((plane(n),), 0xEE, dtype=torch.uint8, device=DEV)
    assert ap.numel() == oz.ozemu_plane_bytes_mixed(m, k, r)
    res = oz.residue_gemm_mixed(m, n, k, r, ap, bp)
    status_ok(oz)
    assert (res[0, :, :n] == 0).all()
    assert (res[1, :, :n] == (64 * k) % 13).all() and (64 * k) % 13 == 1


# ------------------------------------------------------------ full dgemm

def check_dgemm(oz, A, B, r, lda_pad=0, ldc_pad=0):
    m, k = A.shape
    n = B.shape[1]
    Ad = torch.zeros((m, k + lda_pad), dtype=torch.float64, device=DEV)
    Ad[:, :k] = to_dev(A)
    Cd = torch.full((m, n + ldc_pad), 7.0, dtype=torch.float64, device=DEV)
    oz.dgemm_mixed(Ad[:, :k], to_dev(B), r, out=Cd[:, :n])
    status_ok(oz)
    C = Cd.cpu().numpy()
    Cref = oracle.dgemm(A, B, r, ceiling=MIX)
    assert (C[:, :n].view(np.int64) == Cref.view(np.int64)).all()
    if ldc_pad:
        assert (C[:, n:] == 7.0).all()
    return C[:, :n]


@pytest.mark.parametrize("m,n,k,r,dist", [(200, 77, 300, 20, "wide"), (1, 1, 1, 20, "uniform"),
                                          (300, 1, 1000, 19, "normal"), (300, 8, 1000, 19, "normal"),
                                          (129, 129, 129, 18, "uniform"), (64, 64, 20000, 17, "normal")])
def test_dgemm_mixed_shapes(oz, m, n, k, r, dist):
    A, B = make_pair(m, n, k, seed=m * n + k + 19, dist=dist)
    C = check_dgemm(oz, A, B, r, lda_pad=3, ldc_pad=5)
    if dist == "normal" and k >= 1000:
        assert oracle.error_bound_ratio(A, B, C) <= 1.0


@pytest.mark.parametrize("m,n,k,r", [(20, 30, 3, 1), (33, 70, 40, 2), (65, 17, 300, 3), (40, 90, 500, 5),
                                     (130, 80, 1000, 6), (50, 66, 700, 7), (70, 70, 200, 11)])
def test_dgemm_mixed_few_moduli(oz, m, n, k, r):
    # Few moduli leave few bits (r = 1: M = 8, so k <= 3); the CRT's word
    # counts change with the bit length of M: every instance against the oracle.
    A, B = make_pair(m, n, k, seed=m + n + k + r + 1, dist="normal")
    check_dgemm(oz, A, B, r)


def test_dgemm_mixed_special_values(oz):
    A = special_matrix(40, 64, seed=31)
    B = special_matrix(30, 64, seed=32).T.copy()
    check_dgemm(oz, A, B, 20)


def test_dgemm_mixed_subnormal_overflow_nonfinite_k0(oz):
    A = np.full((4, 4), 2.0 ** -540)
    B = np.full((4, 4), 2.0 ** -540) * np.array([1.0, 3.0, 0.75, -1.25])
    check_dgemm(oz, A, B, 20)
    C = check_dgemm(oz, np.full((2, 2), 1.5e154), np.full((2, 2), 1.5e154), 20)
    assert np.isinf(C).all()
    C = oz.dgemm_mixed(to_dev(np.zeros((3, 0))), to_dev(np.zeros((0, 4))), 19)
    status_ok(oz)
    assert (C.cpu().numpy() == 0).all()
    A, B = make_pair(8, 8, 16, seed=2, dist="normal")
    B[3, 5] = np.inf
    oz.dgemm_mixed(to_dev(A), to_dev(B), 19)
    assert oz.get_status() == oz.OZEMU_ERR_NONFINITE
    assert oz.get_status() == oz.OZEMU_OK


@pytest.mark.parametrize("m,n,k,r,dist", [(2100, 300, 500, 19, "wide"), (4100, 70, 300, 17, "normal")])
def test_dgemm_mixed_row_chunked(oz, m, n, k, r, dist):
    A, B = make_pair(m, n, k, seed=m + 7 * n + k, dist=dist)
    C = oz.dgemm_mixed(to_dev(A), to_dev(B), r)
    status_ok(oz)
    rows = np.unique(np.concatenate([sample_indices(m, 40, seed=m + 1), [0, m // 8 - 1, m // 8, m // 4, m - 1]]))
    Cref = oracle.dgemm_block(A, B, r, rows=rows, ceiling=MIX)
    assert (C.cpu().numpy()[rows].view(np.int64) == Cref.view(np.int64)).all()


@pytest.mark.parametrize("m,n,k,r", [(300, 200, 500, 19), (4100, 4200, 200, 19), (3, 5, 0, 19)])
def test_dgemm_host_mixed_matches_device(oz, m, n, k, r):
    A, B = make_pair(m, n, k, seed=m + n + k + 5, dist="wide")
    A_pin = torch.from_numpy(A).pin_memory()
    B_pin = torch.from_numpy(B).pin_memory()
    C = oz.dgemm_host_mixed(A_pin, B_pin, r).numpy()
    status_ok(oz)
    Cd = oz.dgemm_mixed(to_dev(A), to_dev(B), r).cpu().numpy()
    status_ok(oz)
    assert (C.view(np.int64) == Cd.view(np.int64)).all()
    if k == 0:
        assert (C == 0).all()
        return
    rows = np.unique(np.concatenate([sample_indices(m, 12, seed=k + 1), [m - 1]]))
    Cref = oracle.dgemm_block(A, B, r, rows=rows, ceiling=MIX)
    assert (C[rows].view(np.int64) == Cref.view(np.int64)).all()


def test_mixed_and_three_limb_agree_within_bound(oz):
    # r = 19 mixed-digit moduli (58 products) and r = 13 three-limb moduli
    # (117) have the same budget at k = 8192; both meet the bound.
    A, B = make_pair(96, 80, 8192, seed=41, dist="wide")
    Cm = oz.dgemm_mixed(to_dev(A), to_dev(B), 19).cpu().numpy()
    C3 = oz.dgemm(to_dev(A), to_dev(B), 13).cpu().numpy()
    status_ok(oz)
    assert oracle.error_bound_ratio_sliced(A, B, Cm) <= 1.0
    assert oracle.error_bound_ratio_sliced(A, B, C3) <= 1.0
