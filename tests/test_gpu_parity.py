"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer stages (shifts, limb digits, INT32 products, residues) must match
bit for bit; the fp64 product must equal the oracle's single correct
rounding of C' 2^-(s_i + t_j) bit for bit, which also places it within
|C - C_exact| <= 2 K 2^-53 (|A||B|)_ij (checked on the exact product).
"""

import numpy as np
import pytest

import oracle
from planes import decode_planes
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


def status_ok(oz):
    assert oz.get_status() == oz.OZEMU_OK


def special_matrix(rows, k, seed):
    A, _ = make_pair(rows, 1, k, seed=seed, dist="wide")
    vals = [0.5, 1.5, 2.5, -2.5, 3.5, 2.0 ** -1074, -1e-310, 0.0]
    A[0, :min(8, k)] = vals[:min(8, k)]
    if rows > 2:
        A[2] = 0.0
    if rows > 3:
        A[3, :] = 2.0 ** -1060 * np.arange(1, k + 1)  # a subnormal-scale row
    if rows > 4:
        A[4, :] = 1e300 * np.sign(A[4])
    return A


# ---------------------------------------------------------------- splits

# pad: extra columns of the device buffer, so that the row stride is k + pad
# (k = 1000, pad = 2 gives 16-byte but not 32-byte row loads; pad = 1 single
# elements).
@pytest.mark.parametrize("rows,k,p,r,pad", [(300, 1000, 44, 13, 0), (1, 1, 62, 16, 0), (129, 257, 30, 5, 0),
                                           (64, 8192, 44, 13, 0), (77, 1000, 44, 13, 2), (50, 3000, 40, 12, 1)])
def test_split_rows_f64_parity(oz, rows, k, p, r, pad):
    A = special_matrix(rows, k, seed=rows + k)
    Ad = torch.zeros((rows, k + pad), dtype=torch.float64, device=DEV)
    Ad[:, :k] = to_dev(A)
    planes, shifts = oz.split_rows_f64(Ad[:, :k], p, r)
    status_ok(oz)
    ref = oracle.deconstruct(A, p, r)
    assert (shifts.cpu().numpy() == ref["shift"]).all()
    digits, codes = decode_planes(planes.cpu().numpy(), rows, k, r)
    assert (digits[:, :, :rows, :k] == ref["digits"]).all()
    assert (codes[:, :, rows:, :] == 0).all() and (codes[:, :, :, k:] == 0).all()


@pytest.mark.parametrize("k,cols,p,r", [(777, 200, 40, 13), (5, 3, 20, 4), (300, 129, 44, 12)])
def test_split_cols_f64_parity(oz, k, cols, p, r):
    B = special_matrix(cols, k, seed=cols * 3 + k).T.copy()
    planes, shifts = oz.split_cols_f64(to_dev(B), p, r)
    status_ok(oz)
    ref = oracle.deconstruct(B.T, p, r)
    assert (shifts.cpu().numpy() == ref["shift"]).all()
    digits, codes = decode_planes(planes.cpu().numpy(), cols, k, r)
    assert (digits[:, :, :cols, :k] == ref["digits"]).all()
    assert (codes[:, :, cols:, :] == 0).all() and (codes[:, :, :, k:] == 0).all()


@pytest.mark.parametrize("k,cols,pad", [(300, 256, 0), (1000, 200, 3), (129, 64, 1), (4096, 130, 0)])
def test_split_cols_s8_direct(oz, k, cols, pad):
    # Column split without a transposed copy: 4-byte loads when the rows are
    # 4-byte aligned and the 64-column tile is full, byte loads otherwise.
    rng = np.random.default_rng(k + cols)
    B = rng.integers(-128, 128, size=(k, cols), dtype=np.int8)
    B[0, :] = -128
    B[:, -1] = 127
    Bd = torch.zeros((k, cols + pad), dtype=torch.int8, device=DEV)
    Bd[:, :cols] = to_dev(B)
    planes = oz.split_cols_s8(Bd[:, :cols])
    status_ok(oz)
    digits, codes = decode_planes(planes.cpu().numpy(), cols, k, 1)
    assert (digits[0, :, :cols, :k] == oracle.limb_digits(B.T)).all()
    assert (codes[:, :, cols:, :] == 0).all() and (codes[:, :, :, k:] == 0).all()


def test_split_s8_parity(oz):
    A, B = make_pair(150, 90, 333, seed=3, dist="int8")
    A[0, :] = -128
    pa = oz.split_rows_s8(to_dev(A))
    pb = oz.split_cols_s8(to_dev(B))
    status_ok(oz)
    da, _ = decode_planes(pa.cpu().numpy(), 150, 333, 1)
    db, _ = decode_planes(pb.cpu().numpy(), 90, 333, 1)
    assert (da[0, :, :150, :333] == oracle.limb_digits(A)).all()
    assert (db[0, :, :90, :333] == oracle.limb_digits(B.T)).all()


# ----------------------------------------------------------- INT8 product

@pytest.mark.parametrize("m,n,k", [(200, 300, 500), (1, 1, 1), (129, 17, 4097), (256, 128, 256), (7, 1, 130),
                                   (300, 40, 64)])
def test_igemm_s8_parity(oz, m, n, k):
    A, B = make_pair(m, n, k, seed=m * 7 + n + k, dist="int8")
    C = oz.igemm_s8(to_dev(A), to_dev(B))
    status_ok(oz)
    assert (C.cpu().numpy() == oracle.igemm_s8_direct(A, B)).all()


@pytest.mark.parametrize("k", [8192, 8193, 20000])
def test_igemm_s8_exact_accumulation(oz, k):
    # Worst-case digit magnitudes (112 = 8 + 13 * 8) over a whole exact chunk,
    # then a long tail of small addends on top of the large partial sums.
    A = np.full((128, k), 112, dtype=np.int8)
    B = np.full((k, 128), 112, dtype=np.int8)
    B[:, 1::2] = -112
    A[1::3, k // 2:] = 1
    B[k // 3:, 2::5] = 1
    C = oz.igemm_s8(to_dev(A), to_dev(B))
    status_ok(oz)
    assert (C.cpu().numpy() == oracle.igemm_s8_direct(A, B)).all()


def test_igemm_s8_full_range(oz):
    A, B = make_pair(256, 256, 8192, seed=9, dist="int8")
    A[:, :4096] = -128
    B[:4096, :] = -128
    C = oz.igemm_s8(to_dev(A), to_dev(B))
    status_ok(oz)
    assert (C.cpu().numpy() == oracle.igemm_s8_direct(A, B)).all()


# ---------------------------------------------------------- residues, CRT

@pytest.mark.parametrize("m,n,k,r,dist", [(200, 150, 300, 13, "uniform"), (130, 20, 1000, 14, "wide"),
                                          (64, 64, 9000, 12, "normal")])
def test_residue_gemm_parity(oz, m, n, k, r, dist):
    A, B = make_pair(m, n, k, seed=m + n + k, dist=dist)
    pA, pB = oz.ozemu_bit_budget(k, r)
    ap, sa = oz.split_rows_f64(to_dev(A), pA, r)
    bp, sb = oz.split_cols_f64(to_dev(B), pB, r)
    res = oz.residue_gemm(m, n, k, r, ap, bp)
    C = oz.crt_f64(m, n, r, res, sa, sb)
    status_ok(oz)
    Cref, st = oracle.dgemm(A, B, r, stages=True)
    got = res.cpu().numpy()[:, :, :n].astype(np.int64)
    assert (got == st["res"]).all()
    assert (C.cpu().numpy().view(np.int64) == Cref.view(np.int64)).all()


# ------------------------------------------------------------ full dgemm

def check_dgemm(oz, A, B, r, lda_pad=0, ldc_pad=0):
    m, k = A.shape
    n = B.shape[1]
    Ad = torch.zeros((m, k + lda_pad), dtype=torch.float64, device=DEV)
    Ad[:, :k] = to_dev(A)
    Cd = torch.full((m, n + ldc_pad), 7.0, dtype=torch.float64, device=DEV)
    oz.dgemm(Ad[:, :k], to_dev(B), r, out=Cd[:, :n])
    status_ok(oz)
    C = Cd.cpu().numpy()
    Cref = oracle.dgemm(A, B, r)
    assert (C[:, :n].view(np.int64) == Cref.view(np.int64)).all()
    if ldc_pad:
        assert (C[:, n:] == 7.0).all()
    return C[:, :n]


def test_dgemm_256_uniform(oz):
    from workloads import workload_inputs
    A, B, spec = workload_inputs("dgemm_256_uniform")
    C = check_dgemm(oz, A, B, spec["r"])
    assert oracle.error_bound_ratio(A, B, C) <= 1.0


@pytest.mark.parametrize("m,n,k,r,dist", [(200, 77, 300, 14, "wide"), (1, 1, 1, 16, "uniform"),
                                          (300, 1, 1000, 13, "normal"), (300, 8, 1000, 13, "normal"),
                                          (129, 129, 129, 14, "uniform"), (64, 64, 20000, 12, "normal")])
def test_dgemm_shapes(oz, m, n, k, r, dist):
    A, B = make_pair(m, n, k, seed=m * n + k, dist=dist)
    C = check_dgemm(oz, A, B, r, lda_pad=3, ldc_pad=5)
    if m * n * k <= 200 * 77 * 300:
        assert oracle.error_bound_ratio(A, B, C) <= 1.0


def test_dgemm_k1_correctly_rounded(oz):
    A, B = make_pair(50, 40, 1, seed=5, dist="wide")
    C = check_dgemm(oz, A, B, 16)
    assert (C == A * B).all()


def test_dgemm_special_values(oz):
    A = special_matrix(40, 64, seed=11)
    B = special_matrix(30, 64, seed=12).T.copy()
    check_dgemm(oz, A, B, 16)


def test_dgemm_subnormal_results(oz):
    A = np.full((4, 4), 2.0 ** -540)
    B = np.full((4, 4), 2.0 ** -540) * np.array([1.0, 3.0, 0.75, -1.25])
    check_dgemm(oz, A, B, 16)


def test_dgemm_overflow_to_inf(oz):
    A = np.full((2, 2), 1.5e154)
    B = np.full((2, 2), 1.5e154)
    C = check_dgemm(oz, A, B, 16)
    assert np.isinf(C).all()


def test_dgemm_empty_and_k0(oz):
    A = to_dev(np.zeros((3, 0)))
    B = to_dev(np.zeros((0, 4)))
    C = oz.dgemm(A, B, 13)
    status_ok(oz)
    assert (C.cpu().numpy() == 0).all()


def test_dgemm_nonfinite_flag(oz):
    A, B = make_pair(8, 8, 16, seed=1, dist="normal")
    A[3, 5] = np.inf
    oz.dgemm(to_dev(A), to_dev(B), 13)
    assert oz.get_status() == oz.OZEMU_ERR_NONFINITE
    assert oz.get_status() == oz.OZEMU_OK  # cleared


def test_repeated_calls_and_release(oz):
    A, B = make_pair(70, 60, 500, seed=2, dist="uniform")
    Cref = oracle.dgemm(A, B, 13)
    for _ in range(2):
        C = oz.dgemm(to_dev(A), to_dev(B), 13)
        status_ok(oz)
        assert (C.cpu().numpy().view(np.int64) == Cref.view(np.int64)).all()
        oz.ozemu_release()


# ------------------------------------------------- INT8 comparison path

@pytest.mark.parametrize("rows,k,p,r", [(300, 1000, 44, 13), (129, 257, 30, 5)])
def test_split_res8_parity(oz, rows, k, p, r):
    A = special_matrix(rows, k, seed=rows * 5 + k)
    res, shifts = oz.split_rows_f64_res8(to_dev(A), p, r)
    status_ok(oz)
    ref = oracle.deconstruct(A, p, r)
    assert (shifts.cpu().numpy() == ref["shift"]).all()
    rows_p, k_p = (rows + 127) // 128 * 128, (k + 127) // 128 * 128
    got = res.cpu().numpy().reshape(r, rows_p, k_p).astype(np.int64)
    assert (got[:, :rows, :k] == ref["res"]).all()
    assert (got[:, rows:, :] == 0).all() and (got[:, :, k:] == 0).all()


@pytest.mark.parametrize("m,n,k,r,dist", [(200, 150, 300, 13, "uniform"), (130, 20, 1000, 14, "wide"),
                                          (256, 256, 9000, 12, "normal")])
def test_residue_gemm_i8_matches_oracle_and_fp4_path(oz, m, n, k, r, dist):
    A, B = make_pair(m, n, k, seed=m + 2 * n + k, dist=dist)
    pA, pB = oz.ozemu_bit_budget(k, r)
    a8, sa = oz.split_rows_f64_res8(to_dev(A), pA, r)
    b8, sb = oz.split_cols_f64_res8(to_dev(B), pB, r)
    res_i8 = oz.residue_gemm_i8(m, n, k, r, a8, b8)
    ap, _ = oz.split_rows_f64(to_dev(A), pA, r)
    bp, _ = oz.split_cols_f64(to_dev(B), pB, r)
    res_fp4 = oz.residue_gemm(m, n, k, r, ap, bp)
    C = oz.crt_f64(m, n, r, res_i8, sa, sb)
    status_ok(oz)
    Cref, st = oracle.dgemm(A, B, r, stages=True)
    got = res_i8.cpu().numpy()[:, :, :n].astype(np.int64)
    assert (got == st["res"]).all()
    assert torch.equal(res_i8[:, :, :n], res_fp4[:, :, :n])
    assert (C.cpu().numpy().view(np.int64) == Cref.view(np.int64)).all()


@pytest.mark.parametrize("m,n,k,r", [(200, 150, 300, 13), (513, 257, 4000, 12), (256, 65, 8192, 13),
                                     (300, 230, 8193, 13), (130, 250, 20000, 12), (257, 449, 16384, 11)])
def test_pair_and_single_cta_gemm_agree(oz, m, n, k, r, monkeypatch):
    # The CTA-pair kernel (256 x 224 tiles) and the single-CTA kernel (128 x
    # 128 tiles) must produce identical residues, equal to the oracle's; for
    # k > 8192 both accumulate exact chunks of 8192 and add their residues.
    A, B = make_pair(m, n, k, seed=m + n + 7 * k, dist="wide")
    pA, pB = oz.ozemu_bit_budget(k, r)
    ap, _ = oz.split_rows_f64(to_dev(A), pA, r)
    bp, _ = oz.split_cols_f64(to_dev(B), pB, r)
    monkeypatch.setenv("OZEMU_GEMM_PAIR", "1")
    res_pair = oz.residue_gemm(m, n, k, r, ap, bp)
    monkeypatch.setenv("OZEMU_GEMM_PAIR", "0")
    res_one = oz.residue_gemm(m, n, k, r, ap, bp)
    status_ok(oz)
    assert torch.equal(res_pair[:, :, :n], res_one[:, :, :n])
    _, st = oracle.dgemm(A, B, r, stages=True)
    assert (res_pair.cpu().numpy()[:, :, :n].astype(np.int64) == st["res"]).all()
