"""The workloads at their full sizes, through the C ABI, against the oracle.

The GPU computes every output; the oracle computes sampled rows and columns
at the full inner dimension (its row/column exponents always see the whole
row/column).  Sampled fp64 entries must match the oracle bit for bit and lie
within |C - C_exact| <= 2 K 2^-53 (|A||B|)_ij; the shifts of every row and
column and the residues of the sampled block must match exactly.  At full
size, every residue of two moduli (the first and the last) is compared with
the oracle's, and the bound is checked with exact products on 16 full rows,
16 full columns (all columns when there are fewer) and 4096 random entries of
the result ozemu_dgemm returns.  The INT8 product is compared in full.
"""

import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, workload_inputs, sample_indices

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


def run_stages(oz, A_h, B_h, r):
    """Full product through the stage calls; returns device tensors."""
    m, k = A_h.shape
    n = B_h.shape[1]
    A = torch.from_numpy(A_h).to(DEV)
    B = torch.from_numpy(B_h).to(DEV)
    pA, pB = oz.ozemu_bit_budget(k, r)
    ap, sa = oz.split_rows_f64(A, pA, r)
    bp, sb = oz.split_cols_f64(B, pB, r)
    res = oz.residue_gemm(m, n, k, r, ap, bp)
    C = oz.crt_f64(m, n, r, res, sa, sb)
    assert oz.get_status() == oz.OZEMU_OK
    C_direct = oz.dgemm(A, B, r)
    assert oz.get_status() == oz.OZEMU_OK
    assert torch.equal(C.view(torch.int64), C_direct.view(torch.int64))
    del ap, bp, A, B, C_direct
    return sa.cpu().numpy(), sb.cpu().numpy(), res, C.cpu().numpy()


@pytest.mark.parametrize("name,n_rows,n_cols", [
    ("dgemm_8192_wide", 12, 12),
    ("dgemv_16384_n1", 96, 1),
    ("dgemv_16384_n8", 48, 8),
    ("dgemm_4096_k65536", 8, 8),
])
def test_workload_parity_sampled(oz, name, n_rows, n_cols):
    A_h, B_h, spec = workload_inputs(name)
    r = spec["r"]
    m, n, k = spec["m"], spec["n"], spec["k"]
    sa, sb, res, C = run_stages(oz, A_h, B_h, r)
    _, pA, pB = oracle.bit_budget(k, r)
    # shifts of every row of A and every column of B
    assert (sa == oracle.row_shifts(A_h, pA)).all()
    assert (sb == oracle.row_shifts(B_h.T, pB)).all()
    rows = sample_indices(m, n_rows, seed=11)
    cols = sample_indices(n, n_cols, seed=12)
    Cref, st = oracle.dgemm_block(A_h, B_h, r, rows=rows, cols=cols, stages=True)
    got_res = res[:, rows][:, :, cols].cpu().numpy().astype(np.int64)
    assert (got_res == st["res"]).all()
    Cs = C[np.ix_(rows, cols)]
    assert (Cs.view(np.int64) == Cref.view(np.int64)).all()
    ratio = oracle.error_bound_ratio(A_h[rows], B_h[:, cols], Cs)
    print("%s r=%d max |C - C_exact| / bound = %.4f" % (name, r, ratio))
    assert ratio <= 1.0


@pytest.mark.parametrize("name,r,n_rows,n_cols", [
    ("dgemm_8192_wide", 16, 8, 8),
    ("dgemm_4096_k65536", 14, 6, 6),
])
def test_workload_two_limb_sampled(oz, name, r, n_rows, n_cols):
    # The two-limb moduli (<= 113) at full size, with the smallest r whose
    # bit budget reaches the three-limb r's: the device entry point and the
    # stage calls agree bit for bit, and sampled entries equal the oracle's
    # at the same modulus ceiling and meet the bound.
    A_h, B_h, spec = workload_inputs(name)
    m, n, k = spec["m"], spec["n"], spec["k"]
    ceil = oracle.MODULUS_CEILING_2LIMB
    assert sum(oracle.bit_budget(k, r, ceil)[1:]) >= sum(oracle.bit_budget(k, spec["r"])[1:])
    A = torch.from_numpy(A_h).to(DEV)
    B = torch.from_numpy(B_h).to(DEV)
    C = oz.dgemm_2limb(A, B, r)
    assert oz.get_status() == oz.OZEMU_OK
    pA, pB = oz.ozemu_bit_budget_2limb(k, r)
    ap, sa = oz.split_rows_f64_2limb(A, pA, r)
    bp, sb = oz.split_cols_f64_2limb(B, pB, r)
    res = oz.residue_gemm_2limb(m, n, k, r, ap, bp)
    Cs = oz.crt_f64_2limb(m, n, r, res, sa, sb)
    assert oz.get_status() == oz.OZEMU_OK
    assert torch.equal(C.view(torch.int64), Cs.view(torch.int64))
    del ap, bp, A, B, Cs
    rows = sample_indices(m, n_rows, seed=21)
    cols = sample_indices(n, n_cols, seed=22)
    Cref, st = oracle.dgemm_block(A_h, B_h, r, rows=rows, cols=cols, stages=True, ceiling=ceil)
    got_res = res[:, rows][:, :, cols].cpu().numpy().astype(np.int64)
    assert (got_res == st["res"]).all()
    Cg = C.cpu().numpy()[np.ix_(rows, cols)]
    assert (Cg.view(np.int64) == Cref.view(np.int64)).all()
    assert oracle.error_bound_ratio(A_h[rows], B_h[:, cols], Cg) <= 1.0


@pytest.mark.parametrize("name", ["dgemm_8192_wide", "dgemv_16384_n1", "dgemv_16384_n8", "dgemm_4096_k65536"])
def test_workload_full_modulus_and_bound_samples(oz, name):
    A_h, B_h, spec = workload_inputs(name)
    r = spec["r"]
    m, n, k = spec["m"], spec["n"], spec["k"]
    A = torch.from_numpy(A_h).to(DEV)
    B = torch.from_numpy(B_h).to(DEV)
    C = oz.dgemm(A, B, r)
    assert oz.get_status() == oz.OZEMU_OK
    C = C.cpu().numpy()
    # Every residue of two moduli, from the path ozemu_dgemm takes for the shape.
    if n <= oz.ozemu_narrow_max_n():
        res, _, _ = oz.residues_narrow_f64(A, B, r)
    else:
        pA, pB = oz.ozemu_bit_budget(k, r)
        ap, sa = oz.split_rows_f64(A, pA, r)
        bp, sb = oz.split_cols_f64(B, pB, r)
        res = oz.residue_gemm(m, n, k, r, ap, bp)
        del ap, bp
    assert oz.get_status() == oz.OZEMU_OK
    del A, B
    want = oracle.residues_of_moduli(A_h, B_h, r, (0, r - 1))
    for l in (0, r - 1):
        got = res[l, :, :n].cpu().numpy().astype(np.int64)
        assert (got == want[l]).all(), l
    del res
    # The bound, with exact products, on 16 full rows, 16 full columns and
    # 4096 random entries.
    rows = sample_indices(m, 16, seed=31)
    cols = sample_indices(n, 16, seed=32)
    rng = np.random.default_rng(33)
    I = rng.integers(0, m, 4096)
    J = rng.integers(0, n, 4096)
    ratios = (oracle.error_bound_ratio_sliced(A_h[rows], B_h, C[rows]),
              oracle.error_bound_ratio_sliced(A_h, B_h[:, cols], C[:, cols]),
              oracle.error_bound_ratio_pairs(A_h, B_h, C[I, J], I, J))
    print("%s r=%d max |C - C_exact| / bound: rows %.4f, columns %.4f, entries %.4f" % ((name, r) + ratios))
    assert max(ratios) <= 1.0


def test_igemm_s8_4096_full(oz):
    A_h, B_h, spec = workload_inputs("igemm_s8_4096")
    C = oz.igemm_s8(torch.from_numpy(A_h).to(DEV), torch.from_numpy(B_h).to(DEV))
    assert oz.get_status() == oz.OZEMU_OK
    ref = oracle.igemm_s8_direct(A_h, B_h)
    assert (C.cpu().numpy() == ref).all()
    # and the limb path of the oracle on a block of it
    rows = sample_indices(4096, 64, seed=3)
    cols = sample_indices(4096, 64, seed=4)
    assert (oracle.igemm_s8(A_h[rows], B_h[:, cols]) == C.cpu().numpy()[np.ix_(rows, cols)]).all()


def test_workload_table_is_what_the_tests_cover():
    assert set(WORKLOADS) == {"dgemm_256_uniform", "igemm_s8_4096", "dgemm_8192_wide", "dgemv_16384_n1",
                              "dgemv_16384_n8", "dgemm_4096_k65536"}
