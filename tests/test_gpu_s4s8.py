"""Parity of the INT4 x INT8 product in four FP4 products with the oracle.

The library builds its plane tables itself; the planes it writes must equal
the oracle's encoding digit for digit (decoded with the oracle's e2m1
definition), and C32 must equal the exact integer product for every shape,
including several exact K chunks and the largest magnitudes.
"""

import numpy as np
import pytest

import oracle
from oracle import int4_int8 as q
from planes import decode_planes

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


def exact_product(A, B):
    # Integer products below 2^53 in every partial sum: float64 BLAS is exact.
    C = A.astype(np.float64) @ B.astype(np.float64)
    assert np.abs(C).max() < 2.0 ** 31
    return C.astype(np.int64)


def test_a_planes_equal_the_oracle_encoding(oz):
    vals = np.arange(-8, 8, dtype=np.int8)
    X = np.tile(vals, (3, 9))[:, :130]  # 3 rows x 130 elements: every value, a ragged K block
    planes = torch.zeros(oz.ozemu_four_plane_bytes(3, 130), dtype=torch.uint8, device=DEV)
    Xd = to_dev(X)
    st = oz.ozemu_split_rows_s4(3, 130, Xd.data_ptr(), 130, planes.data_ptr(), oz._stream())
    assert st == oz.OZEMU_OK and oz.get_status() == oz.OZEMU_OK
    digits, _ = decode_planes(planes.cpu().numpy(), 3, 130, 1, limbs=4)
    table = q.a_table()
    for i in range(3):
        for kk in range(130):
            assert tuple(digits[0, :, i, kk]) == table[int(X[i, kk])]
    assert (digits[0, :, 3:, :] == 0).all() and (digits[0, :, :, 130:] == 0).all()


def test_b_planes_equal_the_oracle_encoding(oz):
    vals = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    X = vals.reshape(256, 1).repeat(3, axis=1)  # k = 256 x 3 columns
    X[:, 1] = X[::-1, 1]
    planes = torch.zeros(oz.ozemu_four_plane_bytes(3, 256), dtype=torch.uint8, device=DEV)
    Xd = to_dev(X)
    st = oz.ozemu_split_cols_s8_four(256, 3, Xd.data_ptr(), 3, planes.data_ptr(), oz._stream())
    assert st == oz.OZEMU_OK and oz.get_status() == oz.OZEMU_OK
    digits, _ = decode_planes(planes.cpu().numpy(), 3, 256, 1, limbs=4)
    table = q.b_table()
    for j in range(3):
        for kk in range(256):
            assert tuple(digits[0, :, j, kk]) == table[int(X[kk, j])]
    S = set(oracle.S)
    assert all(int(d) in S for d in np.unique(digits))


@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 7, 3), (130, 300, 129), (256, 224, 8192), (300, 450, 8193),
                                   (128, 96, 20000), (257, 1, 1000), (64, 16, 4096), (33, 500, 128)])
def test_s4s8_matches_the_integer_product(oz, shape):
    m, n, k = shape
    rng = np.random.default_rng(m * 7 + n * 13 + k)
    A = rng.integers(-8, 8, (m, k), dtype=np.int8)
    B = rng.integers(-128, 128, (k, n), dtype=np.int16).astype(np.int8)
    C = oz.igemm_s4s8(to_dev(A), to_dev(B)).cpu().numpy().astype(np.int64)
    assert oz.get_status() == oz.OZEMU_OK
    np.testing.assert_array_equal(C, exact_product(A, B))
    if m * n * k <= 300 * 450 * 200:
        np.testing.assert_array_equal(C, q.igemm_s4s8_four(A, B))


def test_s4s8_largest_magnitudes_over_chunks(oz):
    # |a b| = 1024 at every K element across two exact chunks and a tail.
    k = 16384 + 100
    A = np.full((130, k), -8, dtype=np.int8)
    A[1] = 7
    B = np.full((k, 230), -128, dtype=np.int16).astype(np.int8)
    B[:, 1] = 127
    C = oz.igemm_s4s8(to_dev(A), to_dev(B)).cpu().numpy().astype(np.int64)
    np.testing.assert_array_equal(C, exact_product(A, B))
    assert C[0, 0] == 1024 * k


def test_s4s8_range_flag(oz):
    A = np.zeros((4, 64), dtype=np.int8)
    A[2, 5] = 9
    B = np.ones((64, 200), dtype=np.int8)
    oz.igemm_s4s8(to_dev(A), to_dev(B))
    assert oz.get_status() == oz.OZEMU_ERR_RANGE
    assert oz.get_status() == oz.OZEMU_OK  # cleared
    A[2, 5] = 7
    C = oz.igemm_s4s8(to_dev(A), to_dev(B)).cpu().numpy()
    assert oz.get_status() == oz.OZEMU_OK
    np.testing.assert_array_equal(C, exact_product(A, B))


def test_s4s8_4096(oz):
    rng = np.random.default_rng(2)
    A = rng.integers(-8, 8, (4096, 4096), dtype=np.int8)
    B = rng.integers(-128, 128, (4096, 4096), dtype=np.int16).astype(np.int8)
    C = oz.igemm_s4s8(to_dev(A), to_dev(B)).cpu().numpy().astype(np.int64)
    assert oz.get_status() == oz.OZEMU_OK
    np.testing.assert_array_equal(C, exact_product(A, B))


def test_s4s8_degenerate_k(oz):
    B = np.ones((1, 70), dtype=np.int8) * -128
    A = np.full((33, 1), 7, dtype=np.int8)
    C = oz.igemm_s4s8(to_dev(A), to_dev(B)).cpu().numpy()
    assert oz.get_status() == oz.OZEMU_OK
    assert (C == -896).all()
    # k = 0 zeroes C.
    Cd = torch.full((5, 6), 123, dtype=torch.int32, device=DEV)
    st = oz.ozemu_igemm_s4s8(5, 6, 0, 0, 0, Cd.data_ptr(), oz._stream())
    assert st == oz.OZEMU_OK and (Cd.cpu().numpy() == 0).all()


def test_split_rows_s4_padded_leading_dimension(oz):
    rng = np.random.default_rng(5)
    k, ldx = 200, 256
    X = rng.integers(-8, 8, (140, ldx), dtype=np.int8)
    planes = torch.zeros(oz.ozemu_four_plane_bytes(140, k), dtype=torch.uint8, device=DEV)
    st = oz.ozemu_split_rows_s4(140, k, to_dev(X).data_ptr(), ldx, planes.data_ptr(), oz._stream())
    assert st == oz.OZEMU_OK and oz.get_status() == oz.OZEMU_OK
    digits, _ = decode_planes(planes.cpu().numpy(), 140, k, 1, limbs=4)
    table = q.a_table()
    lut = np.array([table[v] for v in range(-8, 8)])  # (16, 4)
    want = lut[X[:, :k].astype(np.int64) + 8]          # (140, k, 4)
    np.testing.assert_array_equal(np.moveaxis(digits[0, :, :140, :k], 0, -1), want)
    assert (digits[0, :, :, k:] == 0).all() and (digits[0, :, 140:, :] == 0).all()
