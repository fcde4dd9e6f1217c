"""CPU checks of bench.py's own measurement helpers (no GPU)."""

import numpy as np

import oracle
from workloads import make_pair


def _dense_parts(m, n):
    I = np.repeat(np.arange(m), n)
    J = np.tile(np.arange(n), m)
    return I, J


def test_bound_ratios_match_the_oracle():
    # bench.py measures accuracy with its own exact products; on every entry
    # of a small block, and on whole rows and columns, it must give the
    # oracle's ratio.
    import bench
    A, B = make_pair(6, 5, 300, seed=17, dist="wide")
    C = A @ B
    C[2, 3] = np.nextafter(C[2, 3], np.inf) * (1 + 2.0 ** -40)  # a larger error on one entry
    want = oracle.error_bound_ratio(A, B, C)
    I, J = _dense_parts(6, 5)
    got = bench.bound_ratios(A, B, [("pairs", (I, J))], {"c": [C[I, J]]})["c"]
    assert abs(got - want) <= 1e-9 * want
    parts = [("rows", np.array([0, 2, 5])), ("cols", np.array([1, 3]))]
    got = bench.bound_ratios(A, B, parts, {"c": [C[[0, 2, 5]], C[:, [1, 3]]]})["c"]
    assert abs(got - want) <= 1e-9 * want


def test_exact_residuals_match_the_oracle_sliced():
    import bench
    A, B = make_pair(5, 700, 900, seed=18, dist="normal")
    C = A @ B
    want = oracle.exact_residual_sliced(A, B, C)
    got, got2 = bench.exact_residuals(A, B, ("rows", np.arange(5)), [C, C * 0.5])
    assert (got == want).all()
    assert (got2 == oracle.exact_residual_sliced(A, B, C * 0.5)).all()
    got, = bench.exact_residuals(A, B, ("cols", np.array([0, 699])), [C[:, [0, 699]]])
    assert (got == want[:, [0, 699]]).all()


def test_bound_ratios_zero_for_the_exact_rounding():
    import bench
    A, B = make_pair(3, 4, 1, seed=5, dist="uniform")
    C = A @ B  # k = 1: each entry is one correctly rounded product
    I = np.array([0, 1, 2, 2])
    J = np.array([0, 3, 1, 2])
    got = bench.bound_ratios(A, B, [("pairs", (I, J))], {"c": [C[I, J]]})["c"]
    assert got <= 0.5  # |fl(ab) - ab| <= 2^-53 |ab| against a bound of 2 * 2^-53 |ab|


def test_accuracy_sample_shape():
    import bench
    parts = bench.accuracy_sample(100, 50, 16, 16, 4096)
    assert [p[0] for p in parts] == ["rows", "cols", "pairs"]
    assert len(parts[0][1]) == 16 and len(parts[1][1]) == 16 and len(parts[2][1][0]) == 4096
    assert bench.sample_size(parts, 100, 50) == 16 * 50 + 16 * 100 + 4096
