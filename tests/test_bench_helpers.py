"""CPU checks of bench.py's own measurement helpers (no GPU)."""

import numpy as np

import oracle
from workloads import make_pair


def test_bound_ratios_match_the_oracle():
    # bench.py measures accuracy with its own exact-rational sum; on every
    # entry of a small block it must give the oracle's ratio.
    import bench
    A, B = make_pair(6, 5, 300, seed=17, dist="wide")
    C = A @ B
    C[2, 3] = np.nextafter(C[2, 3], np.inf) * (1 + 2.0 ** -40)  # a larger error on one entry
    rows = np.repeat(np.arange(6), 5)
    cols = np.tile(np.arange(5), 6)
    got = bench.bound_ratios(A, B, rows, cols, {"c": C[rows, cols]})["c"]
    want = oracle.error_bound_ratio(A, B, C)
    assert abs(got - want) <= 1e-9 * want


def test_bound_ratios_zero_for_the_exact_rounding():
    import bench
    A, B = make_pair(3, 4, 1, seed=5, dist="uniform")
    C = A @ B  # k = 1: each entry is one correctly rounded product
    rows = np.array([0, 1, 2, 2])
    cols = np.array([0, 3, 1, 2])
    got = bench.bound_ratios(A, B, rows, cols, {"c": C[rows, cols]})["c"]
    assert got <= 0.5  # |fl(ab) - ab| <= 2^-53 |ab| against a bound of 2 * 2^-53 |ab|
