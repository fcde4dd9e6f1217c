"""Pins for the INT4 x INT8 four-product encoding (oracle/int4_int8.py), CPU only.

The identity a b = sum_k g_k u_k(a) v_k(b) must hold for every pair of an
INT4 and an INT8 value, every plane value must lie in S, the B planes must
satisfy the linear relation the construction rests on, the four-product
matrix result must equal the integer product, and a planted wrong weight or
relation coefficient must break the identity.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import int4_int8 as q


def _identity_failures(t=q.T, g=q.G):
    ua, vb = q.a_table(t), q.b_table(t, g)
    return [(a, b) for a in range(-8, 8) for b in range(-128, 128)
            if sum(gk * x * y for gk, x, y in zip(g, ua[a], vb[b])) != a * b]


def test_identity_holds_for_every_int4_int8_pair():
    assert _identity_failures() == []


def test_every_plane_value_is_a_digit():
    S = set(oracle.S)
    ua, vb = q.a_table(), q.b_table()
    assert sorted(ua) == list(range(-8, 8)) and sorted(vb) == list(range(-128, 128))
    assert all(x in S for u in ua.values() for x in u)
    assert all(x in S for v in vb.values() for x in v)


def test_b_planes_satisfy_the_relation_and_sum_to_b():
    for b, v in q.b_table().items():
        assert sum(tk * gk * vk for tk, gk, vk in zip(q.T, q.G, v)) == 0
        assert sum(gk * vk for gk, vk in zip(q.G, v)) == b


def test_a_planes_lie_on_the_relation_line():
    # u_k(a) = a + t_k z(a) with one z(a) for all four planes; values of a in
    # S take z = 0 (all four planes equal a).
    for a, u in q.a_table().items():
        z = Fraction(u[0] - a) / q.T[0]
        assert all(Fraction(uk) == a + tk * z for uk, tk in zip(u, q.T))
        if a in set(oracle.S):
            assert u == (a, a, a, a)


@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 300, 5), (64, 1000, 33)])
def test_four_products_equal_the_integer_product(shape):
    m, k, n = shape
    rng = np.random.default_rng(sum(shape))
    A = rng.integers(-8, 8, (m, k))
    B = rng.integers(-128, 128, (k, n))
    A[0, 0], B[0, 0] = -8, -128  # the largest product
    np.testing.assert_array_equal(q.igemm_s4s8_four(A, B), q.igemm_s4s8(A, B))


def test_extreme_matrices():
    A = np.full((3, 4096), -8)
    B = np.full((4096, 2), -128)
    C = q.igemm_s4s8_four(A, B)
    assert (C == 4096 * 1024).all()


def test_running_value_bound_gives_the_exact_chunk():
    # Products added in the order k = 1..4 for each 64-element K block: the
    # accumulator never exceeds (elements so far) x 1024 plus one block's
    # partial prefixes, so K chunks of 8192 stay below 2^24 (exact in fp32).
    assert q.prefix_growth() == 1024
    assert 8192 * 1024 < 2 ** 24 <= 16384 * 1024


@pytest.mark.parametrize("k", range(4))
def test_planted_wrong_weight_breaks_the_identity(k):
    # The planes of (T, G) combined with one weight off by one: the identity
    # must fail somewhere.
    ua, vb = q.a_table(), q.b_table()
    g = list(q.G)
    g[k] += 1
    assert any(sum(gk * x * y for gk, x, y in zip(g, ua[a], vb[b])) != a * b
               for a in range(-8, 8) for b in range(-128, 128))


def test_planted_wrong_relation_is_caught():
    # A relation coefficient changed: a = 7 (outside S) then has no planes.
    with pytest.raises(ValueError):
        q.a_table((Fraction(-12), Fraction(-9), Fraction(-6), Fraction(3)))
    # The other weight set the search found is a valid encoding too.
    assert _identity_failures(q.T, (3, 2, 6, 24)) == []
