"""Pins for the six-product encoding study (oracle/encodings.py), CPU only.

The identity a b = sum_p c_p P_p(a) Q_p(b) must hold for every pair of 8-bit
values; every plane value must lie in S; the weight search must find exactly
the two weight triples that cover [-128, 127]; a planted wrong coefficient must
break the identity.
"""

import numpy as np
import pytest

import oracle
from oracle import encodings as enc


def test_pairwise_closed_triples_are_closed():
    S = set(oracle.S)
    triples = enc.pairwise_closed_triples()
    assert (0, 0, 0) in triples and (12, 0, -12) in triples
    for t in triples:
        assert all(x in S for x in t)
        assert t[0] + t[1] in S and t[0] + t[2] in S and t[1] + t[2] in S


def test_weight_search_finds_the_two_covering_triples():
    found = enc.search_weights(w1_max=40, w2_max=60)
    assert sorted(found) == [((1, 11, 39), 134), ((1, 29, 37), 148)]
    assert enc.coverage((1, 13, 169)) < 128  # base 13 limbs are not pairwise closed


@pytest.mark.parametrize("weights", [(1, 29, 37), (1, 11, 39)])
def test_six_products_reproduce_every_int8_product(weights):
    vals = np.arange(-128, 128, dtype=np.int64)
    C = enc.igemm_s8_six(vals[:, None], vals[None, :], weights)
    assert (C == np.outer(vals, vals)).all()
    P = enc.planes(vals, weights)
    assert len(P) == 6
    S = np.array(sorted(set(oracle.S)))
    for plane in P.values():
        assert np.isin(plane, S).all()


def test_six_products_random_matrices():
    rng = np.random.default_rng(7)
    A = rng.integers(-128, 128, size=(37, 300))
    B = rng.integers(-128, 128, size=(300, 29))
    assert (enc.igemm_s8_six(A, B) == A @ B).all()


def test_planted_wrong_coefficient_fails():
    vals = np.arange(-128, 128, dtype=np.int64)
    w = (1, 29, 37)
    c = enc.coefficients(w)
    assert c == {(0, 0): -65, (1, 1): -261, (2, 2): 259, (0, 1): 29, (0, 2): 37, (1, 2): 1073}
    P = enc.planes(vals, w)
    bad = dict(c)
    bad[(0, 0)] = 65
    C = sum(coef * np.outer(P[k], P[k]) for k, coef in bad.items())
    assert not (C == np.outer(vals, vals)).all()


def test_accumulator_growth_against_the_nine_product_scheme():
    # One accumulator of all six weighted products grows by up to this much per
    # K element; the 9-product scheme's first accumulator grows by 1728.
    growth, cmax = enc.accumulator_growth((1, 29, 37))
    assert cmax == 1073
    assert growth > 16 * 1728
