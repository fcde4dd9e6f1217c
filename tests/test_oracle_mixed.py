"""Pins of the mixed-digit reading (oracle, CPU only).

[AWE] abstract: the digit set S (FP4 values times two) holds every residue
modulo 13, the encodings are searched per input range, and the formulation
holds modulo m.  The mixed-digit list takes first the moduli whose every
residue class holds a member of S, so that each of their residue products is
ONE FP4 product, then the two-limb moduli (two base-13 digits, 4 products).
Everything here is checked by brute force against S as printed.
"""

import itertools
import math

import numpy as np
import pytest

import oracle
from workloads import make_pair


def test_single_digit_moduli_bruteforce(golden):
    S = golden["S"]["value"]
    covering = [m for m in range(2, 200) if {d % m for d in S} == set(range(m))]
    assert covering == [2, 3, 4, 5, 6, 7, 8, 9, 11, 13]
    assert oracle.single_digit_moduli(200) == covering
    # 15 values cannot cover more than 15 classes; 14, 15 and 16 miss some
    for m in (14, 15, 16):
        assert len({d % m for d in S}) < m


def test_single_digit_set_has_the_largest_product():
    cands = [2, 3, 4, 5, 6, 7, 8, 9, 11, 13]
    best = max((c for n in range(1, len(cands) + 1) for c in itertools.combinations(cands, n)
                if all(math.gcd(a, b) == 1 for a, b in itertools.combinations(c, 2))), key=math.prod)
    assert sorted(best) == sorted(oracle.single_digit_set()) == [5, 7, 8, 9, 11, 13]
    assert math.prod(best) == 360360
    assert oracle.single_digit_set()[0] == 8  # the even modulus first


@pytest.mark.parametrize("m", [8, 13, 11, 9, 7, 5])
def test_single_digit_identity_exhaustive(golden, m):
    # For every pair of balanced residues the product of the two digits is
    # congruent to the product of the residues: one FP4 product per modulus.
    S = set(golden["S"]["value"])
    h = m // 2
    res = range(-h, m - h)
    for x in res:
        d = oracle.single_digit(x, m)
        assert d in S and (d - x) % m == 0
        assert abs(d) <= 8
    for x in res:
        for y in res:
            assert (oracle.single_digit(x, m) * oracle.single_digit(y, m) - x * y) % m == 0


def test_single_digit_rule_values():
    # x itself when it lies in S; otherwise the smallest member of its class.
    assert [oracle.single_digit(x, 13) for x in range(-6, 7)] == [-6, 8, -4, -3, -2, -1, 0, 1, 2, 3, 4, -8, 6]
    assert [oracle.single_digit(x, 11) for x in range(-5, 6)] == [6, -4, -3, -2, -1, 0, 1, 2, 3, 4, -6]
    assert [oracle.single_digit(x, 8) for x in range(-4, 4)] == list(range(-4, 4))


def test_mixed_moduli_list():
    mods = oracle.moduli(20, oracle.MIXED)
    assert mods[:6] == [8, 13, 11, 9, 7, 5]
    for i, m in enumerate(mods):
        for j in range(i):
            assert math.gcd(m, mods[j]) == 1
    # after the single-digit set: every integer from 113 down that is coprime
    # to all moduli taken so far, and no other
    taken = mods[:6]
    for c in range(113, mods[-1] - 1, -1):
        if all(math.gcd(c, q) == 1 for q in taken):
            taken.append(c)
    assert taken[:20] == mods
    assert all(m <= 113 for m in mods[6:])  # residues in [-56, 56]: two digits


def test_mixed_digits_reconstruct_residues():
    A, _ = make_pair(9, 1, 300, seed=51, dist="wide")
    r = 20
    _, pA, _ = oracle.bit_budget(300, r, oracle.MIXED)
    d = oracle.deconstruct(A, pA, r, oracle.MIXED)
    mods = oracle.moduli(r, oracle.MIXED)
    for l, m in enumerate(mods):
        dig = d["digits"][l]
        assert (dig[2] == 0).all()
        if l < 6:
            assert (dig[1] == 0).all()
            assert ((dig[0] - d["res"][l]) % m == 0).all()
            assert np.isin(dig[0], oracle.S).all()
        else:
            assert (dig[0] + 13 * dig[1] == d["res"][l]).all()
        assert oracle.products_per_modulus(l, oracle.MIXED) == (1 if l < 6 else 4)


def test_mixed_products_and_bit_budget_against_the_three_limb_list():
    # r = 19 mixed-digit moduli: 6 + 4 * 13 = 58 FP4 products per output
    # reach, at K = 8192, the budget P = 88 that r = 13 three-limb moduli
    # (117 products) reach; [AWE] abstract gives 59 products for the FP64
    # significand.  At K = 65536, r = 17 (50 products) reach the P = 70 of
    # r = 11 three-limb moduli (99 products).
    prods = lambda r: sum(oracle.products_per_modulus(l, oracle.MIXED) for l in range(r))
    assert prods(19) == 58 and prods(17) == 50
    assert oracle.bit_budget(8192, 19, oracle.MIXED)[0] >= oracle.bit_budget(8192, 13)[0] == 88
    assert oracle.bit_budget(65536, 17, oracle.MIXED)[0] >= oracle.bit_budget(65536, 11)[0] == 70
    assert oracle.bit_budget(65536, 16, oracle.MIXED)[0] < 70
    assert oracle.bit_budget(8192, 18, oracle.MIXED)[0] < 88  # one modulus fewer falls short


def test_mixed_single_digit_products_match_direct_modular_product():
    A, B = make_pair(11, 7, 200, seed=52, dist="normal")
    r = 8
    C, st = oracle.dgemm(A, B, r, stages=True, ceiling=oracle.MIXED)
    for l, m in enumerate(st["mods"]):
        direct = oracle.mod_product_direct(st["a"]["res"][l], st["b"]["res"][l].T, m)
        assert (st["res"][l] == direct).all()


def test_mixed_crt_recovers_integer_product_and_bound():
    A, B = make_pair(6, 5, 33, seed=53, dist="uniform")
    C, st = oracle.dgemm(A, B, 20, stages=True, ceiling=oracle.MIXED)
    exact_int = st["a"]["xint"].astype(object) @ st["b"]["xint"].T.astype(object)
    assert (st["Cp"] == exact_int).all()
    A, B = make_pair(24, 20, 2048, seed=54, dist="normal")
    assert oracle.error_bound_ratio(A, B, oracle.dgemm(A, B, 18, ceiling=oracle.MIXED)) <= 1.0
    assert oracle.error_bound_ratio(A, B, oracle.dgemm(A, B, 12, ceiling=oracle.MIXED)) > 1.0


def test_planted_wrong_single_digit_is_caught(monkeypatch):
    # A digit off by one in the single-digit rule must break the identity pin.
    import oracle.ozaki2 as oz
    real = oz.single_digit
    wrong = lambda x, m: real(x, m) + (1 if int(x) == 3 else 0)
    monkeypatch.setattr(oz, "single_digit", wrong)
    monkeypatch.setattr(oracle, "single_digit", wrong)
    with pytest.raises(AssertionError):
        test_single_digit_identity_exhaustive({"S": {"value": list(oz.S)}}, 13)
