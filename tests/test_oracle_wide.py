"""Pins of the wide-moduli reading and of the limb GEMM's exact chunks (CPU).

Three base-13 limbs with the top limb anywhere in S reach every integer of
[-732, 732] ([AWE] abstract's limb algebra), so moduli up to 1465 fit three
limbs (about 10.5 bits for 9 products).  The pins check the list, the digits,
the exact integer product and the bound, and compute by brute force over
every pair of digit triples how fast the FP32 accumulators of the limb GEMM
grow per K element, which fixes the exact K chunk of every family.
"""

import math

import numpy as np

import oracle
from workloads import make_pair

WIDE = oracle.MODULUS_CEILING_WIDE


def test_wide_moduli_list_and_digits():
    mods = oracle.moduli(12, WIDE)
    assert mods[0] == 1465
    for i, m in enumerate(mods):
        for j in range(i):
            assert math.gcd(m, mods[j]) == 1
    A, _ = make_pair(7, 1, 400, seed=61, dist="wide")
    _, pA, _ = oracle.bit_budget(400, 12, WIDE)
    d = oracle.deconstruct(A, pA, 12, WIDE)
    assert np.abs(d["res"]).max() <= 732
    dig = d["digits"]
    assert np.isin(dig, oracle.S).all()
    assert (dig[:, 0] + 13 * dig[:, 1] + 169 * dig[:, 2] == d["res"]).all()


def test_wide_product_exact_and_within_bound():
    A, B = make_pair(6, 5, 40, seed=62, dist="uniform")
    C, st = oracle.dgemm(A, B, 12, stages=True, ceiling=WIDE)
    exact = st["a"]["xint"].astype(object) @ st["b"]["xint"].T.astype(object)
    assert (st["Cp"] == exact).all()
    A, B = make_pair(20, 16, 1024, seed=63, dist="normal")
    assert oracle.error_bound_ratio(A, B, oracle.dgemm(A, B, 11, ceiling=WIDE)) <= 1.0


def test_products_per_output_at_the_8192_budget():
    # P = 88 at K = 8192: three-limb r = 13 (117 products), wide r = 10 (90),
    # two-limb r = 16 (64), mixed-digit r = 19 (58).
    P = oracle.bit_budget(8192, 13)[0]
    assert P == 88

    def budget(r, ceiling):
        try:
            return oracle.bit_budget(8192, r, ceiling)[0]
        except ValueError:  # too few moduli for this k
            return -1

    def fewest(ceiling):
        r = next(r for r in range(1, 21) if budget(r, ceiling) >= P)
        return sum(oracle.products_per_modulus(l, ceiling) for l in range(r))

    assert [fewest(c) for c in (oracle.MODULUS_CEILING, WIDE, oracle.MODULUS_CEILING_2LIMB, oracle.MIXED)] == \
        [117, 90, 64, 58]


def test_accumulator_growth_and_exact_chunks():
    # Two accumulators D1 = A0B0 + 13 (A0B1 + A1B0), D2 = the rest: the
    # int8-range residues grow D1 by at most 1728 per K element (so 8192 K
    # elements stay below 2^24) and D2 by 97; the wide residues grow D2 by
    # 3168 (chunks of 4096 stay exact).  One accumulator for the two-limb
    # residues ([-56, 56]): 3136 per element, 4096 K elements exact.
    assert oracle.accumulator_growth(oracle.MODULUS_CEILING) == (1728, 97)
    assert 1728 * 8192 < 2 ** 24 and 1728 * 16384 >= 2 ** 24
    assert oracle.accumulator_growth(WIDE) == (1728, 3168)
    assert 3168 * 4096 < 2 ** 24 and 3168 * 8192 >= 2 ** 24
    g2 = oracle.accumulator_growth(oracle.MODULUS_CEILING_2LIMB, single_accumulator=True)
    assert g2 == 3136 and g2 * 4096 < 2 ** 24 and g2 * 8192 >= 2 ** 24
    # single-digit moduli: digits of magnitude <= 8, products <= 64 per element
    worst = max(abs(oracle.single_digit(x, m)) for m in oracle.single_digit_set()
                for x in range(-(m // 2), m - m // 2))
    assert worst == 8 and worst * worst * 2 ** 18 == 2 ** 24
