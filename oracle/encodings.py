"""Six-product encodings of 8-bit values over the FP4 digit set (a study).

TEST INFRASTRUCTURE ONLY: nothing on the CUDA path imports this module.

[AWE] abstract: with weights chosen freely (instead of the fixed base 13),
planes that are integer combinations of limbs and stay inside S, an INT8 x
INT8 product takes 6 FP4 GEMMs instead of 9.  The pages do not print the
encoding.  Reading taken here: the 6 products are those of Karatsuba's
three-term identity,

    a b = sum_i c_ii a_i b_i + sum_{i<j} w_i w_j (a_i + a_j)(b_i + b_j),
    c_ii = w_i^2 - w_i sum_{j != i} w_j,

for a = sum_i w_i a_i, b = sum_i w_i b_i, which needs every limb a_i and every
pairwise sum a_i + a_j in S.  A search over weights (1, w1, w2), w1 < 60,
w2 < 200, finds exactly two that cover all of [-128, 127] with such limbs:
(1, 29, 37), covering [-148, 148], and (1, 11, 39), covering [-134, 134].
"""

import itertools

import numpy as np

from .ozaki2 import S

_SSET = frozenset(S)


def pairwise_closed_triples():
    """Limb triples (a0, a1, a2) in S^3 whose pairwise sums are also in S."""
    return [t for t in itertools.product(S, repeat=3)
            if t[0] + t[1] in _SSET and t[0] + t[2] in _SSET and t[1] + t[2] in _SSET]


def coverage(weights):
    """Largest h with every integer in [-h, h] equal to sum_i w_i a_i for a
    pairwise-closed triple."""
    vals = {sum(w * a for w, a in zip(weights, t)) for t in pairwise_closed_triples()}
    h = 0
    while h + 1 in vals and -(h + 1) in vals:
        h += 1
    return h


def search_weights(w1_max=60, w2_max=200, need=128):
    """All weights (1, w1, w2), w1 < w2, whose coverage reaches `need`."""
    triples = pairwise_closed_triples()
    found = []
    for w1 in range(2, w1_max):
        for w2 in range(w1 + 1, w2_max):
            vals = {a0 + w1 * a1 + w2 * a2 for a0, a1, a2 in triples}
            h = 0
            while h + 1 in vals and -(h + 1) in vals:
                h += 1
            if h >= need:
                found.append(((1, w1, w2), h))
    return found


def digit_table(weights, lo=-128, hi=127):
    """For each x in [lo, hi] a pairwise-closed triple with sum w_i a_i = x:
    the one of least sum |a_i|, ties broken by the lexicographic order of
    (|a0|, |a1|, |a2|, a0, a1, a2)."""
    best = {}
    for t in pairwise_closed_triples():
        x = sum(w * a for w, a in zip(weights, t))
        if lo <= x <= hi:
            key = (sum(abs(a) for a in t), abs(t[0]), abs(t[1]), abs(t[2]), t)
            if x not in best or key < best[x][0]:
                best[x] = (key, t)
    missing = [x for x in range(lo, hi + 1) if x not in best]
    if missing:
        raise ValueError("weights do not cover %d..%d (first gap %d)" % (lo, hi, missing[0]))
    return {x: v[1] for x, v in best.items()}


def coefficients(weights):
    """Karatsuba coefficients: {(i, i): c_ii, (i, j): w_i w_j} for i < j."""
    w = weights
    c = {(i, i): w[i] * w[i] - w[i] * sum(w[j] for j in range(3) if j != i) for i in range(3)}
    for i, j in ((0, 1), (0, 2), (1, 2)):
        c[(i, j)] = w[i] * w[j]
    return c


def planes(X, weights):
    """The six planes of an int8 matrix: a0, a1, a2, a0+a1, a0+a2, a1+a2,
    keyed like :func:`coefficients` (all entries in S)."""
    table = digit_table(weights)
    X = np.asarray(X, dtype=np.int64)
    lut = np.array([table[x] for x in range(-128, 128)], dtype=np.int64)  # (256, 3)
    d = lut[X + 128]  # (..., 3)
    out = {(i, i): d[..., i] for i in range(3)}
    for i, j in ((0, 1), (0, 2), (1, 2)):
        out[(i, j)] = d[..., i] + d[..., j]
    return out


def igemm_s8_six(A, B, weights=(1, 29, 37)):
    """Exact int64 A @ B of int8 matrices from the 6 plane products."""
    c = coefficients(weights)
    PA = planes(A, weights)
    PB = planes(np.asarray(B).T, weights)
    C = np.zeros((np.asarray(A).shape[0], np.asarray(B).shape[1]), dtype=np.int64)
    for key, coef in c.items():
        prod = PA[key].astype(np.float64) @ PB[key].astype(np.float64).T  # exact: |sum| < 2^53
        C += coef * prod.astype(np.int64)
    return C


def accumulator_growth(weights):
    """Largest |sum_p c_p P_p Q_p| one element adds to a single accumulator
    holding all six coefficient-weighted products, and the largest |c_p|."""
    c = coefficients(weights)
    table = digit_table(weights)
    biggest = max(abs(a + b) if i != j else abs(a) for t in table.values()
                  for (i, j) in c for a, b in [(t[i], t[j])])
    return sum(abs(v) for v in c.values()) * biggest * biggest, max(abs(v) for v in c.values())
