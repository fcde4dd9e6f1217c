"""INT4 x INT8 products in four FP4 products (exact), the oracle side.

TEST INFRASTRUCTURE ONLY: nothing on the CUDA path imports this module.

[AWE] abstract: with freely chosen weights and planes that stay inside the
FP4 digit set, an INT4 x INT8 product takes 4 FP4 products.  The pages do not
print the encoding; the reading taken here is an identity over the integers

    a b = sum_{k=1..4} g_k u_k(a) v_k(b)    for all a in [-8, 7], b in [-128, 127],

with every plane value u_k(a), v_k(b) in S = {0, +-1, +-2, +-3, +-4, +-6, +-8,
+-12} (twice the FP4 e2m1 values) and positive weights g_k that the block
scales can carry.  Construction: the B planes satisfy one linear relation
sum_k t_k g_k v_k(b) = 0 next to b = sum_k g_k v_k(b); the A planes are
u_k(a) = a + t_k z(a) for a rational z(a) chosen per a.  Then

    sum_k g_k u_k v_k = a sum_k g_k v_k + z sum_k t_k g_k v_k = a b.

A search over relations t with small numerators and denominators, A-side
feasibility for a = +-5, +-7 (the values of [-8, 7] outside S) and weights
g_k <= 32 for the B side found t = (-12, -9, -6, 3/2) with g = (3, 2, 6, 12)
(and g = (3, 2, 6, 24)); the tables below are built from that choice and
pinned exhaustively in tests/test_oracle_int4_int8.py.
"""

from fractions import Fraction

import numpy as np

from .ozaki2 import S

T = (Fraction(-12), Fraction(-9), Fraction(-6), Fraction(3, 2))
G = (3, 2, 6, 12)
A_RANGE = (-8, 7)
B_RANGE = (-128, 127)

_SSET = frozenset(S)


def a_table(t=T):
    """u(a) for a in [-8, 7]: the smallest |z| (then the smaller z) with
    a + t_k z in S for every k; returns {a: (u_1, .., u_4), ...}."""
    zs = sorted({Fraction(n, d) for d in (1, 2, 3, 4, 6) for n in range(-48, 49)}, key=lambda z: (abs(z), z))
    out = {}
    for a in range(A_RANGE[0], A_RANGE[1] + 1):
        for z in zs:
            u = [a + tk * z for tk in t]
            if all(x.denominator == 1 and int(x) in _SSET for x in u):
                out[a] = tuple(int(x) for x in u)
                break
        else:
            raise ValueError("no A planes for a = %d" % a)
    return out


def b_table(t=T, g=G):
    """v(b) for b in [-128, 127]: among the v in S^4 with the relation
    sum_k t_k g_k v_k = 0 and b = sum_k g_k v_k, the one with the smallest
    sum_k |v_k|, ties going to the lexicographically smallest tuple (a rule
    that does not depend on the order S is listed in)."""
    out = {}
    c4 = t[3] * g[3]
    for v1 in S:
        for v2 in S:
            for v3 in S:
                v4 = -(t[0] * g[0] * v1 + t[1] * g[1] * v2 + t[2] * g[2] * v3) / c4
                if v4.denominator != 1 or int(v4) not in _SSET:
                    continue
                v = (v1, v2, v3, int(v4))
                b = sum(gk * vk for gk, vk in zip(g, v))
                if not B_RANGE[0] <= b <= B_RANGE[1]:
                    continue
                key = (sum(abs(x) for x in v), v)
                if b not in out or key < (sum(abs(x) for x in out[b]), out[b]):
                    out[b] = v
    missing = [b for b in range(B_RANGE[0], B_RANGE[1] + 1) if b not in out]
    if missing:
        raise ValueError("no B planes for b in %s" % missing[:8])
    return out


def planes(X, table, lo):
    """The four plane matrices of an integer matrix X (values in the table's
    range starting at lo): int64 array (4, *X.shape)."""
    lut = np.array([table[v] for v in range(lo, lo + len(table))], dtype=np.int64)  # (range, 4)
    idx = np.asarray(X, dtype=np.int64) - lo
    return np.moveaxis(lut[idx], -1, 0)


def igemm_s4s8(A, B):
    """The definition: C = A B in exact integer arithmetic (A in [-8, 7],
    B in [-128, 127])."""
    return np.asarray(A, dtype=np.int64) @ np.asarray(B, dtype=np.int64)


def igemm_s4s8_four(A, B, t=T, g=G):
    """C = sum_k g_k U_k V_k from the four plane products (U_k = u_k(A),
    V_k = v_k(B)); equals igemm_s4s8(A, B)."""
    U = planes(A, a_table(t), A_RANGE[0])
    V = planes(B, b_table(t, g), B_RANGE[0])
    C = np.zeros((U.shape[1], V.shape[2]), dtype=np.int64)
    for k in range(4):
        C += g[k] * (U[k] @ V[k])
    return C


def prefix_growth(t=T, g=G):
    """Largest |sum_{j<=k} g_j u_j(a) v_j(b)| over a, b and k = 1..4: how far
    the running value of one K element can stray while its four products are
    added in order (after the fourth it is a b, at most 1024 in magnitude)."""
    ua, vb = a_table(t), b_table(t, g)
    worst = 0
    for u in ua.values():
        for v in vb.values():
            acc = 0
            for k in range(4):
                acc += g[k] * u[k] * v[k]
                worst = max(worst, abs(acc))
    return worst
