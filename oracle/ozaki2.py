"""Ozaki scheme II over base-13 FP4 limbs: the method's stages, written plainly.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Stage order follows the sources:

1. [TME4] abstract -- each fp64 row of A (column of B) is scaled by a power of
   two, rounded to an integer and reduced modulo each of r moduli.
2. [AWE] abstract -- each residue splits, with carries, into base-13 digits
   drawn from S = {0, +-1, +-2, +-3, +-4, +-6, +-8, +-12} (FP4 e2m1 values
   times two); three limbs with weights (1, 13, 169).
3. [AWE] abstract -- the limbs multiply pairwise: 9 FP4 GEMMs, each exact.
4. [AWE] abstract ("also holds modulo m") and [TME4] abstract (per-output
   reconstruction) -- recombine the 9 products modulo m, rebuild the integer
   product by the Chinese remainder theorem, scale back to fp64.

Readings where the sources are silent (each one also listed in the design
notes): moduli are the greedy pairwise-coprime integers descending from 256;
balanced residues lie in [-floor(m/2), ceil(m/2) - 1]; the bit budget P is the
largest integer with 2 K 2^P < prod(m), split p_A = ceil(P/2), p_B = floor(P/2);
the scale exponent of a row is the frexp exponent of its largest magnitude;
rounding to integer is round-half-to-even; the two digits that have two
representatives in S take the one of smaller magnitude; the fp64 result is the
single correct rounding of C' 2^-(s_i + t_j).

Parity pins (tests/test_oracle_pins.py): S against residues mod 13 and the
e2m1 definition; exhaustive int8 limb round trip; greedy moduli by brute force;
vectorised rounding against exact Fractions; CRT round trips and brute force on
small moduli; limb GEMMs against a triple loop and closed forms; the modular
recombination against a direct modular product; the full product against the
exact rational product, the error bound and exactly representable cases;
single roundings in the subnormal range (hand-derived values where one
rounding and two differ) and at the overflow threshold; the sliced exact
product against Fraction sums, including heavy cancellation.
"""

from fractions import Fraction
import math

import numpy as np

# ----------------------------------------------------------------------------
# Constants fixed by the sources
# ----------------------------------------------------------------------------

#: FP4 (e2m1) values scaled by two -- [AWE] abstract.
S = (0, 1, -1, 2, -2, 3, -3, 4, -4, 6, -6, 8, -8, 12, -12)
#: Digit base and limb weights -- [AWE] abstract.
BASE = 13
LIMB_WEIGHTS = (1, 13, 169)
N_LIMBS = 3
#: Largest modulus: keeps every balanced residue inside int8 (reading).
MODULUS_CEILING = 256
# Two-limb reading ([AWE] abstract: base-13 limbs from S; residues of moduli
# up to 113 lie in [-56, 56], where the 3-limb split's top digit is always 0,
# so 2 limbs and 2 x 2 = 4 FP4 products per modulus suffice).
MODULUS_CEILING_2LIMB = 113


# Wide-moduli reading (a derived variant; [AWE] abstract: base-13 limbs in S
# with weights (1, 13, 169)): with the top limb allowed anywhere in S (up to
# +-12), three limbs reach every integer of [-732, 732] (pinned), so moduli up
# to 1465 fit three limbs: about 10.5 bits per 9 products instead of 8.
MODULUS_CEILING_WIDE = 1465

# Mixed-digit reading ([AWE] abstract: the formulation holds modulo m, and the
# encodings may differ per input range).  A modulus m whose every residue
# class holds a member of S needs ONE digit per residue, so its residue
# product is one FP4 product.  The list starts with such moduli (the set of
# largest product, pairwise coprime) and continues with the two-limb moduli
# (greedy from 113, coprime to all taken).  Passed as ``ceiling=MIXED``.
MIXED = "mixed"


# ----------------------------------------------------------------------------
# Stage 0: moduli and bit budget (reading of [TME4] abstract; configs)
# ----------------------------------------------------------------------------

def single_digit_moduli(limit=16):
    """Every m in [2, limit] for which S meets every residue class mod m."""
    return [m for m in range(2, limit + 1) if len({d % m for d in S}) == m]


def single_digit_set():
    """The pairwise-coprime subset of :func:`single_digit_moduli` with the
    largest product, the even member first, the others descending."""
    cands = single_digit_moduli()
    best, best_prod = (), 1
    for mask in range(1 << len(cands)):
        pick = [m for i, m in enumerate(cands) if mask >> i & 1]
        if all(math.gcd(a, b) == 1 for i, a in enumerate(pick) for b in pick[:i]):
            prod = math.prod(pick)
            if prod > best_prod:
                best, best_prod = pick, prod
    even = [m for m in best if m % 2 == 0]
    return even + sorted((m for m in best if m % 2), reverse=True)


def single_digit(x, m):
    """The digit of residue x modulo a single-digit modulus m: x itself if it
    lies in S, otherwise the member of S in x's class of smallest magnitude."""
    x = int(x)
    if x in S:
        return x
    return min((d for d in S if (d - x) % m == 0), key=abs)


def moduli(r, ceiling=MODULUS_CEILING):
    """First ``r`` greedy pairwise-coprime integers counting down from
    ``ceiling`` (256; 113 for the two-limb reading); with ``ceiling=MIXED``
    the single-digit set first, then the greedy count from 113.

    The sources name no moduli.  Reading: take each integer from the ceiling
    down that is coprime to every modulus already taken.
    """
    if r < 1:
        raise ValueError("r must be >= 1")
    out = []
    if ceiling == MIXED:
        out = single_digit_set()[:r]
        ceiling = MODULUS_CEILING_2LIMB
    m = ceiling
    while len(out) < r:
        if m < 2:
            raise ValueError("ran out of moduli")
        if all(math.gcd(m, q) == 1 for q in out):
            out.append(m)
        m -= 1
    return out


def modulus_product(r, ceiling=MODULUS_CEILING):
    """Product of the first ``r`` moduli, as a Python int."""
    prod = 1
    for m in moduli(r, ceiling):
        prod *= m
    return prod


def bit_budget(k, r, ceiling=MODULUS_CEILING):
    """Return (P, p_A, p_B): P is the largest integer with 2 k 2^P < M.

    |A'| <= 2^p_A and |B'| <= 2^p_B then give |sum_k A'B'| <= k 2^P < M/2,
    so the product is recoverable from its residues.  Raises ValueError when
    not even P = 0 fits.
    """
    if k < 1:
        raise ValueError("k must be >= 1")
    M = modulus_product(r, ceiling)
    if not (2 * k * 1 < M):
        raise ValueError("modulus product too small for this k")
    P = 0
    while 2 * k * 2 ** (P + 1) < M:
        P += 1
    return P, (P + 1) // 2, P // 2


# ----------------------------------------------------------------------------
# Stage 1: scale, round, reduce ([TME4] abstract)
# ----------------------------------------------------------------------------

def frexp_exponent(x):
    """e with 2^(e-1) <= |x| < 2^e (frexp exponent); None for zero."""
    if x == 0:
        return None
    return math.frexp(float(x))[1]


def row_shifts(X, p):
    """Power-of-two shift s_i = p - e_i per row of X (0 for an all-zero row).

    e_i is the frexp exponent of max_k |X_ik|, so |X_ik 2^s_i| < 2^p.
    """
    X = np.asarray(X, dtype=np.float64)
    out = np.zeros(X.shape[0], dtype=np.int64)
    for i in range(X.shape[0]):
        mx = float(np.max(np.abs(X[i]))) if X.shape[1] else 0.0
        e = frexp_exponent(mx)
        out[i] = 0 if e is None else p - e
    return out


def scale_round_scalar(x, s):
    """round-half-to-even(x 2^s), computed exactly with Fractions."""
    return round(Fraction(float(x)) * Fraction(2) ** int(s))


def scale_round(X, shifts):
    """Vectorised round-half-to-even(X_ik 2^s_i) as int64 (|result| <= 2^62).

    Exact integer arithmetic on the significand: x = q 2^(e-53) with q the
    53-bit integer significand from frexp, then a left shift or a rounded right
    shift.  Pinned against :func:`scale_round_scalar`.
    """
    X = np.asarray(X, dtype=np.float64)
    s = np.asarray(shifts, dtype=np.int64).reshape(-1, 1)
    if X.ndim == 2 and X.size > (1 << 20):
        # Large matrices a block of rows at a time (same values, small temporaries).
        step = max(1, (1 << 20) // max(X.shape[1], 1))
        return np.concatenate([scale_round(X[i:i + step], s[i:i + step]) for i in range(0, X.shape[0], step)])
    mant, e = np.frexp(X)
    q = (np.abs(mant) * 2.0 ** 53).astype(np.int64)  # exact, < 2^53
    sh = e.astype(np.int64) - 53 + s
    # Left shifts (sh >= 0): the integer is q 2^sh; it must stay <= 2^62.
    shl = np.clip(sh, 0, 62)
    if np.any((q > 0) & (sh > 0) & ((sh > 62) | (q > (np.int64(1) << 62) >> shl))):
        raise OverflowError("scaled integer exceeds 2^62")
    left = q << shl
    # Right shifts (sh < 0) by d = min(-sh, 62), rounded half to even.
    d = np.clip(-sh, 1, 62)
    qd = q >> d
    rem = q & ((np.int64(1) << d) - 1)
    half = np.int64(1) << (d - 1)
    up = (rem > half) | ((rem == half) & ((qd & 1) == 1))
    out = np.where(sh >= 0, left, qd + up.astype(np.int64))
    return np.where(X < 0, -out, out)


def balanced_residue(x, m):
    """Residue of integer x modulo m in [-floor(m/2), ceil(m/2) - 1]."""
    v = int(x) % m
    if v > (m - 1) // 2:
        v -= m
    return v


def balanced_residue_array(X, m):
    """Element-wise :func:`balanced_residue` on an int64 array."""
    X = np.asarray(X, dtype=np.int64)
    if X.ndim == 2 and X.size > (1 << 20):
        step = max(1, (1 << 20) // max(X.shape[1], 1))
        return np.concatenate([balanced_residue_array(X[i:i + step], m) for i in range(0, X.shape[0], step)])
    v = np.mod(X, m)
    return np.where(v > (m - 1) // 2, v - m, v)


# ----------------------------------------------------------------------------
# Stage 2: base-13 limbs in S and their FP4 codes ([AWE] abstract)
# ----------------------------------------------------------------------------

def digit_of_class(c):
    """The element of S congruent to c mod 13 with the smallest magnitude.

    Classes 1 and 12 have two representatives in S (1 / -12 and 12 / -1);
    the smaller magnitude is taken (reading).
    """
    c %= BASE
    best = None
    for d in S:
        if d % BASE == c and (best is None or abs(d) < abs(best)):
            best = d
    if best is None:
        raise ValueError("S does not cover residue class %d" % c)
    return best


def limb_split(x):
    """Split integer x into (d0, d1, d2), x = d0 + 13 d1 + 169 d2, d_i in S.

    The two low digits are chosen by congruence (with a carry into the next
    digit); the top digit is what remains and must itself lie in S.
    """
    x = int(x)
    digits = []
    for _ in range(N_LIMBS - 1):
        d = digit_of_class(x)
        digits.append(d)
        x = (x - d) // BASE
    if x not in S:
        raise ValueError("top limb %d not in S" % x)
    digits.append(x)
    return tuple(digits)


def limb_table_int8():
    """(256, 3) int64 table: limbs of v for v = -128..127 (row v + 128)."""
    return np.array([limb_split(v) for v in range(-128, 128)], dtype=np.int64)


def limb_digits(X, lo=-128, hi=127):
    """Limb digits of an int array with values in [lo, hi] (int8 range by
    default; [-732, 732] for the wide moduli): shape (3, ...)."""
    X = np.asarray(X, dtype=np.int64)
    if X.size and (X.min() < lo or X.max() > hi):
        raise ValueError("limb_digits expects values in [%d, %d]" % (lo, hi))
    tab = limb_table_int8() if (lo, hi) == (-128, 127) else \
        np.array([limb_split(v) for v in range(lo, hi + 1)], dtype=np.int64)
    d = tab[X - lo]  # (..., 3)
    return np.moveaxis(d, -1, 0)


def e2m1_value(code):
    """Value of a 4-bit FP4 e2m1 code: sign, 2-bit exponent (bias 1), 1-bit mantissa."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        mag = man * 0.5
    else:
        mag = 2.0 ** (exp - 1) * (1.0 + man / 2.0)
    return sign * mag


def e2m1_code(d):
    """The 4-bit e2m1 code holding digit d as the FP4 value d / 2 (0 -> +0)."""
    target = d / 2.0
    for code in range(16):
        if code == 0x8:
            continue  # -0 is never produced
        if e2m1_value(code) == target:
            return code
    raise ValueError("digit %r is not in S" % (d,))


# ----------------------------------------------------------------------------
# Stage 3: the 9 limb products ([AWE] abstract)
# ----------------------------------------------------------------------------

def limb_products(Ad, Bd):
    """P[i][j] = Ad[i] @ Bd[j] for i, j in 0..2, exact, as int64.

    Ad: (3, M, K) digits, Bd: (3, K, N) digits.  Float64 BLAS is exact here
    because every partial sum is an integer below 2^53 (checked).
    """
    Ad = np.asarray(Ad, dtype=np.int64)
    Bd = np.asarray(Bd, dtype=np.int64)
    K = Ad.shape[2]
    amax = int(np.abs(Ad).max()) if Ad.size else 0
    bmax = int(np.abs(Bd).max()) if Bd.size else 0
    if K * amax * bmax >= 2 ** 53:
        raise OverflowError("limb product not exact in float64")
    P = np.zeros((N_LIMBS, N_LIMBS, Ad.shape[1], Bd.shape[2]), dtype=np.int64)
    for i in range(N_LIMBS):
        for j in range(N_LIMBS):
            P[i, j] = np.rint(Ad[i].astype(np.float64) @ Bd[j].astype(np.float64)).astype(np.int64)
    return P


def mod_recombine(P, m):
    """c = (sum_{i,j} 13^(i+j) P_ij) mod m, in [0, m)."""
    acc = np.zeros(P.shape[2:], dtype=np.int64)
    for i in range(N_LIMBS):
        for j in range(N_LIMBS):
            w = LIMB_WEIGHTS[i] * LIMB_WEIGHTS[j]
            acc = (acc + (w % m) * np.mod(P[i, j], m)) % m
    return acc


def mod_product_direct(a, b, m):
    """(a @ b) mod m for int residue matrices, without limbs (cross-check)."""
    a = np.asarray(a, dtype=np.int64)
    b = np.asarray(b, dtype=np.int64)
    prod = np.rint(a.astype(np.float64) @ b.astype(np.float64)).astype(np.int64)
    if a.shape[1] * 128 * 128 >= 2 ** 53:
        raise OverflowError("direct product not exact in float64")
    return np.mod(prod, m)


# ----------------------------------------------------------------------------
# Stage 4: CRT and scale back ([AWE] abstract; [TME4] abstract)
# ----------------------------------------------------------------------------

def crt(residues, mods):
    """Integer C' in (-M/2, M/2) with C' = residues[l] (mod mods[l]).

    Direct form: X = sum_l c_l (M/m_l) ((M/m_l)^-1 mod m_l) mod M, then the
    symmetric lift.  M is even (256 is the first modulus) and |C'| < M/2, so
    X = M/2 cannot occur.
    """
    M = 1
    for m in mods:
        M *= m
    X = 0
    for c, m in zip(residues, mods):
        Mi = M // m
        X += int(c) * Mi * pow(Mi % m, -1, m)
    X %= M
    return X - M if X > M // 2 else X


def crt_array(res, mods):
    """:func:`crt` over an array of residue vectors: res shape (r, ...)."""
    M = 1
    for m in mods:
        M *= m
    X = np.zeros(res.shape[1:], dtype=object)
    for l, m in enumerate(mods):
        Mi = M // m
        w = Mi * pow(Mi % m, -1, m)
        X = X + res[l].astype(object) * w
    X = X % M
    return np.where(X > M // 2, X - M, X)


def scale_back(Cp, S_shift):
    """Single correct rounding of Cp 2^-S_shift to fp64 (+-inf on overflow)."""
    val = Fraction(int(Cp)) / Fraction(2) ** int(S_shift)
    try:
        return float(val)
    except OverflowError:
        return math.inf if val > 0 else -math.inf


def scale_back_array(Cp, sA, sB):
    """:func:`scale_back` over a matrix: entry (i, j) uses sA[i] + sB[j]."""
    out = np.empty(Cp.shape, dtype=np.float64)
    for i in range(Cp.shape[0]):
        for j in range(Cp.shape[1]):
            out[i, j] = scale_back(Cp[i, j], int(sA[i]) + int(sB[j]))
    return out


# ----------------------------------------------------------------------------
# Pipelines
# ----------------------------------------------------------------------------

def digits_of_modulus(res, m, l, ceiling=MODULUS_CEILING):
    """Limb digits (3, ...) of the balanced residues ``res`` of the l-th
    modulus m: base-13 limbs, or for a single-digit modulus of the mixed list
    (d, 0, 0) with d = :func:`single_digit`."""
    if ceiling == MIXED and l < len(single_digit_set()):
        h = m // 2
        table = np.array([single_digit(x, m) for x in range(-h, m - h)], dtype=np.int64)
        d = table[np.asarray(res, dtype=np.int64) + h]
        return np.stack([d, np.zeros_like(d), np.zeros_like(d)])
    if ceiling == MODULUS_CEILING_WIDE:
        return limb_digits(res, -732, 732)
    return limb_digits(res)


def products_per_modulus(l, ceiling=MODULUS_CEILING):
    """FP4 products the l-th modulus takes: 9 (three limbs), 4 (two limbs),
    1 (a single-digit modulus of the mixed list)."""
    if ceiling == MIXED:
        return 1 if l < len(single_digit_set()) else 4
    return 4 if ceiling == MODULUS_CEILING_2LIMB else 9  # three limbs: 256 and the wide 1465


def accumulator_growth(ceiling=MODULUS_CEILING, single_accumulator=False):
    """Largest |increment| one K element adds to the FP32 accumulators of the
    limb GEMM for residues of the given moduli list (brute force over every
    pair of digit triples the split produces): with two accumulators
    D1 = A0B0 + 13 (A0B1 + A1B0) and D2 = the rest (weights 1, 13, 169), or
    one accumulator D = sum 13^(i+j) A_i B_j.  Returns (growth of D1, growth
    of D2) or the single growth; an exact chunk holds (2^24 - 1) // growth
    K elements."""
    lo, hi = {MODULUS_CEILING: (-128, 127), MODULUS_CEILING_2LIMB: (-56, 56),
              MODULUS_CEILING_WIDE: (-732, 732)}[ceiling]  # the balanced residues of each list
    trip = np.array([limb_split(v) for v in range(lo, hi + 1)], dtype=np.int64)
    g1 = g2 = gs = 0
    for a in trip:
        d1 = np.abs(a[0] * trip[:, 0] + 13 * (a[0] * trip[:, 1] + a[1] * trip[:, 0]))
        d2 = np.abs(a[0] * trip[:, 2] + a[1] * trip[:, 1] + a[2] * trip[:, 0]
                    + 13 * (a[1] * trip[:, 2] + a[2] * trip[:, 1]) + 169 * a[2] * trip[:, 2])
        g1, g2 = max(g1, int(d1.max())), max(g2, int(d2.max()))
        full = np.abs(sum(13 ** (i + j) * a[i] * trip[:, j] for i in range(3) for j in range(3)))
        gs = max(gs, int(full.max()))
    return gs if single_accumulator else (g1, g2)


def deconstruct(X, p, r, ceiling=MODULUS_CEILING):
    """Stage 1 + 2 for the rows of X: shifts, integers, residues, limb digits.

    Returns dict(shift=(rows,), xint=(rows, k), res=(r, rows, k),
    digits=(r, 3, rows, k)); with ceiling 113 the top digit is 0 throughout;
    with ceiling MIXED single-digit moduli have digits (d, 0, 0).
    """
    s = row_shifts(X, p)
    xi = scale_round(X, s)
    mods = moduli(r, ceiling)
    res = np.stack([balanced_residue_array(xi, m) for m in mods]) if r else None
    digits = np.stack([digits_of_modulus(res[l], mods[l], l, ceiling) for l in range(r)])
    return dict(shift=s, xint=xi, res=res, digits=digits)


def dgemm_block(A, B, r, rows=None, cols=None, stages=False, ceiling=MODULUS_CEILING):
    """Emulated C[rows][:, cols] = A @ B by the four stages.

    ``rows`` / ``cols`` select a sub-block (default: all).  Row and column
    exponents always see the full row / column.  ``ceiling`` 113 takes the
    two-limb moduli (the same stages; the third limb is 0).
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    rows = np.arange(M) if rows is None else np.asarray(rows)
    cols = np.arange(N) if cols is None else np.asarray(cols)
    mods = moduli(r, ceiling)
    _, pA, pB = bit_budget(K, r, ceiling)
    da = deconstruct(A[rows], pA, r, ceiling)
    db = deconstruct(B[:, cols].T, pB, r, ceiling)  # columns of B as rows
    res = np.zeros((r, len(rows), len(cols)), dtype=np.int64)
    for l, m in enumerate(mods):
        Ad = da["digits"][l]                       # (3, rows, K)
        Bd = np.swapaxes(db["digits"][l], 1, 2)    # (3, K, cols)
        res[l] = mod_recombine(limb_products(Ad, Bd), m)
    Cp = crt_array(res, mods)
    C = scale_back_array(Cp, da["shift"], db["shift"])
    if stages:
        return C, dict(mods=mods, pA=pA, pB=pB, a=da, b=db, res=res, Cp=Cp)
    return C


def dgemm(A, B, r, stages=False, ceiling=MODULUS_CEILING):
    """Emulated fp64 C = A @ B with r moduli (whole matrix)."""
    return dgemm_block(A, B, r, stages=stages, ceiling=ceiling)


def igemm_s8(A, B):
    """Exact int32 C = A @ B of int8 matrices by 9 base-13 limb products."""
    A = np.asarray(A, dtype=np.int64)
    B = np.asarray(B, dtype=np.int64)
    Ad = limb_digits(A)
    Bd = limb_digits(B)
    P = limb_products(Ad, Bd)
    C = np.zeros(P.shape[2:], dtype=np.int64)
    for i in range(N_LIMBS):
        for j in range(N_LIMBS):
            C += LIMB_WEIGHTS[i] * LIMB_WEIGHTS[j] * P[i, j]
    if C.size and (C.max() > 2 ** 31 - 1 or C.min() < -2 ** 31):
        raise OverflowError("int32 overflow")
    return C.astype(np.int32)


def igemm_s8_direct(A, B):
    """A @ B of int8 matrices in one exact float64 product (no limbs)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    if A.shape[1] * 128 * 128 >= 2 ** 53:
        raise OverflowError("not exact in float64")
    return np.rint(A @ B).astype(np.int64)


# ----------------------------------------------------------------------------
# The exact product and the error bound
# ----------------------------------------------------------------------------

def exact_dot_fraction(a, b):
    """Exact sum_k a_k b_k as a Fraction (slow; tiny inputs)."""
    return sum((Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a, b)), Fraction(0))


_SPLITTER = 134217729.0  # 2^27 + 1


def two_product(a, b):
    """Error-free product a*b = p + e (Dekker / Veltkamp), element-wise.

    Exact when no intermediate overflows or underflows (|a|, |b| well inside
    the normal range, |a b| above 2^-969).
    """
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    p = a * b
    ca = _SPLITTER * a
    ah = ca - (ca - a)
    al = a - ah
    cb = _SPLITTER * b
    bh = cb - (cb - b)
    bl = b - bh
    e = ((ah * bh - p) + ah * bl + al * bh) + al * bl
    return p, e


def exact_residual(A, B, C, rows=None, cols=None):
    """RN(sum_k A_ik B_kj - C_ij) for the selected entries (fsum of two-products)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    rows = np.arange(A.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(B.shape[1]) if cols is None else np.asarray(cols)
    out = np.zeros((len(rows), len(cols)), dtype=np.float64)
    for ii, i in enumerate(rows):
        p, e = two_product(A[i][:, None], B[:, cols])  # (K, cols)
        for jj in range(len(cols)):
            out[ii, jj] = math.fsum(p[:, jj].tolist() + e[:, jj].tolist() + [-float(C[ii, jj])])
    return out


def abs_product_sum(A, B, rows=None, cols=None):
    """(|A| |B|)_ij for the selected entries, correctly rounded (fsum)."""
    A = np.abs(np.asarray(A, dtype=np.float64))
    B = np.abs(np.asarray(B, dtype=np.float64))
    rows = np.arange(A.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(B.shape[1]) if cols is None else np.asarray(cols)
    out = np.zeros((len(rows), len(cols)), dtype=np.float64)
    for ii, i in enumerate(rows):
        p, e = two_product(A[i][:, None], B[:, cols])
        for jj in range(len(cols)):
            out[ii, jj] = math.fsum(p[:, jj].tolist() + e[:, jj].tolist())
    return out


def error_bound_ratio(A, B, C, rows=None, cols=None):
    """Max over entries of |C - C_exact| / (2 K 2^-53 (|A||B|)_ij).

    The target bound is ratio <= 1.  Entries whose (|A||B|)_ij is 0 must be
    exact; they count as ratio 0 when exact and inf otherwise.
    """
    K = np.asarray(A).shape[1]
    res = np.abs(exact_residual(A, B, C, rows, cols))
    absum = abs_product_sum(A, B, rows, cols)
    bound = 2.0 * K * 2.0 ** -53 * absum
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, res / np.where(bound > 0, bound, 1.0),
                         np.where(res == 0, 0.0, np.inf))
    return float(ratio.max()) if ratio.size else 0.0


# ----------------------------------------------------------------------------
# The exact product at full size: error-free slices summed by float64 BLAS
# ----------------------------------------------------------------------------
#
# The bound check needs sum_k A_ik B_kj exactly for whole rows and columns of
# the largest workloads, where Fractions are far too slow.  Every fp64 value
# is a dyadic rational, so the product can be taken exactly in pieces: each
# row of A (column of B) is cut into slices whose entries are integers below
# 2^beta times one power of two per row and slice, with beta chosen so that
# K 2^(2 beta) <= 2^53.  Every partial sum of a slice-by-slice product is then
# an integer below 2^53 and float64 BLAS returns it exactly, in any summation
# order.  The exact product is the sum of those exact terms, each scaled by a
# power of two; the residual sum - C is rounded once with math.fsum.  Pinned
# against the Fraction sums above (tests/test_oracle_pins.py).

def _slice_beta(k):
    """Bits per slice entry: the largest beta with k 2^(2 beta) <= 2^53."""
    beta = 26
    while k * 2 ** (2 * beta) > 2 ** 53:
        beta -= 1
    if beta < 1:
        raise ValueError("k too large for exact float64 slices")
    return beta


def _slices(X, beta, max_slices=80):
    """Cut the rows of X into slices: X = sum_s Q_s 2^(e_i - beta (s+1)) with
    every Q_s integer-valued and |Q_s| < 2^beta.  Returns (e, [Q_s])."""
    rem = np.array(X, dtype=np.float64, order="C")  # a contiguous copy
    e = np.zeros(rem.shape[0], dtype=np.int64)
    mx = np.max(np.abs(rem), axis=1) if rem.shape[1] else np.zeros(rem.shape[0])
    for i in range(rem.shape[0]):
        ex = frexp_exponent(float(mx[i]))
        e[i] = 0 if ex is None else ex
    out = []
    lim = 2.0 ** beta
    for s in range(max_slices):
        if not rem.any():
            return e, out
        sc = np.ldexp(1.0, (beta * (s + 1) - e))[:, None]
        q = rem * sc                       # exact: a power-of-two scaling ...
        np.trunc(q, out=q)                 # ... then truncation: an integer below 2^beta
        if np.abs(q).max() >= lim:
            raise ArithmeticError("slice out of range")
        q /= sc                            # exact: fewer than beta significant bits
        rem -= q                           # exact: the bits below the slice's grid
        q *= sc
        out.append(q)
    raise ArithmeticError("values span more bits than %d slices hold" % max_slices)


def _exact_terms_block(A, B):
    """Exact sum_k A_ik B_kj as a list of float64 arrays whose sum (taken
    exactly) is the product, for a block A (R x K) @ B (K x N)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    k = A.shape[1]
    beta = _slice_beta(max(k, 1))
    ea, sa = _slices(A, beta)
    eb, sb = _slices(B.T, beta)
    terms = []
    for s, qa in enumerate(sa):
        for t, qb in enumerate(sb):
            g = qa @ qb.T                  # integer partial sums below 2^53: exact
            ex = (ea[:, None] + eb[None, :]) - beta * (s + t + 2)
            term = np.ldexp(g, ex)
            if not np.array_equal(np.ldexp(term, -ex), g):
                raise ArithmeticError("scaled term not exact (range)")
            terms.append(term)
    return terms


def exact_residual_sliced(A, B, C, block=512):
    """RN(sum_k A_ik B_kj - C_ij) for every entry of C = (A @ B)'s block,
    exactly (see the section comment); A is R x K, B is K x N, C is R x N.
    B is taken ``block`` columns at a time (the same terms, less memory)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    out = np.empty(C.shape, dtype=np.float64)
    for j0 in range(0, C.shape[1], block):
        j1 = min(j0 + block, C.shape[1])
        terms = _exact_terms_block(A, B[:, j0:j1])
        T = np.stack(terms + [-C[:, j0:j1]])
        for i in range(C.shape[0]):
            Ti = T[:, i, :]
            for j in range(j1 - j0):
                out[i, j0 + j] = math.fsum(Ti[:, j].tolist())
    return out


def exact_residual_pairs(A, B, C, rows, cols, block=512):
    """RN(sum_k A_(rows_e) k B_k (cols_e) - C_e) for the entry pairs (rows[e],
    cols[e]), exactly; C holds the entries (length len(rows)).  Taken
    ``block`` pairs at a time."""
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    beta = _slice_beta(max(A.shape[1], 1))
    out = np.empty(len(rows), dtype=np.float64)
    for e0 in range(0, len(rows), block):
        e1 = min(e0 + block, len(rows))
        ea, sa = _slices(A[rows[e0:e1]], beta)
        eb, sb = _slices(B[:, cols[e0:e1]].T, beta)   # entry e: row e of each
        terms = []
        for s, qa in enumerate(sa):
            for t, qb in enumerate(sb):
                g = np.einsum("ek,ek->e", qa, qb)  # integer partial sums below 2^53: exact
                ex = (ea + eb) - beta * (s + t + 2)
                term = np.ldexp(g, ex)
                if not np.array_equal(np.ldexp(term, -ex), g):
                    raise ArithmeticError("scaled term not exact (range)")
                terms.append(term)
        T = np.stack(terms + [-C[e0:e1]])
        for e in range(e1 - e0):
            out[e0 + e] = math.fsum(T[:, e].tolist())
    return out


def bound_ratio_from_residual(res, absum, k):
    """Max of |res| / (2 k 2^-53 absum) (entries with a zero bound must be
    exact: ratio 0 when they are, inf otherwise)."""
    res = np.abs(np.asarray(res, dtype=np.float64))
    bound = 2.0 * k * 2.0 ** -53 * np.asarray(absum, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, res / np.where(bound > 0, bound, 1.0), np.where(res == 0, 0.0, np.inf))
    return float(ratio.max()) if ratio.size else 0.0


def error_bound_ratio_sliced(A, B, C):
    """:func:`error_bound_ratio` for a block with the exact residual from
    slices; (|A||B|)_ij from one float64 product of the magnitudes (all terms
    positive: relative error below K 2^-53, which moves the ratio by that
    relative amount at most)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    res = exact_residual_sliced(A, B, C)
    return bound_ratio_from_residual(res, np.abs(A) @ np.abs(B), A.shape[1])


def error_bound_ratio_pairs(A, B, C, rows, cols):
    """:func:`error_bound_ratio_sliced` for the entry pairs (rows[e], cols[e])."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    res = exact_residual_pairs(A, B, C, rows, cols)
    absum = np.einsum("ek,ek->e", np.abs(A[np.asarray(rows)]), np.abs(B[:, np.asarray(cols)].T))
    return bound_ratio_from_residual(res, absum, A.shape[1])


def residues_of_moduli(A, B, r, ls, ceiling=MODULUS_CEILING):
    """{l: residues in [0, m_l) of C' = A'B' modulo the l-th of r moduli} for
    the whole product and each l in ls, from the balanced residues of A' and
    B' and exact float64 products (as :func:`mod_product_direct`, a block of
    rows at a time); memory is one integer copy of each operand rather than
    all r residues and limb digits."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    k = A.shape[1]
    mods = moduli(r, ceiling)
    _, pA, pB = bit_budget(k, r, ceiling)
    if k * 128 * 128 >= 2 ** 53:
        raise OverflowError("direct product not exact in float64")
    ai = scale_round(A, row_shifts(A, pA))
    Bt = np.ascontiguousarray(B.T)
    bi = scale_round(Bt, row_shifts(Bt, pB))
    del Bt
    out = {}
    for l in ls:
        m = mods[l]
        a = balanced_residue_array(ai, m)
        bf = np.ascontiguousarray(balanced_residue_array(bi, m).T, dtype=np.float64)
        res = np.empty((A.shape[0], B.shape[1]), dtype=np.int64)
        step = 512
        for i in range(0, A.shape[0], step):
            # |residues| <= 128: every partial sum is an integer below 2^53, exact
            prod = a[i:i + step].astype(np.float64) @ bf
            res[i:i + step] = np.mod(np.rint(prod).astype(np.int64), m)
        out[l] = res
    return out


def residues_one_modulus(A, B, r, l, ceiling=MODULUS_CEILING):
    """:func:`residues_of_moduli` for one modulus."""
    return residues_of_moduli(A, B, r, [l], ceiling)[l]
