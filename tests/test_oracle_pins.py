"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against what the sources print (the golden file),
against a definition from outside the method (the e2m1 format, exact rational
arithmetic, brute force), or against a closed form.  None re-types the
oracle's own formula.
"""

import math
from fractions import Fraction
import itertools

import numpy as np
import pytest

import oracle
from workloads import make_pair


# --------------------------------------------------------------------------
# S, limbs, FP4 codes  (Adaptive Weight Encoding abstract)
# --------------------------------------------------------------------------

def test_S_matches_printed_set(golden):
    assert sorted(oracle.S) == sorted(golden["S"]["value"])
    assert oracle.BASE == golden["digit_base"]["value"]
    assert list(oracle.LIMB_WEIGHTS) == golden["limb_weights"]["value"]


def test_S_covers_every_residue_mod_13(golden):
    classes = {d % 13 for d in golden["S"]["value"]}
    assert classes == set(range(13))
    # the oracle's digit choice lands in S and in the right class for all 13
    for c in range(13):
        d = oracle.digit_of_class(c)
        assert d in golden["S"]["value"] and d % 13 == c


def test_S_is_twice_the_e2m1_values(golden):
    # e2m1 per the OCP MX format: 1 sign bit, 2 exponent bits (bias 1),
    # 1 mantissa bit, exponent 0 subnormal.  Decoded independently here.
    vals = set()
    for code in range(16):
        s = -1 if code >> 3 else 1
        e = (code >> 1) & 3
        m = code & 1
        v = (m / 2.0) if e == 0 else (2.0 ** (e - 1)) * (1 + m / 2.0)
        vals.add(s * v * 2)
        assert oracle.e2m1_value(code) == s * v
    assert {int(v) for v in vals} == set(golden["S"]["value"])


def test_e2m1_code_roundtrip():
    for d in oracle.S:
        code = oracle.e2m1_code(d)
        assert 0 <= code < 16 and code != 8
        assert oracle.e2m1_value(code) * 2 == d


def test_int8_limb_roundtrip_exhaustive(golden):
    w = golden["limb_weights"]["value"]
    S = set(golden["S"]["value"])
    for x in range(-128, 128):
        d = oracle.limb_split(x)
        assert len(d) == 3
        assert all(di in S for di in d)
        assert d[0] * w[0] + d[1] * w[1] + d[2] * w[2] == x
        assert abs(d[0]) <= 8 and abs(d[1]) <= 8 and d[2] in (-1, 0, 1)


def _splits(x):
    try:
        oracle.limb_split(x)
        return True
    except ValueError:
        return False


def test_limb_split_range_is_pm732():
    # The greedy 3-digit split (top digit in S) covers every integer of
    # [-732, 732] and neither neighbour: the widest interval around zero.
    assert all(_splits(x) for x in range(-732, 733))
    assert not _splits(733) and not _splits(-733)


def test_limb_sums_leave_S(golden):
    # The printed reason Karatsuba does not apply: limb sums reach +-24.
    S = golden["S"]["value"]
    sums = {a + b for a in S for b in S}
    assert max(sums) == golden["limb_sum_reach"]["value"]
    assert not sums <= set(S)


def test_limb_digits_table_matches_scalar():
    X = np.arange(-128, 128).reshape(16, 16)
    d = oracle.limb_digits(X)
    for idx, x in np.ndenumerate(X):
        assert tuple(int(d[l][idx]) for l in range(3)) == oracle.limb_split(int(x))


# --------------------------------------------------------------------------
# Moduli and bit budget
# --------------------------------------------------------------------------

def test_moduli_greedy_bruteforce():
    mods = oracle.moduli(16)
    assert mods[0] == 256
    for i, m in enumerate(mods):
        for j in range(i):
            assert math.gcd(m, mods[j]) == 1
        # no skipped integer between the previous modulus and this one was usable
        lo, hi = m + 1, (mods[i - 1] - 1 if i else 256)
        for c in range(lo, hi + 1):
            assert any(math.gcd(c, mods[j]) != 1 for j in range(i))


def test_bit_budget_is_tight():
    for k in (1, 2, 3, 255, 256, 8192, 65536):
        for r in (4, 8, 11, 13, 16):
            P, pA, pB = oracle.bit_budget(k, r)
            M = oracle.modulus_product(r)
            assert 2 * k * 2 ** P < M <= 2 * k * 2 ** (P + 1)
            assert pA + pB == P and pA - pB in (0, 1)


def test_bit_budget_rejects_too_few_moduli():
    with pytest.raises(ValueError):
        oracle.bit_budget(200, 1)  # M = 256 <= 2 * 200


# --------------------------------------------------------------------------
# Scaling and rounding
# --------------------------------------------------------------------------

def _check_round_half_even_ties(oz):
    """Ties of the scaled values round to the even integer, in the scalar
    (Fraction) rounding and in the vectorised integer rounding alike."""
    cases = [(2.5, 0, 2), (3.5, 0, 4), (-2.5, 0, -2), (0.5, 0, 0), (1.5, 0, 2), (-1.5, 0, -2),
             (5.0, -1, 2), (7.0, -1, 4), (0.75, 1, 2), (2.0 ** -1074 * 3, 1073, 2)]
    for x, s, want in cases:
        assert oz.scale_round_scalar(x, s) == want, (x, s)
        got = oz.scale_round(np.array([[x]]), np.array([s]))
        assert int(got[0, 0]) == want, (x, s, int(got[0, 0]))


def test_round_half_even_ties():
    import oracle.ozaki2 as oz
    _check_round_half_even_ties(oz)


def _edge_values():
    vals = [0.0, -0.0, 1.0, -1.0, 0.5, 1.5, 2.5, -2.5, 3.5, 2.0 ** -1074, -2.0 ** -1074,
            2.0 ** -1022, 2.0 ** -1022 * 1.5, 1e-310, -3e-320, 1e300, -1.7976931348623157e308,
            np.nextafter(1.0, 2.0), np.nextafter(1.0, 0.0), 0.1, 1 / 3.0]
    return np.array(vals)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_scale_round_vector_matches_fraction(seed):
    rng = np.random.default_rng(seed)
    rows = 6
    X = np.ldexp(rng.uniform(-1, 1, (rows, 40)), rng.integers(-60, 60, (rows, 40)))
    X[0, :len(_edge_values())] = _edge_values()
    X[1, :5] = [0.5, 1.5, 2.5, 3.5, -0.5]
    for p in (0, 1, 7, 30, 53, 62):
        s = oracle.row_shifts(X, p)
        got = oracle.scale_round(X, s)
        for i in range(rows):
            for k in range(X.shape[1]):
                exp = oracle.scale_round_scalar(X[i, k], s[i])
                assert got[i, k] == exp, (i, k, X[i, k], s[i], p)
            assert np.max(np.abs(got[i])) <= 2 ** p


def test_scale_round_zeros_beside_tiny_values():
    # A row of tiny magnitudes takes a shift near 1000; its zeros must stay 0
    # (no overflow), and every element must match the Fraction rounding.
    X = np.array([[0.0, 5e-300, -7e-301, 0.0, 2.0 ** -1074], [1.0, -3.0, 0.0, 0.5, 2.5]])
    for p in (30, 52, 62):
        s = oracle.row_shifts(X, p)
        got = oracle.scale_round(X, s)
        for i in range(2):
            for k in range(X.shape[1]):
                assert got[i, k] == oracle.scale_round_scalar(X[i, k], s[i])


def test_row_shift_scaling_is_tight():
    # After scaling, the largest |X'| of each nonzero row lies in [2^(p-1), 2^p].
    A, _ = make_pair(32, 1, 300, seed=7, dist="wide")
    A[3] = 0.0
    for p in (10, 44, 62):
        s = oracle.row_shifts(A, p)
        X = oracle.scale_round(A, s)
        for i in range(A.shape[0]):
            mx = int(np.max(np.abs(X[i])))
            if i == 3:
                assert mx == 0 and s[i] == 0
            else:
                assert 2 ** (p - 1) <= mx <= 2 ** p


def test_frexp_exponent_definition():
    for x in [1.0, 0.75, 3.0, 2.0 ** -1074, 1e308, 0.1]:
        e = oracle.frexp_exponent(x)
        assert Fraction(2) ** (e - 1) <= Fraction(x) < Fraction(2) ** e


# --------------------------------------------------------------------------
# Residues and CRT
# --------------------------------------------------------------------------

def test_balanced_residue_range_and_congruence():
    rng = np.random.default_rng(3)
    xs = list(rng.integers(-2 ** 62, 2 ** 62, 2000)) + [0, 1, -1, 127, 128, -128, -129, 2 ** 62, -2 ** 62]
    for m in oracle.moduli(16):
        arr = oracle.balanced_residue_array(np.array(xs, dtype=np.int64), m)
        for x, v in zip(xs, arr):
            assert (int(x) - int(v)) % m == 0
            assert -(m // 2) <= v <= (m + 1) // 2 - 1
            assert -128 <= v <= 127
            assert v == oracle.balanced_residue(int(x), m)


def test_crt_small_moduli_bruteforce():
    mods = [4, 3, 5]  # M = 60, symmetric range (-30, 30)
    for x in range(-29, 30):
        res = [x % m for m in mods]
        assert oracle.crt(res, mods) == x


def test_crt_roundtrip_random():
    rng = np.random.default_rng(11)
    for r in (2, 5, 11, 13, 16):
        mods = oracle.moduli(r)
        M = oracle.modulus_product(r)
        for _ in range(200):
            x = int.from_bytes(rng.bytes(18), "little") % M - M // 2
            if abs(x) >= M // 2:
                continue
            assert oracle.crt([x % m for m in mods], mods) == x
            assert oracle.crt([oracle.balanced_residue(x, m) for m in mods], mods) == x


def test_crt_array_matches_scalar():
    mods = oracle.moduli(6)
    rng = np.random.default_rng(5)
    res = np.stack([rng.integers(0, m, (3, 4)) for m in mods])
    arr = oracle.crt_array(res, mods)
    for idx in np.ndindex(3, 4):
        assert arr[idx] == oracle.crt([res[l][idx] for l in range(6)], mods)


# --------------------------------------------------------------------------
# Limb products, INT8 GEMM, modular recombination
# --------------------------------------------------------------------------

def _triple_loop(A, B):
    M, K = len(A), len(A[0])
    N = len(B[0])
    return [[sum(int(A[i][k]) * int(B[k][j]) for k in range(K)) for j in range(N)] for i in range(M)]


def test_igemm_matches_triple_loop_nonsquare(golden):
    A, B = make_pair(5, 7, 11, seed=21, dist="int8")
    A[0, :] = -128
    B[:, 0] = -128
    C = oracle.igemm_s8(A, B)
    assert C.tolist() == _triple_loop(A.tolist(), B.tolist())
    # 9 limb products
    Ad, Bd = oracle.limb_digits(A), oracle.limb_digits(B)
    assert oracle.limb_products(Ad, Bd).shape[:2] == (3, 3)
    assert 3 * 3 == golden["fp4_gemms_int8xint8"]["value"]


def test_igemm_closed_forms():
    K = 256
    A = np.full((4, K), 112, dtype=np.int8)
    B = np.full((K, 3), -112, dtype=np.int8)
    assert (oracle.igemm_s8(A, B) == -112 * 112 * K).all()
    I = np.eye(16, dtype=np.int8)
    X, _ = make_pair(16, 1, 16, seed=4, dist="int8")
    assert (oracle.igemm_s8(I, X) == X.astype(np.int32)).all()
    perm = np.random.default_rng(0).permutation(16)
    Pm = np.eye(16, dtype=np.int8)[:, perm]  # (X @ Pm)[:, j] = X[:, perm[j]]
    assert (oracle.igemm_s8(X, Pm) == X[:, perm].astype(np.int32)).all()


def test_igemm_matches_direct_medium():
    A, B = make_pair(70, 90, 300, seed=22, dist="int8")
    assert (oracle.igemm_s8(A, B) == oracle.igemm_s8_direct(A, B)).all()


def test_mod_recombine_matches_direct_modular_product():
    A, B = make_pair(9, 8, 200, seed=23, dist="int8")
    Ad, Bd = oracle.limb_digits(A), oracle.limb_digits(B)
    P = oracle.limb_products(Ad, Bd)
    for m in oracle.moduli(13):
        a = oracle.balanced_residue_array(A.astype(np.int64), m)
        b = oracle.balanced_residue_array(B.astype(np.int64), m)
        Pa = oracle.limb_products(oracle.limb_digits(a), oracle.limb_digits(b))
        got = oracle.mod_recombine(Pa, m)
        assert (got == oracle.mod_product_direct(a, b, m)).all()
        # and the int8 products themselves, brute force, reduced
        ref = np.mod(np.array(_triple_loop(a.tolist(), b.tolist())), m)
        assert (got == ref).all()
    assert P.dtype == np.int64


# --------------------------------------------------------------------------
# End to end: the fp64 product
# --------------------------------------------------------------------------

def test_crt_recovers_integer_product():
    A, B = make_pair(6, 5, 33, seed=31, dist="uniform")
    C, st = oracle.dgemm(A, B, 13, stages=True)
    exact_int = st["a"]["xint"].astype(object) @ st["b"]["xint"].T.astype(object)
    assert (st["Cp"] == exact_int).all()
    for l, m in enumerate(st["mods"]):
        assert (st["res"][l] == np.mod(exact_int, m).astype(np.int64)).all()


def test_dgemm_exact_on_small_integers():
    rng = np.random.default_rng(8)
    A = rng.integers(-1000, 1000, (7, 13)).astype(np.float64)
    B = rng.integers(-1000, 1000, (13, 9)).astype(np.float64)
    C = oracle.dgemm(A, B, 8)
    assert (C == A @ B).all()  # integers below 2^53: fp64 product is exact


def test_dgemm_k1_is_correctly_rounded_product():
    # K = 1 with p_A, p_B >= 53: C_ij = RN(a_i b_j), which IEEE multiplication gives.
    A, B = make_pair(11, 10, 1, seed=32, dist="wide")
    P, pA, pB = oracle.bit_budget(1, 16)
    assert pB >= 53
    C = oracle.dgemm(A, B, 16)
    assert (C == A * B).all()


def test_dgemm_matches_exact_rational_tiny():
    # K = 5 makes the bound 10u: r = 16 (p_A, p_B about 60 bits) is needed.
    A, B = make_pair(3, 4, 5, seed=33, dist="uniform")
    C, st = oracle.dgemm(A, B, 16, stages=True)
    for i in range(3):
        for j in range(4):
            ex = oracle.exact_dot_fraction(A[i], B[:, j])
            bound = 2 * 5 * Fraction(2) ** -53 * oracle.exact_dot_fraction(np.abs(A[i]), np.abs(B[:, j]))
            assert abs(Fraction(C[i, j]) - ex) <= bound


def test_exact_residual_matches_fraction():
    A, B = make_pair(4, 3, 17, seed=34, dist="wide")
    C = A @ B
    res = oracle.exact_residual(A, B, C)
    for i in range(4):
        for j in range(3):
            ex = oracle.exact_dot_fraction(A[i], B[:, j]) - Fraction(C[i, j])
            assert res[i, j] == float(ex)


@pytest.mark.parametrize("dist,r", [("uniform", 13), ("wide", 14), ("normal", 13)])
def test_dgemm_within_bound(dist, r):
    A, B = make_pair(24, 20, 256, seed=35, dist=dist)
    C = oracle.dgemm(A, B, r)
    assert oracle.error_bound_ratio(A, B, C) <= 1.0


def test_dgemm_too_few_moduli_breaks_bound():
    # With r = 5 (about 39 bits) the product cannot reach fp64 accuracy.
    A, B = make_pair(8, 8, 64, seed=36, dist="uniform")
    C = oracle.dgemm(A, B, 5)
    assert oracle.error_bound_ratio(A, B, C) > 1.0


def test_dgemm_zero_rows_and_cols():
    A, B = make_pair(5, 6, 30, seed=37, dist="normal")
    A[2] = 0.0
    B[:, 4] = 0.0
    C = oracle.dgemm(A, B, 13)
    assert (C[2] == 0).all() and (C[:, 4] == 0).all()
    assert oracle.error_bound_ratio(A, B, C) <= 1.0


def test_dgemm_block_matches_full():
    A, B = make_pair(20, 18, 64, seed=38, dist="wide")
    C = oracle.dgemm(A, B, 13)
    rows, cols = np.array([1, 5, 19]), np.array([0, 7, 17])
    Cb = oracle.dgemm_block(A, B, 13, rows=rows, cols=cols)
    assert (Cb == C[np.ix_(rows, cols)]).all()


# --------------------------------------------------------------------------
# Sensitivity: a planted mistake in the oracle must fail a pin
# --------------------------------------------------------------------------

def test_planted_wrong_weight_is_caught(monkeypatch):
    import oracle.ozaki2 as oz
    monkeypatch.setattr(oz, "LIMB_WEIGHTS", (1, 13, 170))
    A, B = make_pair(5, 7, 11, seed=21, dist="int8")
    A[0, 0] = 127  # a value whose top limb is nonzero
    B[0, 0] = 127
    assert oz.igemm_s8(A, B).tolist() != _triple_loop(A.tolist(), B.tolist())


def test_planted_transposed_operand_is_caught():
    A, B = make_pair(5, 5, 5, seed=24, dist="int8")
    wrong = oracle.igemm_s8(A, B.T.copy())
    assert wrong.tolist() != _triple_loop(A.tolist(), B.tolist())


def test_planted_wrong_rounding_is_caught(monkeypatch):
    # A floor planted inside the oracle's vectorised rounding (the one every
    # pipeline uses) must make the tie pin above fail.
    import oracle.ozaki2 as oz
    real = oz.scale_round

    def floored(X, shifts):
        X = np.asarray(X, dtype=np.float64)
        s = np.asarray(shifts, dtype=np.int64).reshape(-1, 1)
        return np.array([[math.floor(Fraction(float(x)) * Fraction(2) ** int(si)) for x in row]
                         for row, si in zip(X, s[:, 0])], dtype=np.int64)

    monkeypatch.setattr(oz, "scale_round", floored)
    with pytest.raises(AssertionError):
        _check_round_half_even_ties(oz)
    monkeypatch.setattr(oz, "scale_round", real)
    _check_round_half_even_ties(oz)


def test_planted_double_rounding_in_scale_back_is_caught(monkeypatch):
    # Rounding C' to fp64 first and scaling afterwards (two roundings) must
    # fail the subnormal-range pins below.
    import oracle.ozaki2 as oz
    monkeypatch.setattr(oz, "scale_back", lambda Cp, S: math.ldexp(float(int(Cp)), -int(S)))
    with pytest.raises(AssertionError):
        _check_scale_back_subnormal(oz)


# --------------------------------------------------------------------------
# TME time model and OI* (The Missing Fourth Term ..., abstract)
# --------------------------------------------------------------------------

def _bisect_crossing(gap, lo=1e-6, hi=1e6):
    for _ in range(200):
        mid = math.sqrt(lo * hi)
        if gap(mid) > 0:
            lo = mid
        else:
            hi = mid
    return lo


def test_oi_star_is_the_crossing_point():
    # OI* is where deconstruction time (infinite tensor throughput, no HBM
    # limit) equals native fp64 compute time.  Solve that by bisection.
    c_q, r, P_fp64, P_int = 3.0, 13, 1.2e12, 3.0e13
    n_in = 1e9                 # fp64 inputs streamed
    bytes_ = 8 * n_in

    def gap(oi):
        flops = oi * bytes_
        return oracle.deconstruction_time(n_in, c_q, r, P_int) - flops / P_fp64

    lo = _bisect_crossing(gap)
    assert abs(lo - oracle.oi_star(c_q, r, P_fp64, P_int)) / lo < 1e-9


def test_tme_time_crossing_with_unbounded_tensor_and_hbm():
    # The same crossing through the full four-term model: with unbounded
    # tensor and HBM rates and a free reconstruction, the model's emulation
    # time equals native fp64 time exactly at the closed-form OI*, for any
    # problem size ([TME4] abstract: the threshold holds regardless of
    # tensor-core throughput).
    c_q, r, P_fp64, P_int = 2.5, 12, 1.3e12, 4.1e13
    for n_in in (1e6, 3e9):
        def gap(oi):
            flops = oi * 8 * n_in
            t_emu = oracle.tme_time(flops * 9 * r, math.inf, 8 * n_in, math.inf, 1000, 0.0,
                                    n_inputs=n_in, c_q=c_q, r=r, P_int=P_int)
            return t_emu - flops / P_fp64
        lo = _bisect_crossing(gap)
        assert abs(lo - oracle.oi_star(c_q, r, P_fp64, P_int)) / lo < 1e-9


def test_tme_time_terms_and_dense_gemm_unaffected():
    # The model is the larger of the tensor and HBM terms plus the two
    # per-element terms: each term alone is recovered when the others vanish.
    assert oracle.tme_time(6.0, 2.0, 0.0, 1.0, 0, 0.0) == 3.0          # tensor-bound
    assert oracle.tme_time(0.0, 1.0, 10.0, 2.0, 0, 0.0) == 5.0         # HBM-bound
    assert oracle.tme_time(0.0, 1.0, 0.0, 1.0, 4, 0.25) == 1.0          # reconstruction only
    assert oracle.tme_time(0.0, 1.0, 0.0, 1.0, 0, 0.0, n_inputs=8, c_q=2.0, r=3, P_int=4.0) == 12.0
    # [TME4] abstract: dense GEMM is unaffected by the fourth term.  An
    # n x n x n product streams 2 n^2 inputs against 2 n^3 flop, so the
    # fourth term's share of the time halves each time n doubles and
    # vanishes for large n, whatever c_q and the integer rate are.
    r = 13

    def overhead(n, c_q, P_int):
        flops = 9 * r * 2.0 * n ** 3
        t3 = oracle.tme_time(flops, 1e16, 0.0, 1.0, n * n, 0.0)
        t4 = oracle.tme_time(flops, 1e16, 0.0, 1.0, n * n, 0.0, n_inputs=2 * n * n, c_q=c_q, r=r, P_int=P_int)
        return (t4 - t3) / t3

    for c_q, P_int in ((3.0, 1e14), (13.0, 7e13)):
        assert overhead(8192, c_q, P_int) == pytest.approx(2 * overhead(16384, c_q, P_int), rel=1e-12)
        assert 0 < overhead(65536, c_q, P_int) < 0.01


def test_scale_back_overflow_rounds_to_signed_inf():
    # Round to nearest: a value at or beyond the largest finite double plus
    # half an ulp becomes +-inf, with the sign of the exact value.
    big = 2 ** 1100
    assert oracle.scale_back(big, 0) == math.inf
    assert oracle.scale_back(-big, 0) == -math.inf
    assert oracle.scale_back(3, -1100) == math.inf
    assert oracle.scale_back(3, 1100) == 0.0
    # The largest finite double, and the tie just above it, which IEEE
    # round-to-nearest sends to infinity.
    fmax = (2 ** 53 - 1) * 2 ** 971
    assert oracle.scale_back(fmax, 0) == 1.7976931348623157e308
    # fmax + ulp/2 = (2^54 - 1) 2^970 is a tie; the even neighbour is 2^1024.
    assert oracle.scale_back(2 ** 54 - 1, -970) == math.inf
    # a quarter ulp above fmax rounds back down to it
    assert oracle.scale_back(2 ** 55 - 3, -969) == 1.7976931348623157e308


def _check_scale_back_subnormal(oz):
    """Hand-derived single roundings in the subnormal range, where one
    rounding and two (to 53 bits, then to the subnormal grid) differ."""
    tiny = 2.0 ** -1074                       # the subnormal grid
    # 1.5 grid units: a tie, rounded to the even 2 units.
    assert oz.scale_back(3, 1075) == 2 * tiny
    assert oz.scale_back(-3, 1075) == -2 * tiny
    # 0.5 grid units: a tie between 0 and 1 unit, rounded to even 0.
    assert oz.scale_back(1, 1075) == 0.0
    # 0.75 grid units rounds up to one unit.
    assert oz.scale_back(3, 1076) == tiny
    # 2.5 units + 2^-61 units: above the tie, so one rounding gives 3 units.
    # Rounding C' = 5 2^60 + 1 to 53 bits first drops the +1 and leaves the
    # exact tie 2.5 units, which then rounds to even, 2 units.
    cp = 5 * 2 ** 60 + 1
    assert oz.scale_back(cp, 1135) == 3 * tiny
    assert oz.scale_back(-cp, 1135) == -3 * tiny
    # Just below the smallest normal: (2^52 - 0.5) units is a tie that rounds
    # to even 2^52 units, the smallest normal number.
    assert oz.scale_back(2 ** 53 - 1, 1075) == 2.0 ** -1022


def test_scale_back_subnormal_single_rounding():
    import oracle.ozaki2 as oz
    _check_scale_back_subnormal(oz)


# --------------------------------------------------------------------------
# The exact product at full size (error-free slices)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dist,k", [("wide", 300), ("normal", 1000), ("uniform", 4097)])
def test_sliced_residual_matches_fraction(dist, k):
    A, B = make_pair(3, 4, k, seed=40, dist=dist)
    C = A @ B
    C[0, 0] = np.nextafter(C[0, 0], np.inf)   # a residual of one ulp
    res = oracle.exact_residual_sliced(A, B, C, block=3)
    for i in range(3):
        for j in range(4):
            ex = oracle.exact_dot_fraction(A[i], B[:, j]) - Fraction(C[i, j])
            assert res[i, j] == float(ex), (i, j)
    rows, cols = [2, 0, 1, 2], [3, 0, 1, 3]
    pr = oracle.exact_residual_pairs(A, B, C[rows, cols], rows, cols, block=3)
    assert (pr == res[rows, cols]).all()


def test_sliced_residual_exact_under_cancellation():
    # A row built so that the exact dot product is a tiny value far below
    # the terms: x, -x pairs plus one small term (and subnormal-free tails).
    rng = np.random.default_rng(41)
    k = 2048
    a = np.ldexp(rng.uniform(0.5, 1, k), rng.integers(-30, 30, k))
    b = np.ldexp(rng.uniform(0.5, 1, k), rng.integers(-30, 30, k))
    a[k // 2:] = a[:k // 2]
    b[k // 2:] = -b[:k // 2]
    a[0] *= 1 + 2.0 ** -50
    A, B = a[None, :], b[:, None]
    C = np.zeros((1, 1))
    res = oracle.exact_residual_sliced(A, B, C)
    assert res[0, 0] == float(oracle.exact_dot_fraction(a, b)) != 0.0


def test_sliced_bound_ratio_matches_fraction_bound():
    A, B = make_pair(6, 5, 700, seed=42, dist="wide")
    C = oracle.dgemm(A, B, 14)
    assert oracle.error_bound_ratio_sliced(A, B, C) == pytest.approx(oracle.error_bound_ratio(A, B, C), rel=1e-12)
    C[1, 1] = np.nextafter(C[1, 1], np.inf) * (1 + 2.0 ** -30)
    assert oracle.error_bound_ratio_sliced(A, B, C) > 1.0


def test_residues_one_modulus_matches_stages():
    A, B = make_pair(9, 7, 130, seed=43, dist="wide")
    _, st = oracle.dgemm(A, B, 13, stages=True)
    for l in (0, 5, 12):
        assert (oracle.residues_one_modulus(A, B, 13, l) == st["res"][l]).all()
    both = oracle.residues_of_moduli(A, B, 13, (0, 12))
    assert (both[0] == st["res"][0]).all() and (both[12] == st["res"][12]).all()


# --------------------------------------------------------------------------
# Two-limb reading: moduli up to 113, residues in [-56, 56], top digit 0
# --------------------------------------------------------------------------

def test_two_limb_range_is_pm56():
    # Every integer of [-56, 56] splits with d2 = 0 (two limbs in S); 57 and
    # -57 are the first that need the third limb.
    for x in range(-56, 57):
        d0, d1, d2 = oracle.limb_split(x)
        assert d2 == 0 and d0 in oracle.S and d1 in oracle.S and d0 + 13 * d1 == x
    assert oracle.limb_split(57)[2] != 0 and oracle.limb_split(-57)[2] != 0
    # Brute force over all pairs of S: no wider symmetric interval is reachable.
    reach = {a + 13 * b for a in oracle.S for b in oracle.S}
    assert all(x in reach for x in range(-56, 57)) and 57 not in reach


def test_two_limb_moduli_greedy_and_residue_range():
    mods = oracle.moduli(16, oracle.MODULUS_CEILING_2LIMB)
    assert mods[0] == 113 and 2 * (113 // 2) + 1 == 113
    for i, m in enumerate(mods):
        for j in range(i):
            assert math.gcd(m, mods[j]) == 1
        lo, hi = m + 1, (mods[i - 1] - 1 if i else 113)
        for c in range(lo, hi + 1):
            assert any(math.gcd(c, mods[j]) != 1 for j in range(i))
        bal = oracle.balanced_residue_array(np.arange(-3 * m, 3 * m), m)
        assert bal.min() >= -56 and bal.max() <= 56
        assert ((bal - np.arange(-3 * m, 3 * m)) % m == 0).all()


def test_two_limb_deconstruct_has_zero_top_digit():
    A, _ = make_pair(9, 1, 200, seed=38, dist="wide")
    _, pA, _ = oracle.bit_budget(200, 16, oracle.MODULUS_CEILING_2LIMB)
    d = oracle.deconstruct(A, pA, 16, oracle.MODULUS_CEILING_2LIMB)
    assert (d["digits"][:, 2] == 0).all()
    assert (d["digits"][:, 0] + 13 * d["digits"][:, 1] == d["res"]).all()


def test_two_limb_crt_recovers_integer_product_and_bound():
    A, B = make_pair(6, 5, 33, seed=39, dist="uniform")
    C, st = oracle.dgemm(A, B, 16, stages=True, ceiling=oracle.MODULUS_CEILING_2LIMB)
    exact_int = st["a"]["xint"].astype(object) @ st["b"]["xint"].T.astype(object)
    assert (st["Cp"] == exact_int).all()
    # Bits per modulus are fewer (6.8 against 8): at K = 256 on wide-range
    # data 17 two-limb moduli (P = 100) meet the bound as 14 of the 3-limb
    # list (P = 101) do; 16 (P = 94) do not, like 13 of the 3-limb list.
    A, B = make_pair(24, 20, 256, seed=35, dist="wide")
    C = oracle.dgemm(A, B, 17, ceiling=oracle.MODULUS_CEILING_2LIMB)
    assert oracle.error_bound_ratio(A, B, C) <= 1.0
    C = oracle.dgemm(A, B, 16, ceiling=oracle.MODULUS_CEILING_2LIMB)
    assert oracle.error_bound_ratio(A, B, C) > 1.0
