"""The CRT + scale-back stage on its own, through the C ABI.

Residues of chosen integers C' in (-M/2, M/2) go in; the result must be the
oracle's single correct rounding of C' 2^-(s_i + t_j), bit for bit.  The
integers cover the whole range: random ones, small ones, powers of two, and
ones whose C'/M lies within 2^-8 .. 2^-30 of +-1/2 (where the kernel's quotient
estimate is ambiguous and it takes the mixed-radix digits), with shifts that
give normal, subnormal, zero and overflowing results.
"""

import random

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def oz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ozaki_ii_fp64_gb300 as oz
    oz.load()
    return oz


def chosen_integers(M, count, rng):
    half = M // 2
    vals = [0, 1, -1, 2, -2, half - 1, -(half - 1), half - 2, -(half - 2)]
    for e in (8, 9, 10, 11, 12, 20, 30):
        d = M >> (e + 1)  # M 2^-(e+1): C'/M = 1/2 - 2^-(e+1)
        vals += [half - d, -(half - d), half - d - 1, -(half - d) + 1]
    for b in range(0, M.bit_length() - 1, 7):
        vals += [1 << b, -(1 << b), (1 << b) - 1]
    while len(vals) < count:
        kind = rng.random()
        if kind < 0.6:
            v = rng.randrange(-half + 1, half)
        elif kind < 0.8:
            v = rng.randrange(-(1 << 40), 1 << 40)
        else:
            v = rng.choice([1, -1]) * (half - rng.randrange(1, 1 << 20))
        vals.append(v)
    vals = [v for v in vals if -half < v < half][:count]
    while len(vals) < count:
        vals.append(0)
    rng.shuffle(vals)
    return vals


@pytest.mark.parametrize("r,family", [(1, "three"), (2, "three"), (3, "three"), (5, "three"), (8, "three"),
                                      (11, "three"), (12, "three"), (13, "three"), (14, "three"), (16, "three"),
                                      (2, "two"), (3, "two"), (9, "two"), (16, "two"),
                                      (1, "mixed"), (2, "mixed"), (5, "mixed"), (6, "mixed"), (7, "mixed"),
                                      (13, "mixed"), (17, "mixed"), (19, "mixed"), (20, "mixed")])
def test_crt_stage_matches_oracle(oz, r, family):
    # The two-limb list has its even modulus (112) second, the others first:
    # near +-M/2 the mixed-radix fallback must still return C' itself.
    rng = random.Random(1000 + r + {"three": 0, "two": 50, "mixed": 100}[family])
    ceil = {"three": oracle.MODULUS_CEILING, "two": oracle.MODULUS_CEILING_2LIMB, "mixed": oracle.MIXED}[family]
    crt = {"three": oz.crt_f64, "two": oz.crt_f64_2limb, "mixed": oz.crt_f64_mixed}[family]
    mods = oracle.moduli(r, ceil)
    M = 1
    for mm in mods:
        M *= mm
    m, n = 48, 37
    ldr = (n + 15) // 16 * 16
    Cp = np.array(chosen_integers(M, m * n, rng), dtype=object).reshape(m, n)
    res = np.zeros((r, m, ldr), dtype=np.uint8)
    for l, mm in enumerate(mods):
        res[l, :, :n] = np.vectorize(lambda v: int(v) % mm, otypes=[np.int64])(Cp).astype(np.uint8)
    bits = M.bit_length()
    # shifts: results from subnormal to overflow and ordinary magnitudes
    sa = np.array([rng.randrange(-960, bits + 1100) for _ in range(m)], dtype=np.int32)
    sb = np.array([rng.randrange(-40, 40) for _ in range(n)], dtype=np.int32)
    sa[:8] = bits - 60  # ordinary results for the first rows
    expect = oracle.scale_back_array(Cp, sa, sb)
    C = crt(m, n, r, torch.from_numpy(res).to(DEV), torch.from_numpy(sa).to(DEV), torch.from_numpy(sb).to(DEV))
    assert oz.get_status() == oz.OZEMU_OK
    got = C.cpu().numpy()
    bad = np.argwhere(got.view(np.int64) != expect.view(np.int64))
    assert bad.size == 0, [(int(Cp[i, j]), int(sa[i] + sb[j]), got[i, j], expect[i, j]) for i, j in bad[:5]]
