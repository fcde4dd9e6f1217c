"""Test-side readers of the library's documented data layouts.

Decodes limb planes (FP4 e2m1 nibbles, layout of include/ozemu.h) into
integer digits with the oracle's e2m1 definition, and slices residues.
"""

import numpy as np

import oracle


def _digit_table():
    return np.array([int(round(2 * oracle.e2m1_value(c))) for c in range(16)], dtype=np.int64)


def decode_planes(planes, rows, k, r, limbs=3):
    """uint8 plane bytes -> digits (r, limbs, rows_p, k_p) as int64."""
    rows_p = (rows + 127) // 128 * 128
    k_p = (k + 127) // 128 * 128
    # [r][rows_p][k_p/128][limbs][64]: the limbs of each 128-element K block
    # side by side in a row.
    b = np.asarray(planes, dtype=np.uint8).reshape(r, rows_p, k_p // 128, limbs, 64)
    b = b.transpose(0, 3, 1, 2, 4).reshape(r, limbs, rows_p, k_p // 2)
    codes = np.empty((r, limbs, rows_p, k_p), dtype=np.uint8)
    codes[..., 0::2] = b & 0xF
    codes[..., 1::2] = b >> 4
    return _digit_table()[codes], codes


def limb_value(digits):
    """d0 + 13 d1 (+ 169 d2) along axis 1 of (r, limbs, ...)."""
    v = digits[:, 0] + 13 * digits[:, 1]
    if digits.shape[1] > 2:
        v = v + 169 * digits[:, 2]
    return v


def decode_planes_mixed(planes, rows, k, r, single=6):
    """Mixed-digit plane bytes -> digits (r, 2, rows_p, k_p): single-digit
    moduli first ([rows_p][k_p/2] each, second digit reported as 0), then
    two-digit moduli ([rows_p][k_p] each, the two-limb layout)."""
    rows_p = (rows + 127) // 128 * 128
    k_p = (k + 127) // 128 * 128
    ns = min(r, single)
    plane = rows_p * k_p // 2
    b = np.asarray(planes, dtype=np.uint8)
    d1, c1 = decode_planes(b[:ns * plane], rows, k, ns, limbs=1)
    digits = np.zeros((r, 2, rows_p, k_p), dtype=np.int64)
    codes = np.zeros((r, 2, rows_p, k_p), dtype=np.uint8)
    digits[:ns, :1] = d1
    codes[:ns, :1] = c1
    if r > ns:
        d2, c2 = decode_planes(b[ns * plane:], rows, k, r - ns, limbs=2)
        digits[ns:] = d2
        codes[ns:] = c2
    return digits, codes
