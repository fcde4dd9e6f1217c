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
