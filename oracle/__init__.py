"""CPU oracle for Ozaki scheme II FP64 emulation on FP4 tensor cores.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, table or constant generator with the CUDA library; the two meet only
in the seeded input generators of ``workloads.py``.

Sources, cited by title and section:

* [TME4] "The Missing Fourth Term for the Emulation Tensor Memory Equilibrium
  (TME) Model: The Residue Deconstruction Cost" (arXiv 2610.10924), abstract:
  every streamed fp64 operand is scaled, rounded and reduced modulo each of the
  r moduli; the TME time model and the threshold OI* = c_q r P_fp64 / (8 P_int).
* [AWE] arXiv 2609.24519 (Adaptive Weight Encoding for FP4 tensor cores),
  English abstract: the set S of FP4 values times two holds every residue
  modulo 13; base-13 limbs with weights (1, 13, 169); 9 FP4 GEMMs for
  INT8 x INT8; the formulation holds modulo m (Ozaki scheme II residues).

Parity status per function is listed in the module docstrings.  Functions
with no independent pin say "parity unpinned".
"""

from .ozaki2 import (  # noqa: F401
    S, BASE, LIMB_WEIGHTS, N_LIMBS, MODULUS_CEILING, MODULUS_CEILING_2LIMB, MODULUS_CEILING_WIDE, MIXED,
    accumulator_growth,
    single_digit_moduli, single_digit_set, single_digit, digits_of_modulus, products_per_modulus,
    moduli, modulus_product, bit_budget, frexp_exponent, row_shifts,
    scale_round_scalar, scale_round, balanced_residue, balanced_residue_array,
    digit_of_class, limb_split, limb_table_int8, limb_digits,
    e2m1_value, e2m1_code, limb_products, mod_recombine, mod_product_direct,
    crt, crt_array, scale_back, scale_back_array, deconstruct,
    dgemm, dgemm_block, igemm_s8, igemm_s8_direct,
    exact_dot_fraction, two_product, exact_residual, abs_product_sum,
    error_bound_ratio, exact_residual_sliced, exact_residual_pairs,
    error_bound_ratio_sliced, error_bound_ratio_pairs, residues_one_modulus, residues_of_moduli,
)
from .cost_model import oi_star, tme_time, deconstruction_time  # noqa: F401
from . import int4_int8  # noqa: F401  (INT4 x INT8 in four FP4 products)
