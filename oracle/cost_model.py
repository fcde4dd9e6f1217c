"""Tensor-Memory-Equilibrium time model with the deconstruction term.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[TME4] abstract: the TME model takes the time of Ozaki scheme II emulation as
the larger of a tensor-core term and an HBM term, plus a per-output
reconstruction term; the note adds a per-input deconstruction term (c_q r SIMT
instructions for every streamed fp64 input) and derives the threshold
OI* = c_q r P_fp64 / (8 P_int), in flop per byte, below which emulation cannot
match native fp64 whatever the tensor-core throughput.

Reading (units are not printed): c_q is instructions per input element per
modulus, P_int integer instructions per second, P_fp64 native fp64 flop/s,
8 the bytes of one fp64 input.  Pins (tests/test_oracle_pins.py): the closed
form equals the crossing point of the deconstruction time and native fp64
time found by bisection, both from :func:`deconstruction_time` alone and
through the full :func:`tme_time` with unbounded tensor and HBM rates; each
term of :func:`tme_time` is recovered when the others vanish; and the fourth
term's share of a dense n^3 product halves when n doubles (the page's "dense
GEMM is unaffected").  The B300 value 0.56 flop/B is parity unpinned: none of
its constituents is printed.
"""


def deconstruction_time(n_inputs, c_q, r, P_int):
    """Seconds to scale, round and reduce n_inputs fp64 values mod r moduli."""
    return n_inputs * c_q * r / P_int


def tme_time(flop_tensor, P_tensor, bytes_hbm, bw_hbm, n_outputs, t_out,
             n_inputs=0, c_q=0.0, r=0, P_int=1.0):
    """max(tensor term, HBM term) + reconstruction + deconstruction (seconds)."""
    t = max(flop_tensor / P_tensor, bytes_hbm / bw_hbm) + n_outputs * t_out
    if n_inputs:
        t += deconstruction_time(n_inputs, c_q, r, P_int)
    return t


def oi_star(c_q, r, P_fp64, P_int):
    """Operational intensity (flop per fp64 byte) below which emulation loses."""
    return c_q * r * P_fp64 / (8.0 * P_int)
