"""Exhaustive CPU checks of shortcuts the CUDA kernels take in place of the
exact definitions, replayed here in IEEE binary32/binary16 with numpy.

The int8 weight reconstruct computes q_w = RNE(v * 127 / 3.453125) ("exl3xpu"
README, "Prefill: int8 linears and oneDNN fused attention") as one binary32
product v * fp32(127 / 3.453125) rounded to nearest even, instead of exact
rational arithmetic.  That is valid only if the two agree for every codebook
value; here every 16-bit state is checked against the oracle's exact
quantiser.
"""
import numpy as np

import oracle


def test_int8_weight_formula_matches_exact_quantiser_for_every_state():
    v = oracle.codebook_table()                                   # fp16 value of each state
    scale = np.float32(127.0) / np.float32(3.453125)              # the kernel's constant, one RN division
    prod = v.astype(np.float32) * scale                           # one RN binary32 product
    q_formula = np.rint(prod).astype(np.int64)                    # round half to even
    q_exact = oracle.quant_weights(v).astype(np.int64)
    assert np.array_equal(q_formula, q_exact)
    # the exact tie of the rational rounding (byte sum 765: v * 127 / 3.453125
    # = 63.5, even -> 64) is among the states checked, and comes out even
    tie = oracle.bytesum_table() == 765
    assert tie.any() and np.all(q_formula[tie] == 64)


def test_int8_weight_constant_is_correctly_rounded():
    from fractions import Fraction
    c = np.float32(127.0) / np.float32(3.453125)
    exact = Fraction(127) / Fraction(3453125, 1000000)
    up, down = np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(0))
    err = abs(Fraction(float(c)) - exact)
    assert err <= abs(Fraction(float(up)) - exact) and err <= abs(Fraction(float(down)) - exact)
