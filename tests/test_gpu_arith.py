"""Exhaustive device checks of two arithmetic shortcuts in the quantizers,
through the test-only entry point lpq_selftest_arith:

* the block-max division by 6 of the NVFP4 block scale (the product with
  RN(1/6) corrected once by a fused multiply-add of the exact residual, the
  correctly-rounded division by a constant of Markstein, "IA-64 and
  Elementary Functions", 2000, and Brisebarre and Muller, "Correctly rounded
  multiplication by arbitrary precision constants", 2008) equals the IEEE
  quotient x / 6 for every non-negative float;
* the stochastic E2M1 rounding computed on the FMA pipe (two values at a
  time) equals its definition (round up iff float(r >> 8) < frac * 2^24, the
  reading of "stochastic rounding of gradients" in "How to optimize
  Transformer-based models for low-precision training") for every float y in
  [0, 8] and +-inf/NaN at the extreme random words, and for every 24-bit
  threshold word at y values chosen at the binade edges of the E2M1 grid."""
import numpy as np
import pytest

from precision_transformer_gemms_gb300 import lpq

pytestmark = pytest.mark.gpu


def test_div6_equals_ieee_quotient_for_every_nonnegative_float():
    n, first = lpq.selftest_arith(0, 0, 0x7F800001)
    assert n == 0, f"{n} mismatches, first at bits {first:#x}"


def test_sr_rounding_every_y_at_extreme_words():
    top = 0x41000000  # 8.0: covers [0, 6], the saturation edge and beyond
    n, first = lpq.selftest_arith(1, 0, top * 8)
    assert n == 0, f"{n} mismatches, first at y bits {first >> 3:#x}, probe {first & 7}"
    for bits in (0x7F800000, 0x7FC00000, 0x7F800001, 0x7F7FFFFF):  # inf, NaN, signalling NaN, largest float
        n, first = lpq.selftest_arith(1, bits * 8, 8)
        assert n == 0, (hex(bits), first)


def _f32_bits(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


Y_EDGES = [2.0 ** -26, 2.0 ** -25, 0.1, 0.25, 0.3, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0,
           5.5, 6.0]


@pytest.mark.parametrize("y", Y_EDGES)
def test_sr_rounding_every_threshold_word(y):
    """Every 24-bit threshold r >> 8 for y and its float neighbours."""
    b = _f32_bits(y)
    for bits in (b - 1, b, b + 1):
        n, first = lpq.selftest_arith(2, 0, 1 << 24, bits)
        assert n == 0, f"y bits {bits:#x}: {n} mismatches, first at r >> 8 = {first}"
