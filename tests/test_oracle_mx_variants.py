"""Pins of the oracle's MX variants (MXFP8 with E5M2 codes, MXFP4 with packed
E2M1 codes; both with E8M0 scales per 32 values) against their definition,
independently of the oracle's arithmetic: the block exponent is the smallest
e with fmax * 2^e >= block amax (checked in exact rational arithmetic), the
E4M3 case is the already pinned MXFP8 quantizer, a brute-force rebuild of a
small tensor gives the same codes, nothing saturates, and the GEMM operand
kinds decode to code * 2^(scale - 127)."""
from fractions import Fraction

import numpy as np
import pytest

import oracle as o
from precision_transformer_gemms_gb300 import synth

FMAX = {o.E4M3: 448.0, o.E5M2: 57344.0, o.E2M1: 6.0}


def smallest_e(a, fmax):
    """min e in [-127, 127] with fmax * 2^e >= a (exact)."""
    a, f = Fraction(a), Fraction(fmax)
    for e in range(-127, 128):
        if f * Fraction(2) ** e >= a:
            return e
    return 127


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2, o.E2M1])
def test_block_exponent_is_the_smallest_covering_power(fmt):
    fmax = FMAX[fmt]
    cases = [0.0]
    for k in range(-40, 40, 3):
        b = np.float32(fmax * 2.0 ** k)
        cases += [b, np.nextafter(b, np.float32(0)), np.nextafter(b, np.float32(np.inf))]
    rng = np.random.default_rng(0)
    cases += list((rng.standard_normal(200) * 10.0 ** rng.uniform(-6, 6, 200)).astype(np.float32))
    for a in cases:
        a = abs(float(a))
        want = -127 if a == 0.0 else smallest_e(a, fmax)
        assert o.mx_exponent(a, fmt) == want, (fmt, a)
    assert o.mx_exponent(float("inf"), fmt) == 127


def test_e4m3_variant_is_the_pinned_mxfp8():
    x = synth.host_bits(synth.bf16_normal((64, 256), 1.0, 3, "cpu", 0.01, 30.0))
    a, b = o.mx(x, o.E4M3), o.mxfp8(x)
    for k in ("row", "row_sf", "col", "col_sf"):
        assert np.array_equal(a[k], b[k])
    rng = np.random.default_rng(1)
    for v in np.abs(rng.standard_normal(500) * 10.0 ** rng.uniform(-8, 8, 500)).astype(np.float32):
        assert o.lib().orc_mx_exponent_fmt(float(v), o.E4M3) == o.mx_exponent(float(v))


@pytest.mark.parametrize("fmt", [o.E5M2, o.E2M1])
def test_brute_force_rebuild_and_no_saturation(fmt):
    x = synth.host_bits(synth.bf16_normal((8, 64), 1.0, 4, "cpu", 0.05, 100.0))
    q = o.mx(x, fmt)
    vals = (x.astype(np.uint32) << 16).view(np.float32)
    for r in range(8):
        for b in range(2):
            blk = vals[r, 32 * b:32 * b + 32]
            e = smallest_e(float(np.max(np.abs(blk))), FMAX[fmt]) if np.any(blk) else -127
            assert q["row_sf"][r, b] == e + 127
            scaled = (blk.astype(np.float64) * 2.0 ** -e).astype(np.float32)
            assert np.all(np.abs(scaled) <= FMAX[fmt])  # nothing saturates
            codes = o.encode(fmt, scaled)
            if fmt == o.E2M1:
                packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)  # low nibble: even column
                assert np.array_equal(q["row"][r, 16 * b:16 * b + 16], packed)
            else:
                assert np.array_equal(q["row"][r, 32 * b:32 * b + 32], codes)
    # the column-wise copy is the transpose re-blocked, not the transposed codes
    t = o.mx(np.ascontiguousarray(x.T), fmt, rowwise=True, colwise=False)
    assert np.array_equal(q["col"], t["row"]) and np.array_equal(q["col_sf"], t["row_sf"])


@pytest.mark.parametrize("fmt,kind", [(o.E5M2, o.K_MXFP8_E5M2), (o.E2M1, o.K_MXFP4)])
def test_gemm_operand_kinds(fmt, kind):
    M, N, K = 4, 3, 64
    xa = synth.host_bits(synth.bf16_normal((M, K), 1.0, 5, "cpu"))
    xb = synth.host_bits(synth.bf16_normal((N, K), 0.5, 6, "cpu"))
    qa, qb = o.mx(xa, fmt, colwise=False), o.mx(xb, fmt, colwise=False)

    def deq(q, rows):
        c = q["row"]
        if fmt == o.E2M1:
            c = np.stack([c & 0xF, c >> 4], axis=-1).reshape(rows, K)
        v = o.decode(fmt, c)
        return v * np.ldexp(1.0, np.repeat(q["row_sf"].astype(np.int64) - 127, 32, axis=1))

    A, B = o.Operand(kind, qa["row"], qa["row_sf"]), o.Operand(kind, qb["row"], qb["row_sf"])
    assert np.array_equal(o.dequant(A, K, 0, M), deq(qa, M))
    c, bound = o.gemm(A, B, M, N, K)
    assert np.allclose(c, deq(qa, M) @ deq(qb, N).T, rtol=1e-12, atol=0)
    # closed form: all-ones operands give K everywhere (1 is exact after the block scaling)
    ones = np.full((M, K), 0x3F80, np.uint16)
    q1 = o.mx(ones, fmt, colwise=False)
    O1 = o.Operand(kind, q1["row"], q1["row_sf"])
    c1, _ = o.gemm(O1, O1, M, M, K)
    assert np.all(c1 == K)
