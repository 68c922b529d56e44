"""Pins of the oracle's format codecs (CPU only).

The decode tables are checked against torch's independent float8 dtypes and
against the E2M1 magnitude set fixed by its 1/2/1 bit split and +-6 range
(Accelerate LLM training with NVFP4, 'technical deep dive'); the encoder is
pinned at every code point, at every midpoint between neighbouring codes
(ties to even) and just either side of it, and by hand-worked values.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as o

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")))


def _torch_table(dtype):
    return torch.arange(256, dtype=torch.uint8).view(dtype).double().numpy()


@pytest.mark.parametrize("fmt,dtype", [(o.E4M3, torch.float8_e4m3fn), (o.E5M2, torch.float8_e5m2)])
def test_fp8_decode_all_256_codes_match_torch(fmt, dtype):
    ref = _torch_table(dtype)
    got = o.decode(fmt, np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_fp8_special_values():
    e4 = o.decode(o.E4M3, np.arange(256))
    e5 = o.decode(o.E5M2, np.arange(256))
    assert np.nanmax(e4) == GOLD["e4m3_max"] and np.isnan(e4).sum() == 2  # only S.1111.111
    assert np.nanmax(e5[np.isfinite(e5)]) == GOLD["e5m2_max"] and np.isinf(e5).sum() == 2
    assert o.decode(o.E4M3, [1])[0] == 2.0 ** -9  # smallest subnormal


def test_e2m1_decode_is_the_1_2_1_magnitude_set():
    mags = GOLD["e2m1_magnitudes"]
    got = o.decode(o.E2M1, np.arange(16))
    assert list(got[:8]) == mags
    assert list(-got[8:]) == mags and all(np.signbit(got[8:]))
    assert got.max() == 6.0  # "about +-6"


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2, o.E2M1])
def test_encode_roundtrips_every_code(fmt):
    n = 16 if fmt == o.E2M1 else 256
    vals = o.decode(fmt, np.arange(n))
    finite = np.isfinite(vals)
    codes = o.encode(fmt, vals[finite].astype(np.float32))
    assert np.array_equal(codes, np.arange(n)[finite].astype(np.uint8))


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2, o.E2M1])
def test_encode_midpoints_tie_to_even_and_neighbours(fmt):
    top = {o.E4M3: 0x7E, o.E5M2: 0x7B, o.E2M1: 0x7}[fmt]
    vals = o.decode(fmt, np.arange(top + 1))
    for c in range(top):
        lo, hi = vals[c], vals[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # representable in fp32
        even = c if c % 2 == 0 else c + 1
        assert o.encode(fmt, [mid])[0] == even
        assert o.encode(fmt, [np.nextafter(mid, np.float32(np.inf))])[0] == c + 1
        assert o.encode(fmt, [np.nextafter(mid, np.float32(-np.inf))])[0] == c
        sgn = 0x8 if fmt == o.E2M1 else 0x80
        assert o.encode(fmt, [-mid])[0] == (even | sgn)


@pytest.mark.parametrize("fmt,dtype,fmax", [(o.E4M3, torch.float8_e4m3fn, 448.0),
                                            (o.E5M2, torch.float8_e5m2, 57344.0)])
def test_encode_random_in_range_matches_torch_rne(fmt, dtype, fmax):
    rng = np.random.default_rng(1)
    y = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, np.log(fmax), 200000))).astype(np.float32)
    y = np.clip(y, -fmax, fmax)
    ref = torch.from_numpy(y).to(dtype).view(torch.uint8).numpy()
    assert np.array_equal(o.encode(fmt, y), ref)


@pytest.mark.parametrize("fmt,dtype,fmax", [(o.E4M3, torch.float8_e4m3fn, 448.0),
                                            (o.E5M2, torch.float8_e5m2, 57344.0)])
def test_encode_saturates_beyond_max(fmt, dtype, fmax):
    y = np.array([fmax * 1.01, fmax * 1e3, np.inf, -np.inf, -fmax * 2], np.float32)
    codes = o.encode(fmt, y)
    top = 0x7E if fmt == o.E4M3 else 0x7B
    assert list(codes) == [top, top, top, top | 0x80, top | 0x80]


def test_encode_nan_codes():
    assert o.encode(o.E4M3, [np.nan])[0] == 0x7F
    assert o.encode(o.E5M2, [np.nan])[0] == 0x7F
    assert o.encode(o.E2M1, [np.nan])[0] == 0x7


def test_hand_worked_e2m1_and_e4m3():
    for v, c in GOLD["e2m1_rne"]:
        assert o.encode(o.E2M1, [v])[0] == c, v
    for v, c in GOLD["e4m3_rne"]:
        assert o.encode(o.E4M3, [v])[0] == c, v


def test_all_bf16_times_scales_brute_force():
    """Every bf16 pattern times a set of fp32 scales: the encoder agrees with
    torch's RNE cast of the clamped product (saturation is the clamp)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = o.bf16_to_f32(bits)
    ok = np.isfinite(x)
    for fmt, dtype, fmax in [(o.E4M3, torch.float8_e4m3fn, 448.0), (o.E5M2, torch.float8_e5m2, 57344.0)]:
        for scale in (1.0, 0.37109375, 448.0 / 3.0, 2.0 ** 20, 1e-30):
            with np.errstate(over="ignore"):
                y = (x[ok] * np.float32(scale)).astype(np.float32)
            ref = torch.from_numpy(np.clip(y, -fmax, fmax)).to(dtype).view(torch.uint8).numpy()
            assert np.array_equal(o.encode(fmt, y), ref), (fmt, scale)
