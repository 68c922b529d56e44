"""Pins of the oracle's quantizers (CPU only): hand-worked blocks, closed
forms and invariants fixed by the format definitions."""
import json
import os

import numpy as np
import pytest

import oracle as o
from precision_transformer_gemms_gb300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")))


def bf16_bits(values):
    """float array -> bf16 bit patterns (values must be bf16-exact)."""
    f = np.asarray(values, np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(o.bf16_to_f32(b), f), "test values must be exactly representable in bf16"
    return b


def rand_bits(shape, std=1.0, seed=0, outlier_frac=0.0, outlier_scale=1.0):
    return synth.host_bits(synth.bf16_normal(shape, std, seed, "cpu", outlier_frac, outlier_scale))


def ulp_half(fmt, q):
    """Half the spacing of the format around |value(q)| (for error bounds)."""
    v = np.abs(o.decode(fmt, q))
    top = {o.E4M3: 0x7E, o.E5M2: 0x7B, o.E2M1: 0x7}[fmt]
    table = o.decode(fmt, np.arange(top + 1))
    gaps = np.diff(table)
    idx = np.clip(np.searchsorted(table, v, side="right") - 1, 0, top - 1)
    left = np.concatenate([[gaps[0]], gaps])[idx]
    return np.maximum(gaps[idx], left) / 2


# ------------------------------------------------------------------ per-tensor FP8
@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_current_scaling_maps_amax_to_fmax_and_bounds_error(fmt):
    x = rand_bits((64, 96), std=3.0, seed=4)
    r = o.fp8_pertensor(x, fmt)
    xf = o.bf16_to_f32(x).astype(np.float64)
    fmax = o.FMAX[fmt]
    assert r["amax"] == np.abs(xf).max()
    assert r["scale"] == np.float32(np.float32(fmax) / np.float32(r["amax"]))
    assert r["scale_inv"] == np.float32(1.0) / np.float32(r["scale"])
    deq = o.decode(fmt, r["row"]) * r["scale_inv"]
    i = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    assert abs(abs(o.decode(fmt, [r["row"][i]])[0]) - fmax) <= 2 * ulp_half(fmt, [r["row"][i]])[0]
    y = np.abs(o.bf16_to_f32(x) * np.float32(r["scale"])).astype(np.float64)  # fp32 product
    ok = y <= fmax
    err = np.abs(deq - xf)
    bound = ulp_half(fmt, r["row"]) * r["scale_inv"] + 2.0 ** -22 * np.abs(xf)
    assert np.all(err[ok] <= bound[ok])
    assert np.array_equal(r["col"], r["row"].T)
    assert r["saturated"] == int(np.sum(y > fmax))


def test_current_scaling_zero_tensor_gives_unit_scale():
    x = np.zeros((8, 32), np.uint16)
    r = o.fp8_pertensor(x, o.E4M3)
    assert r["scale"] == 1.0 and r["scale_inv"] == 1.0 and r["amax"] == 0.0
    assert not r["row"].any()


def test_delayed_scaling_hand_worked_three_steps():
    """State starts at scale 1; each step quantizes with the scale made from
    earlier steps, then pushes its amax; scale = 448 / max(history)."""
    st = o.DelayedState(16)
    amaxes = [2.0, 8.0, 4.0]
    scales_used = []
    for a in amaxes:
        x = bf16_bits([[a, -a / 2, 0.0, 1.0] * 8])
        r = o.fp8_pertensor(x, o.E4M3, scale=float(st.scale[0]))
        scales_used.append(r["scale"])
        assert r["amax"] == a
        st.update(r["amax"], 448.0)
    assert scales_used == [1.0, 224.0, 56.0]
    assert st.scale[0] == 56.0 and st.scale_inv[0] == np.float32(1 / 56.0) and st.pos[0] == 3
    assert list(st.hist[:4]) == [2.0, 8.0, 4.0, 0.0]


def test_delayed_history_wraps_and_forgets():
    st = o.DelayedState(16)
    st.update(100.0, 448.0)
    for _ in range(15):
        st.update(1.0, 448.0)
    assert st.scale[0] == np.float32(448.0 / 100.0)
    st.update(1.0, 448.0)  # the 100 leaves the ring
    assert st.scale[0] == 448.0 and st.pos[0] == 1


def test_delayed_saturation_count_brute_force():
    x = rand_bits((32, 64), std=4.0, seed=9)
    scale = 448.0 / 3.0
    r = o.fp8_pertensor(x, o.E4M3, scale=scale)
    y = np.abs(o.bf16_to_f32(x) * np.float32(scale))
    assert r["saturated"] == int(np.sum(y > 448.0)) > 0
    assert np.all(np.abs(o.decode(o.E4M3, r["row"])) <= 448.0)


def test_delayed_checkpoint_resume_bit_exact():
    """20 steps equal 10 steps, a save/restore of the state arrays, 10 steps."""
    xs = [rand_bits((16, 32), std=synth.drift_std(t), seed=10 * t) for t in range(20)]

    def run(st, steps):
        out = []
        for t in steps:
            r = o.fp8_pertensor(xs[t], o.E4M3, scale=float(st.scale[0]))
            out.append(r["row"].copy())
            st.update(r["amax"], 448.0)
        return out

    a = o.DelayedState()
    full = run(a, range(20))
    b = o.DelayedState()
    first = run(b, range(10))
    saved = [arr.copy() for arr in (b.hist, b.pos, b.scale, b.scale_inv)]
    c = o.DelayedState()
    c.hist[:], c.pos[:], c.scale[:], c.scale_inv[:] = saved
    second = run(c, range(10, 20))
    assert all(np.array_equal(p, q) for p, q in zip(full, first + second))
    assert np.array_equal(a.hist, c.hist) and a.scale[0] == c.scale[0]


# ------------------------------------------------------------------ MXFP8
def test_mxfp8_all_zero_block():
    r = o.mxfp8(np.zeros((32, 32), np.uint16))
    assert not r["row"].any() and not r["row_sf"].any() and not r["col_sf"].any()


def test_mxfp8_single_outlier_block():
    g = GOLD["mxfp8_outlier_block"]
    vals = np.zeros((1, 32), np.float32)
    vals[0, 5] = g["amax"]
    vals[0, 6] = 1.0
    r = o.mxfp8(bf16_bits(vals), colwise=False)
    assert o.mx_exponent(g["amax"]) == g["exponent"]
    assert r["row_sf"][0, 0] == g["e8m0"]
    assert r["row"][0, 5] == g["outlier_code"]
    assert o.decode(o.E4M3, [r["row"][0, 5]])[0] * 2.0 ** g["exponent"] == g["outlier_dequant"]
    assert o.decode(o.E4M3, [r["row"][0, 6]])[0] == 8.0  # 1 * 2^3 exactly


def test_mxfp8_powers_of_two():
    for amax, e, sf, code in GOLD["mxfp8_power_of_two"]:
        vals = np.full((1, 32), amax / 4, np.float32)
        vals[0, 0] = amax
        r = o.mxfp8(bf16_bits(vals), colwise=False)
        assert r["row_sf"][0, 0] == sf and r["row"][0, 0] == code


def test_mxfp8_exponent_is_smallest_covering_power():
    rng = np.random.default_rng(0)
    for a in np.concatenate([rng.uniform(1e-6, 1e6, 2000), [448 * 2.0 ** k for k in range(-20, 20)],
                             [np.nextafter(448.0, 1e9), np.nextafter(448.0, 0)]]).astype(np.float32):
        e = o.mx_exponent(a)
        assert 448.0 * 2.0 ** e >= a and 448.0 * 2.0 ** (e - 1) < a


def test_mxfp8_no_saturation_error_bound_and_colwise_reblocking():
    x = rand_bits((64, 128), std=1.0, seed=1, outlier_frac=0.01, outlier_scale=50)
    r = o.mxfp8(x)
    xf = o.bf16_to_f32(x).astype(np.float64)
    e = r["row_sf"].astype(np.int64) - 127
    scale = np.repeat(2.0 ** e, 32, axis=1)
    assert np.all(np.abs(xf / scale) <= 448.0)
    deq = o.decode(o.E4M3, r["row"]) * scale
    assert np.all(np.abs(deq - xf) <= ulp_half(o.E4M3, r["row"]) * scale)
    # the column-wise copy is quantized along the other dimension: it is the
    # row-wise quantization of the transpose, not the transpose of the codes
    t = o.mxfp8(np.ascontiguousarray(x.T), colwise=False)
    assert np.array_equal(r["col"], t["row"]) and np.array_equal(r["col_sf"], t["row_sf"])
    assert not np.array_equal(r["col"], r["row"].T)


# ------------------------------------------------------------------ NVFP4
def unpack(codes):
    lo = codes & 0xF
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def nv_deq(codes, sf, ts):
    q = o.decode(o.E2M1, unpack(codes).ravel()).reshape(codes.shape[0], -1)
    s = np.repeat(o.decode(o.E4M3, sf.ravel()).reshape(sf.shape), 16, axis=1)
    return q * s * ts


def test_nvfp4_all_zero():
    r = o.nvfp4(np.zeros((16, 32), np.uint16), o.NV_ROW | o.NV_COL)
    assert not r["row"].any() and not r["row_sf"].any() and r["row_ts"] == 1.0 and r["row_amax"] == 0


def test_nvfp4_single_outlier_block():
    for k in (-3, 0, 4):
        vals = np.zeros((1, 32), np.float32)
        vals[0, 0] = 6.0 * 2.0 ** k
        vals[0, 17] = 0.75 * 2.0 ** k  # another block: d = 56 exactly, element -> 6
        r = o.nvfp4(bf16_bits(vals), o.NV_ROW)
        assert (r["row"][0, 0] & 0xF) == 0x7  # the outlier encodes as 6
        assert r["row_sf"][0, 0] == 0x7E  # its block scale is 448 (= 2688 / 6)
        assert o.decode(o.E4M3, [r["row_sf"][0, 1]])[0] == 56.0
        assert r["row_ts"] == np.float32(np.float32(6.0 * 2.0 ** k) / np.float32(2688.0))
        deq = nv_deq(r["row"], r["row_sf"], r["row_ts"])
        assert deq[0, 0] == pytest.approx(6.0 * 2.0 ** k, rel=1e-6)
        assert deq[0, 17] == pytest.approx(0.75 * 2.0 ** k, rel=1e-6)
        # a block whose scale rounds down (d = 74.67 -> 72) saturates its max to 6
        vals[0, 17] = 2.0 ** k
        r = o.nvfp4(bf16_bits(vals), o.NV_ROW)
        assert o.decode(o.E4M3, [r["row_sf"][0, 1]])[0] == 72.0 and (r["row"][0, 8] >> 4) == 0x7


def test_nvfp4_error_bound_and_storage():
    x = rand_bits((64, 256), std=1.0, seed=2)
    r = o.nvfp4(x, o.NV_ROW)
    xf = o.bf16_to_f32(x).astype(np.float64)
    deq = nv_deq(r["row"], r["row_sf"], r["row_ts"])
    S = np.repeat(o.decode(o.E4M3, r["row_sf"].ravel()).reshape(r["row_sf"].shape), 16, axis=1)
    q = unpack(r["row"])
    # half an E2M1 ulp at the code, in units of the block's dequant scale, plus
    # the fp32 rounding of the scaled value
    bound = ulp_half(o.E2M1, q) * S * r["row_ts"] * (1 + 1e-5) + 1e-12
    y = xf / (S * r["row_ts"])
    ok = np.abs(y) <= 6.0
    assert np.all(np.abs(deq - xf)[ok] <= bound[ok])
    # block scale covers the block max: the E4M3 rounding of d at most loses 1/16
    bmax = np.abs(xf).reshape(64, -1, 16).max(-1)
    assert np.all(o.decode(o.E4M3, r["row_sf"].ravel()).reshape(bmax.shape) * 6 * r["row_ts"] >= bmax * (1 - 1 / 16))
    # storage: 4 bits per value + 8 bits per 16 values = 4.5 bits per value
    bits = (r["row"].size + r["row_sf"].size) * 8 / x.size
    assert bits == GOLD["nvfp4_bits_per_value"]


def test_nvfp4_colwise_is_reblocked_transpose_without_rht():
    x = rand_bits((32, 64), seed=3)
    r = o.nvfp4(x, o.NV_ROW | o.NV_COL)
    t = o.nvfp4(np.ascontiguousarray(x.T), o.NV_ROW)
    assert np.array_equal(r["col"], t["row"]) and np.array_equal(r["col_sf"], t["row_sf"])
    assert r["col_ts"] == t["row_ts"]


def test_nvfp4_rht_colwise_matches_transform_then_quantize():
    x = rand_bits((32, 48), seed=6)
    r = o.nvfp4(x, o.NV_COL | o.NV_RHT, rht_seed=5)
    signs = o.rht_sign_mask(5)
    xf = o.bf16_to_f32(x)
    v = np.empty((48, 32), np.float32)
    for c in range(48):
        for m0 in range(0, 32, 16):
            v[c, m0:m0 + 16] = o.rht16(xf[m0:m0 + 16, c], signs)
    assert r["col_amax"] == np.abs(v).max()
    deq = nv_deq(r["col"], r["col_sf"], r["col_ts"])
    S = np.repeat(o.decode(o.E4M3, r["col_sf"].ravel()).reshape(r["col_sf"].shape), 16, axis=1)
    assert np.all(np.abs(deq - v) <= ulp_half(o.E2M1, unpack(r["col"])) * S * r["col_ts"] * (1 + 1e-5) + 1e-12)


def test_nvfp4_sr_is_deterministic_and_rounds_to_neighbours():
    x = rand_bits((16, 64), std=1e-3, seed=7)
    a = o.nvfp4(x, o.NV_ROW | o.NV_COL | o.NV_SR, seed=42, counter_offset=8)
    b = o.nvfp4(x, o.NV_ROW | o.NV_COL | o.NV_SR, seed=42, counter_offset=8)
    c = o.nvfp4(x, o.NV_ROW | o.NV_COL | o.NV_SR, seed=43, counter_offset=8)
    rne = o.nvfp4(x, o.NV_ROW | o.NV_COL)
    assert np.array_equal(a["row"], b["row"]) and np.array_equal(a["col"], b["col"])
    assert not np.array_equal(a["row"], c["row"])
    assert np.array_equal(a["row_sf"], rne["row_sf"])  # block scales never stochastic
    # SR codes differ from RNE codes by at most one step of the magnitude table
    qa, qr = unpack(a["row"]), unpack(rne["row"])
    assert np.all(np.abs((qa & 7).astype(int) - (qr & 7).astype(int)) <= 1)


def test_nvfp4_2d_transpose_and_reduction_to_1d():
    x = rand_bits((64, 48), std=0.02, seed=8)
    r = o.nvfp4(x, o.NV_ROW | o.NV_COL | o.NV_2D)
    assert np.array_equal(unpack(r["col"]), unpack(r["row"]).T)
    # column copy scales [48, 64/16]: entry (c, rb) is the scale of tile (rb, c // 16)
    want = np.array([[r["row_sf"][rb * 16, c // 16] for rb in range(4)] for c in range(48)], np.uint8)
    assert np.array_equal(r["col_sf"], want)
    # every row of a 16x16 tile carries the same scale
    sf = r["row_sf"].reshape(4, 16, 3)
    assert np.all(sf == sf[:, :1, :])
    # a tile whose 16 rows are identical reduces to the 1D quantizer of that row
    row = rand_bits((1, 32), std=0.02, seed=9)
    same = np.repeat(row, 16, axis=0)
    r2 = o.nvfp4(same, o.NV_ROW | o.NV_2D)
    r1 = o.nvfp4(same, o.NV_ROW)
    assert np.array_equal(r2["row"], r1["row"]) and np.array_equal(r2["row_sf"], r1["row_sf"])


# ------------------------------------------------------------------ sub-channel FP8
@pytest.mark.parametrize("block_rows", [1, 128])
def test_fp8_block_scales_and_error(block_rows):
    x = rand_bits((128, 256), std=1.0, seed=11, outlier_frac=0.001, outlier_scale=100)
    r = o.fp8_block(x, block_rows)
    xf = o.bf16_to_f32(x).astype(np.float64)
    sinv = np.repeat(np.repeat(r["row_sinv"], block_rows, axis=0)[:128], 128, axis=1)
    blocks = np.abs(xf).reshape(128 // block_rows, block_rows, 2, 128).max(axis=(1, 3))
    want = np.float32(1) / (np.float32(448) / blocks.astype(np.float32))
    assert np.array_equal(r["row_sinv"], want.astype(np.float32))
    deq = o.decode(o.E4M3, r["row"]) * sinv
    # half an E4M3 ulp in scaled units, plus the two fp32 roundings (x * scale, 1 / scale)
    assert np.all(np.abs(deq - xf) <= ulp_half(o.E4M3, r["row"]) * sinv + 2.0 ** -22 * np.abs(xf))
    if block_rows == 128:
        assert np.array_equal(r["col"], r["row"].T) and np.array_equal(r["col_sinv"], r["row_sinv"].T)
    else:
        t = o.fp8_block(np.ascontiguousarray(x.T), 1, colwise=False)
        assert np.array_equal(r["col"], t["row"]) and np.array_equal(r["col_sinv"], t["row_sinv"])


# ------------------------------------------------------------------ tiny amax: scale quotients clamped
FLT_MAX = np.float32(3.4028234663852886e38)


def _torch_fp8_code(y, fmt):
    """RNE float8 code of float32 values by torch's own conversion (in range only)."""
    import torch
    dt = torch.float8_e4m3fn if fmt == o.E4M3 else torch.float8_e5m2
    return torch.tensor(np.asarray(y, np.float32)).to(dt).view(torch.uint8).numpy()


def _nearest_e2m1(y):
    """E2M1 code of |y| < 6 by exhaustive nearest search (no ties in the values used)."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    return int(np.argmin(np.abs(grid - abs(float(y)))))


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_tiny_amax_fp8_scale_clamped_to_largest_float(fmt):
    """An amax below fmax / FLT_MAX (bf16 holds it: 2^-123 ~ 9.4e-38) makes
    fmax / amax overflow; the scale is then the largest finite float (the
    reading for a case the pages leave open).  Worked with numpy float32
    arithmetic and torch's float8 conversion: zeros stay +0 instead of becoming
    NaN codes, the tiny value encodes as RNE(t * FLT_MAX), scale_inv is the
    float32 1 / FLT_MAX rather than 0."""
    t = np.float32(2.0 ** -123)
    x = np.zeros((4, 32), np.float32)
    x[1, 5], x[2, 7] = t, -t
    bits = bf16_bits(x)
    with np.errstate(over="ignore"):
        assert np.isinf(np.float32(o.FMAX[fmt]) / t)  # the unclamped quotient overflows
    r = o.fp8_pertensor(bits, fmt)
    assert r["amax"] == t and r["scale"] == FLT_MAX
    assert r["scale_inv"] == np.float32(1) / FLT_MAX and r["scale_inv"] > 0
    want = _torch_fp8_code(x * FLT_MAX, fmt)
    assert np.array_equal(r["row"], want) and np.array_equal(r["col"], want.T)
    assert (r["row"] == 0).sum() == x.size - 2  # every zero encodes as +0
    # delayed scaling: a history whose max is t gives the same clamped scale
    st = o.DelayedState(16)
    st.update(t, o.FMAX[fmt])
    assert st.scale[0] == FLT_MAX and st.scale_inv[0] == np.float32(1) / FLT_MAX
    assert np.array_equal(o.fp8_pertensor(bits, fmt, scale=float(st.scale[0]))["row"], want)


def test_tiny_amax_nvfp4_encode_and_block_factors_clamped():
    """NVFP4 with A = 2^-123: s_enc = 2688 / A overflows and is clamped to
    FLT_MAX; a block whose max is the smallest bf16 subnormal 2^-133 gets a
    subnormal E4M3 scale S, whose factor s_enc / dec(S) overflows too and is
    clamped.  Zeros stay 0 in both blocks (an infinite factor would make them
    NaN, encoded as +6)."""
    t, u = np.float32(2.0 ** -123), np.float32(2.0 ** -133)
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 16] = t, u
    r = o.nvfp4(bf16_bits(x), o.NV_ROW)
    assert r["row_amax"] == t and r["row_ts"] == t / np.float32(2688)
    s_enc = FLT_MAX  # 2688 / t overflows
    want_sf, want_codes = [], []
    for v in (t, u):
        d = (v / np.float32(6)) * s_enc
        S = int(_torch_fp8_code([d], o.E4M3)[0])
        dec = np.float32(o.decode(o.E4M3, [S])[0])
        with np.errstate(over="ignore"):
            f = np.float32(s_enc / dec)
        f = min(f, FLT_MAX)
        want_sf.append(S)
        want_codes.append(_nearest_e2m1(v * f))
    assert want_sf[1] < 8  # the second block's scale is an E4M3 subnormal
    assert list(r["row_sf"][0]) == want_sf
    codes = [(r["row"][0, j // 2] >> (4 * (j % 2))) & 0xF for j in range(32)]
    assert codes[0] == want_codes[0] == 7 and codes[16] == want_codes[1] == 0
    assert all(c == 0 for j, c in enumerate(codes) if j not in (0, 16))


def test_tiny_amax_subchannel_scale_clamped():
    """1x128 block whose max is 2^-123: 448 / m overflows, the block scale is
    FLT_MAX and its FP32 factor 1 / FLT_MAX; zeros encode as +0."""
    t = np.float32(2.0 ** -123)
    x = np.zeros((2, 128), np.float32)
    x[0, 3] = t
    r = o.fp8_block(bf16_bits(x), 1, colwise=False)
    assert r["row_sinv"][0, 0] == np.float32(1) / FLT_MAX
    assert np.array_equal(r["row"][0], _torch_fp8_code(x[0] * FLT_MAX, o.E4M3))
    assert r["row_sinv"][1, 0] == 1.0 and not r["row"][1].any()  # all-zero block: scale 1


def test_delayed_position_outside_ring_is_taken_modulo_len():
    """A state restored with pos outside [0, len) writes slot pos mod len."""
    st = o.DelayedState(16)
    st.pos[0] = 37
    st.update(2.0, 448.0)
    assert st.hist[5] == 2.0 and int(st.pos[0]) == 6 and st.hist.sum() == 2.0
    st.pos[0] = -1
    st.update(4.0, 448.0)
    assert st.hist[15] == 4.0 and int(st.pos[0]) == 0
    assert st.scale[0] == np.float32(448.0) / np.float32(4.0)
