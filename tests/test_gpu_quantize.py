"""GPU parity of the quantizers: codes, scales, amax and tensor scales from the
CUDA kernels (through the C ABI) must equal the CPU oracle bit for bit on the
same seeded bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle as o
from precision_transformer_gemms_gb300 import lpq, synth
from lpq_testutil import bf16_input, codes, plain_scales, scalar

pytestmark = pytest.mark.gpu

BOTH = lpq.ROWWISE | lpq.COLWISE

# (rows, cols): small, ragged against the 64x128 / 128x128 CTA tiles, several tiles.
SHAPES_16 = [(64, 128), (176, 272), (256, 512), (400, 1040)]
SHAPES_32 = [(64, 128), (160, 288), (256, 512), (384, 1056)]


def eq(a, b):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    if not np.array_equal(a, b):
        idx = np.argwhere(a != b)
        raise AssertionError(f"{len(idx)} mismatches, first at {idx[0].tolist()}: {a[tuple(idx[0])]} vs {b[tuple(idx[0])]}")


@pytest.mark.parametrize("shape", SHAPES_16)
@pytest.mark.parametrize("fmt", [lpq.FP8_E4M3, lpq.FP8_E5M2])
def test_fp8_current_scaling(shape, fmt):
    x, bits = bf16_input(shape, std=3.0, seed=1, outlier_frac=0.001, outlier_scale=50)
    q = lpq.quantize(x, fmt, BOTH)
    ref = o.fp8_pertensor(bits, o.E4M3 if fmt == lpq.FP8_E4M3 else o.E5M2)
    eq(codes(q.row), ref["row"])
    eq(codes(q.col), ref["col"])
    assert scalar(q.row.amax) == ref["amax"] and scalar(q.col.amax) == ref["amax"]
    assert scalar(q.row.tensor_scale) == np.float32(ref["scale_inv"]) == scalar(q.col.tensor_scale)


def test_fp8_delayed_scaling_20_steps_with_drift():
    """Activation std drifting 1 -> 4 over 20 steps, history 16: every step's
    codes, amax and the state after each update match the oracle."""
    st_gpu = lpq.DelayedState(16)
    st_ref = o.DelayedState(16)
    for t in range(20):
        x, bits = bf16_input((128, 256), std=synth.drift_std(t), seed=10 * t)
        q = lpq.quantize(x, lpq.FP8_E4M3, BOTH, scaling=lpq.SCALING_DELAYED, state=st_gpu)
        ref = o.fp8_pertensor(bits, o.E4M3, scale=float(st_ref.scale[0]))
        eq(codes(q.row), ref["row"])
        eq(codes(q.col), ref["col"])
        assert scalar(q.row.amax) == ref["amax"]
        assert scalar(q.row.tensor_scale) == np.float32(1.0) / np.float32(st_ref.scale[0])
        lpq.scale_update(st_gpu, q.row.amax, 448.0)
        st_ref.update(ref["amax"], 448.0)
        eq(st_gpu.hist.cpu().numpy(), st_ref.hist)
        assert int(st_gpu.pos.item()) == int(st_ref.pos[0])
        assert scalar(st_gpu.scale) == st_ref.scale[0] and scalar(st_gpu.scale_inv) == st_ref.scale_inv[0]


@pytest.mark.parametrize("layout", [lpq.SF_PLAIN, lpq.SF_GEMM])
@pytest.mark.parametrize("shape", SHAPES_32)
def test_mxfp8(shape, layout):
    x, bits = bf16_input(shape, std=1.0, seed=2, outlier_frac=0.001, outlier_scale=50)
    q = lpq.quantize(x, lpq.MXFP8, BOTH, sf_layout=layout)
    ref = o.mxfp8(bits)
    eq(codes(q.row), ref["row"])
    eq(plain_scales(q.row), ref["row_sf"])
    eq(codes(q.col), ref["col"])
    eq(plain_scales(q.col), ref["col_sf"])


def test_mxfp8_gemm_layout_padding_is_zero():
    x, _ = bf16_input((160, 288), seed=3)
    q = lpq.quantize(x, lpq.MXFP8, lpq.ROWWISE, sf_layout=lpq.SF_GEMM)
    buf = q.row.scales.cpu().numpy().copy()
    kt = (288 + 127) // 128
    from lpq_testutil import sf_gemm_to_plain
    used = np.zeros(buf.size, bool)
    r = np.arange(160)[:, None]
    kb = np.arange(288 // 32)[None, :]
    used[(((r >> 7) * kt + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3)).ravel()] = True
    assert not buf[~used].any()


MX_VARIANTS = {lpq.MXFP8_E5M2: (o.E5M2, 1e-3), lpq.MXFP4: (o.E2M1, 1.0)}  # element format, input std


@pytest.mark.parametrize("layout", [lpq.SF_PLAIN, lpq.SF_GEMM])
@pytest.mark.parametrize("shape", SHAPES_32)
@pytest.mark.parametrize("fmt", [lpq.MXFP8_E5M2, lpq.MXFP4])
def test_mx_variants(fmt, shape, layout):
    """MXFP8 with E5M2 codes (gradients, std 1e-3 like dY) and MXFP4 (packed
    E2M1): both copies, codes and E8M0 scales bit for bit."""
    efmt, std = MX_VARIANTS[fmt]
    x, bits = bf16_input(shape, std=std, seed=12, outlier_frac=0.001, outlier_scale=50)
    q = lpq.quantize(x, fmt, BOTH, sf_layout=layout)
    ref = o.mx(bits, efmt)
    eq(codes(q.row), ref["row"])
    eq(plain_scales(q.row), ref["row_sf"])
    eq(codes(q.col), ref["col"])
    eq(plain_scales(q.col), ref["col_sf"])


@pytest.mark.parametrize("fmt", [lpq.MXFP8_E5M2, lpq.MXFP4])
def test_mx_variants_special_values(fmt):
    """Zeros (E8M0 code 0), a block whose max sits exactly on fmax * 2^e, a
    tiny negative beside a large value (negative-zero code), and infinities
    (saturated codes in a block of exponent 127)."""
    efmt, _ = MX_VARIANTS[fmt]
    z = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    fmax = {o.E5M2: 57344.0, o.E2M1: 6.0}[efmt]
    z[1, 0:32] = 0.5
    z[1, 5] = fmax / 4  # block max exactly fmax * 2^-2
    z[7, 9] = -1e-30
    z[7, 10] = 5.0
    z[9, 40] = float("inf")
    z[12, 70] = float("-inf")
    bits = synth.host_bits(z)
    q = lpq.quantize(z, fmt, BOTH)
    ref = o.mx(bits, efmt)
    for name in ("row", "col"):
        eq(codes(getattr(q, name)), ref[name])
        eq(plain_scales(getattr(q, name)), ref[name + "_sf"])
    assert plain_scales(q.row)[1, 0] == 127 - 2
    assert plain_scales(q.row)[0, 0] == 0


def test_mxfp4_gemm_layout_padding_is_zero():
    x, _ = bf16_input((160, 288), seed=3)
    q = lpq.quantize(x, lpq.MXFP4, lpq.ROWWISE, sf_layout=lpq.SF_GEMM)
    buf = q.row.scales.cpu().numpy().copy()
    kt = 2 * ((288 + 255) // 256)
    used = np.zeros(buf.size, bool)
    r = np.arange(160)[:, None]
    kb = np.arange(288 // 32)[None, :]
    used[(((r >> 7) * kt + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3)).ravel()] = True
    assert buf.size == 2 * kt * 512
    assert not buf[~used].any()


@pytest.mark.parametrize("layout", [lpq.SF_PLAIN, lpq.SF_GEMM])
@pytest.mark.parametrize("shape", SHAPES_16)
@pytest.mark.parametrize("variant", ["rne", "rht", "sr", "rht_sr"])
def test_nvfp4_1d(shape, variant, layout):
    std = 1e-3 if "sr" in variant else 1.0
    x, bits = bf16_input(shape, std=std, seed=4)
    flags = BOTH | (lpq.RHT_COLWISE if "rht" in variant else 0) | (lpq.STOCHASTIC if "sr" in variant else 0)
    q = lpq.quantize(x, lpq.NVFP4, flags, seed=1234567, counter_offset=8, rht_seed=77, sf_layout=layout)
    oflags = o.NV_ROW | o.NV_COL | (o.NV_RHT if "rht" in variant else 0) | (o.NV_SR if "sr" in variant else 0)
    ref = o.nvfp4(bits, oflags, seed=1234567, counter_offset=8, rht_seed=77)
    eq(codes(q.row), ref["row"])
    eq(plain_scales(q.row), ref["row_sf"])
    eq(codes(q.col), ref["col"])
    eq(plain_scales(q.col), ref["col_sf"])
    assert scalar(q.row.amax) == ref["row_amax"] and scalar(q.col.amax) == ref["col_amax"]
    assert scalar(q.row.tensor_scale) == ref["row_ts"] and scalar(q.col.tensor_scale) == ref["col_ts"]


@pytest.mark.parametrize("layout", [lpq.SF_PLAIN, lpq.SF_GEMM])
@pytest.mark.parametrize("shape", [(64, 128), (176, 272), (512, 384)])
def test_nvfp4_2d(shape, layout):
    x, bits = bf16_input(shape, std=0.02, seed=5)
    q = lpq.quantize(x, lpq.NVFP4_2D, BOTH, sf_layout=layout)
    ref = o.nvfp4(bits, o.NV_ROW | o.NV_COL | o.NV_2D)
    eq(codes(q.row), ref["row"])
    eq(plain_scales(q.row), ref["row_sf"])
    eq(codes(q.col), ref["col"])
    eq(plain_scales(q.col), ref["col_sf"])
    assert scalar(q.row.tensor_scale) == ref["row_ts"] == scalar(q.col.tensor_scale)


@pytest.mark.parametrize("layout", [lpq.SF_PLAIN, lpq.SF_GEMM])
@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (384, 1024)])
def test_fp8_block_1x128(shape, layout):
    x, bits = bf16_input(shape, std=1.0, seed=6, outlier_frac=0.001, outlier_scale=100)
    q = lpq.quantize(x, lpq.FP8_BLOCK_1x128, BOTH, sf_layout=layout)
    ref = o.fp8_block(bits, 1)
    eq(codes(q.row), ref["row"])
    eq(plain_scales(q.row), ref["row_sinv"])
    eq(codes(q.col), ref["col"])
    eq(plain_scales(q.col), ref["col_sinv"])


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (200, 256)])
def test_fp8_block_128x128(shape):
    x, bits = bf16_input(shape, std=1.0, seed=7, outlier_frac=0.001, outlier_scale=100)
    flags = BOTH if shape[0] % 128 == 0 else lpq.ROWWISE
    q = lpq.quantize(x, lpq.FP8_BLOCK_128x128, flags)
    ref = o.fp8_block(bits, 128, colwise=bool(flags & lpq.COLWISE))
    eq(codes(q.row), ref["row"])
    eq(plain_scales(q.row), ref["row_sinv"])
    if flags & lpq.COLWISE:
        eq(codes(q.col), ref["col"])
        eq(q.col.scales.cpu().numpy()[: ref["col_sinv"].size].reshape(ref["col_sinv"].shape), ref["col_sinv"])


@pytest.mark.parametrize("shape", [(64, 128), (176, 272)])
def test_bf16_transpose(shape):
    x, bits = bf16_input(shape, seed=8)
    q = lpq.quantize(x, lpq.BF16, BOTH)
    assert torch.equal(q.row.codes, x)
    assert torch.equal(q.col.codes, x.t().contiguous())


def test_special_values_zero_tensor_and_signed_zero():
    z = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    z[3, 5] = -0.0
    bits = synth.host_bits(z)
    # an all-zero tensor (signed zeros included): scale 1, codes keep the sign
    q = lpq.quantize(z, lpq.FP8_E4M3, BOTH)
    ref = o.fp8_pertensor(bits, o.E4M3)
    eq(codes(q.row), ref["row"])
    assert scalar(q.row.tensor_scale) == 1.0 and scalar(q.row.amax) == 0.0
    q = lpq.quantize(z, lpq.NVFP4, BOTH)
    ref = o.nvfp4(bits, o.NV_ROW | o.NV_COL)
    eq(codes(q.row), ref["row"])
    assert scalar(q.row.tensor_scale) == 1.0
    # a tiny negative value next to a large one rounds to the negative-zero code
    z[7, 9] = -1e-30
    z[7, 10] = 5.0
    bits = synth.host_bits(z)
    for fmt, ref in [(lpq.FP8_E4M3, o.fp8_pertensor(bits, o.E4M3)), (lpq.MXFP8, o.mxfp8(bits))]:
        q = lpq.quantize(z, fmt, BOTH)
        eq(codes(q.row), ref["row"])
        eq(codes(q.col), ref["col"])
        assert codes(q.row)[7, 9] == 0x80
    q = lpq.quantize(z, lpq.NVFP4, BOTH)
    ref = o.nvfp4(bits, o.NV_ROW | o.NV_COL)
    eq(codes(q.row), ref["row"])
    eq(plain_scales(q.row), ref["row_sf"])


def test_nonfinite_inputs_follow_the_oracle():
    x, _ = bf16_input((64, 128), seed=9)
    x[1, 2] = float("nan")
    x[4, 6] = float("inf")
    x[10, 70] = float("-inf")
    bits = synth.host_bits(x)
    for fmt, ref in [(lpq.MXFP8, o.mxfp8(bits))]:
        q = lpq.quantize(x, fmt, BOTH)
        eq(codes(q.row), ref["row"])
        eq(plain_scales(q.row), ref["row_sf"])
        eq(codes(q.col), ref["col"])
    q = lpq.quantize(x, lpq.FP8_E4M3, BOTH, scaling=lpq.SCALING_DELAYED, state=lpq.DelayedState())
    ref = o.fp8_pertensor(bits, o.E4M3, scale=1.0)
    eq(codes(q.row), ref["row"])


def test_nvfp4_nonfinite_inputs_follow_the_oracle():
    """NaN and infinities in an NVFP4 input: the amax skips NaN, an infinite
    amax gives tensor scale 1, NaN values encode as +6 and infinities
    saturate; the RHT spreads a NaN over its 16-value run.  Row-wise with
    stochastic rounding, column-wise with RHT (+ SR), and the 2D copies."""
    x, _ = bf16_input((64, 128), seed=19)
    x[1, 2] = float("nan")
    x[4, 6] = float("inf")
    x[40, 70] = float("-inf")
    bits = synth.host_bits(x)
    for flags, ref_flags in [(BOTH, o.NV_ROW | o.NV_COL),
                             (BOTH | lpq.STOCHASTIC, o.NV_ROW | o.NV_COL | o.NV_SR),
                             (BOTH | lpq.RHT_COLWISE, o.NV_ROW | o.NV_COL | o.NV_RHT),
                             (BOTH | lpq.RHT_COLWISE | lpq.STOCHASTIC, o.NV_ROW | o.NV_COL | o.NV_RHT | o.NV_SR)]:
        q = lpq.quantize(x, lpq.NVFP4, flags, seed=3, rht_seed=7)
        ref = o.nvfp4(bits, ref_flags, seed=3, rht_seed=7)
        for name in ("row", "col"):
            eq(codes(getattr(q, name)), ref[name])
            eq(plain_scales(getattr(q, name)), ref[name + "_sf"])
    x2 = x.clone()
    x2[4, 6] = 1.0
    x2[40, 70] = -2.0  # only the NaN: a finite amax
    bits2 = synth.host_bits(x2)
    for t, b in ((x, bits), (x2, bits2)):
        q = lpq.quantize(t, lpq.NVFP4_2D, BOTH)
        ref = o.nvfp4(b, o.NV_ROW | o.NV_COL | o.NV_2D)
        for name in ("row", "col"):
            eq(codes(getattr(q, name)), ref[name])
            eq(plain_scales(getattr(q, name)), ref[name + "_sf"])
        assert scalar(q.row.tensor_scale) == np.float32(ref["row_ts"])


def test_tiny_amax_scales_follow_the_oracle():
    """Tensors whose amax is below fmax / FLT_MAX (2^-123, and a block max at
    the smallest bf16 subnormal 2^-133): every scale quotient that overflows
    is clamped to the largest finite float on both sides, so zeros stay +0 and
    the dequantization factors stay positive.  Per-tensor FP8 (current and
    delayed, after a scale update with that amax), NVFP4 (plain, RHT, SR, 2D),
    and sub-channel FP8, bit-exact against the oracle."""
    z = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    z[1, 5], z[2, 7], z[33, 16], z[40, 100] = 2.0 ** -123, -(2.0 ** -123), 2.0 ** -133, 2.0 ** -130
    bits = synth.host_bits(z)
    for fmt, of in ((lpq.FP8_E4M3, o.E4M3), (lpq.FP8_E5M2, o.E5M2)):
        q = lpq.quantize(z, fmt, BOTH)
        ref = o.fp8_pertensor(bits, of)
        eq(codes(q.row), ref["row"])
        eq(codes(q.col), ref["col"])
        assert scalar(q.row.tensor_scale) == np.float32(ref["scale_inv"]) > 0
        st, st_ref = lpq.DelayedState(16), o.DelayedState(16)
        lpq.scale_update(st, q.row.amax, lpq.FMAX[fmt])
        st_ref.update(ref["amax"], o.FMAX[of])
        assert scalar(st.scale) == st_ref.scale[0] and scalar(st.scale_inv) == st_ref.scale_inv[0]
        q = lpq.quantize(z, fmt, BOTH, scaling=lpq.SCALING_DELAYED, state=st)
        eq(codes(q.row), o.fp8_pertensor(bits, of, scale=float(st_ref.scale[0]))["row"])
    for flags, ref_flags in [(BOTH, o.NV_ROW | o.NV_COL),
                             (BOTH | lpq.RHT_COLWISE | lpq.STOCHASTIC, o.NV_ROW | o.NV_COL | o.NV_RHT | o.NV_SR)]:
        q = lpq.quantize(z, lpq.NVFP4, flags, seed=3, rht_seed=7)
        ref = o.nvfp4(bits, ref_flags, seed=3, rht_seed=7)
        for name in ("row", "col"):
            eq(codes(getattr(q, name)), ref[name])
            eq(plain_scales(getattr(q, name)), ref[name + "_sf"])
            assert scalar(getattr(q, name).tensor_scale) == np.float32(ref[name + "_ts"])
    q = lpq.quantize(z, lpq.NVFP4_2D, BOTH)
    ref = o.nvfp4(bits, o.NV_ROW | o.NV_COL | o.NV_2D)
    for name in ("row", "col"):
        eq(codes(getattr(q, name)), ref[name])
        eq(plain_scales(getattr(q, name)), ref[name + "_sf"])
    for fmt, br in ((lpq.FP8_BLOCK_1x128, 1), (lpq.FP8_BLOCK_128x128, 128)):
        zz = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
        zz[1, 5], zz[100, 200] = 2.0 ** -123, 2.0 ** -133
        b2 = synth.host_bits(zz)
        q = lpq.quantize(zz, fmt, BOTH, sf_layout=lpq.SF_PLAIN)
        ref = o.fp8_block(b2, br)
        eq(codes(q.row), ref["row"])
        eq(plain_scales(q.row), ref["row_sinv"])
        eq(codes(q.col), ref["col"])


def test_mx_amax_outputs_for_either_view():
    """The MX formats' optional amax: written for whichever view asks (row,
    column or both), each starting from zero rather than a stale value."""
    x, bits = bf16_input((64, 128), std=2.0, seed=23)
    want = np.float32(o.amax(bits))
    for flags in (lpq.ROWWISE, lpq.COLWISE, BOTH):
        q = lpq.alloc(lpq.MXFP8, 64, 128, flags)
        for c in (q.row, q.col):
            if c is not None:
                c.amax = torch.full((1,), 1e30, dtype=torch.float32, device="cuda")  # stale
        lpq.quantize(x, lpq.MXFP8, flags, out=q)
        for c in (q.row, q.col):
            if c is not None:
                assert scalar(c.amax) == want


def test_delayed_position_outside_the_ring_wraps():
    """A restored state whose pos is outside [0, len) writes slot pos mod len
    (as the oracle does) and never outside the history."""
    st, ref = lpq.DelayedState(16), o.DelayedState(16)
    st.pos.fill_(37)
    ref.pos[0] = 37
    a = torch.tensor([3.0], device="cuda")
    lpq.scale_update(st, a, 448.0)
    ref.update(3.0, 448.0)
    eq(st.hist.cpu().numpy(), ref.hist)
    assert int(st.pos.item()) == int(ref.pos[0]) == 6


@pytest.mark.parametrize("shape", [(64, 128), (176, 272), (4096, 1040)])
def test_amax_entry_point(shape):
    """lpq_amax: max |x| and the column-wise RHT amax equal the oracle's (the
    amax an NVFP4 copy records), overwriting whatever the outputs held."""
    x, bits = bf16_input(shape, std=2.0, seed=31, outlier_frac=0.001, outlier_scale=40)
    stale = torch.full((1,), 1e30, dtype=torch.float32, device="cuda")
    a, r = lpq.amax(x, rht=True, rht_seed=7, out=stale.clone(), rht_out=stale.clone())
    ref = o.nvfp4(bits, o.NV_ROW | o.NV_COL | o.NV_RHT, rht_seed=7)
    assert scalar(a) == np.float32(o.amax(bits)) == ref["row_amax"]
    assert scalar(r) == ref["col_amax"]
    a2, none = lpq.amax(x)
    assert none is None and scalar(a2) == scalar(a)
    e = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    assert scalar(lpq.amax(e, out=stale.clone())[0]) == 0.0


def test_empty_input():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    q = lpq.quantize(x, lpq.NVFP4, lpq.ROWWISE)
    torch.cuda.synchronize()
    assert scalar(q.row.tensor_scale) == 1.0 and scalar(q.row.amax) == 0.0


@pytest.mark.parametrize("fmt,shape", [(lpq.MXFP8, (15872, 4096)), (lpq.NVFP4, (15872, 4096)),
                                       (lpq.MXFP8_E5M2, (15872, 4096)), (lpq.MXFP4, (15872, 4096)),
                                       (lpq.FP8_E4M3, (15872, 4096)), (lpq.NVFP4_2D, (4096, 4096))])
def test_full_size_whole_tensor(fmt, shape):
    """At the layer's full size, in the tensor-core scale layout the benchmark
    uses, the whole outputs are compared."""
    std = 0.02 if fmt == lpq.NVFP4_2D else 1.0
    x, bits = bf16_input(shape, std=std, seed=11)
    if fmt == lpq.NVFP4:
        q = lpq.quantize(x, fmt, BOTH | lpq.RHT_COLWISE | lpq.STOCHASTIC, seed=5, rht_seed=3)
        ref = o.nvfp4(bits, o.NV_ROW | o.NV_COL | o.NV_RHT | o.NV_SR, seed=5, rht_seed=3)
        pairs = [("row", "row_sf"), ("col", "col_sf")]
    elif fmt == lpq.NVFP4_2D:
        q = lpq.quantize(x, fmt, BOTH)
        ref = o.nvfp4(bits, o.NV_ROW | o.NV_COL | o.NV_2D)
        pairs = [("row", "row_sf"), ("col", "col_sf")]
    elif fmt == lpq.MXFP8:
        q = lpq.quantize(x, fmt, BOTH)
        ref = o.mxfp8(bits)
        pairs = [("row", "row_sf"), ("col", "col_sf")]
    elif fmt in MX_VARIANTS:
        q = lpq.quantize(x, fmt, BOTH)
        ref = o.mx(bits, MX_VARIANTS[fmt][0])
        pairs = [("row", "row_sf"), ("col", "col_sf")]
    else:
        q = lpq.quantize(x, fmt, BOTH)
        ref = o.fp8_pertensor(bits, o.E4M3)
        pairs = [("row", None), ("col", None)]
    for cname, sname in pairs:
        copy = getattr(q, cname)
        eq(codes(copy), ref[cname])
        if sname:
            eq(plain_scales(copy), ref[sname])


def test_delayed_state_checkpoint_resume():
    """The delayed-scaling state is raw arrays (history, position, scale,
    1/scale): 10 steps, a save to host memory, a restore into a fresh state
    and 10 more steps give the same codes, amaxes and state, bit for bit, as
    20 uninterrupted steps."""
    def run(state, t0, t1):
        out = []
        for t in range(t0, t1):
            x, _ = bf16_input((128, 256), std=synth.drift_std(t), seed=10 * t)
            q = lpq.quantize(x, lpq.FP8_E4M3, BOTH, scaling=lpq.SCALING_DELAYED, state=state)
            lpq.scale_update(state, q.row.amax, 448.0)
            out.append((codes(q.row), codes(q.col), scalar(q.row.amax), scalar(q.row.tensor_scale)))
        return out

    whole = lpq.DelayedState(16)
    ref = run(whole, 0, 20)
    first = lpq.DelayedState(16)
    part = run(first, 0, 10)
    saved = {k: getattr(first, k).cpu().numpy().copy() for k in ("hist", "pos", "scale", "scale_inv")}
    resumed = lpq.DelayedState(16)
    for k, v in saved.items():
        getattr(resumed, k).copy_(torch.from_numpy(v))
    part += run(resumed, 10, 20)
    for t, (a, b) in enumerate(zip(ref, part)):
        eq(a[0], b[0])
        eq(a[1], b[1])
        assert a[2:] == b[2:], t
    for k in ("hist", "pos", "scale", "scale_inv"):
        eq(getattr(whole, k).cpu().numpy(), getattr(resumed, k).cpu().numpy())
