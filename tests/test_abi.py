"""CPU checks of the C ABI library: it loads, exports every entry point the
header declares, its host-only helpers agree with the oracle and the pages,
and argument validation returns the documented status codes without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as o
from precision_transformer_gemms_gb300 import lpq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lpq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lpq_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 9
    L = lpq.lib()
    for n in names:
        assert hasattr(L, n), n


def test_layer_shapes_match_oracle():
    got = lpq.layer_shapes(4096, 16384, 31, 512)
    want = o.layer_shapes(4096, 16384, 31, 512)
    assert [(n, m, k, nn) for n, _, m, k, nn in got] == want
    assert [lay for _, lay, *_ in got] == [0, 1, 2] * 4


def test_copy_bytes():
    assert lpq.copy_bytes(lpq.NVFP4, 15872, 4096, lpq.SF_PLAIN) == (15872 * 2048, 15872 * 256)
    # 4 bits per value + one byte per 16 values = 4.5 bits per value
    cb, sb = lpq.copy_bytes(lpq.NVFP4, 1024, 4096, lpq.SF_PLAIN)
    assert (cb + sb) * 8 / (1024 * 4096) == 4.5
    assert lpq.copy_bytes(lpq.MXFP8, 256, 512, lpq.SF_GEMM) == (256 * 512, 2 * 4 * 512)
    assert lpq.copy_bytes(lpq.NVFP4, 300, 544, lpq.SF_GEMM)[1] == 3 * (4 * 3) * 512
    assert lpq.copy_bytes(lpq.FP8_BLOCK_1x128, 256, 512, lpq.SF_GEMM) == (256 * 512, 4 * 256 * 4)
    assert lpq.copy_bytes(lpq.BF16, 3, 16, lpq.SF_PLAIN) == (96, 0)
    with pytest.raises(lpq.LpqError) as e:
        lpq.copy_bytes(lpq.MXFP8, 4, 48)
    assert e.value.status == lpq.ERR_SHAPE


def test_copy_bytes_mx_variants():
    """MXFP8 with E5M2 codes has MXFP8's sizes; MXFP4 packs two codes a byte
    with one E8M0 scale per 32 values (4.25 bits per value) and two scale atoms
    per 256 columns in the tensor-core layout."""
    for layout in (lpq.SF_PLAIN, lpq.SF_GEMM):
        assert lpq.copy_bytes(lpq.MXFP8_E5M2, 300, 544, layout) == lpq.copy_bytes(lpq.MXFP8, 300, 544, layout)
    cb, sb = lpq.copy_bytes(lpq.MXFP4, 1024, 4096, lpq.SF_PLAIN)
    assert (cb, sb) == (1024 * 2048, 1024 * 128)
    assert (cb + sb) * 8 / (1024 * 4096) == 4.25
    assert lpq.copy_bytes(lpq.MXFP4, 300, 544, lpq.SF_GEMM) == (300 * 272, 3 * (2 * 3) * 512)
    for fmt in (lpq.MXFP8_E5M2, lpq.MXFP4):
        with pytest.raises(lpq.LpqError) as e:
            lpq.copy_bytes(fmt, 4, 48)
        assert e.value.status == lpq.ERR_SHAPE
    with pytest.raises(lpq.LpqError) as e:
        lpq.copy_bytes(lpq.MXFP4 + 1, 4, 64)
    assert e.value.status == lpq.ERR_INVALID_ARG


def _quantize_raw(x_ptr, rows, cols, fmt, flags, scaling=0, ctr=0, out=None, state=None):
    out = out or lpq.QTensorC()
    return lpq.lib().lpq_quantize(x_ptr, rows, cols, fmt, scaling, flags, 0, ctr, 0, state, ctypes.byref(out), None)


def test_quantize_validation_codes():
    assert _quantize_raw(None, 4, 32, 99, lpq.ROWWISE) == lpq.ERR_INVALID_ARG
    assert _quantize_raw(None, 4, 32, lpq.MXFP8, 0) == lpq.ERR_INVALID_ARG
    assert _quantize_raw(None, 4, 32, lpq.MXFP8, lpq.ROWWISE | lpq.STOCHASTIC) == lpq.ERR_UNSUPPORTED
    assert _quantize_raw(None, 4, 32, lpq.NVFP4, lpq.ROWWISE | lpq.RHT_COLWISE) == lpq.ERR_INVALID_ARG
    assert _quantize_raw(None, 4, 32, lpq.NVFP4, lpq.ROWWISE, ctr=2) == lpq.ERR_INVALID_ARG
    assert _quantize_raw(None, 4, 32, lpq.MXFP8, lpq.ROWWISE, scaling=1) == lpq.ERR_UNSUPPORTED
    assert _quantize_raw(None, 4, 32, lpq.FP8_E4M3, lpq.ROWWISE, scaling=1) == lpq.ERR_INVALID_ARG  # no state
    assert _quantize_raw(None, 4, 32, lpq.MXFP8, lpq.ROWWISE) == lpq.ERR_INVALID_ARG  # x NULL
    assert _quantize_raw(ctypes.c_void_p(8), 4, 32, lpq.MXFP8, lpq.ROWWISE) == lpq.ERR_ALIGN
    assert _quantize_raw(ctypes.c_void_p(16), 4, 40, lpq.MXFP8, lpq.ROWWISE) == lpq.ERR_SHAPE
    assert _quantize_raw(ctypes.c_void_p(16), 40, 32, lpq.MXFP8, lpq.COLWISE) == lpq.ERR_SHAPE  # rows % 32
    for fmt in (lpq.MXFP8_E5M2, lpq.MXFP4):
        assert _quantize_raw(None, 4, 32, fmt, lpq.ROWWISE | lpq.STOCHASTIC) == lpq.ERR_UNSUPPORTED
        assert _quantize_raw(ctypes.c_void_p(16), 4, 48, fmt, lpq.ROWWISE) == lpq.ERR_SHAPE
        assert _quantize_raw(ctypes.c_void_p(16), 48, 32, fmt, lpq.COLWISE) == lpq.ERR_SHAPE
    # a view that does not match the request
    out = lpq.QTensorC()
    out.row = lpq.QView(16, 16, 16, 16, 4, 64, lpq.MXFP8, lpq.SF_GEMM, 0, 0)
    assert _quantize_raw(ctypes.c_void_p(16), 4, 32, lpq.MXFP8, lpq.ROWWISE, out=out) == lpq.ERR_SHAPE
    assert "expected" in lpq.last_error()


def test_gemm_validation_codes():
    L = lpq.lib()

    def view(fmt, rows, cols, colwise=0):
        return lpq.QView(16, 16, 16, 16, rows, cols, fmt, lpq.SF_GEMM, colwise, 0)

    a, b = view(lpq.MXFP8, 128, 256), view(lpq.NVFP4, 64, 256)
    call = lambda lay, a, b, m, n, k, c=16: L.lpq_gemm(lay, ctypes.byref(a), ctypes.byref(b), c, 0, m, n, k, None)
    assert call(0, a, b, 128, 64, 256) == lpq.ERR_UNSUPPORTED  # mixed formats never fall back
    assert call(0, a, view(lpq.MXFP8, 64, 256), 128, 64, 128) == lpq.ERR_SHAPE  # k mismatch
    assert call(1, a, view(lpq.MXFP8, 64, 256), 128, 64, 256) == lpq.ERR_INVALID_ARG  # dgrad wants b col-wise
    assert call(7, a, a, 128, 128, 256) == lpq.ERR_INVALID_ARG
    assert call(0, view(lpq.MXFP8, 128, 48), view(lpq.MXFP8, 64, 48), 128, 64, 48) == lpq.ERR_SHAPE
    assert call(0, a, view(lpq.MXFP8, 64, 256), 128, 64, 256, c=8) == lpq.ERR_ALIGN
    # MX variants: E5M2 gradients pair with E4M3 MXFP8 either way; MXFP4 only with MXFP4
    f4 = view(lpq.MXFP4, 64, 256)
    for fa, fb in ((lpq.MXFP4, lpq.NVFP4), (lpq.NVFP4, lpq.MXFP4), (lpq.MXFP4, lpq.MXFP8), (lpq.MXFP8, lpq.MXFP4),
                   (lpq.MXFP8_E5M2, lpq.FP8_E5M2)):
        assert call(0, view(fa, 128, 256), view(fb, 64, 256), 128, 64, 256) == lpq.ERR_UNSUPPORTED, (fa, fb)
    validated = (lpq.ERR_UNSUPPORTED, lpq.ERR_SHAPE, lpq.ERR_INVALID_ARG, lpq.ERR_ALIGN)
    for fa, fb in ((lpq.MXFP8_E5M2, lpq.MXFP8), (lpq.MXFP8, lpq.MXFP8_E5M2), (lpq.MXFP4, lpq.MXFP4)):
        # legal pairings pass validation and stop at the device check (no GPU here)
        assert call(0, view(fa, 128, 256), view(fb, 64, 256), 128, 64, 256) not in validated, (fa, fb)
    assert call(0, view(lpq.MXFP4, 128, 48), view(lpq.MXFP4, 64, 48), 128, 64, 48) == lpq.ERR_SHAPE
    f4.sf_layout = lpq.SF_PLAIN
    assert call(0, view(lpq.MXFP4, 128, 256), f4, 128, 64, 256) == lpq.ERR_INVALID_ARG  # plain scales


def test_scale_update_and_selftest_validation():
    L = lpq.lib()
    st = lpq.DelayedStateC(None, None, None, None, 16)
    assert L.lpq_scale_update(ctypes.byref(st), None, 448.0, None) == lpq.ERR_INVALID_ARG
    assert L.lpq_selftest_wait(0, None) == lpq.ERR_INVALID_ARG
    assert L.lpq_selftest_wait(5_000_000_000, None) == lpq.ERR_INVALID_ARG


def test_amax_validation():
    """lpq_amax checks flags, outputs, shapes and alignment before any device call."""
    L = lpq.lib()
    f = 16  # a 16-byte aligned fake device address: validation stops before the device check
    assert L.lpq_amax(f, 4, 32, 8, 0, f, None, None) == lpq.ERR_INVALID_ARG      # unknown flag
    assert L.lpq_amax(f, 4, 32, 0, 0, None, None, None) == lpq.ERR_INVALID_ARG   # no output
    assert L.lpq_amax(f, 4, 32, lpq.RHT_COLWISE, 0, f, None, None) == lpq.ERR_INVALID_ARG  # RHT without output
    assert L.lpq_amax(f, 4, 24, 0, 0, f, None, None) == lpq.ERR_SHAPE            # cols % 16
    assert L.lpq_amax(f, 8, 32, lpq.RHT_COLWISE, 0, f, f, None) == lpq.ERR_SHAPE  # rows % 16 for the RHT amax
    assert L.lpq_amax(8, 4, 32, 0, 0, f, None, None) == lpq.ERR_ALIGN           # x not 16-byte aligned
    assert L.lpq_amax(None, 4, 32, 0, 0, f, None, None) == lpq.ERR_INVALID_ARG
    ok = L.lpq_amax(f, 16, 32, lpq.RHT_COLWISE, 0, f, f, None)
    assert ok not in (lpq.ERR_INVALID_ARG, lpq.ERR_SHAPE, lpq.ERR_ALIGN)


def test_selftest_arith_validation():
    L = lpq.lib()
    assert L.lpq_selftest_arith(3, 0, 1, 0, 16, None) == lpq.ERR_INVALID_ARG        # no such check
    assert L.lpq_selftest_arith(0, 0, 0x7F800002, 0, 16, None) == lpq.ERR_INVALID_ARG  # past +inf
    assert L.lpq_selftest_arith(2, 1, 1 << 24, 0, 16, None) == lpq.ERR_INVALID_ARG  # past 2^24 words
    assert L.lpq_selftest_arith(0, 0, 1, 0, None, None) == lpq.ERR_INVALID_ARG
    assert L.lpq_selftest_arith(0, 0, 1, 0, 12, None) == lpq.ERR_INVALID_ARG        # result not 8-byte aligned


def test_mma_peak_validation():
    """Rate-probe arguments are checked before any device call."""
    L = lpq.lib()
    assert L.lpq_mma_peak(4, 10, 0, None) == lpq.ERR_INVALID_ARG     # no such kind
    assert L.lpq_mma_peak(3, 0, 0, None) == lpq.ERR_INVALID_ARG      # iters
    assert L.lpq_mma_peak(3, 10, 9, None) == lpq.ERR_INVALID_ARG     # no such mode
    assert L.lpq_mma_peak(2, 10, 4, None) == lpq.ERR_INVALID_ARG     # modes 2..5 are NVFP4 only
    assert L.lpq_mma_peak(0, 10, 7, None) == lpq.ERR_INVALID_ARG     # mode 7 is for the block-scaled kinds
    assert L.lpq_mma_peak(1, 10, -1, None) == lpq.ERR_INVALID_ARG


def test_gemm_options_validation():
    """lpq_gemm_ex checks its kernel-path options before anything else; the
    default options (all zero, or NULL) validate like lpq_gemm."""
    L = lpq.lib()
    v = lambda rows, cols: lpq.QView(16, 16, 16, 16, rows, cols, lpq.MXFP8, lpq.SF_GEMM, 0, 0)
    a, b = v(128, 256), v(64, 256)
    bad = [lpq.GemmOpts(single_cta=2), lpq.GemmOpts(tile_n=64), lpq.GemmOpts(scale_copies=-1),
           lpq.GemmOpts(direct_store=3), lpq.GemmOpts(whole_tiles=2),
           lpq.GemmOpts(reserved=(ctypes.c_int32 * 3)(0, 1, 0))]
    for opts in bad:
        assert L.lpq_gemm_ex(0, ctypes.byref(a), ctypes.byref(b), 16, 0, 128, 64, 256, ctypes.byref(opts),
                             None) == lpq.ERR_INVALID_ARG
    validated = (lpq.ERR_UNSUPPORTED, lpq.ERR_SHAPE, lpq.ERR_INVALID_ARG, lpq.ERR_ALIGN)
    for name, opts in lpq.GEMM_PATHS.items():  # legal options pass validation and stop at the device check
        assert L.lpq_gemm_ex(0, ctypes.byref(a), ctypes.byref(b), 16, 0, 128, 64, 256, ctypes.byref(opts),
                             None) not in validated, name
    assert L.lpq_gemm_ex(0, ctypes.byref(a), ctypes.byref(b), 16, 0, 128, 64, 256, None, None) not in validated


def test_given_amax_validation():
    """LPQ_GIVEN_AMAX applies to current-scaled per-tensor FP8 and NVFP4 only."""
    assert _quantize_raw(None, 4, 32, lpq.MXFP8, lpq.ROWWISE | lpq.GIVEN_AMAX) == lpq.ERR_UNSUPPORTED
    for fmt in (lpq.MXFP8_E5M2, lpq.MXFP4):
        assert _quantize_raw(None, 4, 32, fmt, lpq.ROWWISE | lpq.GIVEN_AMAX) == lpq.ERR_UNSUPPORTED
    assert _quantize_raw(None, 4, 128, lpq.FP8_BLOCK_1x128, lpq.ROWWISE | lpq.GIVEN_AMAX) == lpq.ERR_UNSUPPORTED
    assert _quantize_raw(None, 4, 32, lpq.FP8_E4M3, lpq.ROWWISE | lpq.GIVEN_AMAX, scaling=1) == lpq.ERR_UNSUPPORTED
    assert _quantize_raw(None, 4, 32, lpq.NVFP4, lpq.ROWWISE | 32) == lpq.ERR_INVALID_ARG  # unknown bit


def test_binding_constants_match_the_header():
    """Every LPQ_* enum value the header declares has the same value in the
    Python binding (LPQ_X <-> lpq.X), and the binding's format names cover
    every format."""
    text = open(os.path.join(ROOT, "include", "lpq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    values = {name: int(v) for name, v in re.findall(r"\bLPQ_([A-Z0-9_a-z]+)\s*=\s*(\d+)", text)}
    assert len(values) >= 30
    for name, v in values.items():
        assert hasattr(lpq, name), name
        assert getattr(lpq, name) == v, (name, getattr(lpq, name), v)
    formats = [n for n in ("BF16", "FP8_E4M3", "FP8_E5M2", "MXFP8", "NVFP4", "NVFP4_2D", "FP8_BLOCK_1x128",
                           "FP8_BLOCK_128x128", "MXFP8_E5M2", "MXFP4")]
    assert sorted(getattr(lpq, n) for n in formats) == list(range(len(formats)))
    assert set(lpq.FORMAT_NAMES) == set(range(len(formats)))
