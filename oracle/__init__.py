"""CPU oracle for the low-precision quantize-then-GEMM path — TEST INFRASTRUCTURE.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It wraps the plain C++ statement of every format,
quantizer and the FP64 GEMM in ``lpq_oracle.cpp`` (see that file for the
passages each function follows) with numpy-level helpers.  It never imports the
CUDA library and the CUDA library never imports it.
"""
import ctypes
import os

import numpy as np

from . import build as _build

E4M3, E5M2, E2M1 = 0, 1, 2
FMAX = {E4M3: 448.0, E5M2: 57344.0, E2M1: 6.0}

# Operand kinds of the FP64 GEMM (see OrcOperand in lpq_oracle.cpp).
K_BF16, K_FP8_E4M3, K_FP8_E5M2, K_MXFP8, K_NVFP4, K_FP8_BLOCK, K_MXFP8_E5M2, K_MXFP4 = range(8)

_lib = None


class _Operand(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("block_rows", ctypes.c_int32),
                ("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("ts", ctypes.c_double)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I64, F, U8, U32, U64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_uint8,
                                   ctypes.c_uint32, ctypes.c_uint64)
        L.orc_decode.restype = ctypes.c_double
        L.orc_decode.argtypes = [ctypes.c_int, U8]
        L.orc_encode.restype = U8
        L.orc_encode.argtypes = [ctypes.c_int, F]
        L.orc_encode_array.argtypes = [ctypes.c_int, P, I64, P]
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_sr_word.restype = U32
        L.orc_sr_word.argtypes = [U64, U64, U32]
        L.orc_rht_sign_mask.restype = U32
        L.orc_rht_sign_mask.argtypes = [U32]
        L.orc_rht16.argtypes = [P, U32, P]
        L.orc_sr_encode_e2m1.restype = U8
        L.orc_sr_encode_e2m1.argtypes = [F, U32]
        L.orc_mx_exponent.restype = ctypes.c_int
        L.orc_mx_exponent.argtypes = [F]
        L.orc_amax_bf16.restype = F
        L.orc_amax_bf16.argtypes = [P, I64]
        L.orc_fp8_pertensor.restype = I64
        L.orc_fp8_pertensor.argtypes = [P, I64, I64, ctypes.c_int, P, P, P, P, P, P]
        L.orc_scale_update.argtypes = [P, ctypes.c_int32, P, P, P, F, F]
        L.orc_mxfp8.argtypes = [P, I64, I64, P, P, P, P]
        L.orc_mx.argtypes = [P, I64, I64, ctypes.c_int, P, P, P, P]
        L.orc_mx_exponent_fmt.restype = ctypes.c_int
        L.orc_mx_exponent_fmt.argtypes = [F, ctypes.c_int]
        L.orc_nvfp4.argtypes = [P, I64, I64, ctypes.c_uint, U64, U64, U32, P, P, P, P, P, P, P, P]
        L.orc_fp8_block.argtypes = [P, I64, I64, ctypes.c_int, P, P, P, P]
        L.orc_gemm.argtypes = [ctypes.POINTER(_Operand), ctypes.POINTER(_Operand), I64, I64, I64, P, I64, P, P]
        L.orc_dequant.argtypes = [ctypes.POINTER(_Operand), I64, I64, I64, P]
        L.orc_layer_shapes.argtypes = [I64, I64, I64, I64, P]
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _bits(x):
    """bf16 input as a contiguous uint16 array of its bit patterns."""
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "oracle inputs are bf16 bit patterns (uint16)"
    return x


def num_threads():
    return lib().orc_num_threads()


def set_threads(n):
    lib().orc_set_threads(int(n))


# ------------------------------------------------------------------ codecs
def decode(fmt, codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return np.array([lib().orc_decode(fmt, int(c)) for c in codes.ravel()]).reshape(codes.shape)


def encode(fmt, y):
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    out = np.empty(y.shape, np.uint8)
    lib().orc_encode_array(fmt, y.ctypes.data, y.size, out.ctypes.data)
    return out


def bf16_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ random / transform
def philox(ctr, key):
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.empty(4, np.uint32)
    lib().orc_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def sr_word(seed, j, copy_id):
    return lib().orc_sr_word(seed, j, copy_id)


def rht_sign_mask(rht_seed):
    return lib().orc_rht_sign_mask(rht_seed)


def rht16(x, signs):
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(16, np.float32)
    lib().orc_rht16(x.ctypes.data, signs, out.ctypes.data)
    return out


def sr_encode_e2m1(y, r):
    return lib().orc_sr_encode_e2m1(float(y), int(r))


def mx_exponent(a, fmt=E4M3):
    """The MX block exponent: the smallest e with fmax(fmt) * 2^e >= a."""
    if fmt == E4M3:
        return lib().orc_mx_exponent(float(a))
    return lib().orc_mx_exponent_fmt(float(a), fmt)


def amax(x_bits):
    x = _bits(x_bits)
    return lib().orc_amax_bf16(x.ctypes.data, x.size)


# ------------------------------------------------------------------ quantizers
def fp8_pertensor(x_bits, fmt, scale=None, rowwise=True, colwise=True):
    """Per-tensor FP8; scale=None is current scaling, a float is delayed scaling.

    Returns dict(row, col, scale, scale_inv, amax, saturated)."""
    x = _bits(x_bits)
    R, C = x.shape
    row = np.empty((R, C), np.uint8) if rowwise else None
    col = np.empty((C, R), np.uint8) if colwise else None
    s_in = None if scale is None else np.array([scale], np.float32)
    s, si, am = (np.zeros(1, np.float32) for _ in range(3))
    sat = lib().orc_fp8_pertensor(x.ctypes.data, R, C, fmt, _p(s_in), _p(row), _p(col), s.ctypes.data,
                                  si.ctypes.data, am.ctypes.data)
    return dict(row=row, col=col, scale=float(s[0]), scale_inv=float(si[0]), amax=float(am[0]),
                saturated=int(sat))


class DelayedState:
    """Delayed-scaling state: amax ring, position, scale and its inverse."""

    def __init__(self, length=16):
        self.hist = np.zeros(length, np.float32)
        self.pos = np.zeros(1, np.int32)
        self.scale = np.ones(1, np.float32)
        self.scale_inv = np.ones(1, np.float32)

    def update(self, amax_value, fmax):
        lib().orc_scale_update(self.hist.ctypes.data, len(self.hist), self.pos.ctypes.data,
                               self.scale.ctypes.data, self.scale_inv.ctypes.data, float(amax_value),
                               float(fmax))


def mxfp8(x_bits, rowwise=True, colwise=True):
    x = _bits(x_bits)
    R, C = x.shape
    out = {}
    rc = np.empty((R, C), np.uint8) if rowwise else None
    rs = np.empty((R, C // 32), np.uint8) if rowwise else None
    cc = np.empty((C, R), np.uint8) if colwise else None
    cs = np.empty((C, R // 32), np.uint8) if colwise else None
    lib().orc_mxfp8(x.ctypes.data, R, C, _p(rc), _p(rs), _p(cc), _p(cs))
    out.update(row=rc, row_sf=rs, col=cc, col_sf=cs)
    return out


def mx(x_bits, fmt, rowwise=True, colwise=True):
    """MX quantization with element format fmt (E4M3, E5M2, or E2M1 packed two
    per byte); returns dict(row, row_sf, col, col_sf) in plain layouts."""
    x = _bits(x_bits)
    R, C = x.shape
    per = 2 if fmt == E2M1 else 1
    rc = np.zeros((R, C // per), np.uint8) if rowwise else None
    rs = np.zeros((R, C // 32), np.uint8) if rowwise else None
    cc = np.zeros((C, R // per), np.uint8) if colwise else None
    cs = np.zeros((C, R // 32), np.uint8) if colwise else None
    lib().orc_mx(x.ctypes.data, R, C, fmt, _p(rc), _p(rs), _p(cc), _p(cs))
    return dict(row=rc, row_sf=rs, col=cc, col_sf=cs)


NV_ROW, NV_COL, NV_RHT, NV_SR, NV_2D = 1, 2, 4, 8, 16


def nvfp4(x_bits, flags, seed=0, counter_offset=0, rht_seed=0):
    x = _bits(x_bits)
    R, C = x.shape
    rc = np.zeros((R, C // 2), np.uint8) if flags & NV_ROW else None
    rs = np.zeros((R, C // 16), np.uint8) if flags & NV_ROW else None
    cc = np.zeros((C, R // 2), np.uint8) if flags & NV_COL else None
    cs = np.zeros((C, R // 16), np.uint8) if flags & NV_COL else None
    rts, ram, cts, cam = (np.zeros(1, np.float32) for _ in range(4))
    lib().orc_nvfp4(x.ctypes.data, R, C, flags, seed, counter_offset, rht_seed, _p(rc), _p(rs),
                    rts.ctypes.data, ram.ctypes.data, _p(cc), _p(cs), cts.ctypes.data, cam.ctypes.data)
    return dict(row=rc, row_sf=rs, row_ts=float(rts[0]), row_amax=float(ram[0]), col=cc, col_sf=cs,
                col_ts=float(cts[0]), col_amax=float(cam[0]))


def fp8_block(x_bits, block_rows, rowwise=True, colwise=True):
    x = _bits(x_bits)
    R, C = x.shape
    rc = np.empty((R, C), np.uint8) if rowwise else None
    rs = np.empty(((R + block_rows - 1) // block_rows, C // 128), np.float32) if rowwise else None
    cc = np.empty((C, R), np.uint8) if colwise else None
    if block_rows == 1:
        cs = np.empty((C, R // 128), np.float32) if colwise else None
    else:
        cs = np.empty((C // 128, (R + 127) // 128), np.float32) if colwise else None
    lib().orc_fp8_block(x.ctypes.data, R, C, block_rows, _p(rc), _p(rs), _p(cc), _p(cs))
    return dict(row=rc, row_sinv=rs, col=cc, col_sinv=cs)


# ------------------------------------------------------------------ GEMM
class Operand:
    """A quantized operand [rows, K] contiguous along K, as the GEMM reads it."""

    def __init__(self, kind, codes, sf=None, ts=1.0, block_rows=1):
        self.kind, self.codes, self.sf, self.ts, self.block_rows = kind, np.ascontiguousarray(codes), \
            (None if sf is None else np.ascontiguousarray(sf)), float(ts), int(block_rows)

    def _c(self):
        return _Operand(self.kind, self.block_rows, self.codes.ctypes.data,
                        None if self.sf is None else self.sf.ctypes.data, self.ts)


def gemm(a, b, M, N, K, pairs=None):
    """FP64 C[m, n] = sum_k deq(a)[m, k] deq(b)[n, k] and the bound sum |.|.

    pairs: None (all, returns [M, N] arrays) or an int64 array [P, 2]."""
    ca, cb = a._c(), b._c()
    if pairs is None:
        c = np.empty((M, N), np.float64)
        bd = np.empty((M, N), np.float64)
        lib().orc_gemm(ctypes.byref(ca), ctypes.byref(cb), M, N, K, None, 0, c.ctypes.data, bd.ctypes.data)
        return c, bd
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64))
    n = pairs.shape[0]
    c = np.empty(n, np.float64)
    bd = np.empty(n, np.float64)
    lib().orc_gemm(ctypes.byref(ca), ctypes.byref(cb), M, N, K, pairs.ctypes.data, n, c.ctypes.data, bd.ctypes.data)
    return c, bd


def dequant(op, K, r0, r1):
    out = np.empty((r1 - r0, K), np.float64)
    lib().orc_dequant(ctypes.byref(op._c()), K, r0, r1, out.ctypes.data)
    return out


# ------------------------------------------------------------------ shapes
LINEARS = ("qkv", "attn_out", "mlp_up", "mlp_down")
PASSES = ("fprop", "dgrad", "wgrad")


def layer_shapes(hidden, intermediate, micro_batch, seq):
    out = np.zeros((12, 3), np.int64)
    lib().orc_layer_shapes(hidden, intermediate, micro_batch, seq, out.ctypes.data)
    names = [f"{l}_{p}" for l in LINEARS for p in PASSES]
    return [(names[i], int(out[i, 0]), int(out[i, 1]), int(out[i, 2])) for i in range(12)]
