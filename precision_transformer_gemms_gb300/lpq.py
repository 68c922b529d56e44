"""Python binding of liblpq (ctypes; argument marshalling only).

Every step of the quantize / GEMM path runs in liblpq's CUDA kernels.  This
module only allocates output buffers with torch, builds the C views and passes
pointers and the current CUDA stream.  If the shared library cannot be built or
loaded, every call raises: there is no CPU or PyTorch fallback.
"""
import ctypes
import os

import torch

from . import build as _build

# ----------------------------------------------------------------- enums (mirror include/lpq.h)
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_ARCH, ERR_CUDA, ERR_TIMEOUT = range(8)
(BF16, FP8_E4M3, FP8_E5M2, MXFP8, NVFP4, NVFP4_2D, FP8_BLOCK_1x128, FP8_BLOCK_128x128, MXFP8_E5M2,
 MXFP4) = range(10)
SCALING_CURRENT, SCALING_DELAYED = 0, 1
ROWWISE, COLWISE, RHT_COLWISE, STOCHASTIC, GIVEN_AMAX = 1, 2, 4, 8, 16
SF_PLAIN, SF_GEMM = 0, 1
FPROP, DGRAD, WGRAD = 0, 1, 2

STATUS_NAMES = {OK: "OK", ERR_INVALID_ARG: "INVALID_ARG", ERR_SHAPE: "SHAPE", ERR_ALIGN: "ALIGN",
                ERR_UNSUPPORTED: "UNSUPPORTED", ERR_ARCH: "ARCH", ERR_CUDA: "CUDA", ERR_TIMEOUT: "TIMEOUT"}
FORMAT_NAMES = {BF16: "bf16", FP8_E4M3: "fp8_e4m3", FP8_E5M2: "fp8_e5m2", MXFP8: "mxfp8", NVFP4: "nvfp4",
                NVFP4_2D: "nvfp4_2d", FP8_BLOCK_1x128: "fp8_block_1x128", FP8_BLOCK_128x128: "fp8_block_128x128",
                MXFP8_E5M2: "mxfp8_e5m2", MXFP4: "mxfp4"}
PACKED_FP4 = (NVFP4, NVFP4_2D, MXFP4)  # two E2M1 codes per byte
FMAX = {FP8_E4M3: 448.0, FP8_E5M2: 57344.0}


class LpqError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"lpq status {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class QView(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("fmt", ctypes.c_int32), ("sf_layout", ctypes.c_int32), ("colwise", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class QTensorC(ctypes.Structure):
    _fields_ = [("row", QView), ("col", QView)]


class DelayedStateC(ctypes.Structure):
    _fields_ = [("amax_history", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("scale_inv", ctypes.c_void_p), ("len", ctypes.c_int32)]


class GemmOpts(ctypes.Structure):
    """Kernel-path options of lpq_gemm_ex (all zero: the default path)."""
    _fields_ = [("single_cta", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("scale_copies", ctypes.c_int32),
                ("direct_store", ctypes.c_int32), ("whole_tiles", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]


# Named kernel paths of the GEMM (every one computes the same result).
GEMM_PATHS = {
    "default": GemmOpts(),
    "pair": GemmOpts(),                               # CTA pairs where m >= 256 (the default)
    "pair_direct": GemmOpts(direct_store=1),          # CTA pairs, bf16 C stored from registers
    "pair_whole": GemmOpts(whole_tiles=1),            # CTA pairs, no 256 x 128 halves in the last round
    "pair_cp": GemmOpts(scale_copies=1),              # CTA pairs, scale factors copied by the MMA thread
    "single": GemmOpts(single_cta=1),                 # one CTA per 128 x 256 tile
    "single_cp": GemmOpts(single_cta=1, scale_copies=1),  # scale factors copied by the MMA thread
    "single_bn128": GemmOpts(single_cta=1, tile_n=128),   # one CTA per 128 x 128 tile
    "single_bn128_cp": GemmOpts(single_cta=1, tile_n=128, scale_copies=1),  # the same, scales copied
}


class TransformerCfg(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("intermediate", ctypes.c_int64), ("heads", ctypes.c_int64),
                ("layers", ctypes.c_int64), ("micro_batch", ctypes.c_int64), ("seq", ctypes.c_int64)]


class GemmShape(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("layout", ctypes.c_int32), ("m", ctypes.c_int64),
                ("k", ctypes.c_int64), ("n", ctypes.c_int64)]


_lib = None


def lib():
    """Loads liblpq.so (building it from source if it is not there yet)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            path = _build.build()
        L = ctypes.CDLL(path)
        P, I32, I64, U32, U64, F = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                    ctypes.c_uint64, ctypes.c_float)
        L.lpq_copy_bytes.argtypes = [I32, I64, I64, I32, ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_size_t)]
        L.lpq_quantize.argtypes = [P, I64, I64, I32, I32, U32, U64, U64, U32, ctypes.POINTER(DelayedStateC),
                                   ctypes.POINTER(QTensorC), P]
        L.lpq_scale_update.argtypes = [ctypes.POINTER(DelayedStateC), P, F, P]
        L.lpq_amax.argtypes = [P, I64, I64, U32, U32, P, P, P]
        L.lpq_gemm.argtypes = [I32, ctypes.POINTER(QView), ctypes.POINTER(QView), P, I32, I64, I64, I64, P]
        L.lpq_gemm_ex.argtypes = [I32, ctypes.POINTER(QView), ctypes.POINTER(QView), P, I32, I64, I64, I64,
                                  ctypes.POINTER(GemmOpts), P]
        L.lpq_layer_shapes.argtypes = [ctypes.POINTER(TransformerCfg), ctypes.POINTER(GemmShape),
                                       ctypes.POINTER(I32)]
        L.lpq_last_error.restype = ctypes.c_char_p
        L.lpq_device_status.argtypes = [P, ctypes.POINTER(I32)]
        L.lpq_selftest_wait.argtypes = [U64, P]
        L.lpq_mma_peak.argtypes = [I32, I32, I32, P]
        L.lpq_selftest_arith.argtypes = [I32, U64, U64, U32, P, P]
        L.lpq_version.restype = I32
        for name in ("lpq_copy_bytes", "lpq_quantize", "lpq_scale_update", "lpq_gemm", "lpq_gemm_ex", "lpq_amax", "lpq_layer_shapes",
                     "lpq_device_status", "lpq_selftest_wait", "lpq_mma_peak", "lpq_selftest_arith"):
            getattr(L, name).restype = I32
        _lib = L
    return _lib


def _check(status):
    if status != OK:
        raise LpqError(status, lib().lpq_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def last_error():
    return lib().lpq_last_error().decode(errors="replace")


def version():
    return lib().lpq_version()


# ----------------------------------------------------------------- host-only helpers
def copy_bytes(fmt, rows, cols, sf_layout=SF_GEMM):
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().lpq_copy_bytes(fmt, rows, cols, sf_layout, ctypes.byref(cb), ctypes.byref(sb)))
    return cb.value, sb.value


def layer_shapes(hidden, intermediate, micro_batch, seq, heads=32, layers=1):
    cfg = TransformerCfg(hidden, intermediate, heads, layers, micro_batch, seq)
    out = (GemmShape * 12)()
    n = ctypes.c_int32()
    _check(lib().lpq_layer_shapes(ctypes.byref(cfg), out, ctypes.byref(n)))
    return [(s.name.decode(), s.layout, s.m, s.k, s.n) for s in out[:n.value]]


# ----------------------------------------------------------------- device buffers
class Copy:
    """One quantized copy: torch-owned device buffers plus its C view."""

    def __init__(self, fmt, rows, cols, colwise, sf_layout=SF_GEMM, device="cuda"):
        self.fmt, self.rows, self.cols, self.colwise, self.sf_layout = fmt, rows, cols, int(colwise), sf_layout
        cb, sb = copy_bytes(fmt, rows, cols, sf_layout)
        if fmt == BF16:
            self.codes = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
        else:
            self.codes = torch.empty(max(cb, 1), dtype=torch.uint8, device=device)
        if fmt in (FP8_BLOCK_1x128, FP8_BLOCK_128x128):
            self.scales = torch.empty(max(sb // 4, 1), dtype=torch.float32, device=device)
        elif sb:
            self.scales = torch.empty(sb, dtype=torch.uint8, device=device)
        else:
            self.scales = None
        # per-tensor factor and amax only where the format has them
        scalar = fmt in (FP8_E4M3, FP8_E5M2, NVFP4, NVFP4_2D)
        self.tensor_scale = torch.ones(1, dtype=torch.float32, device=device) if scalar else None
        self.amax = torch.zeros(1, dtype=torch.float32, device=device) if scalar else None

    @classmethod
    def of_bf16(cls, x, colwise=False):
        """Wraps an existing contiguous bf16 tensor [rows, cols] as a bf16 operand."""
        c = cls.__new__(cls)
        c.fmt, c.rows, c.cols, c.colwise, c.sf_layout = BF16, x.shape[0], x.shape[1], int(colwise), SF_PLAIN
        c.codes, c.scales, c.tensor_scale, c.amax = x.contiguous(), None, None, None
        return c

    def view(self):
        return QView(_ptr(self.codes), _ptr(self.scales), _ptr(self.tensor_scale), _ptr(self.amax), self.rows,
                     self.cols, self.fmt, self.sf_layout, self.colwise, 0)

    def codes_matrix(self):
        """Codes as a [rows, bytes per row] uint8 tensor (packed for NVFP4 and MXFP4)."""
        if self.fmt == BF16:
            return self.codes
        per_row = self.cols // 2 if self.fmt in PACKED_FP4 else self.cols
        return self.codes[: self.rows * per_row].view(self.rows, per_row)


class QTensor:
    def __init__(self, row=None, col=None):
        self.row, self.col = row, col


class DelayedState:
    """Delayed-scaling state on the device: amax ring, position, scale, 1/scale."""

    def __init__(self, length=16, device="cuda"):
        self.hist = torch.zeros(length, dtype=torch.float32, device=device)
        self.pos = torch.zeros(1, dtype=torch.int32, device=device)
        self.scale = torch.ones(1, dtype=torch.float32, device=device)
        self.scale_inv = torch.ones(1, dtype=torch.float32, device=device)

    def c(self):
        return DelayedStateC(_ptr(self.hist), _ptr(self.pos), _ptr(self.scale), _ptr(self.scale_inv),
                             self.hist.numel())


def alloc(fmt, rows, cols, flags, sf_layout=SF_GEMM, device="cuda"):
    return QTensor(Copy(fmt, rows, cols, False, sf_layout, device) if flags & ROWWISE else None,
                   Copy(fmt, cols, rows, True, sf_layout, device) if flags & COLWISE else None)


def quantize(x, fmt, flags, scaling=SCALING_CURRENT, seed=0, counter_offset=0, rht_seed=0, state=None,
             sf_layout=SF_GEMM, out=None, stream=None):
    """lpq_quantize on a bf16 CUDA tensor x [rows, cols]; returns a QTensor."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    if out is None:
        out = alloc(fmt, rows, cols, flags, sf_layout, x.device)
    qt = QTensorC(out.row.view() if out.row is not None else QView(),
                  out.col.view() if out.col is not None else QView())
    st = ctypes.byref(state.c()) if state is not None else None
    _check(lib().lpq_quantize(_ptr(x), rows, cols, fmt, scaling, flags, seed, counter_offset, rht_seed, st,
                              ctypes.byref(qt), _stream(stream)))
    return out


def amax(x, rht=False, rht_seed=0, out=None, rht_out=None, stream=None):
    """lpq_amax on a bf16 CUDA tensor x [rows, cols]: max |x| into `out` (and,
    with rht, the column-wise RHT amax into `rht_out`); returns (out, rht_out)
    as 1-element FP32 device tensors."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    if rht and rht_out is None:
        rht_out = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().lpq_amax(_ptr(x), x.shape[0], x.shape[1], RHT_COLWISE if rht else 0, rht_seed, _ptr(out),
                          _ptr(rht_out) if rht else None, _stream(stream)))
    return out, (rht_out if rht else None)


def scale_update(state, amax, fmax, stream=None):
    _check(lib().lpq_scale_update(ctypes.byref(state.c()), _ptr(amax), float(fmax), _stream(stream)))


def gemm(layout, a, b, c=None, out_fp32=False, stream=None, path=None):
    """lpq_gemm: C[m, n] = sum_k deq(a)[m, k] deq(b)[n, k]; a, b are Copy objects.
    `path` (a GEMM_PATHS name or a GemmOpts) selects a kernel path through
    lpq_gemm_ex; None is lpq_gemm's default."""
    m, k, n = a.rows, a.cols, b.rows
    if c is None:
        c = torch.empty((m, n), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=a.codes.device)
    va, vb = a.view(), b.view()
    if path is None:
        _check(lib().lpq_gemm(layout, ctypes.byref(va), ctypes.byref(vb), _ptr(c), int(out_fp32), m, n, k,
                              _stream(stream)))
    else:
        opts = GEMM_PATHS[path] if isinstance(path, str) else path
        _check(lib().lpq_gemm_ex(layout, ctypes.byref(va), ctypes.byref(vb), _ptr(c), int(out_fp32), m, n, k,
                                 ctypes.byref(opts), _stream(stream)))
    return c


def device_status(stream=None):
    code = ctypes.c_int32()
    _check(lib().lpq_device_status(_stream(stream), ctypes.byref(code)))
    return code.value


def selftest_wait(limit_ns, stream=None):
    _check(lib().lpq_selftest_wait(int(limit_ns), _stream(stream)))


def selftest_arith(which, begin, count, param=0, stream=None):
    """lpq_selftest_arith: (mismatches, first mismatching index or -1)."""
    out = torch.empty(2, dtype=torch.int64, device="cuda")
    _check(lib().lpq_selftest_arith(which, begin, count, param, _ptr(out), _stream(stream)))
    torch.cuda.synchronize()
    n, first = out.tolist()
    return n, (-1 if n == 0 else first)


MMA_KINDS = {"bf16": 0, "fp8": 1, "mxfp8": 2, "nvfp4": 3}
MMA_K = {0: 16, 1: 32, 2: 32, 3: 64}


def mma_peak(kind, iters=20000, with_scale_copies=True, stream=None):
    """Dense tcgen05 rate in TFLOP/s for `kind` (see lpq_mma_peak; modes 6 to
    8 run on CTA pairs)."""
    k = MMA_KINDS[kind] if isinstance(kind, str) else kind
    mode = int(with_scale_copies)
    st = stream if stream is not None else torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _check(lib().lpq_mma_peak(k, 64, mode, _stream(st)))  # warm-up
    e0.record(st)
    _check(lib().lpq_mma_peak(k, iters, mode, _stream(st)))  # mode 0..7
    e1.record(st)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    ctas = sms & ~1 if mode >= 6 else sms
    flops = ctas * iters * 4 * 2 * 128 * 256 * MMA_K[k]
    return flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
