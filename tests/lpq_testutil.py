"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and the CPU oracle on the same seeded bf16 input, and bring tensors
back to numpy in the oracle's plain layouts.  Pure index bookkeeping; no
format arithmetic."""
import numpy as np
import torch

import oracle as o
from precision_transformer_gemms_gb300 import lpq, synth


def np_u8(t):
    return t.detach().cpu().numpy()


def sf_gemm_to_plain(buf, rows, nblocks, kt):
    """Tensor-core scale layout -> plain [rows, nblocks] (see lpq_copy_bytes)."""
    buf = np.asarray(buf)
    r = np.arange(rows)[:, None]
    kb = np.arange(nblocks)[None, :]
    off = ((r >> 7) * kt + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3)
    return buf[off]


MX_FORMATS = (lpq.MXFP8, lpq.MXFP8_E5M2, lpq.MXFP4)


def kt_atoms(fmt, cols):
    if fmt in (lpq.MXFP8, lpq.MXFP8_E5M2):
        return (cols + 127) // 128
    if fmt == lpq.MXFP4:
        return ((cols + 255) // 256) * 2
    return ((cols + 255) // 256) * 4


def codes(copy):
    return np_u8(copy.codes_matrix())


def plain_scales(copy):
    """Scales of a Copy in the oracle's plain layout."""
    f = copy.fmt
    if f in MX_FORMATS + (lpq.NVFP4, lpq.NVFP4_2D):
        blk = 32 if f in MX_FORMATS else 16
        nb = copy.cols // blk
        buf = np_u8(copy.scales)
        if copy.sf_layout == lpq.SF_GEMM:
            return sf_gemm_to_plain(buf, copy.rows, nb, kt_atoms(f, copy.cols))
        return buf[: copy.rows * nb].reshape(copy.rows, nb)
    if f == lpq.FP8_BLOCK_1x128:
        nb = copy.cols // 128
        buf = copy.scales.cpu().numpy()
        if copy.sf_layout == lpq.SF_GEMM:
            return buf[: nb * copy.rows].reshape(nb, copy.rows).T.copy()
        return buf[: copy.rows * nb].reshape(copy.rows, nb)
    if f == lpq.FP8_BLOCK_128x128:
        nb = copy.cols // 128
        nr = (copy.rows + 127) // 128
        return copy.scales.cpu().numpy()[: nr * nb].reshape(nr, nb)
    return None


def scalar(t):
    return float(t.cpu().numpy()[0])


def bf16_input(shape, std=1.0, seed=0, outlier_frac=0.0, outlier_scale=1.0):
    x = synth.bf16_normal(shape, std, seed, "cuda", outlier_frac, outlier_scale)
    return x, synth.host_bits(x)


def oracle_operand(copy, fmt_override=None):
    """An oracle GEMM operand built from the GPU's codes (to check the GEMM
    alone, given codes the quantizer tests have already checked)."""
    f = fmt_override if fmt_override is not None else copy.fmt
    if f == lpq.BF16:
        return o.Operand(o.K_BF16, copy.codes.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
    if f in (lpq.FP8_E4M3, lpq.FP8_E5M2):
        return o.Operand(o.K_FP8_E4M3 if f == lpq.FP8_E4M3 else o.K_FP8_E5M2, codes(copy), ts=scalar(copy.tensor_scale))
    if f == lpq.MXFP8:
        return o.Operand(o.K_MXFP8, codes(copy), plain_scales(copy))
    if f == lpq.MXFP8_E5M2:
        return o.Operand(o.K_MXFP8_E5M2, codes(copy), plain_scales(copy))
    if f == lpq.MXFP4:
        return o.Operand(o.K_MXFP4, codes(copy), plain_scales(copy))
    if f in (lpq.NVFP4, lpq.NVFP4_2D):
        return o.Operand(o.K_NVFP4, codes(copy), plain_scales(copy), scalar(copy.tensor_scale))
    if f == lpq.FP8_BLOCK_1x128:
        return o.Operand(o.K_FP8_BLOCK, codes(copy), plain_scales(copy), block_rows=1)
    if f == lpq.FP8_BLOCK_128x128:
        return o.Operand(o.K_FP8_BLOCK, codes(copy), plain_scales(copy), block_rows=128)
    raise ValueError(f)


def gemm_gate(c_gpu, c_ref, bound, bf16_out):
    """|C - C_ref| <= 1e-3 * sum|a b| (+ half a bf16 ulp of C for bf16 output)."""
    c = c_gpu.float().cpu().numpy().astype(np.float64)
    tol = 1e-3 * bound
    if bf16_out:
        mag = np.abs(c_ref)
        ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.maximum(mag, 1e-300))) - 7), 0.0)
        tol = tol + 0.5 * ulp * (1 + 2 ** -6)
    err = np.abs(c - c_ref)
    bad = err > tol
    return int(bad.sum()), float(np.max(err / np.maximum(tol, 1e-300)))
