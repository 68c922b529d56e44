"""Token-sharded data parallelism emulated on one GPU: the rows (tokens) of X
and dY are split into slabs, each slab measures its amax, the amaxes are
combined with a MAX on the device (the all-reduce a multi-GPU run would do),
and each slab is quantized with that global amax (LPQ_GIVEN_AMAX).  Codes,
block scales and tensor scales must then be bit-identical to the unsharded
quantization; the Wgrad partials of the slabs, summed on the device (the
all-reduce SUM of dW), must meet the GEMM gate against the oracle's FP64 GEMM
of the whole tensors' operands."""
import numpy as np
import pytest
import torch

import oracle as o
from precision_transformer_gemms_gb300 import lpq
from lpq_testutil import bf16_input, codes, gemm_gate, oracle_operand, plain_scales, scalar

pytestmark = pytest.mark.gpu

M, C, G = 1024, 512, 2  # tokens, features, shards


def shard_quantize(x, fmt, flags, rows_per, counter_row_offset, sf_layout=lpq.SF_PLAIN):
    """Slab-by-slab: amax pass, device MAX, quantize with the global amax."""
    slabs = [x[g * rows_per:(g + 1) * rows_per].contiguous() for g in range(G)]
    # the amax pass of each slab (same Hadamard signs as the quantization)
    first = [lpq.quantize(s, fmt, flags, seed=5, rht_seed=9, sf_layout=sf_layout) for s in slabs]
    out = []
    for g, s in enumerate(slabs):
        q = lpq.alloc(fmt, rows_per, x.shape[1], flags, sf_layout)
        for copy_name in ("row", "col"):
            dst = getattr(q, copy_name)
            if dst is None:
                continue
            amax = torch.stack([getattr(f, copy_name).amax for f in first]).max(dim=0).values
            dst.amax.copy_(amax)
        off = g * rows_per * x.shape[1] if counter_row_offset else 0
        out.append(lpq.quantize(s, fmt, flags | lpq.GIVEN_AMAX, seed=5, counter_offset=off, rht_seed=9,
                                sf_layout=sf_layout, out=q))
    return out


@pytest.mark.parametrize("fmt,flags", [
    (lpq.FP8_E4M3, lpq.ROWWISE | lpq.COLWISE),
    (lpq.FP8_E5M2, lpq.ROWWISE | lpq.COLWISE),
    (lpq.NVFP4, lpq.ROWWISE | lpq.COLWISE),
    (lpq.NVFP4, lpq.ROWWISE | lpq.STOCHASTIC),
    (lpq.NVFP4, lpq.COLWISE | lpq.RHT_COLWISE),
])
def test_sharded_quantize_is_bit_identical(fmt, flags):
    x, _ = bf16_input((M, C), std=1.0, seed=21, outlier_frac=0.001, outlier_scale=40)
    whole = lpq.quantize(x, fmt, flags, seed=5, rht_seed=9, sf_layout=lpq.SF_PLAIN)
    rows_per = M // G
    shards = shard_quantize(x, fmt, flags, rows_per, counter_row_offset=bool(flags & lpq.STOCHASTIC))
    torch.cuda.synchronize()
    assert lpq.device_status() == 0
    for g, q in enumerate(shards):
        r0, r1 = g * rows_per, (g + 1) * rows_per
        if whole.row is not None:
            assert np.array_equal(codes(q.row), codes(whole.row)[r0:r1])
            if fmt == lpq.NVFP4:
                assert np.array_equal(plain_scales(q.row), plain_scales(whole.row)[r0:r1])
            assert scalar(q.row.tensor_scale) == scalar(whole.row.tensor_scale)
        if whole.col is not None:
            per = 2 if fmt == lpq.NVFP4 else 1  # values per code byte
            assert np.array_equal(codes(q.col), codes(whole.col)[:, r0 // per:r1 // per])
            if fmt == lpq.NVFP4:
                assert np.array_equal(plain_scales(q.col), plain_scales(whole.col)[:, r0 // 16:r1 // 16])
            assert scalar(q.col.tensor_scale) == scalar(whole.col.tensor_scale)


@pytest.mark.parametrize("fmt,flags", [(lpq.NVFP4, lpq.COLWISE | lpq.RHT_COLWISE),
                                       (lpq.FP8_E4M3, lpq.COLWISE)])
def test_sharded_wgrad_sum_meets_gate(fmt, flags):
    """dW = sum over slabs of dY_g^T X_g, each from the slab's column copies."""
    N = 384
    x, _ = bf16_input((M, C), std=1.0, seed=22)
    dy, _ = bf16_input((M, N), std=1e-3, seed=23)
    rows_per = M // G
    qx = shard_quantize(x, fmt, flags, rows_per, False, lpq.SF_GEMM)  # the GEMM reads tensor-core scales
    qd = shard_quantize(dy, fmt, flags, rows_per, False, lpq.SF_GEMM)
    dw = None
    for g in range(G):
        part = lpq.gemm(lpq.WGRAD, qd[g].col, qx[g].col, out_fp32=True)
        dw = part if dw is None else dw + part  # the all-reduce SUM, on the device
    whole_x = lpq.quantize(x, fmt, flags, seed=5, rht_seed=9, sf_layout=lpq.SF_PLAIN)
    whole_d = lpq.quantize(dy, fmt, flags, seed=5, rht_seed=9, sf_layout=lpq.SF_PLAIN)
    torch.cuda.synchronize()
    assert lpq.device_status() == 0
    ref, bound = o.gemm(oracle_operand(whole_d.col), oracle_operand(whole_x.col), N, C, M)
    nbad, worst = gemm_gate(dw, ref, bound, False)
    assert nbad == 0, f"{nbad} elements outside the gate (worst {worst:.3g}x)"


@pytest.mark.parametrize("fmt", [lpq.FP8_E4M3, lpq.FP8_E5M2, lpq.NVFP4])
def test_empty_shard_takes_tensor_scale_from_given_amax(fmt):
    """A rank with no tokens still publishes the tensor scales of the global amax."""
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q = lpq.alloc(fmt, 0, 64, lpq.ROWWISE, lpq.SF_PLAIN)
    q.row.amax.fill_(3.5)
    lpq.quantize(x, fmt, lpq.ROWWISE | lpq.GIVEN_AMAX, out=q)
    torch.cuda.synchronize()
    ts = scalar(q.row.tensor_scale)
    a = np.float32(3.5)
    if fmt == lpq.NVFP4:
        want = np.float32(a / np.float32(2688.0))
    else:
        fmax = np.float32(448.0 if fmt == lpq.FP8_E4M3 else 57344.0)
        want = np.float32(np.float32(1.0) / np.float32(fmax / a))
    assert ts == want and scalar(q.row.amax) == 3.5
