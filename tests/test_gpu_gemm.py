"""GPU parity of the tensor-core GEMMs: every checked output element must satisfy
|C - C_ref| <= 1e-3 * sum_k |a b| against the oracle's FP64 GEMM of the
dequantized operands (plus half a bf16 ulp of C for bf16 output)."""
import numpy as np
import pytest
import torch

import oracle as o
from precision_transformer_gemms_gb300 import lpq
from lpq_testutil import bf16_input, gemm_gate, oracle_operand

pytestmark = pytest.mark.gpu

# (M, K, N): tiny, the MXFP8 tiny case, ragged M/N/K tails, several tiles in every dimension
SHAPES = [(4, 32, 16), (256, 512, 384), (300, 544, 200), (520, 1056, 776)]


def quantize_pair(fmt_a, fmt_b, M, K, N, seed=0):
    xa, _ = bf16_input((M, K), std=1.0, seed=seed, outlier_frac=0.001, outlier_scale=50)
    xb, _ = bf16_input((N, K), std=0.02, seed=seed + 1)
    if fmt_a == lpq.BF16:
        return lpq.Copy.of_bf16(xa), lpq.Copy.of_bf16(xb)
    qa = lpq.quantize(xa, fmt_a, lpq.ROWWISE)
    qb = lpq.quantize(xb, fmt_b, lpq.ROWWISE)
    return qa.row, qb.row


def check(a, b, M, N, K, out_fp32, layout=lpq.FPROP, path=None):
    c = lpq.gemm(layout, a, b, out_fp32=out_fp32, path=path)
    torch.cuda.synchronize()
    assert lpq.device_status() == 0
    ref, bound = o.gemm(oracle_operand(a), oracle_operand(b), M, N, K)
    nbad, worst = gemm_gate(c, ref, bound, not out_fp32)
    assert nbad == 0, f"{nbad} elements outside the gate (worst {worst:.3g}x)"


@pytest.mark.parametrize("path", ["single", "pair", "pair_whole", "pair_direct", "pair_cp", "single_cp",
                                  "single_bn128", "single_bn128_cp"])
@pytest.mark.parametrize("out_fp32", [True, False])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmts", [(lpq.BF16, lpq.BF16), (lpq.FP8_E4M3, lpq.FP8_E4M3), (lpq.FP8_E5M2, lpq.FP8_E4M3),
                                  (lpq.FP8_E4M3, lpq.FP8_E5M2), (lpq.FP8_E5M2, lpq.FP8_E5M2),
                                  (lpq.MXFP8, lpq.MXFP8), (lpq.MXFP8_E5M2, lpq.MXFP8), (lpq.MXFP8, lpq.MXFP8_E5M2),
                                  (lpq.MXFP8_E5M2, lpq.MXFP8_E5M2), (lpq.MXFP4, lpq.MXFP4),
                                  (lpq.NVFP4, lpq.NVFP4), (lpq.NVFP4, lpq.NVFP4_2D), (lpq.NVFP4_2D, lpq.NVFP4)])
def test_gemm_parity(fmts, shape, out_fp32, path):
    """Every kernel path: one CTA per 128 x 256 tile (block scales stored into
    TMEM by scale warps, or copied by the MMA thread: single_cp, pair_cp), one CTA per
    128 x 128 tile with two accumulators (block-scaled kinds: single_bn128), and
    CTA pairs (cta_group::2) per 256 x 256 tile, whose bf16 output leaves
    through TMA tile stores (pair) or direct stores (pair_direct).  These
    shapes have fewer tiles than half the CTA pairs, so pair and pair_direct
    run every tile as two 256 x 128 halves; pair_whole keeps whole tiles."""
    if path in ("single_cp", "pair_cp") and fmts[0] not in (lpq.NVFP4, lpq.MXFP4, lpq.MXFP8, lpq.MXFP8_E5M2):
        pytest.skip("scale-copy variant exists for the block-scaled kinds only")
    if path in ("single_bn128", "single_bn128_cp") and fmts[0] not in (lpq.NVFP4, lpq.MXFP8, lpq.MXFP8_E5M2,
                                                                      lpq.MXFP4):
        pytest.skip("128-wide tiles exist for the block-scaled kinds only")
    M, K, N = shape
    if fmts[1] == lpq.NVFP4_2D and N % 16:
        pytest.skip("2D weight tiles need N % 16 == 0")
    if fmts[0] == lpq.NVFP4_2D and M % 16:
        pytest.skip("2D tiles need M % 16 == 0")
    a, b = quantize_pair(*fmts, M, K, N)
    check(a, b, M, N, K, out_fp32, path=path)


BLOCK_SHAPES = [(4, 128, 16), (256, 512, 384), (300, 640, 200), (520, 1024, 776)]


@pytest.mark.parametrize("out_fp32", [True, False])
@pytest.mark.parametrize("shape", BLOCK_SHAPES)
@pytest.mark.parametrize("fmts", [(lpq.FP8_BLOCK_1x128, lpq.FP8_BLOCK_128x128),
                                  (lpq.FP8_BLOCK_1x128, lpq.FP8_BLOCK_1x128),
                                  (lpq.FP8_BLOCK_128x128, lpq.FP8_BLOCK_128x128),
                                  (lpq.FP8_BLOCK_128x128, lpq.FP8_BLOCK_1x128)])
def test_subchannel_gemm_parity(fmts, shape, out_fp32):
    """Sub-channel FP8: per 128-deep slice the tensor-core partial is scaled by
    the FP32 block factors and accumulated in FP32."""
    M, K, N = shape
    a, b = quantize_pair(*fmts, M, K, N, seed=7)
    check(a, b, M, N, K, out_fp32)


def test_gemm_closed_form_all_ones():
    """All-ones operands: every output is exactly K (MXFP8 scales are exact
    powers of two, so the products are exact)."""
    M, K, N = 256, 1024, 256
    x = torch.ones((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.ones((N, K), dtype=torch.bfloat16, device="cuda")
    for fmt in (lpq.MXFP8, lpq.MXFP8_E5M2, lpq.MXFP4, lpq.NVFP4, lpq.BF16):
        if fmt == lpq.BF16:
            a, b = lpq.Copy.of_bf16(x), lpq.Copy.of_bf16(y)
        else:
            a, b = lpq.quantize(x, fmt, lpq.ROWWISE).row, lpq.quantize(y, fmt, lpq.ROWWISE).row
        c = lpq.gemm(lpq.FPROP, a, b, out_fp32=True)
        torch.cuda.synchronize()
        ref, _ = o.gemm(oracle_operand(a), oracle_operand(b), 1, 1, K, pairs=np.array([[0, 0]]))
        assert float(ref[0]) == pytest.approx(K, rel=1e-6)
        if fmt != lpq.NVFP4:
            assert float(ref[0]) == K  # power-of-two scales: exact
        if fmt == lpq.NVFP4:  # the FP32 tensor scales 1/2688 are rounded: K up to a few ulps
            assert torch.allclose(c, torch.full_like(c, float(ref[0])), rtol=1e-6, atol=0), fmt
        else:
            assert torch.all(c == float(ref[0])), (fmt, float(ref[0]), c.flatten()[:4])


def test_gemm_single_nonzero_k():
    M, K, N = 128, 256, 256
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    x[:, 77] = 3.0
    y[:, 77] = -2.0
    for fmt in (lpq.MXFP8, lpq.MXFP8_E5M2, lpq.MXFP4, lpq.FP8_E4M3, lpq.NVFP4, lpq.BF16):
        if fmt == lpq.BF16:
            a, b = lpq.Copy.of_bf16(x), lpq.Copy.of_bf16(y)
        else:
            a, b = lpq.quantize(x, fmt, lpq.ROWWISE).row, lpq.quantize(y, fmt, lpq.ROWWISE).row
        c = lpq.gemm(lpq.FPROP, a, b, out_fp32=True)
        torch.cuda.synchronize()
        ref, _ = o.gemm(oracle_operand(a), oracle_operand(b), 1, 1, K, pairs=np.array([[0, 0]]))
        assert torch.allclose(c, torch.full_like(c, float(ref[0])), rtol=1e-6), fmt


@pytest.mark.parametrize("fmt", [lpq.MXFP8, lpq.MXFP8_E5M2, lpq.MXFP4, lpq.NVFP4, lpq.FP8_E4M3, lpq.BF16,
                                 lpq.FP8_BLOCK_1x128])
def test_fprop_dgrad_wgrad_layouts(fmt):
    """The three GEMMs of a linear layer on the copies each one reads."""
    M, K, N = 256, 512, 384
    X, _ = bf16_input((M, K), std=1.0, seed=20)
    W, _ = bf16_input((N, K), std=0.02, seed=21)
    dY, _ = bf16_input((M, N), std=1e-3, seed=22)
    both = lpq.ROWWISE | lpq.COLWISE
    if fmt == lpq.BF16:
        qx, qw, qd = (lpq.quantize(t, fmt, both) for t in (X, W, dY))
    elif fmt == lpq.NVFP4:
        qx = lpq.quantize(X, fmt, both | lpq.RHT_COLWISE, rht_seed=9)
        qw = lpq.quantize(W, lpq.NVFP4_2D, both)
        qd = lpq.quantize(dY, fmt, both | lpq.RHT_COLWISE | lpq.STOCHASTIC, seed=3, rht_seed=9)
    elif fmt == lpq.FP8_BLOCK_1x128:
        qx = lpq.quantize(X, fmt, both)
        qw = lpq.quantize(W, lpq.FP8_BLOCK_128x128, both)
        qd = lpq.quantize(dY, fmt, both)
    elif fmt == lpq.FP8_E4M3:
        qx = lpq.quantize(X, fmt, both)
        qw = lpq.quantize(W, fmt, both)
        qd = lpq.quantize(dY, lpq.FP8_E5M2, both)
    elif fmt == lpq.MXFP8_E5M2:  # MXFP8 with E5M2 gradients: dY in E5M2, X and W in E4M3
        qx = lpq.quantize(X, lpq.MXFP8, both)
        qw = lpq.quantize(W, lpq.MXFP8, both)
        qd = lpq.quantize(dY, fmt, both)
    else:
        qx, qw, qd = (lpq.quantize(t, fmt, both) for t in (X, W, dY))
    check(qx.row, qw.row, M, N, K, True, lpq.FPROP)      # Y  [M, N]
    check(qd.row, qw.col, M, K, N, True, lpq.DGRAD)      # dX [M, K]
    check(qd.col, qx.col, N, K, M, True, lpq.WGRAD)      # dW [N, K]


@pytest.mark.parametrize("fmt", [lpq.NVFP4, lpq.MXFP8, lpq.MXFP4, lpq.FP8_E4M3, lpq.BF16])
def test_full_size_sampled(fmt):
    """QKV Fprop at the layer's size (15872 x 4096 x 12288): the first and last
    128 x 128 output tiles and 4096 uniformly sampled elements."""
    M, K, N = 15872, 4096, 12288
    X, _ = bf16_input((M, K), std=1.0, seed=30)
    W, _ = bf16_input((N, K), std=0.02, seed=31)
    if fmt == lpq.BF16:
        qx, qw = lpq.QTensor(lpq.Copy.of_bf16(X)), lpq.QTensor(lpq.Copy.of_bf16(W))
    else:
        qx = lpq.quantize(X, fmt, lpq.ROWWISE)
        qw = lpq.quantize(W, lpq.NVFP4_2D if fmt == lpq.NVFP4 else fmt, lpq.ROWWISE)
    c = lpq.gemm(lpq.FPROP, qx.row, qw.row)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    first = np.array([(m, n) for m in range(128) for n in range(128)])
    last = np.array([(M - 128 + m, N - 128 + n) for m in range(128) for n in range(128)])
    rand = np.stack([rng.integers(0, M, 4096), rng.integers(0, N, 4096)], 1)
    pairs = np.concatenate([first, last, rand]).astype(np.int64)
    ref, bound = o.gemm(oracle_operand(qx.row), oracle_operand(qw.row), M, N, K, pairs)
    got = c[torch.from_numpy(pairs[:, 0]).cuda(), torch.from_numpy(pairs[:, 1]).cuda()]
    nbad, worst = gemm_gate(got, ref, bound, True)
    assert nbad == 0, f"{nbad} bad (worst {worst:.3g}x)"


def test_empty_and_zero_k():
    a = lpq.Copy(lpq.MXFP8, 0, 128, False)
    b = lpq.Copy(lpq.MXFP8, 64, 128, False)
    c = lpq.gemm(lpq.FPROP, a, b)
    assert c.shape == (0, 64)
    x = torch.empty((64, 0), dtype=torch.bfloat16, device="cuda")
    c = lpq.gemm(lpq.FPROP, lpq.Copy.of_bf16(x), lpq.Copy.of_bf16(torch.empty((32, 0), dtype=torch.bfloat16,
                                                                               device="cuda")), out_fp32=True)
    torch.cuda.synchronize()
    assert torch.all(c == 0)


def test_no_fallback_on_mixed_formats():
    x, _ = bf16_input((128, 128), seed=40)
    a = lpq.quantize(x, lpq.MXFP8, lpq.ROWWISE).row
    b = lpq.quantize(x, lpq.NVFP4, lpq.ROWWISE).row
    with pytest.raises(lpq.LpqError) as e:
        lpq.gemm(lpq.FPROP, a, b)
    assert e.value.status == lpq.ERR_UNSUPPORTED
    # MXFP4 pairs with MXFP4 only (not with NVFP4, nor with MXFP8)
    c = lpq.quantize(x, lpq.MXFP4, lpq.ROWWISE).row
    for a2, b2 in ((c, b), (b, c), (c, a)):
        with pytest.raises(lpq.LpqError) as e:
            lpq.gemm(lpq.FPROP, a2, b2)
        assert e.value.status == lpq.ERR_UNSUPPORTED


def test_bounded_wait_reports_timeout_and_context_survives():
    assert lpq.device_status() == 0
    lpq.selftest_wait(20_000_000)  # 20 ms
    assert lpq.device_status() == lpq.ERR_TIMEOUT
    assert lpq.device_status() == 0  # read clears it
    x, bits = bf16_input((64, 128), seed=41)
    q = lpq.quantize(x, lpq.MXFP8, lpq.ROWWISE)
    assert np.array_equal(q.row.codes_matrix().cpu().numpy(), o.mxfp8(bits, colwise=False)["row"])


@pytest.mark.parametrize("kind,mode", [("bf16", 0), ("fp8", 0), ("mxfp8", 0), ("mxfp8", 1), ("nvfp4", 0), ("nvfp4", 1),
                                       ("nvfp4", 2), ("nvfp4", 3), ("nvfp4", 4), ("nvfp4", 5),
                                       ("bf16", 6), ("fp8", 6), ("mxfp8", 6), ("nvfp4", 6), ("mxfp8", 7),
                                       ("nvfp4", 7), ("bf16", 8), ("fp8", 8), ("mxfp8", 8), ("nvfp4", 8)])
def test_mma_peak_modes_run(kind, mode):
    """Every rate-probe mode runs to completion with a clean device status and
    a rate below the nominal dense peak of its kind (x1.2 for clock slack)."""
    rate = lpq.mma_peak(kind, iters=256, with_scale_copies=mode)
    torch.cuda.synchronize()
    assert lpq.device_status() == 0
    nominal = {"bf16": 2250, "fp8": 4500, "mxfp8": 4500, "nvfp4": 13500}[kind]
    assert 0 < rate < 1.2 * nominal


@pytest.mark.parametrize("fmts", [(lpq.BF16, lpq.BF16), (lpq.FP8_E4M3, lpq.FP8_E4M3), (lpq.MXFP8, lpq.MXFP8),
                                  (lpq.MXFP4, lpq.MXFP4)])
def test_pair_gemm_ragged_n_direct_stores(fmts):
    """N not a multiple of 8: no tensor map fits the output rows, so the pair
    kernel's epilogue stores directly (bf16 and FP32 outputs)."""
    M, K, N = 512, 256, 100
    a, b = quantize_pair(*fmts, M, K, N, seed=11)
    for out_fp32 in (False, True):
        check(a, b, M, N, K, out_fp32, path="pair")


@pytest.mark.parametrize("fmts", [(lpq.BF16, lpq.BF16), (lpq.FP8_E4M3, lpq.FP8_E4M3), (lpq.MXFP8, lpq.MXFP8),
                                  (lpq.MXFP4, lpq.MXFP4), (lpq.NVFP4, lpq.NVFP4_2D)])
def test_pair_gemm_whole_and_half_tiles_mixed(fmts):
    """Two tiles more than there are CTA pairs (M = 512: two tile rows): the
    pair kernel runs one round of whole 256 x 256 tiles and splits the two
    tiles of the last round (the last tile column) into four 256 x 128 halves
    (N = 128 MMAs on 64 B rows per CTA, with the half's one group of B scale
    atoms); whole_tiles = 1 runs them as whole tiles.  Every output of the last
    tile column and 4096 others (seed 0) against the oracle, bf16 and FP32
    outputs, both paths."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    M, K, N = 512, 256, (pairs + 2) // 2 * 256 + (128 if pairs % 2 else 0)
    a, b = quantize_pair(*fmts, M, K, N, seed=5)
    n0 = (N - 1) // 256 * 256
    rng = np.random.default_rng(0)
    last = np.array([(m, n) for m in range(M) for n in range(n0, N)])
    rand = np.stack([rng.integers(0, M, 4096), rng.integers(0, N, 4096)], 1)
    pairs_mn = np.concatenate([last, rand]).astype(np.int64)
    ref, bound = o.gemm(oracle_operand(a), oracle_operand(b), M, N, K, pairs_mn)
    rows, cols = torch.from_numpy(pairs_mn[:, 0]).cuda(), torch.from_numpy(pairs_mn[:, 1]).cuda()
    for out_fp32 in (False, True):
        for path in ("pair", "pair_whole") + (("pair_cp",) if fmts[0] in (lpq.MXFP8, lpq.MXFP4, lpq.NVFP4) else ()):
            c = lpq.gemm(lpq.FPROP, a, b, out_fp32=out_fp32, path=path)
            torch.cuda.synchronize()
            assert lpq.device_status() == 0
            nbad, worst = gemm_gate(c[rows, cols], ref, bound, not out_fp32)
            assert nbad == 0, f"{path} fp32={out_fp32}: {nbad} outside the gate (worst {worst:.3g}x)"
