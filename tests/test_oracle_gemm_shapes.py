"""Pins of the oracle's FP64 GEMM and of the layer's 12 GEMM shapes (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle as o
from precision_transformer_gemms_gb300 import synth

LAYER = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "codonfm5b_layer.json")))


def rand_bits(shape, std=1.0, seed=0):
    return synth.host_bits(synth.bf16_normal(shape, std, seed, "cpu"))


def naive(a, b, M, N, K):
    """Brute-force triple loop over dequantized values (independent of the
    oracle's GEMM loop; dequantization is checked separately)."""
    A = o.dequant(a, K, 0, M)
    B = o.dequant(b, K, 0, N)
    C = [[0.0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(A[m, k]) * float(B[n, k])
            C[m][n] = s
    return np.array(C), A, B


def test_brute_force_4x32x16_mxfp8_and_nvfp4():
    M, K, N = 4, 32, 16
    xa, xb = rand_bits((M, K), seed=1), rand_bits((N, K), std=0.02, seed=2)
    for make in ("mx", "nv"):
        if make == "mx":
            ra, rb = o.mxfp8(xa, colwise=False), o.mxfp8(xb, colwise=False)
            a = o.Operand(o.K_MXFP8, ra["row"], ra["row_sf"])
            b = o.Operand(o.K_MXFP8, rb["row"], rb["row_sf"])
        else:
            ra, rb = o.nvfp4(xa, o.NV_ROW), o.nvfp4(xb, o.NV_ROW)
            a = o.Operand(o.K_NVFP4, ra["row"], ra["row_sf"], ra["row_ts"])
            b = o.Operand(o.K_NVFP4, rb["row"], rb["row_sf"], rb["row_ts"])
        C, Bd = o.gemm(a, b, M, N, K)
        ref, A, B = naive(a, b, M, N, K)
        assert np.allclose(C, ref, rtol=1e-14, atol=0)
        assert np.allclose(C, A @ B.T, rtol=1e-12, atol=0)
        assert np.allclose(Bd, np.abs(A) @ np.abs(B).T, rtol=1e-12)
        # quantized GEMM is close to the bf16 GEMM (information, loose)
        xf = o.bf16_to_f32(xa).astype(np.float64) @ o.bf16_to_f32(xb).astype(np.float64).T
        assert np.all(np.abs(C - xf) <= 0.35 * Bd)


def test_dequant_matches_format_definitions():
    x = rand_bits((4, 64), seed=3)
    r = o.mxfp8(x, colwise=False)
    d = o.dequant(o.Operand(o.K_MXFP8, r["row"], r["row_sf"]), 64, 0, 4)
    want = o.decode(o.E4M3, r["row"]) * np.repeat(2.0 ** (r["row_sf"].astype(int) - 127), 32, axis=1)
    assert np.array_equal(d, want)
    n = o.nvfp4(x, o.NV_ROW)
    d = o.dequant(o.Operand(o.K_NVFP4, n["row"], n["row_sf"], n["row_ts"]), 64, 0, 4)
    q = np.stack([n["row"] & 15, n["row"] >> 4], -1).reshape(4, 64)
    want = o.decode(o.E2M1, q) * np.repeat(o.decode(o.E4M3, n["row_sf"]), 16, axis=1) * n["row_ts"]
    assert np.array_equal(d, want)


def test_all_ones_closed_form_and_single_nonzero_k():
    M, N, K = 3, 5, 64
    ones = np.full((M, K), 0x3F80, np.uint16)  # bf16 1.0
    onesb = np.full((N, K), 0x3F80, np.uint16)
    ra, rb = o.fp8_pertensor(ones, o.E4M3, rowwise=True, colwise=False), \
        o.fp8_pertensor(onesb, o.E4M3, rowwise=True, colwise=False)
    a = o.Operand(o.K_FP8_E4M3, ra["row"], ts=ra["scale_inv"])
    b = o.Operand(o.K_FP8_E4M3, rb["row"], ts=rb["scale_inv"])
    C, Bd = o.gemm(a, b, M, N, K)
    closed = K * (448.0 * ra["scale_inv"]) * (448.0 * rb["scale_inv"])
    assert np.allclose(C, closed, rtol=1e-14, atol=0) and np.array_equal(C, Bd)
    assert abs(closed - K) < 1e-4 * K  # each operand dequantizes to 1 up to the fp32 scale
    # single nonzero k: C is that single product exactly
    xa = np.zeros((M, K), np.uint16)
    xa[:, 7] = 0x4040  # 3.0
    xb = np.zeros((N, K), np.uint16)
    xb[:, 7] = 0xC000  # -2.0
    A = o.Operand(o.K_BF16, xa)
    B = o.Operand(o.K_BF16, xb)
    C, Bd = o.gemm(A, B, M, N, K)
    assert np.all(C == -6.0) and np.all(Bd == 6.0)


def test_block_fp8_gemm_equals_blockwise_promotion():
    """Sub-channel: C = sum_kb sa[m,kb] sb[nb,kb] sum_{k in kb} qa qb."""
    M, N, K = 4, 128, 256
    xa, xb = rand_bits((M, K), seed=4), rand_bits((N, K), seed=5)
    ra, rb = o.fp8_block(xa, 1, colwise=False), o.fp8_block(xb, 128, colwise=False)
    a = o.Operand(o.K_FP8_BLOCK, ra["row"], ra["row_sinv"], block_rows=1)
    b = o.Operand(o.K_FP8_BLOCK, rb["row"], rb["row_sinv"], block_rows=128)
    C, _ = o.gemm(a, b, M, N, K)
    qa, qb = o.decode(o.E4M3, ra["row"]), o.decode(o.E4M3, rb["row"])
    ref = np.zeros((M, N))
    for kb in range(K // 128):
        part = qa[:, kb * 128:(kb + 1) * 128] @ qb[:, kb * 128:(kb + 1) * 128].T
        ref += part * ra["row_sinv"][:, kb][:, None].astype(np.float64) * rb["row_sinv"][0, kb]
    assert np.allclose(C, ref, rtol=1e-12)


def test_sampled_pairs_equal_dense():
    M, N, K = 8, 8, 64
    xa, xb = rand_bits((M, K), seed=6), rand_bits((N, K), seed=7)
    a, b = o.Operand(o.K_BF16, xa), o.Operand(o.K_BF16, xb)
    C, Bd = o.gemm(a, b, M, N, K)
    pairs = np.array([[0, 0], [7, 3], [2, 6]], np.int64)
    c, bd = o.gemm(a, b, M, N, K, pairs)
    assert np.array_equal(c, C[pairs[:, 0], pairs[:, 1]]) and np.array_equal(bd, Bd[pairs[:, 0], pairs[:, 1]])


# ------------------------------------------------------------------ shapes
def test_layer_shapes_match_the_pages():
    cfg = LAYER["config"]
    shapes = o.layer_shapes(cfg["hidden_size"], cfg["intermediate_size"], cfg["micro_batch_size"],
                            cfg["sequence_length"])
    M = LAYER["tokens_M"]
    assert cfg["micro_batch_size"] * cfg["sequence_length"] == M
    d = {n: (m, k, nn) for n, m, k, nn in shapes}
    assert d["qkv_fprop"] == (M, LAYER["qkv_fprop_K"], LAYER["qkv_fprop_N"])
    assert d["qkv_dgrad"] == (M, LAYER["qkv_fprop_N"], LAYER["qkv_fprop_K"])  # K and N swap
    assert d["attn_out_fprop"][1:] == tuple(LAYER["attn_out_weight"])
    for lin in ("qkv", "attn_out", "mlp_up", "mlp_down"):
        m, k, n = d[f"{lin}_fprop"]
        assert d[f"{lin}_dgrad"] == (m, n, k) and d[f"{lin}_wgrad"] == (n, m, k)
    flops = sum(2 * m * k * n for _, m, k, n in shapes)
    assert round(flops / 1e12, 3) == 19.173


def test_pages_fprop_ratios_are_consistent():
    """The per-shape NVFP4/MXFP8 ratios printed on the page are the quotients
    of the printed times, and the sums give the blended 1.47x."""
    t = LAYER["fprop_ms_b300"]
    for v in t.values():
        assert round(v["mxfp8"] / v["nvfp4"], 2) == v["ratio"]
    blended = sum(v["mxfp8"] for v in t.values()) / sum(v["nvfp4"] for v in t.values())
    assert round(blended, 2) == LAYER["blended_fprop_ratio"]
