"""Every GEMM of the CodonFM-5B layer (M = 31 x 512, hidden 4096, intermediate
16384) at full size, with the operand copies, scale layouts and kernel paths the
benchmark uses: the first and last 128 x 128 output tiles and 4096 uniformly
sampled elements (seed 0) of each GEMM against the oracle's FP64 GEMM of the
dequantized operands, |C - C_ref| <= 1e-3 sum_k |a b| (+ half a bf16 ulp of C).

NVFP4 follows the layer recipe: 1D 16-value blocks for X and dY, 16x16 tiles for
W, the random Hadamard transform on the Wgrad operands (the column-wise copies
of X and dY) and stochastic rounding of dY; MXFP8 quantizes every tensor with
E4M3 codes and E8M0 scales per 32 values (the E5M2 variant gives dY E5M2
codes); MXFP4 every tensor with packed E2M1 codes and E8M0 scales per 32."""
import numpy as np
import pytest
import torch

import oracle as o
from precision_transformer_gemms_gb300 import lpq
from lpq_testutil import bf16_input, gemm_gate, oracle_operand

pytestmark = pytest.mark.gpu


def layer_shapes():
    return lpq.layer_shapes(4096, 16384, 31, 512)


def linear_dims(layout, m, k, n):
    """(tokens, K_lin, N_lin) of the linear a GEMM belongs to."""
    if layout == lpq.FPROP:
        return m, k, n
    if layout == lpq.DGRAD:
        return m, n, k
    return k, n, m  # Wgrad: (N_lin, M, K_lin)


def quantize_copy(t, recipe, role, colwise, seed):
    """The copy of tensor t (role X, W or dY) one GEMM reads, as the layer quantizes it."""
    flags = lpq.COLWISE if colwise else lpq.ROWWISE
    if recipe == "mxfp8":
        q = lpq.quantize(t, lpq.MXFP8, flags)
    elif recipe == "mxfp8_e5m2":  # E5M2 codes for the gradients, E4M3 for X and W
        q = lpq.quantize(t, lpq.MXFP8_E5M2 if role == "dY" else lpq.MXFP8, flags)
    elif recipe == "mxfp4":
        q = lpq.quantize(t, lpq.MXFP4, flags)
    elif role == "W":
        q = lpq.quantize(t, lpq.NVFP4_2D, flags)
    else:
        if colwise:
            flags |= lpq.RHT_COLWISE
        if role == "dY":
            flags |= lpq.STOCHASTIC
        q = lpq.quantize(t, lpq.NVFP4, flags, seed=seed, rht_seed=1234)
    return q.col if colwise else q.row


@pytest.mark.parametrize("recipe", ["nvfp4", "mxfp8", "mxfp8_e5m2", "mxfp4"])
@pytest.mark.parametrize("index", range(12))
def test_layer_gemm_sampled(recipe, index):
    name, layout, M, K, N = layer_shapes()[index]
    tokens, k_lin, n_lin = linear_dims(layout, M, K, N)
    lin = index // 3
    # operands of the pass: (role, column-wise) for a and b
    roles = {lpq.FPROP: (("X", False), ("W", False)), lpq.DGRAD: (("dY", False), ("W", True)),
             lpq.WGRAD: (("dY", True), ("X", True))}[layout]
    shapes = {"X": (tokens, k_lin), "W": (n_lin, k_lin), "dY": (tokens, n_lin)}
    stds = {"X": 1.0, "W": 0.02, "dY": 1e-3}
    seeds = {"X": 100 * lin, "W": 100 * lin + 1, "dY": 100 * lin + 2}
    copies = []
    for role, col in roles:
        t, _ = bf16_input(shapes[role], std=stds[role], seed=seeds[role])
        copies.append(quantize_copy(t, recipe, role, col, seed=7 + index))
        del t
    a, b = copies
    assert (a.rows, a.cols, b.rows, b.cols) == (M, K, N, K), name
    c = lpq.gemm(layout, a, b)
    torch.cuda.synchronize()
    assert lpq.device_status() == 0
    rng = np.random.default_rng(0)
    first = np.array([(m, n) for m in range(128) for n in range(128)])
    last = np.array([(M - 128 + m, N - 128 + n) for m in range(128) for n in range(128)])
    rand = np.stack([rng.integers(0, M, 4096), rng.integers(0, N, 4096)], 1)
    pairs = np.concatenate([first, last, rand]).astype(np.int64)
    ref, bound = o.gemm(oracle_operand(a), oracle_operand(b), M, N, K, pairs)
    got = c[torch.from_numpy(pairs[:, 0]).cuda(), torch.from_numpy(pairs[:, 1]).cuda()]
    nbad, worst = gemm_gate(got, ref, bound, True)
    assert nbad == 0, f"{name}: {nbad} sampled outputs outside the gate (worst {worst:.3g}x)"
