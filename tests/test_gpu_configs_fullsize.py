"""Full-size GEMM gates of the two workloads the layer tests do not cover,
with the operand copies and kernel paths their benchmarks use; the first and
last 128 x 128 output tiles and 4096 uniformly sampled elements (seed 0) of
each GEMM against the oracle's FP64 GEMM of the dequantized operands,
|C - C_ref| <= 1e-3 sum_k |a b| (+ half a bf16 ulp of C).

* Per-tensor FP8 drift ("Faster training throughput in FP8 with NVIDIA NeMo",
  per-tensor current and delayed scaling; "Optimizing Transformer models for
  low-precision training", E4M3 forward / E5M2 gradients): the attention-out
  GEMMs (M = 15872, 4096 x 4096) with X's std drifting 1 -> 4 over 20 steps,
  the Fprop, Dgrad and Wgrad of the first and the last step, under current and
  under delayed scaling (history 16; the state advanced through all 20 steps).
* The scaling-granularity K-sweep at its largest K ("Faster training
  throughput in FP8 with NVIDIA NeMo", scaling up recipe granularity):
  8192 x 16384 x 8192 with sub-channel FP8 (1x128 activations, 128x128
  weights), per-tensor FP8, MXFP8, NVFP4 (1D activations, 2D weights) and
  MXFP4, inputs ~N(0,1) with 0.1% entries x100."""
import numpy as np
import pytest
import torch

import oracle as o
from precision_transformer_gemms_gb300 import lpq, synth
from lpq_testutil import gemm_gate, oracle_operand

pytestmark = pytest.mark.gpu

BOTH = lpq.ROWWISE | lpq.COLWISE


def sampled_gate(c, a, b, M, N, K, label):
    rng = np.random.default_rng(0)
    first = np.array([(m, n) for m in range(128) for n in range(128)])
    last = np.array([(M - 128 + m, N - 128 + n) for m in range(128) for n in range(128)])
    rand = np.stack([rng.integers(0, M, 4096), rng.integers(0, N, 4096)], 1)
    pairs = np.concatenate([first, last, rand]).astype(np.int64)
    ref, bound = o.gemm(oracle_operand(a), oracle_operand(b), M, N, K, pairs)
    got = c[torch.from_numpy(pairs[:, 0]).cuda(), torch.from_numpy(pairs[:, 1]).cuda()]
    nbad, worst = gemm_gate(got, ref, bound, True)
    assert nbad == 0, f"{label}: {nbad} sampled outputs outside the gate (worst {worst:.3g}x)"


@pytest.mark.parametrize("scaling", [lpq.SCALING_CURRENT, lpq.SCALING_DELAYED])
def test_fp8_drift_attention_out_gemms_first_and_last_step(scaling):
    M = 15872
    K = N = 4096
    delayed = scaling == lpq.SCALING_DELAYED
    W = synth.bf16_normal((N, K), synth.WEIGHT_STD, 1, "cuda")
    st = {r: lpq.DelayedState(16) for r in ("X", "W", "dY")}
    q = {"X": lpq.alloc(lpq.FP8_E4M3, M, K, BOTH), "W": lpq.alloc(lpq.FP8_E4M3, N, K, BOTH),
         "dY": lpq.alloc(lpq.FP8_E5M2, M, N, BOTH)}
    for t in range(20):
        X = synth.bf16_normal((M, K), synth.drift_std(t), 10 * t, "cuda")
        dY = synth.bf16_normal((M, N), synth.GRAD_STD, 10 * t + 2, "cuda")
        for role, x, fmt in (("X", X, lpq.FP8_E4M3), ("W", W, lpq.FP8_E4M3), ("dY", dY, lpq.FP8_E5M2)):
            lpq.quantize(x, fmt, BOTH, scaling=scaling, state=st[role] if delayed else None, out=q[role])
            if delayed:
                lpq.scale_update(st[role], q[role].row.amax, lpq.FMAX[fmt])
        if t not in (0, 19):
            continue
        for layout, a, b, m, n, k, name in ((lpq.FPROP, q["X"].row, q["W"].row, M, N, K, "fprop"),
                                            (lpq.DGRAD, q["dY"].row, q["W"].col, M, K, N, "dgrad"),
                                            (lpq.WGRAD, q["dY"].col, q["X"].col, N, K, M, "wgrad")):
            c = lpq.gemm(layout, a, b)
            torch.cuda.synchronize()
            assert lpq.device_status() == 0
            sampled_gate(c, a, b, m, n, k, f"step {t} {name}")
            del c


@pytest.mark.parametrize("recipe", ["fp8_subchannel", "fp8_current", "mxfp8", "nvfp4", "mxfp4"])
def test_ksweep_largest_k(recipe):
    M = N = 8192
    K = 16384
    fa, fb = {"fp8_subchannel": (lpq.FP8_BLOCK_1x128, lpq.FP8_BLOCK_128x128),
              "fp8_current": (lpq.FP8_E4M3, lpq.FP8_E4M3), "mxfp8": (lpq.MXFP8, lpq.MXFP8),
              "nvfp4": (lpq.NVFP4, lpq.NVFP4_2D), "mxfp4": (lpq.MXFP4, lpq.MXFP4)}[recipe]
    A = synth.bf16_normal((M, K), 1.0, 50, "cuda", 0.001, 100.0)
    B = synth.bf16_normal((N, K), 1.0, 51, "cuda", 0.001, 100.0)
    qa = lpq.quantize(A, fa, lpq.ROWWISE)
    qb = lpq.quantize(B, fb, lpq.ROWWISE)
    del A, B
    c = lpq.gemm(lpq.FPROP, qa.row, qb.row)
    torch.cuda.synchronize()
    assert lpq.device_status() == 0
    sampled_gate(c, qa.row, qb.row, M, N, K, recipe)
