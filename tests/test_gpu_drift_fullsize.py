"""Per-tensor FP8 over 20 steps at the attention-output size (X [15872, 4096]
whose std drifts 1 -> 4, W [4096, 4096], dY [15872, 4096]), current and
delayed scaling (history 16), as the drift workload runs them: every step's
X codes (both copies), the amax and the tensor scale, and the delayed state
after each update, equal the oracle's; dY's codes are compared on the first
and the last step."""
import numpy as np
import pytest
import torch

import oracle as o
from precision_transformer_gemms_gb300 import lpq, synth

pytestmark = pytest.mark.gpu

M, K = 15872, 4096
BOTH = lpq.ROWWISE | lpq.COLWISE


@pytest.mark.parametrize("scaling", [lpq.SCALING_CURRENT, lpq.SCALING_DELAYED])
def test_fp8_drift_20_steps_full_size(scaling):
    delayed = scaling == lpq.SCALING_DELAYED
    st_x, st_dy = lpq.DelayedState(16), lpq.DelayedState(16)
    ref_x, ref_dy = o.DelayedState(16), o.DelayedState(16)
    qx = lpq.alloc(lpq.FP8_E4M3, M, K, BOTH)
    qd = lpq.alloc(lpq.FP8_E5M2, M, K, BOTH)
    for t in range(20):
        X = synth.bf16_normal((M, K), synth.drift_std(t), 10 * t, "cuda")
        dY = synth.bf16_normal((M, K), synth.GRAD_STD, 10 * t + 2, "cuda")
        lpq.quantize(X, lpq.FP8_E4M3, BOTH, scaling=scaling, state=st_x if delayed else None, out=qx)
        lpq.quantize(dY, lpq.FP8_E5M2, BOTH, scaling=scaling, state=st_dy if delayed else None, out=qd)
        if delayed:
            lpq.scale_update(st_x, qx.row.amax, 448.0)
            lpq.scale_update(st_dy, qd.row.amax, 57344.0)
        torch.cuda.synchronize()
        rx = o.fp8_pertensor(synth.host_bits(X), o.E4M3, scale=float(ref_x.scale[0]) if delayed else None)
        assert np.array_equal(qx.row.codes_matrix().cpu().numpy(), rx["row"]), t
        assert np.array_equal(qx.col.codes_matrix().cpu().numpy(), rx["col"]), t
        assert float(qx.row.amax.item()) == rx["amax"], t
        assert float(qx.row.tensor_scale.item()) == np.float32(rx["scale_inv"]), t
        if t in (0, 19) or delayed:
            rd = o.fp8_pertensor(synth.host_bits(dY), o.E5M2, scale=float(ref_dy.scale[0]) if delayed else None)
            if t in (0, 19):
                assert np.array_equal(qd.row.codes_matrix().cpu().numpy(), rd["row"]), t
                assert np.array_equal(qd.col.codes_matrix().cpu().numpy(), rd["col"]), t
        if delayed:
            ref_x.update(rx["amax"], 448.0)
            ref_dy.update(rd["amax"], 57344.0)
            assert np.array_equal(st_x.hist.cpu().numpy(), ref_x.hist), t
            assert float(st_x.scale.item()) == ref_x.scale[0] and float(st_dy.scale.item()) == ref_dy.scale[0], t
        del X, dY
