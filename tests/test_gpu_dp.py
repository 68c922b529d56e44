"""Token-sharded data parallelism (precision_transformer_gemms_gb300.dp) on the
GPU: two ranks, each a process with its own token shard, exchange through a
real torch.distributed process group (gloo, which stages the two all-reduces
through host memory, so no kernel ever waits on another rank).  The shards'
codes and scales must be bit-identical to the unsharded quantization (the
global amax reached every rank), and the all-reduced Wgrad must meet the GEMM
gate against the oracle's FP64 sum of the shards' Wgrad partials; Fprop and
Dgrad rows against the oracle on sampled outputs."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle as o
from precision_transformer_gemms_gb300 import dp, lpq, synth
from lpq_testutil import codes, gemm_gate, oracle_operand, plain_scales, scalar

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, K, N = 512, 256, 384  # tokens (two shards of 256), in features, out features


def _inputs(device):
    X = synth.bf16_normal((M, K), 1.0, 3, device, 0.001, 40.0)
    W = synth.bf16_normal((N, K), 0.02, 4, device)
    dY = synth.bf16_normal((M, N), 1e-3, 5, device)
    return X, W, dY


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_worker(rank, world, port, recipe, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, W, dY = _inputs("cuda")
        r0, r1 = dp.shard_rows(M, world, rank)
        lin = dp.TokenShardedLinear(recipe, X[r0:r1].contiguous(), W, dY[r0:r1].contiguous(), first_row=r0)
        for s in range(2):  # two steps: the second re-runs every exchange on reused buffers
            Y, dX, dW = lin.step(seed=11)
        torch.cuda.synchronize()
        status = lpq.device_status()
        out = {"status": status, "r0": r0, "r1": r1, "Y": Y.float().cpu().numpy(), "dX": dX.float().cpu().numpy(),
               "dW": dW.cpu().numpy()}
        if recipe != "bf16":
            for role in ("X", "W", "dY"):
                for c in ("row", "col"):
                    cp = getattr(lin.q[role], c)
                    out[f"{role}_{c}"] = codes(cp)
                    out[f"{role}_{c}_sf"] = plain_scales(cp)
                    out[f"{role}_{c}_ts"] = scalar(cp.tensor_scale) if cp.tensor_scale is not None else None
                    out[f"{role}_{c}_op"] = oracle_operand(cp)
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def _run(recipe, world=2):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_worker, args=(r, world, port, recipe, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs)
    return res


@pytest.mark.parametrize("recipe", ["nvfp4", "fp8_current"])
def test_two_rank_exchange_matches_unsharded(recipe):
    res = _run(recipe)
    assert all(r["status"] == 0 for r in res.values())
    X, W, dY = _inputs("cuda")
    both = lpq.ROWWISE | lpq.COLWISE
    fx, ex, _ = dp.quant_config(recipe, "X")
    fd, ed, _ = dp.quant_config(recipe, "dY")
    whole_x = lpq.quantize(X, fx, both | ex, seed=11, rht_seed=1234, sf_layout=lpq.SF_PLAIN)
    whole_d = lpq.quantize(dY, fd, both | ed, seed=11, rht_seed=1234, sf_layout=lpq.SF_PLAIN)
    per = 2 if fx == lpq.NVFP4 else 1
    for rank, r in res.items():
        r0, r1 = r["r0"], r["r1"]
        # the global amax reached both ranks: shard codes are the unsharded tensor's rows
        assert np.array_equal(r["X_row"], codes(whole_x.row)[r0:r1])
        assert np.array_equal(r["X_col"], codes(whole_x.col)[:, r0 // per:r1 // per])
        assert np.array_equal(r["dY_row"], codes(whole_d.row)[r0:r1])  # SR counters continue the global order
        assert r["X_row_ts"] == scalar(whole_x.row.tensor_scale) and r["X_col_ts"] == scalar(whole_x.col.tensor_scale)
        assert r["dY_row_ts"] == scalar(whole_d.row.tensor_scale) and r["dY_col_ts"] == scalar(whole_d.col.tensor_scale)
        if fx == lpq.NVFP4:
            assert np.array_equal(r["X_row_sf"], plain_scales(whole_x.row)[r0:r1])
            assert np.array_equal(r["X_col_sf"], plain_scales(whole_x.col)[:, r0 // 16:r1 // 16])
        # Fprop / Dgrad of the shard's rows against the oracle
        for name, a, b, n, k in (("Y", "X_row", "W_row", N, K), ("dX", "dY_row", "W_col", K, N)):
            ref, bound = o.gemm(r[a + "_op"], r[b + "_op"], r1 - r0, n, k)
            nbad, worst = gemm_gate(torch.from_numpy(r[name]), ref, bound, True)
            assert nbad == 0, f"rank {rank} {name}: {nbad} outside the gate ({worst:.3g}x)"
    # the all-reduced Wgrad: the same on both ranks, and the sum of the partials within the gate
    assert np.array_equal(res[0]["dW"], res[1]["dW"])
    ref = np.zeros((N, K))
    bound = np.zeros((N, K))
    for r in res.values():
        p, b = o.gemm(r["dY_col_op"], r["X_col_op"], N, K, r["r1"] - r["r0"])
        ref += p
        bound += b
    nbad, worst = gemm_gate(torch.from_numpy(res[0]["dW"]), ref, bound, False)
    assert nbad == 0, f"dW: {nbad} outside the gate ({worst:.3g}x)"


def test_single_rank_step_equals_unsharded_quantization():
    """Without a process group the exchanges are no-ops and the step is the
    unsharded fused-producer layer step."""
    X, W, dY = _inputs("cuda")
    lin = dp.TokenShardedLinear("nvfp4", X, W, dY)
    Y, dX, dW = lin.step(seed=2)
    torch.cuda.synchronize()
    assert lpq.device_status() == 0
    both = lpq.ROWWISE | lpq.COLWISE | lpq.RHT_COLWISE
    wx = lpq.quantize(X, lpq.NVFP4, both, rht_seed=1234, sf_layout=lpq.SF_PLAIN)
    wd = lpq.quantize(dY, lpq.NVFP4, both | lpq.STOCHASTIC, seed=2, rht_seed=1234, sf_layout=lpq.SF_PLAIN)
    assert np.array_equal(codes(lin.q["X"].col), codes(wx.col))
    assert np.array_equal(codes(lin.q["dY"].col), codes(wd.col))
    ref, bound = o.gemm(oracle_operand(lin.q["dY"].col), oracle_operand(lin.q["X"].col), N, K, M)
    assert gemm_gate(dW, ref, bound, False)[0] == 0


@pytest.mark.parametrize("recipe", ["fp8_delayed", "mxfp8", "bf16"])
def test_two_rank_exchange_other_recipes(recipe):
    """The other branches of the exchange: delayed scaling all-reduces the amax
    its quantize pass measured before the history update (both ranks then hold
    the same state and tensor scales), MXFP8 exchanges no amax (block-local
    scales; shard codes equal the unsharded tensor's rows), bf16 only sums
    dW.  In every recipe the all-reduced dW is the same on both ranks and
    within the gate of the oracle's FP64 sum of the shards' partials."""
    res = _run(recipe)
    assert all(r["status"] == 0 for r in res.values())
    assert np.array_equal(res[0]["dW"], res[1]["dW"])
    if recipe != "bf16":
        for role in ("X", "dY"):
            assert res[0][f"{role}_row_ts"] == res[1][f"{role}_row_ts"]
        ref = np.zeros((N, K))
        bound = np.zeros((N, K))
        for r in res.values():
            p, b = o.gemm(r["dY_col_op"], r["X_col_op"], N, K, r["r1"] - r["r0"])
            ref += p
            bound += b
        nbad, worst = gemm_gate(torch.from_numpy(res[0]["dW"]), ref, bound, False)
        assert nbad == 0, f"dW: {nbad} outside the gate ({worst:.3g}x)"
    if recipe == "mxfp8":
        X, W, dY = _inputs("cuda")
        whole = lpq.quantize(X, lpq.MXFP8, lpq.ROWWISE | lpq.COLWISE, sf_layout=lpq.SF_PLAIN)
        for r in res.values():
            assert np.array_equal(r["X_row"], codes(whole.row)[r["r0"]:r["r1"]])
            assert np.array_equal(r["X_col"], codes(whole.col)[:, r["r0"]:r["r1"]])
    if recipe == "bf16":
        X, W, dY = _inputs("cuda")
        ref, bound = o.gemm(o.Operand(o.K_BF16, synth.host_bits(dY.t().contiguous())),
                            o.Operand(o.K_BF16, synth.host_bits(X.t().contiguous())), N, K, M)
        nbad, worst = gemm_gate(torch.from_numpy(res[0]["dW"]), ref, bound, False)
        assert nbad == 0, f"bf16 dW: {nbad} outside the gate ({worst:.3g}x)"
