"""World-size-2 gloo tests (CPU) of the host logic of the data-parallel path:
the benchmark's max-over-ranks timing, and the token-sharded quantize + Wgrad
through the product module's shard split and its two exchange steps
(precision_transformer_gemms_gb300.dp: exchange_amax = all-reduce MAX of the
shard amaxes, exchange_wgrad = all-reduce SUM of dW), with the oracle standing
in for the CUDA kernels, checked against the unsharded oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _timing_worker(rank, world, port, q):
    _init(rank, world, port)
    import bench
    got = bench.max_over_ranks(10.0 + rank, world)
    bench.barrier(world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_timing_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    res = dict(q.get(timeout=5) for _ in range(world))
    assert res == {0: 11.0, 1: 11.0}
    assert all(p.exitcode == 0 for p in procs)


def _shard_worker(rank, world, port, q):
    _init(rank, world, port)
    import oracle as o
    from precision_transformer_gemms_gb300 import dp, synth
    M, K, N = 64, 32, 16
    X = synth.host_bits(synth.bf16_normal((M, K), 1.0, 1, "cpu"))
    dY = synth.host_bits(synth.bf16_normal((M, N), 1e-3, 2, "cpu"))
    r0, r1 = dp.shard_rows(M, world, rank, granule=16)
    xs, ds = np.ascontiguousarray(X[r0:r1]), np.ascontiguousarray(dY[r0:r1])
    # exchange 1: all-reduce MAX of the shard amaxes (X raw, X RHT column, dY raw) in one call
    a = torch.tensor([o.amax(xs), o.nvfp4(xs, o.NV_COL | o.NV_RHT, rht_seed=9)["col_amax"], o.amax(ds)],
                     dtype=torch.float32)
    dp.exchange_amax(a)
    scale = float(np.float32(448.0) / np.float32(a[0].item()))
    codes = o.fp8_pertensor(xs, o.E4M3, scale=scale, colwise=False)["row"]
    # exchange 2: all-reduce SUM of the shard's dW = dY^T X (FP64 oracle GEMM on bf16)
    A = o.Operand(o.K_BF16, np.ascontiguousarray(ds.T))
    B = o.Operand(o.K_BF16, np.ascontiguousarray(xs.T))
    dw, _ = o.gemm(A, B, N, K, xs.shape[0])
    t = torch.from_numpy(dw.copy())
    dp.exchange_wgrad(t)
    q.put((rank, a.numpy().copy(), codes, t.numpy()))
    dist.destroy_process_group()


def test_sharded_quantize_and_wgrad_match_unsharded():
    import oracle as o
    from precision_transformer_gemms_gb300 import synth
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    res = {r: (a, c, dw) for r, a, c, dw in (q.get(timeout=5) for _ in range(world))}
    assert all(p.exitcode == 0 for p in procs)
    M, K, N = 64, 32, 16
    X = synth.host_bits(synth.bf16_normal((M, K), 1.0, 1, "cpu"))
    dY = synth.host_bits(synth.bf16_normal((M, N), 1e-3, 2, "cpu"))
    full = o.fp8_pertensor(X, o.E4M3, colwise=False)
    want = [full["amax"], o.nvfp4(X, o.NV_COL | o.NV_RHT, rht_seed=9)["col_amax"], o.amax(dY)]
    assert np.array_equal(res[0][0], np.float32(want)) and np.array_equal(res[1][0], res[0][0])
    assert np.array_equal(np.concatenate([res[0][1], res[1][1]]), full["row"])  # codes bit-identical
    ref, _ = o.gemm(o.Operand(o.K_BF16, np.ascontiguousarray(dY.T)), o.Operand(o.K_BF16, np.ascontiguousarray(X.T)),
                    N, K, M)
    assert np.allclose(res[0][2], ref, rtol=1e-12, atol=1e-18)  # only the summation order differs
    assert np.array_equal(res[0][2], res[1][2])


def test_shard_rows_cover_the_tokens_in_whole_groups():
    from precision_transformer_gemms_gb300 import dp
    for total, world in ((15872, 1), (15872, 2), (15872, 4), (15872, 8), (300, 3), (64, 8), (0, 2)):
        spans = [dp.shard_rows(total, world, r) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == total
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        assert all(r0 % 128 == 0 for r0, r1 in spans if r1 > r0)  # empty shards sit at the end
        sizes = [r1 - r0 for r0, r1 in spans]
        assert max(sizes) - min(sizes) <= 128
    assert dp.shard_rows(15872, 8, 0) == (0, 2048) and dp.shard_rows(15872, 8, 7) == (13952, 15872)
    with pytest.raises(ValueError):
        dp.shard_rows(128, 2, 2)


def test_exchanges_are_noops_without_a_process_group():
    from precision_transformer_gemms_gb300 import dp
    a = torch.tensor([1.0, 2.0])
    assert dp.exchange_amax(a) is a and a.tolist() == [1.0, 2.0]
    assert dp.exchange_wgrad(a) is a and a.tolist() == [1.0, 2.0]
