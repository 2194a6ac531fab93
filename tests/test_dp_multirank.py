"""Data-parallel Wgrad's exchange step on two gloo ranks (CPU): each rank holds the FP32
partial dW of its own token shard (computed here by the oracle, standing in for the
GPU partial, which tests/test_gpu_dp.py checks), dp.reduce_scatter_rows sums the
partials and hands each rank its rows.  The reassembled dW must equal the oracle's
data-parallel dW bit for bit (two FP32 addends: the sum is exact-commutative) and the
single-rank dW within the GEMM tolerance (only the FP32 addition order across the
shard boundary differs)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synth
from tests.gpu_util import assert_gemm_close


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SHAPE = dict(T=1024, Cout=256, Cin=392)


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from fp8_fine_grained_27_b300 import dp
        oracle.build()
        d = synth.wgrad(**SHAPE)
        t0, t1 = dp.token_shard(SHAPE["T"], world, rank)
        qd, sd = oracle.quant_1x128_cols(d["dY"][t0:t1])
        qx, sx = oracle.quant_1x128_cols(d["X"][t0:t1])
        part = torch.from_numpy(oracle.gemm_blockscaled(qd, sd, qx, sx, 1))
        mine = dp.reduce_scatter_rows(part)
        rows = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(rows, mine)
        q.put((rank, (t0, t1), torch.cat(rows).numpy()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_scatter_the_wgrad_partials(orc):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=300) for _ in range(2)), key=lambda g: g[0])
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    d = synth.wgrad(**SHAPE)
    ref, _ = orc.wgrad_dp(d["dY"], d["X"], 2)
    assert [g[1] for g in got] == orc.token_shards(SHAPE["T"], 2)
    for _, _, dW in got:
        assert np.array_equal(dW, ref)
    qd, sd = orc.quant_1x128_cols(d["dY"])
    qx, sx = orc.quant_1x128_cols(d["X"])
    assert_gemm_close(got[0][2], orc.gemm_blockscaled(qd, sd, qx, sx, 1), "dp vs single rank")


def test_token_shard_bounds():
    from fp8_fine_grained_27_b300 import dp
    assert [dp.token_shard(1024, 3, r) for r in range(3)] == [(0, 256), (256, 640), (640, 1024)]
    for bad in [(100, 2, 0), (1024, 2, 2), (1024, 0, 0)]:
        try:
            dp.token_shard(*bad)
        except ValueError:
            continue
        raise AssertionError(bad)
