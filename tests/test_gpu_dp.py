"""GPU parity of data-parallel Wgrad's local step (fp8_fine_grained_27_b300.dp.wgrad_local):
each shard's FP32 partial against the oracle's partial, and the rank-order FP32 sum of the
shards' partials against the oracle's data-parallel dW, within the GEMM tolerance.  The
ranks run one after the other on the one GPU (their kernels never wait on each other);
the collective is tested on two gloo ranks in tests/test_dp_multirank.py."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import assert_gemm_close, dev, host_bits, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 3])
def test_shard_partials_and_their_sum(orc, world):
    from fp8_fine_grained_27_b300 import dp
    d = synth.wgrad(T=1024, Cout=256, Cin=392)
    ref, ref_parts = orc.wgrad_dp(d["dY"], d["X"], world)
    total = None
    for r in range(world):
        t0, t1 = dp.token_shard(1024, world, r)
        part = dp.wgrad_local(dev(d["dY"][t0:t1]), dev(d["X"][t0:t1]))
        torch.cuda.synchronize()
        assert_gemm_close(host_bits(part), ref_parts[r], f"partial {r}")
        total = part.clone() if total is None else total + part
    torch.cuda.synchronize()
    assert_gemm_close(host_bits(total), ref, f"dp sum, {world} ranks")


def test_full_size_two_ranks_sampled_rows(orc):
    """Workload 4 (16384 tokens, dW 2048 x 7168) split over two ranks; 64 rows of dW."""
    from fp8_fine_grained_27_b300 import dp
    d = synth.wgrad()
    T = d["dY"].shape[0]
    rows = sample_rows(2048, 64, seed=13, must=(0, 2047))
    ref = None
    total = None
    for r in range(2):
        t0, t1 = dp.token_shard(T, 2, r)
        part = dp.wgrad_local(dev(d["dY"][t0:t1]), dev(d["X"][t0:t1]))
        total = part if total is None else total + part
        qd, sd = orc.quant_1x128_cols(d["dY"][t0:t1])
        qx, sx = orc.quant_1x128_cols(d["X"][t0:t1])
        p = orc.gemm_blockscaled(qd, sd, qx, sx, 1, rows=rows)
        ref = p if ref is None else np.add(ref, p, dtype=np.float32)
    torch.cuda.synchronize()
    assert_gemm_close(host_bits(total[torch.from_numpy(rows).cuda()]), ref, "dp full size")
