"""Pins of the oracle's data-parallel Wgrad (V3 report §7: ZeRO-1 data parallelism over
the batch; §6: Wgrad in FP8, FP32 out): token shards of whole 128-token tiles, one
partial per shard by the single-rank rule, partials summed in FP32 in rank order.

Checked against: the tiling itself (shards cover every tile once, contiguously, as evenly
as possible); the single-rank oracle for one rank; and, for inputs whose quantisation is
lossless and whose every partial sum is exact, the exact integer product (a missing,
repeated or transposed shard would change it)."""
import numpy as np
import torch

import synth


def test_token_shards_tile_the_tokens(orc):
    for T, world in [(1024, 2), (1024, 3), (16384, 8), (128, 1), (384, 4)]:
        sh = orc.token_shards(T, world)
        assert len(sh) == world and sh[0][0] == 0 and sh[-1][1] == T
        assert all(a[1] == b[0] for a, b in zip(sh, sh[1:]))
        sizes = [t1 - t0 for t0, t1 in sh]
        assert all(s % 128 == 0 for s in sizes) and max(sizes) - min(sizes) <= 128


def test_one_rank_is_the_single_rank_wgrad(orc):
    d = synth.wgrad(T=512, Cout=256, Cin=136)
    dW, parts = orc.wgrad_dp(d["dY"], d["X"], 1)
    qd, sd = orc.quant_1x128_cols(d["dY"])
    qx, sx = orc.quant_1x128_cols(d["X"])
    assert len(parts) == 1 and np.array_equal(dW, orc.gemm_blockscaled(qd, sd, qx, sx, 1))


def _exact_inputs(rng, T, C):
    """BF16 [T, C]: small integers times 2^-8, every 128-token tile of a channel holding
    +-448 * 2^-8 (so its scale is 2^-8 and its codes are exact)."""
    v = rng.integers(-4, 5, (T, C)).astype(np.float64)
    for t0 in range(0, T, 128):
        rows = t0 + rng.integers(0, 128, C)
        v[rows, np.arange(C)] = rng.choice([-448.0, 448.0], C)
    v *= 2.0 ** -8
    bits = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(synth.bf16_to_f32(bits).astype(np.float64), v)
    return bits, v


def test_shards_sum_to_the_exact_product(orc):
    rng = np.random.default_rng(12)
    T, Cout, Cin = 1024, 256, 392
    dy, vy = _exact_inputs(rng, T, Cout)
    x, vx = _exact_inputs(rng, T, Cin)
    exact = (vy.T @ vx).astype(np.float32)          # every partial sum fits FP32 exactly
    assert np.array_equal(exact.astype(np.float64), vy.T @ vx)
    for world in (1, 2, 3, 8):
        dW, parts = orc.wgrad_dp(dy, x, world)
        assert len(parts) == world
        assert np.array_equal(dW, exact), world
    # a shard boundary off by one tile would drop or repeat 128 tokens
    qd, sd = orc.quant_1x128_cols(dy[128:])
    qx, sx = orc.quant_1x128_cols(x[128:])
    assert not np.array_equal(orc.gemm_blockscaled(qd, sd, qx, sx, 1), exact)


def test_rank_order_sum_in_fp32(orc):
    d = synth.wgrad(T=768, Cout=128, Cin=64)
    dW, parts = orc.wgrad_dp(d["dY"], d["X"], 3)
    p = [torch.from_numpy(q) for q in parts]
    assert np.array_equal(dW, ((p[0] + p[1]) + p[2]).numpy())
