"""GPU parity of the power-of-two (UE8M0) scale variant through the C ABI.

- Quantisers: codes and scales bit-exact against the oracle's power-of-two mode, including
  tiles whose scale is clamped at 2^-127, all-zero tiles and -0.
- fp8_gemm_ue8m0 (the tensor cores' block-scaled MMA, FP32 accumulation over the whole K)
  against the oracle's exact double sum of the scaled products, under the GEMM tolerance of
  tests/gpu_util.py.
- fp8_gemm_blockscaled on power-of-two scales (per-chunk promotion) against the oracle's
  promotion rule, under the same tolerance.
"""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import assert_gemm_close, dev, host_bits, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    import fp8_fine_grained_27_b300 as fb
    assert torch.cuda.is_available()
    return fb


@pytest.fixture(params=[0, 192], ids=["bn256", "bn192"])
def mx_tile(request, fb):
    """The block-scaled GEMM's tile width: 256 (one accumulator, the default) or 192 (two)."""
    fb.set_gemm_tile_n(request.param)
    yield request.param
    fb.set_gemm_tile_n(0)


def _rows(fb, orc, x_bits):
    q, s = fb.quant_1x128_ue8m0(dev(x_bits))
    torch.cuda.synchronize()
    oq, os_ = orc.quant_1x128_rows_pow2(x_bits)
    assert np.array_equal(s.cpu().numpy(), os_), "scales differ"
    assert np.count_nonzero(q.cpu().numpy() != oq) == 0, "codes differ"
    return q, s


def _block(fb, orc, w_bits):
    q, s = fb.quant_128x128_ue8m0(dev(w_bits))
    torch.cuda.synchronize()
    oq, os_ = orc.quant_128x128_pow2(w_bits)
    assert np.array_equal(s.cpu().numpy(), os_), "scales differ"
    assert np.count_nonzero(q.cpu().numpy() != oq) == 0, "codes differ"
    return q, s


def test_quant_rows_ragged_and_wide_range(fb, orc):
    for (M, K, seed) in [(1, 128, 1), (129, 384, 2), (300, 1024, 3)]:
        _rows(fb, orc, synth.fill_bf16(synth.OUTLIER, synth.key(50, seed), (M, K), 1.0, 0.02, 30.0,
                                       k2=synth.key(51, seed)))
    rng = np.random.default_rng(3)
    x = rng.standard_normal((256, 2048)).astype(np.float32)
    x *= np.exp2(rng.integers(-60, 60, (256, 16))).repeat(128, axis=1).astype(np.float32)
    x[3, :128] = 0.0
    x[4, 128:256] = -0.0
    x[5, 256:384] = 1e-38   # scale clamped at 2^-127
    x[6, 384:512] = 3e38    # near the top of the range
    _rows(fb, orc, (x.view(np.uint32) >> 16).astype(np.uint16))


def test_quant_block_and_full_tensors(fb, orc):
    for (N, K, seed) in [(1, 128, 1), (200, 256, 2), (576, 512, 3)]:
        _block(fb, orc, synth.fill_bf16(synth.NORMAL, synth.key(52, seed), (N, K), 0.02))
    d = synth.mla()
    _rows(fb, orc, d["A"])
    _block(fb, orc, d["Wkv"])


def _mx(fb, orc, a, w, out_dtype=torch.bfloat16, rows=None, what=""):
    qa, sa = fb.quant_1x128_ue8m0(dev(a))
    qb, sb = fb.quant_128x128_ue8m0(dev(w))
    C = fb.gemm_ue8m0(qa, sa, qb, sb, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    oqa, osa = orc.quant_1x128_rows_pow2(a)
    oqb, osb = orc.quant_128x128_pow2(w)
    if rows is None:
        rows = np.arange(a.shape[0])
    ref = orc.gemm_exact_sum(oqa, osa, oqb, osb, 0, rows=rows)
    if out_dtype == torch.bfloat16:
        ref = orc.bf16_round(ref)
    got = host_bits(C[torch.from_numpy(rows).cuda()])
    return assert_gemm_close(got, ref, what)


def test_mx_tiny(fb, orc, mx_tile):
    d = synth.tiny()
    _mx(fb, orc, d["A"], d["B"], what="tiny")
    _mx(fb, orc, d["A"], d["B"], out_dtype=torch.float32, what="tiny fp32")


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (300, 392, 640), (129, 72, 256), (257, 520, 384), (64, 128, 1024)])
def test_mx_ragged_shapes(fb, orc, mx_tile, M, N, K):
    a = synth.fill_bf16(synth.OUTLIER, synth.key(53, M), (M, K), 1.0, 0.01, 50.0, k2=synth.key(54, M))
    w = synth.fill_bf16(synth.NORMAL, synth.key(55, N), (N, K), 0.02)
    _mx(fb, orc, a, w, what=f"{M}x{N}x{K}")
    _mx(fb, orc, a, w, out_dtype=torch.float32, what=f"{M}x{N}x{K} fp32")


def test_mx_raster_groups_with_a_partial_last_group(fb, orc, mx_tile):
    """40 M tiles at a K whose raster group is 32 tiles (one full group, a
    partial one, ragged last M and N tiles); the first and last row of every M
    tile plus a seeded sample are checked."""
    M, N, K = 40 * 128 - 37, 520, 256
    a = synth.fill_bf16(synth.OUTLIER, synth.key(93, M), (M, K), 1.0, 0.01, 50.0, k2=synth.key(94, M))
    w = synth.fill_bf16(synth.NORMAL, synth.key(95, N), (N, K), 0.02)
    must = [r for t in range(40) for r in (t * 128, min(t * 128 + 127, M - 1))]
    _mx(fb, orc, a, w, rows=sample_rows(M, 64, seed=11, must=must), what="mx raster groups")


def test_mx_mla_full(fb, orc, mx_tile):
    d = synth.mla()
    _mx(fb, orc, d["A"], np.concatenate([d["Wq"], d["Wkv"]]), what="mla")


def test_mx_ffn_sampled(fb, orc):
    d = synth.ffn()
    rows = sample_rows(16384, 128, seed=8, must=(0, 127, 128, 16383))
    _mx(fb, orc, d["A"], d["B"], rows=rows, what="ffn")


def test_promoted_gemm_on_power_of_two_scales(fb, orc):
    d = synth.tiny()
    qa, sa = fb.quant_1x128_ue8m0(dev(d["A"]))
    qb, sb = fb.quant_128x128_ue8m0(dev(d["B"]))
    C = fb.gemm_blockscaled(qa, sa, qb, sb, 0)
    torch.cuda.synchronize()
    oqa, osa = orc.quant_1x128_rows_pow2(d["A"])
    oqb, osb = orc.quant_128x128_pow2(d["B"])
    assert_gemm_close(host_bits(C), orc.bf16_round(orc.gemm_blockscaled(oqa, osa, oqb, osb, 0)), "promoted pow2")
