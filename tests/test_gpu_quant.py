"""GPU parity: E4M3 conversion and the 1x128 / 128x128 quantisers, bit-exact
against the oracle (codes and scales), through the C ABI.

Sizes: small ragged cases that span several tiles plus the full tensors of
every workload (tiny, MLA, MoE sampled experts, Wgrad, FFN, Dgrad weights)."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    import fp8_fine_grained_27_b300 as fb
    assert torch.cuda.is_available()
    return fb


def _rows(fb, orc, x_bits):
    q, s = fb.quant_1x128(dev(x_bits))
    torch.cuda.synchronize()
    qr, sr = orc.quant_1x128_rows(x_bits)
    assert np.array_equal(s.cpu().numpy(), sr), "scales differ"
    bad = np.count_nonzero(q.cpu().numpy() != qr)
    assert bad == 0, f"{bad} codes differ"


def _block(fb, orc, w_bits):
    q, s = fb.quant_128x128(dev(w_bits))
    torch.cuda.synchronize()
    qr, sr = orc.quant_128x128(w_bits)
    assert np.array_equal(s.cpu().numpy(), sr), "scales differ"
    bad = np.count_nonzero(q.cpu().numpy() != qr)
    assert bad == 0, f"{bad} codes differ"


def _cols(fb, orc, x_bits):
    q, s = fb.quant_1x128(dev(x_bits), along=1)
    torch.cuda.synchronize()
    qr, sr = orc.quant_1x128_cols(x_bits)
    assert np.array_equal(s.cpu().numpy(), sr), "scales differ"
    bad = np.count_nonzero(q.cpu().numpy() != qr)
    assert bad == 0, f"{bad} codes differ"


def _block_t(fb, orc, w_bits, straight=True):
    q, s, qt, st = fb.quant_128x128_t(dev(w_bits), straight=straight)
    torch.cuda.synchronize()
    qr, sr, qtr, str_ = orc.quant_128x128_t(w_bits)
    assert np.array_equal(st.cpu().numpy(), str_), "transposed scales differ"
    bad = np.count_nonzero(qt.cpu().numpy() != qtr)
    assert bad == 0, f"{bad} transposed codes differ"
    if straight:
        assert np.array_equal(s.cpu().numpy(), sr), "scales differ"
        bad = np.count_nonzero(q.cpu().numpy() != qr)
        assert bad == 0, f"{bad} codes differ"


def _wide_range(rng, R, C):
    """Tiles whose scales span ~2^-60 .. 2^60, with exact zeros, -0 and subnormal inputs."""
    x = rng.standard_normal((R, C)).astype(np.float32)
    x *= np.exp2(rng.integers(-60, 60, (R // 128 + 1, C // 128))).repeat(128, axis=0)[:R].repeat(
        128, axis=1).astype(np.float32)
    return x


def test_fast_quotient_equals_ieee_divide_on_whole_bf16_domain(fb):
    """The quantisers divide by the tile scale with a per-tile reciprocal and
    one Markstein correction; on the device, encode that quotient and the IEEE
    quotient to E4M3 for every BF16 amax and every BF16 x with |x| <= amax:
    the codes must agree everywhere (the FP32 quotients may differ in the
    last bit near underflow, where both encode to zero)."""
    code_mismatches, quotient_mismatches = fb.selftest_division()
    assert code_mismatches == 0
    assert quotient_mismatches < 2 ** 31 // 100


def test_encode_exhaustive(fb, orc):
    """Every non-NaN FP32 bit pattern through the kernels' E4M3 conversion."""
    chunk = 1 << 28
    for lo in range(0, 1 << 32, chunk):
        pat = torch.arange(lo, lo + chunk, dtype=torch.int64, device="cuda").to(torch.int32)
        x = pat.view(torch.float32)
        q = fb.e4m3_encode(x).cpu().numpy()
        ref = orc.e4m3_encode_patterns(lo, chunk)
        xs = np.arange(lo, lo + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        keep = ~np.isnan(xs)
        bad = np.count_nonzero(q[keep] != ref[keep])
        assert bad == 0, f"patterns {lo:#x}..: {bad} codes differ"


def test_rows_small_ragged(fb, orc):
    for (M, K, seed) in [(1, 128, 1), (127, 256, 2), (129, 384, 3), (300, 1024, 4)]:
        a = synth.fill_bf16(synth.OUTLIER, synth.key(90, seed), (M, K), 1.0, 0.02, 30.0, k2=synth.key(91, seed))
        _rows(fb, orc, a)


def test_rows_wide_dynamic_range(fb, orc):
    """Tiles whose scales span ~2^-60 .. 2^60, with exact zeros and -0."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal((256, 2048)).astype(np.float32)
    x *= np.exp2(rng.integers(-60, 60, (256, 16))).repeat(128, axis=1).astype(np.float32)
    x[3, :128] = 0.0
    x[4, 128:256] = -0.0
    x[5, 256:384] = 1e-38  # subnormal inputs: the tile scale is subnormal too
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    _rows(fb, orc, bits)


def test_rows_tiny_workload(fb, orc):
    _rows(fb, orc, synth.tiny()["A"])


def test_block_small_ragged(fb, orc):
    for (N, K, seed) in [(1, 128, 1), (200, 256, 2), (576, 512, 3)]:
        _block(fb, orc, synth.fill_bf16(synth.NORMAL, synth.key(92, seed), (N, K), 0.02))


def test_block_tiny_workload(fb, orc):
    _block(fb, orc, synth.tiny()["B"])


def test_mla_full(fb, orc):
    d = synth.mla()
    _rows(fb, orc, d["A"])
    _block(fb, orc, d["Wq"])
    _block(fb, orc, d["Wkv"])  # 576 rows: last block is 64 rows


def test_cols_small_ragged(fb, orc):
    for (T, C, seed) in [(128, 8, 1), (384, 200, 2), (512, 1032, 3)]:
        _cols(fb, orc, synth.fill_bf16(synth.NORMAL, synth.key(93, seed), (T, C), 1e-2))


def test_cols_wide_dynamic_range(fb, orc):
    rng = np.random.default_rng(1)
    x = _wide_range(rng, 384, 1024)
    x[:128, 3] = 0.0
    x[128:256, 130] = -0.0
    x[256:, 260] = 1e-38
    _cols(fb, orc, (x.view(np.uint32) >> 16).astype(np.uint16))


def test_block_t_small_ragged(fb, orc):
    for (N, K, seed) in [(16, 128, 1), (144, 256, 2), (576, 512, 3), (384, 1024, 4)]:
        w = synth.fill_bf16(synth.OUTLIER, synth.key(98, seed), (N, K), 0.02, 0.01, 40.0, k2=synth.key(99, seed))
        _block_t(fb, orc, w)
        _block_t(fb, orc, w, straight=False)


def test_block_t_wide_dynamic_range(fb, orc):
    rng = np.random.default_rng(2)
    x = _wide_range(rng, 400, 640)
    x[:128, :128] = 0.0
    x[128:256, 128:256] = -0.0
    x[256:384, 256:384] = 1e-38
    _block_t(fb, orc, (x.view(np.uint32) >> 16).astype(np.uint16))


def test_block_t_strided(fb, orc):
    """Leading dimensions larger than the used widths (16-byte multiples)."""
    w = synth.fill_bf16(synth.NORMAL, synth.key(94, 1), (160, 400), 0.02)
    x = dev(w)[:, :256]
    qt = torch.zeros((256, 176), dtype=torch.uint8, device="cuda")[:, :160]
    st = torch.zeros((2, 4), dtype=torch.float32, device="cuda")[:, :2]
    q = torch.zeros((160, 272), dtype=torch.uint8, device="cuda")[:, :256]
    s = torch.zeros((2, 4), dtype=torch.float32, device="cuda")[:, :2]
    fb.quant_128x128_t(x, q=q, s=s, qt=qt, st=st)
    torch.cuda.synchronize()
    qr, sr, qtr, str_ = orc.quant_128x128_t(np.ascontiguousarray(w[:, :256]))
    assert np.array_equal(qt.cpu().numpy(), qtr) and np.array_equal(st.cpu().numpy(), str_)
    assert np.array_equal(q.cpu().numpy(), qr) and np.array_equal(s.cpu().numpy(), sr)


def test_block_t_full_weights(fb, orc):
    d = synth.mla()
    _block_t(fb, orc, d["Wq"])
    _block_t(fb, orc, d["Wkv"])  # 576 rows: last block is 64 rows
    _block_t(fb, orc, synth.dgrad(T=128)["W"])  # 18432 x 7168


def test_wgrad_full(fb, orc):
    d = synth.wgrad()
    _cols(fb, orc, d["dY"])
    _cols(fb, orc, d["X"])


def test_ffn_full(fb, orc):
    d = synth.ffn()
    _rows(fb, orc, d["A"])
    _block(fb, orc, d["B"])


def test_moe_tokens_and_sampled_experts(fb, orc):
    _rows(fb, orc, synth.moe_tokens())
    _rows(fb, orc, synth.moe_down_input())
    for which in ("up", "down"):
        for e in (0, 1, 128, 255):
            w = synth.moe_weights(which, e, e + 1)[0]
            _block(fb, orc, w)


def test_strided_views(fb, orc):
    """Leading dimensions larger than the used width (16-byte multiples)."""
    a = synth.fill_bf16(synth.NORMAL, synth.key(94, 0), (200, 520), 1.0)
    x = dev(a)[:, :384]
    q = torch.zeros((200, 400), dtype=torch.uint8, device="cuda")[:, :384]
    s = torch.zeros((3, 208), dtype=torch.float32, device="cuda")[:, :200]
    fb.quant_1x128(x, q=q, s=s)
    torch.cuda.synchronize()
    qr, sr = orc.quant_1x128_rows(np.ascontiguousarray(a[:, :384]))
    assert np.array_equal(q.cpu().numpy(), qr) and np.array_equal(s.cpu().numpy(), sr)



@pytest.mark.parametrize("ue8m0", [False, True], ids=["amax448", "ue8m0"])
def test_act_weight_in_one_launch(fb, orc, ue8m0):
    """The fused launch gives the separate quantisers' codes and scales bit for bit."""
    d = synth.mla()
    A, W = d["A"], np.concatenate([d["Wq"], d["Wkv"]])
    qx, sx, qw, sw = fb.quant_act_weight(dev(A), dev(W), ue8m0=ue8m0)
    torch.cuda.synchronize()
    if ue8m0:
        rx, rsx = orc.quant_1x128_rows_pow2(A)
        rw, rsw = orc.quant_128x128_pow2(W)
    else:
        rx, rsx = orc.quant_1x128_rows(A)
        rw, rsw = orc.quant_128x128(W)
    assert np.array_equal(qx.cpu().numpy(), rx) and np.array_equal(sx.cpu().numpy(), rsx)
    assert np.array_equal(qw.cpu().numpy(), rw) and np.array_equal(sw.cpu().numpy(), rsw)
    # an empty activation leaves only the weight's tiles
    e = torch.empty((0, 7168), dtype=torch.bfloat16, device="cuda")
    _, _, qw2, sw2 = fb.quant_act_weight(e, dev(W), ue8m0=ue8m0)
    torch.cuda.synchronize()
    assert np.array_equal(qw2.cpu().numpy(), rw) and np.array_equal(sw2.cpu().numpy(), rsw)
