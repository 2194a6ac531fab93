"""Pins of the oracle's power-of-two (UE8M0) scale variant: the exponent rule checked on
every positive BF16 amax, the codes against torch's independent E4M3 conversion of the
exactly scaled values, the exact-sum GEMM against numpy's double product of the dequantised
operands, and an accuracy comparison of the two scale rules against the exact product of
the BF16 inputs."""
import numpy as np
import torch

import synth


def _f32(bits):
    return synth.bf16_to_f32(np.asarray(bits, np.uint16))


def test_exponent_rule_on_every_bf16_amax(orc):
    for b in range(1, 0x7F80):
        amax = float(_f32(b))
        e = orc.pow2_exponent(amax)
        assert e >= -127
        assert amax <= np.ldexp(448.0, e), (b, e)
        assert e == -127 or amax > np.ldexp(448.0, e - 1), (b, e)  # the smallest such e
    assert orc.pow2_exponent(0.0) == 0


def _torch_codes(v64):
    return torch.from_numpy(v64.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_rows_codes_and_scales(orc):
    x = synth.fill_bf16(synth.OUTLIER, synth.key(40, 0), (64, 512), 1.0, 0.02, 40.0, k2=synth.key(41, 0))
    x[3, :128] = 0
    x[4, 128:256] = 0x8000  # -0
    q, s = orc.quant_1x128_rows_pow2(x)
    xf = _f32(x).astype(np.float64)
    for kb in range(4):
        amax = np.abs(xf[:, kb * 128:(kb + 1) * 128]).max(axis=1)
        e = np.array([orc.pow2_exponent(a) for a in amax])
        assert np.array_equal(s[kb], np.ldexp(1.0, e).astype(np.float32))
        scaled = xf[:, kb * 128:(kb + 1) * 128] * np.ldexp(1.0, -e)[:, None]
        assert np.array_equal(q[:, kb * 128:(kb + 1) * 128], _torch_codes(scaled))
        nz = amax > 0
        top = amax[nz] / np.ldexp(1.0, e[nz])
        assert np.all((top > 224) & (top <= 448))  # the largest element uses the top binade
    assert np.all(q[4, 128:256] == 0x80)


def test_block_codes_and_partial_block(orc):
    w = synth.fill_bf16(synth.NORMAL, synth.key(42, 0), (200, 256), 0.02)
    q, s = orc.quant_128x128_pow2(w)
    wf = _f32(w).astype(np.float64)
    for nb in range(2):
        for kb in range(2):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            e = orc.pow2_exponent(np.abs(blk).max())
            assert s[nb, kb] == np.float32(np.ldexp(1.0, e))
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128],
                                  _torch_codes(blk * np.ldexp(1.0, -e)))


def _dq(codes, scale_rows):
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * scale_rows


def test_exact_sum_gemm_is_the_double_product(orc):
    a = synth.fill_bf16(synth.NORMAL, synth.key(43, 0), (24, 384), 1.0)
    w = synth.fill_bf16(synth.NORMAL, synth.key(44, 0), (136, 384), 0.02)
    qa, sa = orc.quant_1x128_rows_pow2(a)
    qb, sb = orc.quant_128x128_pow2(w)
    da = _dq(qa, np.repeat(sa.T.astype(np.float64), 128, axis=1))
    db = _dq(qb, np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0)[:136], 128, axis=1))
    ref = (da @ db.T).astype(np.float32)
    got = orc.gemm_exact_sum(qa, sa, qb, sb, 0)
    assert np.max(np.abs(got.astype(np.float64) - ref) / (np.abs(ref) + 1e-30)) <= 2.0 ** -23


def test_accuracy_of_the_two_scale_rules(orc):
    """Against the exact product of the BF16 inputs, the amax/448 rule is at least as
    accurate as the power-of-two rule, and the power-of-two rule loses at most a factor of
    two (its scaled values use between half and all of E4M3's range)."""
    d = synth.tiny()
    A, B = d["A"], d["B"]
    exact = _f32(A).astype(np.float64) @ _f32(B).astype(np.float64).T
    qa, sa = orc.quant_1x128_rows(A)
    qb, sb = orc.quant_128x128(B)
    c_f32 = orc.gemm_blockscaled(qa, sa, qb, sb, 0).astype(np.float64)
    pa, psa = orc.quant_1x128_rows_pow2(A)
    pb, psb = orc.quant_128x128_pow2(B)
    c_p2 = orc.gemm_exact_sum(pa, psa, pb, psb, 0).astype(np.float64)
    err = lambda c: np.linalg.norm(c - exact) / np.linalg.norm(exact)  # noqa: E731
    e_f32, e_p2 = err(c_f32), err(c_p2)
    assert e_f32 < 0.05 and e_p2 < 0.05
    assert e_f32 <= e_p2 <= 2.0 * e_f32, (e_f32, e_p2)
