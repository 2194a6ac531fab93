"""Pins for the oracle's 1x128 / 128x128 quantisers (V3 report §6.1).

Checked against invariants that the method fixes (each tile's amax element
maps to +-448, every code is finite and |q| <= 448, scales are the correctly
rounded amax/448), power-of-two equivariance, identities between the tile
shapes, the dequantisation error bound, and an independent numpy + torch
restatement on small inputs.
"""
from fractions import Fraction

import numpy as np
import torch

import synth


def _f32(bits):
    return synth.bf16_to_f32(bits)


def _indep_rows(x_bits):
    """Independent restatement: numpy float32 amax/448 and x/s, torch's E4M3 conversion."""
    x = _f32(x_bits).astype(np.float32)
    M, K = x.shape
    t = x.reshape(M, K // 128, 128)
    amax = np.abs(t).max(axis=2).astype(np.float32)
    s = np.where(amax == 0, np.float32(1), amax / np.float32(448)).astype(np.float32)
    y = (t / s[:, :, None]).astype(np.float32)
    y = np.clip(y, -448, 448)  # torch turns >= 464 into NaN; the method saturates
    q = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q.reshape(M, K), s.T.copy()


def test_rows_match_independent_restatement(orc):
    x = synth.tiny()["A"]
    q, s = orc.quant_1x128_rows(x)
    q2, s2 = _indep_rows(x)
    assert np.array_equal(s, s2)
    assert np.array_equal(q, q2)


def test_scale_is_correctly_rounded_quotient(orc):
    x = synth.tiny()["A"]
    _, s = orc.quant_1x128_rows(x)
    amax = np.abs(_f32(x)).reshape(128, 4, 128).max(axis=2).T
    for sc, am in zip(s.ravel()[:256], amax.ravel()[:256]):
        exact = Fraction(float(am)) / 448
        here = abs(Fraction(float(sc)) - exact)
        for nb in (np.nextafter(sc, np.float32(0)), np.nextafter(sc, np.float32(1e30))):
            assert here <= abs(Fraction(float(nb)) - exact)


def test_invariants_rows(orc):
    x = synth.tiny()["A"]
    q, s = orc.quant_1x128_rows(x)
    dec = orc.decode_table()
    v = dec[q]
    assert not np.isnan(v).any() and np.abs(v).max() <= 448
    xf = _f32(x).reshape(128, 4, 128)
    at_amax = np.abs(xf) == np.abs(xf).max(axis=2, keepdims=True)
    qq = q.reshape(128, 4, 128)
    assert np.all((qq[at_amax] & 0x7F) == 0x7E)


def test_dequant_error_bound(orc):
    x = synth.tiny()["A"]
    q, s = orc.quant_1x128_rows(x)
    dec = orc.decode_table()
    xf = _f32(x).astype(np.float64).reshape(128, 4, 128)
    sc = s.T.astype(np.float64)[:, :, None]
    y = dec[q].reshape(128, 4, 128)
    # |dec(q) - x/s| <= 2^-4 |x/s| (normal range) or 2^-10 (subnormal range), plus the divide's rounding
    err = np.abs(y - xf / sc)
    bound = np.maximum(2.0 ** -4 * np.abs(xf / sc), 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(err <= bound)


def test_power_of_two_equivariance(orc):
    x = synth.tiny()["A"]
    q, s = orc.quant_1x128_rows(x)
    for j in (-20, -3, 5, 40):
        xs = (_f32(x).astype(np.float64) * 2.0 ** j).astype(np.float32)
        bits = (xs.view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal(_f32(bits), xs)  # exact in BF16
        q2, s2 = orc.quant_1x128_rows(bits)
        assert np.array_equal(q2, q)
        assert np.array_equal(s2, (s.astype(np.float64) * 2.0 ** j).astype(np.float32))


def test_zero_tile_and_negative_zero(orc):
    x = np.zeros((2, 256), np.uint16)
    x[1, :128] = 0x8000  # -0.0 in BF16
    x[1, 128] = 0x3F80  # 1.0
    q, s = orc.quant_1x128_rows(x)
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0 and s[1, 0] == 1.0
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0x80)
    assert q[1, 128] == 0x7E and np.all(q[1, 129:] == 0)


def test_gather_commutes_with_row_quant(orc):
    x = synth.tiny()["A"]
    idx = np.random.default_rng(3).integers(0, 128, 300)
    q, s = orc.quant_1x128_rows(x)
    q2, s2 = orc.quant_1x128_rows(np.ascontiguousarray(x[idx]))
    assert np.array_equal(q[idx], q2) and np.array_equal(s[:, idx], s2)


def test_cols_equal_rows_of_transpose(orc):
    d = synth.wgrad(T=384, Cout=96, Cin=160)
    for X in (d["dY"], d["X"]):
        qc, sc = orc.quant_1x128_cols(X)
        qr, sr = orc.quant_1x128_rows(np.ascontiguousarray(X.T))
        assert np.array_equal(qc, qr) and np.array_equal(sc, sr)


def test_block_equals_rows_when_row_amax_uniform(orc):
    """If every 1x128 row tile of a 128x128 block has the same amax, the block
    scale equals each row scale and the codes coincide."""
    rng = np.random.default_rng(5)
    w = rng.standard_normal((256, 256)).astype(np.float32) * 0.02
    w = np.clip(w, -0.06, 0.06)
    w[:, 7] = 0.0625
    w[:, 200] = -0.0625
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)
    qb, sb = orc.quant_128x128(bits)
    qr, sr = orc.quant_1x128_rows(bits)
    assert np.array_equal(qb, qr)
    assert np.all(sb == sr[0, 0]) and np.all(sr == sr[0, 0])


def test_partial_block_uses_present_rows_only(orc):
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((192, 128)) * 0.01).astype(np.float32)
    w[5, 3] = 4.0  # only in the first block
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)
    q, s = orc.quant_128x128(bits)
    amax1 = np.abs(_f32(bits[128:])).max()
    assert s[1, 0] == np.float32(amax1) / np.float32(448)
    assert s[0, 0] == np.float32(4.0) / np.float32(448)
    # block invariants: the block's amax element maps to 448
    assert (q[5, 3] & 0x7F) == 0x7E
    i, j = np.unravel_index(np.argmax(np.abs(_f32(bits[128:]))), (64, 128))
    assert (q[128 + i, j] & 0x7F) == 0x7E


def test_block_matches_independent_restatement(orc):
    w = synth.tiny()["B"]
    q, s = orc.quant_128x128(w)
    x = _f32(w)
    N, K = x.shape
    for nb in range(N // 128):
        for kb in range(K // 128):
            blk = x[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            sc = np.float32(np.abs(blk).max()) / np.float32(448)
            assert s[nb, kb] == sc
            y = np.clip((blk / sc).astype(np.float32), -448, 448)
            ref = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128], ref)


def test_block_transpose_is_quantisation_of_transpose(orc):
    """Quantising W^T directly gives the transposed codes and block scales (a 128x128 block
    is the same set of elements either way); the partial last block row survives the swap."""
    for N, K, seed in ((256, 384, 1), (384, 128, 2)):
        w = synth.fill_bf16(synth.OUTLIER, synth.key(95, seed), (N, K), 0.02, 0.02, 40.0, k2=synth.key(96, seed))
        q, s, qt, st = orc.quant_128x128_t(w)
        q2, s2 = orc.quant_128x128(np.ascontiguousarray(w.T))
        assert np.array_equal(qt, q2) and np.array_equal(st, s2)
        assert np.array_equal(qt.T, q) and np.array_equal(st.T, s)
    w = synth.fill_bf16(synth.NORMAL, synth.key(97, 0), (144, 256), 0.02)
    q, s, qt, st = orc.quant_128x128_t(w)
    assert qt.shape == (256, 144) and st.shape == (2, 2)
    assert np.array_equal(qt[:, 128:], orc.quant_128x128(w[128:])[0].T)
