"""Pins for the oracle's block-scaled GEMM (V3 report §6, §6.2).

- exact rational brute force (Fractions) of the per-chunk promotion rule on a
  tiny case spanning two K chunks and two B blocks, both scale modes;
- all-ones scales reduce to a plain FP8 GEMM with FP32 accumulation of
  per-128 partials (numpy matmul of torch-decoded codes);
- lossless inputs (E4M3 values times a per-tile power of two with the tile
  amax at 448*2^j) give the exact double GEMM of the BF16 inputs, up to FP32
  accumulation;
- the grouped form equals per-expert GEMMs stitched together.
"""
from fractions import Fraction

import numpy as np
import torch

import synth


def _dec_torch(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _rne_f32(fr: Fraction) -> np.float32:
    """Round a rational to the nearest float32, ties to even (normal range)."""
    if fr == 0:
        return np.float32(0.0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # a in [2^e, 2^(e+1)); 24-bit significand
    scale = Fraction(2) ** (23 - e)
    m = a * scale
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return np.float32(sign * float(Fraction(fl) / scale))


def _brute(A, sa, B, sb, b_mode):
    M, K = A.shape
    N = B.shape[0]
    dA = _dec_torch(A)
    dB = _dec_torch(B)
    out = np.zeros((M, N), np.float32)
    for m in range(M):
        for n in range(N):
            acc = np.float32(0)
            for kb in range(K // 128):
                P = sum((Fraction(float(dA[m, k])) * Fraction(float(dB[n, k]))
                         for k in range(kb * 128, kb * 128 + 128)), Fraction(0))
                P32 = _rne_f32(P)
                sbv = sb[n // 128, kb] if b_mode == 0 else sb[kb, n]
                sc = np.float32(sa[kb, m]) * np.float32(sbv)
                acc = _rne_f32(Fraction(float(sc)) * Fraction(float(P32)) + Fraction(float(acc)))
            out[m, n] = acc
    return out


def _tiny_quantised(orc, M=3, N=130, K=256, seed=11):
    rng = np.random.default_rng(seed)
    a = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-3, 4, (M, K)))).astype(np.float32)
    b = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    ab = (a.view(np.uint32) >> 16).astype(np.uint16)
    bb = (b.view(np.uint32) >> 16).astype(np.uint16)
    qa, sa = orc.quant_1x128_rows(ab)
    qb, sb = orc.quant_128x128(bb)
    return qa, sa, qb, sb, bb


def test_exact_bruteforce_block_mode(orc):
    qa, sa, qb, sb, _ = _tiny_quantised(orc)
    out = orc.gemm_blockscaled(qa, sa, qb, sb, 0)
    ref = _brute(qa, sa, qb, sb, 0)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


def test_exact_bruteforce_row_mode(orc):
    qa, sa, _, _, bb = _tiny_quantised(orc, N=40)
    qb, sbr = orc.quant_1x128_rows(bb)  # per-row 1x128 scales on B: [K/128, N]
    out = orc.gemm_blockscaled(qa, sa, qb, sbr, 1)
    ref = _brute(qa, sa, qb, sbr, 1)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


def test_ones_scales_reduce_to_plain_fp8_gemm(orc):
    rng = np.random.default_rng(2)
    M, N, K = 64, 300, 512
    qa = rng.integers(0, 256, (M, K)).astype(np.uint8)
    qb = rng.integers(0, 256, (N, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    qb[(qb & 0x7F) == 0x7F] = 0x7E
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones(((N + 127) // 128, K // 128), np.float32)
    out = orc.gemm_blockscaled(qa, sa, qb, sb, 0)
    dA, dB = _dec_torch(qa), _dec_torch(qb)
    acc = np.zeros((M, N), np.float32)
    for kb in range(K // 128):
        P = dA[:, kb * 128:(kb + 1) * 128] @ dB[:, kb * 128:(kb + 1) * 128].T  # exact in double
        acc = (acc + P.astype(np.float32)).astype(np.float32)
    assert np.array_equal(out, acc)


def test_lossless_inputs_give_exact_gemm(orc):
    rng = np.random.default_rng(9)
    M, N, K = 32, 256, 384
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    ca = rng.choice(finite, (M, K))
    cb = rng.choice(finite, (N, K))
    ca[:, ::128] = 0x7E  # every 1x128 tile holds +448
    cb[::128, ::128] = 0xFE  # every 128x128 block holds -448
    ja = rng.integers(-6, 6, (M, K // 128))
    jb = rng.integers(-12, -4, (N // 128, K // 128))
    va = _dec_torch(ca) * np.exp2(np.repeat(ja, 128, axis=1))
    vb = _dec_torch(cb) * np.exp2(np.repeat(np.repeat(jb, 128, axis=0), 128, axis=1))
    ab = (va.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bb = (vb.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(synth.bf16_to_f32(ab), va.astype(np.float32))
    qa, sa = orc.quant_1x128_rows(ab)
    qb, sb = orc.quant_128x128(bb)
    assert np.array_equal(qa, ca) and np.array_equal(qb, cb)
    assert np.array_equal(sa, np.exp2(ja.T).astype(np.float32))
    assert np.array_equal(sb, np.exp2(jb).astype(np.float32))
    out = orc.gemm_blockscaled(qa, sa, qb, sb, 0).astype(np.float64)
    exact = va @ vb.T
    # three chunk partials each rounded once to FP32 and accumulated in FP32
    tol = 4 * 2.0 ** -24 * (np.abs(va) @ np.abs(vb).T)
    assert np.all(np.abs(out - exact) <= tol)


def test_dgrad_lossless_inputs_give_exact_product(orc):
    """dX = dY W from dY's 1x128 codes and the transposed 128x128 weight codes: with
    lossless inputs it is the exact double product (a transposed operand or scale grid
    would not be)."""
    rng = np.random.default_rng(10)
    T, Cout, Cin = 16, 256, 384
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    cy = rng.choice(finite, (T, Cout))
    cw = rng.choice(finite, (Cout, Cin))
    cy[:, ::128] = 0x7E
    cw[::128, ::128] = 0xFE
    jy = rng.integers(-6, 6, (T, Cout // 128))
    jw = rng.integers(-12, -4, (Cout // 128, Cin // 128))
    vy = _dec_torch(cy) * np.exp2(np.repeat(jy, 128, axis=1))
    vw = _dec_torch(cw) * np.exp2(np.repeat(np.repeat(jw, 128, axis=0), 128, axis=1))
    yb = (vy.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    wb = (vw.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qy, sy = orc.quant_1x128_rows(yb)
    _, _, qwt, swt = orc.quant_128x128_t(wb)
    out = orc.gemm_blockscaled(qy, sy, qwt, swt, 0).astype(np.float64)
    exact = vy @ vw
    tol = 4 * 2.0 ** -24 * (np.abs(vy) @ np.abs(vw))
    assert np.all(np.abs(out - exact) <= tol)


def test_row_subset_matches_full(orc):
    qa, sa, qb, sb, _ = _tiny_quantised(orc, M=20, N=200, K=256)
    full = orc.gemm_blockscaled(qa, sa, qb, sb, 0)
    rows = np.array([19, 0, 7, 7, 3])
    sub = orc.gemm_blockscaled(qa, sa, qb, sb, 0, rows=rows)
    assert np.array_equal(sub, full[rows])


def test_grouped_equals_per_expert(orc):
    rng = np.random.default_rng(4)
    G, N, K = 4, 256, 256
    offs = np.array([0, 5, 5, 140, 150])
    M = offs[-1]
    a = (rng.standard_normal((M, K))).astype(np.float32)
    ab = (a.view(np.uint32) >> 16).astype(np.uint16)
    qa, sa = orc.quant_1x128_rows(ab)
    qb = np.empty((G, N, K), np.uint8)
    sb = np.empty((G, 2, 2), np.float32)
    for e in range(G):
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        qb[e], sb[e] = orc.quant_128x128((w.view(np.uint32) >> 16).astype(np.uint16))
    out = orc.grouped_gemm(qa, sa, qb, sb, offs)
    for e in range(G):
        rows = np.arange(offs[e], offs[e + 1])
        if rows.size:
            ref = orc.gemm_blockscaled(qa, sa, qb[e], sb[e], 0, rows=rows)
            assert np.array_equal(out[rows], ref)
