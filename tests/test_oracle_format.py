"""Pins for the oracle's E4M3 decode/encode and BF16 rounding.

The oracle's encoder is checked against (a) hand-worked values from the
format definition (tests/golden/e4m3_closed_forms.txt), (b) torch's own
float8_e4m3fn conversion, an independent implementation, over every FP32 bit
pattern, and (c) a brute-force nearest-value search over all finite codes.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_closed_forms.txt")


def _parse_value(tok):
    if tok.lstrip("-").startswith("0x"):
        return float.fromhex(tok)
    return float(tok)


def test_decode_all_codes_against_torch(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = orc.decode_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], mine[~nan])


def test_decode_closed_forms(orc):
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0xFE) == -448.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert orc.e4m3_decode(0x08) == 2.0 ** -6
    assert orc.e4m3_decode(0x38) == 1.0
    assert orc.e4m3_decode(0x80) == 0.0 and np.signbit(orc.e4m3_decode(0x80))
    mags = orc.decode_table()[:127]
    assert np.all(np.diff(mags) > 0), "codes 0..126 must be increasing magnitudes"


def test_encode_golden_closed_forms(orc):
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            val, code = line.split()[:2]
            y = np.float32(_parse_value(val))
            assert orc.e4m3_encode(y) == int(code, 16), (val, code)
            n += 1
    assert n >= 20


def test_encode_nan(orc):
    assert orc.e4m3_encode(float("nan")) == 0x7F


def test_encode_exhaustive_against_torch(orc):
    """Every FP32 bit pattern.  torch's conversion rounds to nearest even but
    turns |y| >= 464 into NaN instead of saturating, so that band is checked
    against the saturation rule instead."""
    chunk = 1 << 26
    for lo in range(0, 1 << 32, chunk):
        pat = np.arange(lo, lo + chunk, dtype=np.uint64).astype(np.uint32)
        x = pat.view(np.float32)
        mine = orc.e4m3_encode_patterns(lo, chunk)
        ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        ax = np.abs(x)
        nan = np.isnan(x)
        sat = (ax >= 448.0) & ~nan
        normal = ~nan & ~sat
        bad = np.nonzero(mine[normal] != ref[normal])[0]
        assert bad.size == 0, (lo, x[normal][bad[:5]], mine[normal][bad[:5]], ref[normal][bad[:5]])
        expect_sat = np.where(np.signbit(x[sat]), 0xFE, 0x7E).astype(np.uint8)
        assert np.array_equal(mine[sat], expect_sat)
        expect_nan = np.where(np.signbit(x[nan]), 0xFF, 0x7F).astype(np.uint8)
        assert np.array_equal(mine[nan], expect_nan)


def _brute_nearest(y):
    """Nearest finite E4M3 code by scanning all 254 finite codes (decoded by
    torch), ties to the even code; exact in double for 2^-40 <= |y| < 448."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    y = y.astype(np.float64)
    d = np.abs(y[:, None] - vals[None, :])
    # a code of the wrong sign is never nearer than the same-signed one; only
    # keep same-signed codes so that +0/-0 are separated by sign.
    same = (np.signbit(vals)[None, :] == np.signbit(y)[:, None])
    d = np.where(same, d, np.inf)
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    even = (codes % 2 == 0)[None, :]
    pick_even = cand & even
    has_even = pick_even.any(axis=1)
    idx = np.where(has_even, np.argmax(pick_even, axis=1), np.argmax(cand, axis=1))
    return codes[idx]


def test_encode_against_brute_force_nearest(orc):
    rng = np.random.default_rng(1234)
    # random magnitudes over the whole range, every midpoint, and 1-ulp neighbours
    r = np.exp2(rng.uniform(-40, np.log2(447.9), 200_000)).astype(np.float32)
    mags = orc.decode_table()[:127]
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                           mags[1:].astype(np.float32)])
    y = np.concatenate([r, near]).astype(np.float32)
    y = np.concatenate([y, -y])
    y = y[np.abs(y) < 448]
    for part in np.array_split(y, 40):
        assert np.array_equal(orc.e4m3_encode_array(part), _brute_nearest(part))


def test_bf16_rne(orc):
    # ties to even at the 16-bit boundary, and ordinary rounding
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -3.0], np.float32)
    y = orc.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, ref)
    rng = np.random.default_rng(7)
    z = (rng.standard_normal(1_000_000) * np.exp2(rng.uniform(-30, 30, 1_000_000))).astype(np.float32)
    ref = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_round(z), ref)
