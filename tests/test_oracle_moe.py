"""Pins of the oracle's MoE chain (V3 report §2 DeepSeekMoE, §4 aux-loss-free routing):
routing logits, top-k selection and gates, grouping, SwiGLU + 1x128 quantisation, combine.

Each is checked against something other than itself: the exact rational value of the
logits with an error bound, numpy's double product, exactly representable cases, a
brute-force ranking in numpy, the grouping invariants, and closed forms of SwiGLU."""
import numpy as np
import torch

import synth


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_route_logits_match_exact_rational_sum(orc):
    """The double logits against the exact value of the dot product (Python
    fractions over the exact BF16 and FP32 inputs): within D * 2^-53 * sum|u c|."""
    from fractions import Fraction
    rng = np.random.default_rng(1)
    T, D, E = 3, 96, 5
    xb = _bf16(rng.standard_normal((T, D)))
    c = (rng.standard_normal((E, D)) / np.sqrt(D)).astype(np.float32)
    l = orc.route_logits(xb, c)
    assert l.dtype == np.float64
    u = synth.bf16_to_f32(xb)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(u[t, k])) * Fraction(float(c[e, k])) for k in range(D))
            mag = sum(abs(float(u[t, k]) * float(c[e, k])) for k in range(D))
            assert abs(Fraction(float(l[t, e])) - exact) <= Fraction(D * mag) * Fraction(2) ** -53


def test_route_logits_against_numpy_double_product(orc):
    rng = np.random.default_rng(11)
    T, D, E = 24, 700, 40
    xb = _bf16(rng.standard_normal((T, D)))
    c = (rng.standard_normal((E, D)) / np.sqrt(D)).astype(np.float32)
    l = orc.route_logits(xb, c)
    u = synth.bf16_to_f32(xb).astype(np.float64)
    ref = u @ c.astype(np.float64).T
    bound = 2 * D * 2.0 ** -53 * (np.abs(u) @ np.abs(c.astype(np.float64)).T)
    assert np.all(np.abs(l - ref) <= bound)
    # a transposed or shifted operand would be far off
    assert not np.allclose(l[:, 1:], ref[:, :-1], atol=1e-3)


def test_route_logits_exact_when_every_partial_sum_is_representable(orc):
    rng = np.random.default_rng(2)
    T, D, E = 8, 256, 16
    u = rng.integers(-8, 9, (T, D)).astype(np.float32)      # small integers: exact in BF16
    c = (rng.integers(-16, 17, (E, D)) / 64.0).astype(np.float32)
    l = orc.route_logits(_bf16(u), c)
    exact = u.astype(np.float64) @ c.astype(np.float64).T     # every partial sum exact in double
    assert np.array_equal(l, exact)


def test_route_select_matches_brute_force_ranking(orc):
    rng = np.random.default_rng(3)
    T, E, k = 64, 32, 5
    l = rng.standard_normal((T, E))
    b = (rng.standard_normal(E) * 0.5).astype(np.float32)
    sel, gate = orc.route_select(l, b, k)
    s = 1.0 / (1.0 + np.exp(-l))
    key = s + b.astype(np.float64)
    for t in range(T):
        order = np.argsort(-key[t], kind="stable")[:k]      # stable: lower index first on ties
        assert np.array_equal(sel[t], np.sort(order))
        ch = np.sort(order)
        assert np.array_equal(gate[t], (s[t, ch] / s[t, ch].sum()).astype(np.float32))
    assert np.allclose(gate.sum(axis=1), 1.0, atol=1e-6)
    # the gates of a given selection follow the same rule
    assert np.array_equal(orc.route_gates(l, sel), gate)
    other = np.sort(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]), axis=1).astype(np.int32)
    s_o = np.take_along_axis(s, other, axis=1)
    assert np.array_equal(orc.route_gates(l, other), (s_o / s_o.sum(axis=1, keepdims=True)).astype(np.float32))


def test_route_select_ties_go_to_the_lower_index(orc):
    l = np.zeros((2, 6))
    b = np.array([0.1, 0.3, 0.3, 0.3, 0.0, 0.3], np.float32)
    sel, gate = orc.route_select(l, b, 2)
    assert sel.tolist() == [[1, 2], [1, 2]]
    assert np.allclose(gate, 0.5)
    sel, _ = orc.route_select(l, b, 4)
    assert sel.tolist()[0] == [1, 2, 3, 5]


def test_route_permute_groups_by_expert_then_token(orc):
    rng = np.random.default_rng(4)
    T, E, k = 50, 12, 3
    sel = np.sort(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]), axis=1).astype(np.int32)
    offs, tor, row_of = orc.route_permute(sel, E)
    counts = np.bincount(sel.reshape(-1), minlength=E)
    assert offs[0] == 0 and np.array_equal(np.diff(offs), counts)
    for e in range(E):
        toks = tor[offs[e]:offs[e + 1]]
        assert np.array_equal(toks, np.sort(np.nonzero((sel == e).any(axis=1))[0]))
    for t in range(T):
        for j in range(k):
            r = row_of[t, j]
            assert tor[r] == t
            assert np.searchsorted(offs, r, side="right") - 1 == sel[t, j]


def test_swiglu_quant_closed_forms_and_bound(orc):
    rng = np.random.default_rng(5)
    R, Nh = 6, 256
    acc = (rng.standard_normal((R, 2 * Nh)) * 3).astype(np.float32)
    acc[0, :128] = 0.0                          # g = 0 -> h = 0: zero tile, scale 1
    acc[1, :128] = 40.0                         # sigmoid(40) = 1 in double to 1e-17: h = 40 u
    q, s = orc.swiglu_quant(acc)
    assert s[0, 0] == 1.0 and np.all((q[0, :128] & 0x7F) == 0)
    g = acc[:, :Nh].astype(np.float64)
    u = acc[:, Nh:].astype(np.float64)
    h = g / (1.0 + np.exp(-g)) * u
    h32 = h.astype(np.float32)
    assert np.array_equal(h32[1, :128], (40.0 * u[1, :128]).astype(np.float32))
    for kb in range(Nh // 128):
        amax = np.abs(h32[:, kb * 128:(kb + 1) * 128]).max(axis=1)
        exp_s = np.where(amax == 0, np.float32(1), (amax / np.float32(448)).astype(np.float32))
        assert np.array_equal(s[kb], exp_s)
    dq = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    sc = np.repeat(s.T.astype(np.float64), 128, axis=1)
    err = np.abs(dq * sc - h)
    # E4M3 half-step: 2^-4 relative in the normal range, 2^-10 * scale below it
    assert np.all(err <= np.maximum(np.abs(h) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-6))


def test_combine_is_the_gate_weighted_sum(orc):
    rng = np.random.default_rng(6)
    R, N, T, k = 40, 96, 10, 4
    Y = _bf16(rng.standard_normal((R, N)))
    row_of = np.stack([rng.choice(R, k, replace=False) for _ in range(T)]).astype(np.int32)
    gate = rng.random((T, k)).astype(np.float32)
    gate /= gate.sum(axis=1, keepdims=True)
    out = synth.bf16_to_f32(orc.moe_combine(Y, row_of, gate)).astype(np.float64)
    y = synth.bf16_to_f32(Y).astype(np.float64)
    exact = np.einsum("tk,tkn->tn", gate.astype(np.float64), y[row_of])
    bound = np.abs(exact) * 2.0 ** -8 + k * 2.0 ** -23 * np.einsum("tk,tkn->tn", gate, np.abs(y[row_of]))
    assert np.all(np.abs(out - exact) <= bound)
