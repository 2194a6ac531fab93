"""GPU parity of the routed-expert chain (V3 report §2 DeepSeekMoE, §4 aux-loss-free
routing) against the oracle, through the C ABI.

- Routing.  The oracle forms the affinity logits in double (exact products, a double sum),
  independent of any GPU summation order; the kernel forms them in FP32 with one fused
  multiply-add per term in increasing k.  The device logits must lie within the FP32
  error bound of that summation (u * sum_k |s_k| over the exact prefix sums s_k, u = 2^-24)
  of the exact ones, and every logit within the order-free bound gamma_D * sum |u c|.
  Through the sigmoid (slope <= 1/4) that bounds each selection key.  A token whose
  chosen experts' keys clear its other experts' keys by more than these bounds has one
  correct selection: the device's must equal the oracle's.  For the few others (counted
  and reported) the device's selection must be a valid top-k within the bounds.  The
  grouping (offsets, rows, row_of) must be the oracle's grouping of the device's
  selection, bit for bit; the gates the oracle's gates of that selection, within the
  propagated logit bound plus two FP32 ulps.
- Gather + quantise: bit-exact.
- Up projection with fused SwiGLU + 1x128 quantisation: the oracle forms h in double from
  its own FP32 GEMM results, the kernel in FP32 from the tensor-core partials, so h differs
  in its last bits.  Scales agree to 1e-5 relative; a code may differ only where h / s lies
  next to a rounding boundary: by one step, in at most 1e-3 of the codes.
- Down projection and combine: the GEMM tolerance (tests/gpu_util.py); the oracle chain
  runs on the device's (validated) routing.
Sizes: small ragged configurations checked in full, and the 4096-token, 256-expert layer
of workload 3 with the routing checked in full and the chain on sampled tokens.
"""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import assert_gemm_close, dev, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    import fp8_fine_grained_27_b300 as fb
    assert torch.cuda.is_available()
    return fb


def _router_inputs(T, D, E, seed):
    x = synth.fill_bf16(synth.NORMAL, synth.key(70, seed), (T, D), 1.0)
    cent = synth.fill_f32(synth.NORMAL, synth.key(71, seed), (E, D), 1.0 / np.sqrt(D))
    bias = synth.fill_f32(synth.NORMAL, synth.key(72, seed), (E,), 0.5)
    return x, cent, bias


def _cent_t(cent):
    """Centroids in the kernel's k-major layout [D, E] (device)."""
    return torch.from_numpy(np.ascontiguousarray(cent.T)).cuda()


U32 = 2.0 ** -24


def _apriori_bound(x, cent):
    """|FP32 dot product - exact| for any summation order: gamma_D * sum_k |u_k c_k|."""
    u = synth.bf16_to_f32(x).astype(np.float64)
    D = u.shape[1]
    return D * U32 / (1 - D * U32) * (np.abs(u) @ np.abs(cent.astype(np.float64)).T)


def _sequential_bound(x, cent, pairs):
    """|FP32 sum - exact| of a chain of fused multiply-adds in increasing k: at most
    u * sum_k |s_k| over the partial sums, taken here as the exact prefix sums s_k with
    a relative allowance of 2^-20 for their own rounding.  pairs: (t, e) index arrays."""
    ts, es = pairs
    out = np.empty(ts.size)
    u = synth.bf16_to_f32(x).astype(np.float64)
    c = cent.astype(np.float64)
    for i in range(0, ts.size, 256):
        p = u[ts[i:i + 256]] * c[es[i:i + 256]]
        np.cumsum(p, axis=1, out=p)
        out[i:i + 256] = U32 * (1 + 2.0 ** -20) * np.abs(p).sum(axis=1)
    return out


def _decided(key, delta, k):
    """Tokens whose top-k by `key` stays the top-k for every key within +-delta."""
    if key.shape[1] <= k:
        return np.ones(key.shape[0], bool)
    idx = np.argsort(-key, axis=1, kind="stable")
    lo = np.take_along_axis(key - delta, idx[:, :k], 1).min(axis=1)
    hi = np.take_along_axis(key + delta, idx[:, k:], 1).max(axis=1)
    return lo > hi


def _check_route(fb, orc, x, cent, bias, k, r=None):
    """Check a device routing (run here unless given) against the oracle; return the
    oracle's view of it: (exact logits, selection, gates, offsets, token_of_row, row_of),
    the last four being the oracle's grouping and gates of the device's selection."""
    T, E = x.shape[0], cent.shape[0]
    if r is None:
        r = fb.moe_route(dev(x), _cent_t(cent), torch.from_numpy(bias).cuda(), k)
        torch.cuda.synchronize()
    ol = orc.route_logits(x, cent)
    gl = r["logits"].cpu().numpy().astype(np.float64)
    bound = _apriori_bound(x, cent)
    assert np.all(np.abs(gl - ol) <= bound), "logits outside the order-free FP32 bound"
    key = 1.0 / (1.0 + np.exp(-ol)) + bias.astype(np.float64)[None, :]
    delta = bound / 4  # the sigmoid's slope is at most 1/4
    decided = _decided(key, delta, k)
    if not decided.all():
        # tighten the bound of the experts that keep a token undecided
        und = np.nonzero(~decided)[0]
        idx = np.argsort(-key[und], axis=1, kind="stable")
        lo = np.take_along_axis(key[und] - delta[und], idx[:, :k], 1).min(axis=1)
        hi = np.take_along_axis(key[und] + delta[und], idx[:, k:], 1).max(axis=1)
        near = (key[und] - delta[und] <= hi[:, None]) & (key[und] + delta[und] >= lo[:, None])
        ti, ei = np.nonzero(near)
        tb = _sequential_bound(x, cent, (und[ti], ei))
        assert np.all(np.abs(gl[und[ti], ei] - ol[und[ti], ei]) <= tb), "logits outside the sequential FP32 bound"
        delta[und[ti], ei] = tb / 4
        decided = _decided(key, delta, k)
    gsel = r["expert_idx"].cpu().numpy()
    osel, _ = orc.route_select(ol, bias, k)
    assert np.array_equal(gsel[decided], osel[decided]), "a decided token's selection differs"
    excluded = np.nonzero(~decided)[0]
    for t in excluded:
        ch = gsel[t]
        assert len(set(ch.tolist())) == k and np.all(np.diff(ch) > 0)
        rest = np.setdiff1d(np.arange(E), ch)
        assert (key[t, ch] + delta[t, ch]).min() >= (key[t, rest] - delta[t, rest]).max(), \
            f"token {t}: not a top-{k} within the bounds"
    print(f"routing: {excluded.size} of {T} tokens within the FP32 bounds of a near-tie "
          f"(selection checked for validity only)")
    assert excluded.size <= max(2, T // 256)
    ogate = orc.route_gates(ol, gsel)
    g = r["gate"].cpu().numpy().astype(np.float64)
    s = np.take_along_axis(1.0 / (1.0 + np.exp(-ol)), gsel.astype(np.int64), 1)
    dmax = np.take_along_axis(delta, gsel.astype(np.int64), 1).max(axis=1, keepdims=True)
    gbound = dmax * (1 + k) / s.sum(axis=1, keepdims=True) + 2 * U32
    assert np.all(np.abs(g - ogate) <= gbound), "gates outside the propagated bound"
    offs, tor, row_of = orc.route_permute(gsel, E)
    assert np.array_equal(r["offsets"].cpu().numpy(), offs)
    assert np.array_equal(r["token_of_row"].cpu().numpy(), tor)
    assert np.array_equal(r["row_of"].cpu().numpy(), row_of)
    return r, (ol, gsel, ogate, offs, tor, row_of)


@pytest.mark.parametrize("T,D,E,k", [(300, 512, 40, 6), (64, 256, 64, 1), (129, 128, 300, 16), (1, 32, 8, 8)])
def test_route_small(fb, orc, T, D, E, k):
    x, cent, bias = _router_inputs(T, D, E, seed=T + E)
    _check_route(fb, orc, x, cent, bias, k)


def test_route_empty_batch(fb):
    E = 16
    r = fb.moe_route(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"),
                     torch.zeros((64, E), device="cuda"), torch.zeros(E, device="cuda"), 2)
    torch.cuda.synchronize()
    assert r["offsets"].cpu().numpy().tolist() == [0] * (E + 1)


def test_route_full_layer(fb, orc):
    """The router of workload 3: 4096 tokens, D 7168, 256 experts, top-8."""
    tok = synth.moe_tokens()
    cent, bias = synth.moe_router()
    _check_route(fb, orc, tok, cent, bias, 8)


def test_gather_quant_bit_exact(fb, orc):
    T, K = 200, 512
    x = synth.fill_bf16(synth.OUTLIER, synth.key(73, 0), (T, K), 1.0, 0.02, 30.0, k2=synth.key(74, 0))
    rng = np.random.default_rng(0)
    row_map = rng.integers(0, T, 700).astype(np.int32)
    row_map[[5, 77, 699]] = [-1, T, 1 << 30]  # outside the source: quantised as zeros
    q, s = fb.quant_1x128_gather(dev(x), torch.from_numpy(row_map).cuda())
    torch.cuda.synchronize()
    src = np.where(((row_map >= 0) & (row_map < T))[:, None], x[np.clip(row_map, 0, T - 1)], 0).astype(np.uint16)
    oq, os_ = orc.quant_1x128_rows(src)
    assert np.array_equal(q.cpu().numpy(), oq) and np.array_equal(s.cpu().numpy(), os_)


def _compare_swiglu_codes(q, s, oq, os_, what):
    assert np.all(np.abs(s.astype(np.float64) / os_.astype(np.float64) - 1.0) <= 1e-5), f"{what}: scales"
    diff = q != oq
    n = int(diff.sum())
    assert n <= max(2, 1e-3 * q.size), f"{what}: {n} of {q.size} codes differ"
    if n:
        dq = torch.from_numpy(q[diff]).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        dr = torch.from_numpy(oq[diff]).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        # adjacent codes of the same sign: one E4M3 step (2^-3 relative, 2^-9 absolute below 2^-6)
        assert np.all(np.sign(dq) * np.sign(dr) >= 0), what
        step = np.maximum(np.abs(dr) * 2.0 ** -3, 2.0 ** -9)
        assert np.all(np.abs(dq - dr) <= step * (1 + 1e-9)), f"{what}: a code moved by more than one step"


def _quant_experts(fb, w_bits):
    """128x128 quantisation of G experts' weights [G, N, K] (device codes, scales)."""
    G, N, K = w_bits.shape
    q, s = fb.quant_128x128(dev(w_bits.reshape(G * N, K)))
    return q.view(G, N, K), s.view(G, N // 128, K // 128)


def test_swiglu_gemm_small_skewed(fb, orc):
    G, Nh, K = 3, 256, 384
    sizes = [130, 0, 257]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M = int(offs[-1]) + 5  # rows past offs[G] stay untouched
    a = synth.fill_bf16(synth.OUTLIER, synth.key(75, 0), (M, K), 1.0, 0.01, 20.0, k2=synth.key(76, 0))
    w = synth.fill_bf16(synth.NORMAL, synth.key(77, 0), (G, 2 * Nh, K), 0.05)
    qa, sa = fb.quant_1x128(dev(a))
    qb, sb = _quant_experts(fb, w)
    Q = torch.full((M, Nh), 0x7F, dtype=torch.uint8, device="cuda")
    S = torch.full((Nh // 128, M), -1.0, dtype=torch.float32, device="cuda")
    fb.grouped_gemm_moe_swiglu(qa, sa, qb, sb, torch.from_numpy(offs).cuda(), Q=Q, s=S)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    q, s = Q.cpu().numpy(), S.cpu().numpy()
    oqa, osa = orc.quant_1x128_rows(a)
    oqb = [orc.quant_128x128(w[e]) for e in range(G)]
    rows = np.arange(offs[-1])
    acc = orc.grouped_gemm(oqa, osa, np.stack([b[0] for b in oqb]), np.stack([b[1] for b in oqb]), offs, rows=rows)
    oq, os_ = orc.swiglu_quant(acc)
    _compare_swiglu_codes(q[:offs[-1]], s[:, :offs[-1]], oq, os_, "swiglu small")
    assert np.all(q[offs[-1]:] == 0x7F) and np.all(s[:, offs[-1]:] == -1.0)


def _gpu_chain(fb, x, cent, bias, k, qwu, swu, qwd, swd):
    """The whole layer on the device; returns every intermediate."""
    T = x.shape[0]
    r = fb.moe_route(x, cent, bias, k)
    qa, sa = fb.quant_1x128_gather(x, r["token_of_row"])
    h, sh = fb.grouped_gemm_moe_swiglu(qa, sa, qwu, swu, r["offsets"])
    Y = fb.grouped_gemm_moe(h, sh, qwd, swd, r["offsets"])
    out = fb.moe_combine(Y, r["row_of"], r["gate"])
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    assert out.shape[0] == T
    return r, h, sh, Y, out


def test_chain_small(fb, orc):
    T, D, E, k, Nh = 256, 512, 16, 4, 256
    x, cent, bias = _router_inputs(T, D, E, seed=9)
    wu = synth.fill_bf16(synth.NORMAL, synth.key(78, 0), (E, 2 * Nh, D), 0.05)
    wd = synth.fill_bf16(synth.NORMAL, synth.key(79, 0), (E, D, Nh), 0.05)
    qwu, swu = _quant_experts(fb, wu)
    qwd, swd = _quant_experts(fb, wd)
    r, h, sh, Y, out = _gpu_chain(fb, dev(x), _cent_t(cent), torch.from_numpy(bias).cuda(), k,
                                  qwu, swu, qwd, swd)
    _, (ol, osel, ogate, offs, tor, row_of) = _check_route(fb, orc, x, cent, bias, k, r=r)
    oqa, osa = orc.quant_1x128_rows(x[tor])
    ou = [orc.quant_128x128(wu[e]) for e in range(E)]
    od = [orc.quant_128x128(wd[e]) for e in range(E)]
    acc = orc.grouped_gemm(oqa, osa, np.stack([u[0] for u in ou]), np.stack([u[1] for u in ou]), offs)
    oh, osh = orc.swiglu_quant(acc)
    _compare_swiglu_codes(h.cpu().numpy(), sh.cpu().numpy(), oh, osh, "chain h")
    oY = orc.bf16_round(orc.grouped_gemm(oh, osh, np.stack([d[0] for d in od]), np.stack([d[1] for d in od]), offs))
    assert_gemm_close(host_bits(Y), oY, "chain down")
    oout = orc.moe_combine(oY, row_of, ogate)
    assert_gemm_close(host_bits(out), oout, "chain combine")


def test_chain_full_layer_sampled_tokens(fb, orc):
    """Workload 3's layer: 4096 tokens, 256 experts (up 2 x 2048 x 7168, down 7168 x 2048),
    top-8; the routing in full, the chain on 4 sampled tokens (32 expert rows)."""
    E, k, D, Nh = 256, 8, 7168, 2048
    tok = synth.moe_tokens()
    cent, bias = synth.moe_router()
    qwu = torch.empty((E, 2 * Nh, D), dtype=torch.uint8, device="cuda")
    swu = torch.empty((E, 2 * Nh // 128, D // 128), dtype=torch.float32, device="cuda")
    qwd = torch.empty((E, D, Nh), dtype=torch.uint8, device="cuda")
    swd = torch.empty((E, D // 128, Nh // 128), dtype=torch.float32, device="cuda")
    for e0 in range(0, E, 16):
        wu = dev(synth.moe_weights("up", e0, e0 + 16))
        fb.quant_128x128(wu.view(-1, D), q=qwu[e0:e0 + 16].view(-1, D), s=swu[e0:e0 + 16].view(-1, D // 128))
        wd = dev(synth.moe_weights("down", e0, e0 + 16))
        fb.quant_128x128(wd.view(-1, Nh), q=qwd[e0:e0 + 16].view(-1, Nh), s=swd[e0:e0 + 16].view(-1, Nh // 128))
        del wu, wd
    r, h, sh, Y, out = _gpu_chain(fb, dev(tok), _cent_t(cent), torch.from_numpy(bias).cuda(), k,
                                  qwu, swu, qwd, swd)
    _, (ol, osel, ogate, offs, tor, row_of) = _check_route(fb, orc, tok, cent, bias, k, r=r)
    toks = np.array([0, 1234, 2048, 4095])
    rows = row_of[toks].reshape(-1)
    oqa, osa = orc.quant_1x128_rows(tok[tor[rows]])
    gh, gsh = h.cpu().numpy()[rows], sh.cpu().numpy()[:, rows]
    Yrows = np.empty((rows.size, D), np.uint16)
    cache = {}
    for i, row in enumerate(rows):
        e = int(np.searchsorted(offs, row, side="right") - 1)
        if e not in cache:
            cache[e] = (orc.quant_128x128(synth.moe_weights("up", e, e + 1)[0]),
                        orc.quant_128x128(synth.moe_weights("down", e, e + 1)[0]))
        (qu, su), (qd, sd) = cache[e]
        acc = orc.gemm_blockscaled(oqa[i:i + 1], osa[:, i:i + 1], qu, su, 0)
        oh, osh = orc.swiglu_quant(acc)
        _compare_swiglu_codes(gh[i:i + 1], gsh[:, i:i + 1], oh, osh, f"h row {row}")
        Yrows[i] = orc.bf16_round(orc.gemm_blockscaled(oh, osh, qd, sd, 0))[0]
    assert_gemm_close(host_bits(Y[torch.from_numpy(rows).cuda()]), Yrows, "full down rows")
    local = np.arange(rows.size, dtype=np.int32).reshape(toks.size, k)
    oout = orc.moe_combine(Yrows, local, ogate[toks])
    assert_gemm_close(host_bits(out[torch.from_numpy(toks).cuda()]), oout, "full combine")
