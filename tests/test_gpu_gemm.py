"""GPU parity: block-scaled GEMM and grouped MoE GEMM against the oracle,
through the C ABI, within the tolerance stated in tests/gpu_util.py.

Each side quantises the same seeded BF16 inputs with its own quantiser (the
quantisers are bit-exact, see test_gpu_quant.py) and multiplies its own codes.
Small cases span several tiles and ragged edges and are checked in full;
the full-size workloads are checked on seeded row samples (the tolerance is
per row, so a row sample checks it exactly for those rows)."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import (assert_canaries_untouched, assert_gemm_close, canary_output, dev, host_bits,
                            sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    import fp8_fine_grained_27_b300 as fb
    assert torch.cuda.is_available()
    return fb


@pytest.fixture(params=[0, 128, 192, 256], ids=["auto", "bn128", "bn192", "bn256"])
def tile_n(request, fb):
    fb.set_gemm_tile_n(request.param)
    yield request.param
    fb.set_gemm_tile_n(0)


def _dense(fb, orc, a_bits, w_bits, out_dtype=torch.bfloat16, rows=None, what=""):
    qa, sa = fb.quant_1x128(dev(a_bits))
    qb, sb = fb.quant_128x128(dev(w_bits))
    C, buf, rs, cs = canary_output(a_bits.shape[0], w_bits.shape[0], out_dtype)
    fb.gemm_blockscaled(qa, sa, qb, sb, 0, C=C)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    assert_canaries_untouched(buf, rs, cs, what)
    oqa, osa = orc.quant_1x128_rows(a_bits)
    oqb, osb = orc.quant_128x128(w_bits)
    if rows is None:
        rows = np.arange(a_bits.shape[0])
    ref = orc.gemm_blockscaled(oqa, osa, oqb, osb, 0, rows=rows)
    got = host_bits(C[torch.from_numpy(rows).cuda()])
    if out_dtype == torch.bfloat16:
        ref = orc.bf16_round(ref)
    return assert_gemm_close(got, ref, what)


def test_tiny_workload(fb, orc):
    d = synth.tiny()
    _dense(fb, orc, d["A"], d["B"], what="tiny")


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (300, 392, 640), (129, 72, 256), (257, 520, 384), (64, 128, 1024)])
def test_ragged_shapes(fb, orc, tile_n, M, N, K):
    a = synth.fill_bf16(synth.OUTLIER, synth.key(80, M), (M, K), 1.0, 0.01, 50.0, k2=synth.key(81, M))
    w = synth.fill_bf16(synth.NORMAL, synth.key(82, N), (N, K), 0.02)
    _dense(fb, orc, a, w, what=f"{M}x{N}x{K}")
    _dense(fb, orc, a, w, out_dtype=torch.float32, what=f"{M}x{N}x{K} fp32")


def test_raster_groups_with_a_partial_last_group(fb, orc, tile_n):
    """40 M tiles at a K whose raster group is 32 tiles: one full group, a
    partial group of 8, a ragged last tile, and a ragged last N tile.  Two rows
    of every M tile (its first and last) are checked, plus a seeded sample."""
    M, N, K = 40 * 128 - 37, 520, 256
    a = synth.fill_bf16(synth.OUTLIER, synth.key(90, M), (M, K), 1.0, 0.01, 50.0, k2=synth.key(91, M))
    w = synth.fill_bf16(synth.NORMAL, synth.key(92, N), (N, K), 0.02)
    must = [r for t in range(40) for r in (t * 128, min(t * 128 + 127, M - 1))]
    rows = sample_rows(M, 64, seed=10, must=must)
    _dense(fb, orc, a, w, rows=rows, what="raster groups")
    _dense(fb, orc, a, w, out_dtype=torch.float32, rows=rows, what="raster groups fp32")


def test_mla_full(fb, orc, tile_n):
    """Both MLA down-projections, every output checked."""
    d = synth.mla()
    _dense(fb, orc, d["A"], d["Wq"], what="mla q")
    _dense(fb, orc, d["A"], d["Wkv"], what="mla kv")


FFN_ROWS = sample_rows(16384, 512, seed=5, must=(0, 127, 128, 255, 256, 16255, 16256, 16383))


@pytest.fixture(scope="module")
def ffn_case(orc):
    """The FFN inputs and the oracle's BF16 result on 512 seeded rows (computed
    once for every tile width)."""
    d = synth.ffn()
    oqa, osa = orc.quant_1x128_rows(d["A"])
    oqb, osb = orc.quant_128x128(d["B"])
    ref = orc.bf16_round(orc.gemm_blockscaled(oqa, osa, oqb, osb, 0, rows=FFN_ROWS))
    return d, ref


def test_ffn_sampled_rows(fb, tile_n, ffn_case):
    """The full 16384x18432x7168 FFN GEMM at every tile width, checked on 512
    seeded rows (including the first and last rows of the first, second and
    last M tiles, and both sides of a 256-row pair-tile boundary)."""
    d, ref = ffn_case
    qa, sa = fb.quant_1x128(dev(d["A"]))
    qb, sb = fb.quant_128x128(dev(d["B"]))
    C, buf, rs, cs = canary_output(16384, 18432, torch.bfloat16)
    fb.gemm_blockscaled(qa, sa, qb, sb, 0, C=C)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    assert_canaries_untouched(buf, rs, cs, "ffn")
    got = host_bits(C[torch.from_numpy(FFN_ROWS).cuda()])
    assert_gemm_close(got, ref, f"ffn tile_n={tile_n}")


def _dgrad(fb, orc, dY, W, rows=None, what=""):
    """dX = dY W: dY quantised 1x128 along its channels, W through the transposed block quantiser."""
    qdy, sdy = fb.quant_1x128(dev(dY))
    _, _, qwt, swt = fb.quant_128x128_t(dev(W), straight=False)
    C, buf, rs, cs = canary_output(dY.shape[0], W.shape[1], torch.bfloat16)
    fb.gemm_blockscaled(qdy, sdy, qwt, swt, 0, C=C)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    assert_canaries_untouched(buf, rs, cs, what)
    oqdy, osdy = orc.quant_1x128_rows(dY)
    _, _, oqwt, oswt = orc.quant_128x128_t(W)
    if rows is None:
        rows = np.arange(dY.shape[0])
    ref = orc.bf16_round(orc.gemm_blockscaled(oqdy, osdy, oqwt, oswt, 0, rows=rows))
    got = host_bits(C[torch.from_numpy(rows).cuda()])
    return assert_gemm_close(got, ref, what)


@pytest.mark.parametrize("T,Cout,Cin", [(200, 384, 384), (129, 256, 128), (1, 1536, 640)])
def test_dgrad_small(fb, orc, tile_n, T, Cout, Cin):
    d = synth.dgrad(T=T, Cout=Cout, Cin=Cin)
    _dgrad(fb, orc, d["dY"], d["W"], what=f"dgrad {T}x{Cin}x{Cout}")


def test_dgrad_full_size_sampled(fb, orc):
    d = synth.dgrad()
    rows = sample_rows(16384, 128, seed=7, must=(0, 127, 128, 16383))
    _dgrad(fb, orc, d["dY"], d["W"], rows=rows, what="dgrad")


def _wgrad(fb, orc, dY, X, rows=None, what=""):
    qdy, sdy = fb.quant_1x128(dev(dY), along=1)   # [Cout, T], [T/128, Cout]
    qx, sx = fb.quant_1x128(dev(X), along=1)      # [Cin, T],  [T/128, Cin]
    C, buf, rs, cs = canary_output(dY.shape[1], X.shape[1], torch.float32)
    fb.gemm_blockscaled(qdy, sdy, qx, sx, 1, C=C)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    assert_canaries_untouched(buf, rs, cs, what)
    oqdy, osdy = orc.quant_1x128_cols(dY)
    oqx, osx = orc.quant_1x128_cols(X)
    if rows is None:
        rows = np.arange(oqdy.shape[0])
    ref = orc.gemm_blockscaled(oqdy, osdy, oqx, osx, 1, rows=rows)
    got = host_bits(C[torch.from_numpy(rows).cuda()])
    return assert_gemm_close(got, ref, what)


def test_wgrad_small_full(fb, orc, tile_n):
    d = synth.wgrad(T=1024, Cout=256, Cin=392)
    _wgrad(fb, orc, d["dY"], d["X"], what="wgrad small")


@pytest.mark.parametrize("Cout,Cin,T", [(128, 8, 128), (384, 264, 384), (256, 136, 256), (200, 264, 256)])
def test_wgrad_ragged(fb, orc, tile_n, Cout, Cin, T):
    """Per-row B scales on output widths that end inside a tile (and, at Cout = 200, a last
    row tile of 72 rows, whose row scales are bulk-copied short)."""
    d = synth.wgrad(T=T, Cout=Cout, Cin=Cin)
    _wgrad(fb, orc, d["dY"], d["X"], what=f"wgrad {Cout}x{Cin}x{T}")


@pytest.mark.parametrize("layout", ["odd_ld", "offset"])
def test_wgrad_row_scales_global_path(fb, tile_n, layout):
    """A row-scale layout that cannot be bulk-copied into shared memory (a row pitch that is
    not a multiple of 4 floats, or a base 4 bytes off a 16-byte boundary) takes the
    global-load path; the result must be bit-identical to the staged path's."""
    d = synth.wgrad(T=1024, Cout=256, Cin=392)
    qdy, sdy = fb.quant_1x128(dev(d["dY"]), along=1)
    qx, sx = fb.quant_1x128(dev(d["X"]), along=1)
    C0 = torch.empty((256, 392), dtype=torch.float32, device="cuda")
    fb.gemm_blockscaled(qdy, sdy, qx, sx, 1, C=C0)
    nkb, M = sdy.shape
    if layout == "odd_ld":
        buf = torch.full((nkb, M + 1), float("nan"), dtype=torch.float32, device="cuda")
        s2 = buf[:, :M]
    else:
        buf = torch.full((nkb * (M + 4) + 1,), float("nan"), dtype=torch.float32, device="cuda")
        s2 = buf[1:].view(nkb, M + 4)[:, :M]
    s2.copy_(sdy)
    C1 = torch.full_like(C0, float("nan"))
    fb.gemm_blockscaled(qdy, s2, qx, sx, 1, C=C1)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    assert torch.equal(C0.view(torch.int32), C1.view(torch.int32)), f"{layout}: staged and global row scales differ"


def test_wgrad_full_size(fb, orc):
    """Workload 4 (dW = dY^T X, 2048 x 7168 from 16384 tokens, FP32 out): every output."""
    d = synth.wgrad()
    _wgrad(fb, orc, d["dY"], d["X"], what="wgrad")


def _split_vs_whole(fb, run, M, N, what):
    """run(C) into a canary-guarded FP32 output twice: with the last round of
    tiles shared out by K chunks (the default) and with whole tiles.  The two
    results must be bit-identical, and neither may write outside C."""
    outs = []
    for split in (True, False):
        fb.set_gemm_split_last_round(split)
        try:
            C, buf, rs, cs = canary_output(M, N, torch.float32)
            run(C)
            torch.cuda.synchronize()
            assert fb.get_device_error() == 0
            assert_canaries_untouched(buf, rs, cs, f"{what} split={split}")
            outs.append(C.clone())
        finally:
            fb.set_gemm_split_last_round(True)
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32)), f"{what}: split result differs"
    return outs[0]


@pytest.mark.parametrize("bn", [0, 128, 256])
def test_split_last_round_wgrad_full(fb, bn):
    """Workload 4 has 608 tiles of 128x192 (896 of 128x128, 448 of 128x256) on
    148 CTAs: its last round is shared out by K chunks, and the result must
    equal the whole-tile result bit for bit."""
    d = synth.wgrad()
    qdy, sdy = fb.quant_1x128(dev(d["dY"]), along=1)
    qx, sx = fb.quant_1x128(dev(d["X"]), along=1)
    fb.set_gemm_tile_n(bn)
    try:
        _split_vs_whole(fb, lambda C: fb.gemm_blockscaled(qdy, sdy, qx, sx, 1, C=C), 2048, 7168, f"wgrad bn={bn}")
    finally:
        fb.set_gemm_tile_n(0)


@pytest.mark.parametrize("bn", [0, 128, 256])
@pytest.mark.parametrize("mode", ["row_scales", "block_scales"])
def test_split_last_round_small(fb, orc, bn, mode):
    """160 (or 320) tiles and 3 K chunks: every CTA's run crosses tiles, so
    most tiles are split between two CTAs.  Bit-identical to whole tiles, and
    every output against the oracle."""
    if mode == "row_scales":
        d = synth.wgrad(T=384, Cout=2048, Cin=2560)
        qa, sa = fb.quant_1x128(dev(d["dY"]), along=1)
        qb, sb = fb.quant_1x128(dev(d["X"]), along=1)
        oqa, osa = orc.quant_1x128_cols(d["dY"])
        oqb, osb = orc.quant_1x128_cols(d["X"])
        M, N, bmode = 2048, 2560, 1
    else:
        a = synth.fill_bf16(synth.OUTLIER, synth.key(100, 0), (2560, 384), 1.0, 0.01, 50.0, k2=synth.key(101, 0))
        w = synth.fill_bf16(synth.NORMAL, synth.key(102, 0), (2048, 384), 0.02)
        qa, sa = fb.quant_1x128(dev(a))
        qb, sb = fb.quant_128x128(dev(w))
        oqa, osa = orc.quant_1x128_rows(a)
        oqb, osb = orc.quant_128x128(w)
        M, N, bmode = 2560, 2048, 0
    fb.set_gemm_tile_n(bn)
    try:
        got = _split_vs_whole(fb, lambda C: fb.gemm_blockscaled(qa, sa, qb, sb, bmode, C=C), M, N,
                              f"{mode} bn={bn}")
    finally:
        fb.set_gemm_tile_n(0)
    ref = orc.gemm_blockscaled(oqa, osa, oqb, osb, bmode)
    assert_gemm_close(host_bits(got), ref, f"split {mode} bn={bn}")


@pytest.mark.parametrize("workload,launches,bn", [("wgrad", 300, 0), ("wgrad", 200, 128), ("wgrad", 200, 256),
                                                  ("mla", 300, 0), ("ffn", 40, 0)])
def test_repeated_launches_are_bit_identical(fb, workload, launches, bn):
    """The same GEMM launched many times into a NaN-filled output gives the
    same bits every time.  A race between a partial buffer's release and its
    reads showed up only this way: a few 8x4 blocks of the Wgrad output were
    off by one chunk's contribution in about one launch in 20."""
    if workload == "wgrad":
        d = synth.wgrad()
        qa, sa = fb.quant_1x128(dev(d["dY"]), along=1)
        qb, sb = fb.quant_1x128(dev(d["X"]), along=1)
        bmode, dtype = 1, torch.float32
    else:
        d = synth.mla() if workload == "mla" else synth.ffn()
        w = np.concatenate([d["Wq"], d["Wkv"]]) if workload == "mla" else d["B"]
        qa, sa = fb.quant_1x128(dev(d["A"]))
        qb, sb = fb.quant_128x128(dev(w))
        bmode, dtype = 0, torch.bfloat16
    C = torch.empty((qa.shape[0], qb.shape[0]), dtype=dtype, device="cuda")
    bits = torch.int32 if dtype == torch.float32 else torch.int16
    first, differ = None, 0
    fb.set_gemm_tile_n(bn)
    try:
        for _ in range(launches):
            C.fill_(float("nan"))
            fb.gemm_blockscaled(qa, sa, qb, sb, bmode, C=C)
            if first is None:
                first = C.view(bits).clone()
            elif not torch.equal(C.view(bits), first):
                differ += 1
    finally:
        fb.set_gemm_tile_n(0)
    assert fb.get_device_error() == 0
    assert differ == 0, f"{workload} bn={bn}: {differ} of {launches - 1} launches differ from the first"


@pytest.mark.parametrize("kind", ["grouped", "grouped_swiglu", "ue8m0_bf16", "ue8m0_fp32"])
def test_repeated_launches_are_bit_identical_other_kernels(fb, kind):
    """The grouped GEMM, the fused SwiGLU grouped GEMM and the UE8M0 GEMM (both
    output types), each launched 100 times: identical bits every time."""
    if kind.startswith("grouped"):
        G, K = 16, 2048
        sizes = np.array([0, 700, 5, 129, 1100, 0, 257, 64, 900, 1, 380, 0, 2048, 33, 500, 128])
        offs = torch.from_numpy(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)).cuda()
        M = int(sizes.sum())
        a = synth.fill_bf16(synth.NORMAL, synth.key(110, 0), (M, K), 1.0)
        N = 2 * 1024 if kind == "grouped_swiglu" else 1536
        w = synth.fill_bf16(synth.NORMAL, synth.key(111, 0), (G, N, K), 0.02)
        qa, sa = fb.quant_1x128(dev(a))
        wd = dev(w)
        qb = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
        sb = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda")
        for e in range(G):
            fb.quant_128x128(wd[e], q=qb[e], s=sb[e])
        if kind == "grouped":
            C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            def run():
                C.fill_(float("nan"))
                fb.grouped_gemm_moe(qa, sa, qb, sb, offs, C=C)
                return C.view(torch.int16)
        else:
            Q = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda")
            S = torch.empty((N // 2 // 128, M), dtype=torch.float32, device="cuda")
            def run():
                Q.fill_(0xFF)
                S.fill_(float("nan"))
                fb.grouped_gemm_moe_swiglu(qa, sa, qb, sb, offs, Q=Q, s=S)
                return torch.cat([Q.view(torch.int32).flatten(), S.view(torch.int32).flatten()])
    else:
        d = synth.mla()
        qa, sa = fb.quant_1x128_ue8m0(dev(d["A"]))
        qb, sb = fb.quant_128x128_ue8m0(dev(np.concatenate([d["Wq"], d["Wkv"]])))
        dtype = torch.bfloat16 if kind == "ue8m0_bf16" else torch.float32
        C = torch.empty((qa.shape[0], qb.shape[0]), dtype=dtype, device="cuda")
        bits = torch.int16 if dtype == torch.bfloat16 else torch.int32
        def run():
            C.fill_(float("nan"))
            fb.gemm_ue8m0(qa, sa, qb, sb, C=C)
            return C.view(bits)
    first, differ = None, 0
    for _ in range(100):
        out = run()
        if first is None:
            first = out.clone()
        elif not torch.equal(out, first):
            differ += 1
    assert fb.get_device_error() == 0
    assert differ == 0, f"{kind}: {differ} of 99 launches differ from the first"


def _grouped(fb, orc, a_bits, offs, w_bits, rows=None, what=""):
    G, N, K = w_bits.shape
    qa, sa = fb.quant_1x128(dev(a_bits))
    wd = dev(w_bits)
    qb = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sb = torch.empty((G, (N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    for e in range(G):  # per expert: a 128x128 block never spans two experts
        fb.quant_128x128(wd[e], q=qb[e], s=sb[e])
    offs_d = torch.from_numpy(offs.astype(np.int32)).cuda()
    C = torch.full((a_bits.shape[0], N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fb.grouped_gemm_moe(qa, sa, qb, sb, offs_d, C=C)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    oqa, osa = orc.quant_1x128_rows(a_bits)
    oqb = np.empty((G, N, K), np.uint8)
    osb = np.empty((G, (N + 127) // 128, K // 128), np.float32)
    for e in range(G):
        oqb[e], osb[e] = orc.quant_128x128(w_bits[e])
    M = a_bits.shape[0]
    if rows is None:
        rows = np.arange(offs[0], offs[-1])
    ref = orc.bf16_round(orc.grouped_gemm(oqa, osa, oqb, osb, offs, rows=rows))
    got = host_bits(C[torch.from_numpy(rows).cuda()])
    assert_gemm_close(got, ref, what)
    # rows outside every group are left untouched
    outside = np.setdiff1d(np.arange(M), np.arange(offs[0], offs[-1]))
    if outside.size:
        assert torch.isnan(C[torch.from_numpy(outside).cuda()].float()).all()


@pytest.mark.parametrize("N", [256, 136, 64])
def test_grouped_small_skewed(fb, orc, tile_n, N):
    sizes = [0, 5, 0, 128, 129, 1, 300, 0, 64, 256, 0, 0, 77, 2, 0, 31]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    M = int(offs[-1]) + 10  # trailing rows belong to no expert
    K = 384
    a = synth.fill_bf16(synth.NORMAL, synth.key(70, N), (M, K), 1.0)
    w = synth.fill_bf16(synth.NORMAL, synth.key(71, N), (len(sizes), N, K), 0.02)
    _grouped(fb, orc, a, offs, w, what=f"grouped N={N}")


def test_grouped_256_experts_routed(fb, orc, tile_n):
    """256 experts, top-8 routing of 512 tokens (skewed groups, many empty)."""
    tok = synth.moe_tokens(T=512, D=256)
    offs, token_of_row = synth.moe_route(tok, E=256, topk=8)
    a = np.ascontiguousarray(tok[token_of_row])
    w = synth.fill_bf16(synth.NORMAL, synth.key(72, 0), (256, 256, 256), 0.02)
    _grouped(fb, orc, a, offs.astype(np.int64), w, what="grouped 256")


def moe_check_rows(offs, n_total=512, seed=3):
    """Rows checked in the full-size grouped GEMMs: the first and the last row
    of every non-empty expert, plus seeded rows up to n_total in all."""
    sizes = np.diff(offs)
    must = []
    for e in np.nonzero(sizes)[0]:
        must += [int(offs[e]), int(offs[e + 1]) - 1]
    must = sorted(set(must))
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(offs[0], offs[-1]), must)
    extra = rng.choice(rest, size=max(0, min(rest.size, n_total - len(must))), replace=False)
    return np.array(sorted(set(must) | set(int(r) for r in extra)), dtype=np.int64)


def test_moe_full_size_sampled(fb, orc):
    """Config-3 shapes: 4096 tokens routed top-8 over 256 experts -> 32768 rows;
    up (N=4096, K=7168) and down (N=7168, K=2048) grouped GEMMs, checked on the
    first and last row of every non-empty expert plus seeded rows (512 rows
    in all), so that every expert's offset into B and its scales is exercised."""
    tok = synth.moe_tokens()
    offs, token_of_row = synth.moe_route(tok)
    offs = offs.astype(np.int64)
    rows = moe_check_rows(offs)
    expert_of_row = np.searchsorted(offs, rows, side="right") - 1
    assert len(np.unique(expert_of_row)) == np.count_nonzero(np.diff(offs))

    for which, A_bits in (("up", np.ascontiguousarray(tok[token_of_row])), ("down", synth.moe_down_input())):
        G = 256
        qa, sa = fb.quant_1x128(dev(A_bits))
        N, K = (4096, 7168) if which == "up" else (7168, 2048)
        qb = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
        sb = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda")
        for e0 in range(0, G, 16):
            w = dev(synth.moe_weights(which, e0, e0 + 16))
            fb.quant_128x128(w.reshape(16 * N, K), q=qb[e0:e0 + 16].view(16 * N, K),
                             s=sb[e0:e0 + 16].view(16 * N // 128, K // 128))
            del w
        C = fb.grouped_gemm_moe(qa, sa, qb, sb, torch.from_numpy(offs.astype(np.int32)).cuda())
        torch.cuda.synchronize()
        assert fb.get_device_error() == 0
        got = host_bits(C[torch.from_numpy(rows).cuda()])
        del qb, sb, C
        oqa, osa = orc.quant_1x128_rows(A_bits)
        ref = np.empty((rows.size, N), np.float32)
        for e in np.unique(expert_of_row):
            sel = np.nonzero(expert_of_row == e)[0]
            oqb, osb = orc.quant_128x128(synth.moe_weights(which, int(e), int(e) + 1)[0])
            ref[sel] = orc.gemm_blockscaled(oqa, osa, oqb, osb, 0, rows=rows[sel])
        assert_gemm_close(got, orc.bf16_round(ref), f"moe {which}")


def test_timeout_path_reports_and_recovers(fb):
    """A wait that nothing completes ends after ~1 ms with FP8BS_ETIMEOUT recorded;
    the context stays usable and the error word is cleared by the read."""
    fb.selftest_timeout(1_000_000)
    assert fb.get_device_error() == fb.binding.ETIMEOUT
    assert fb.get_device_error() == 0
    x = torch.ones((128, 128), dtype=torch.bfloat16, device="cuda")
    q, s = fb.quant_1x128(x)
    torch.cuda.synchronize()
    assert int(q[0, 0]) == 0x7E and float(s[0, 0]) == float(np.float32(1) / np.float32(448))


def test_gemm_after_an_uncleared_timeout_is_complete(fb, orc):
    """A timeout recorded by an earlier launch and not yet read does not make
    later launches give up: a GEMM run after it is complete and correct, the
    earlier error is still reported once, and the word is then clear."""
    fb.selftest_timeout(1_000_000)
    d = synth.tiny()
    _dense_no_error_check(fb, orc, d["A"], d["B"])
    assert fb.get_device_error() == fb.binding.ETIMEOUT
    assert fb.get_device_error() == 0


def _dense_no_error_check(fb, orc, a_bits, w_bits):
    qa, sa = fb.quant_1x128(dev(a_bits))
    qb, sb = fb.quant_128x128(dev(w_bits))
    C = fb.gemm_blockscaled(qa, sa, qb, sb, 0)
    torch.cuda.synchronize()
    oqa, osa = orc.quant_1x128_rows(a_bits)
    oqb, osb = orc.quant_128x128(w_bits)
    ref = orc.bf16_round(orc.gemm_blockscaled(oqa, osa, oqb, osb, 0))
    assert_gemm_close(host_bits(C), ref, "after an uncleared timeout")


def test_mla_stacked_weight_equals_separate(fb, orc):
    """W_q (1536 rows) and W_kv (576 rows) stacked into one 2112-row weight:
    the 128x128 blocks never straddle the two, so the stacked quantisation and
    the single GEMM reproduce the separate ones bit for bit."""
    d = synth.mla()
    qa, sa = fb.quant_1x128(dev(d["A"]))
    qq, sq = fb.quant_128x128(dev(d["Wq"]))
    qk, sk = fb.quant_128x128(dev(d["Wkv"]))
    qw, sw = fb.quant_128x128(dev(np.concatenate([d["Wq"], d["Wkv"]])))
    assert torch.equal(qw[:1536], qq) and torch.equal(qw[1536:], qk)
    assert torch.equal(sw[:12], sq) and torch.equal(sw[12:], sk)
    C = fb.gemm_blockscaled(qa, sa, qw, sw, 0)
    Cq = fb.gemm_blockscaled(qa, sa, qq, sq, 0)
    Ck = fb.gemm_blockscaled(qa, sa, qk, sk, 0)
    torch.cuda.synchronize()
    assert torch.equal(C[:, :1536], Cq) and torch.equal(C[:, 1536:], Ck)
    rows = sample_rows(4096, 64, seed=8, must=(0, 4095))
    oqa, osa = orc.quant_1x128_rows(d["A"])
    oqw, osw = orc.quant_128x128(np.concatenate([d["Wq"], d["Wkv"]]))
    ref = orc.bf16_round(orc.gemm_blockscaled(oqa, osa, oqw, osw, 0, rows=rows))
    assert_gemm_close(host_bits(C[torch.from_numpy(rows).cuda()]), ref, "mla stacked")


@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32_scales", "ue8m0"])
def test_quantiser_then_gemm_back_to_back(fb, orc, ue8m0):
    """The GEMMs are launched so that their set-up overlaps the quantiser before
    them, and wait on the device for its codes.  Quantiser -> GEMM pairs issued
    back to back into shared code buffers, on inputs that change every
    iteration, give bit for bit the outputs of the same pairs run with a full
    synchronisation between the two launches; the first is also checked against
    the oracle."""
    d = synth.mla()
    A0 = dev(d["A"])
    W = dev(np.concatenate([d["Wq"], d["Wkv"]]))
    n = 6
    A = [torch.roll(A0, shifts=37 * i, dims=0) for i in range(n)]
    qa = torch.empty((4096, 7168), dtype=torch.uint8, device="cuda")
    qw = torch.empty((2112, 7168), dtype=torch.uint8, device="cuda")
    sa = torch.empty((56, 4096), dtype=torch.float32, device="cuda")
    sw = torch.empty((17, 56), dtype=torch.float32, device="cuda")
    gemm = fb.gemm_ue8m0 if ue8m0 else (lambda a, s, b, t, C: fb.gemm_blockscaled(a, s, b, t, 0, C=C))

    def pair(i, C, sync):
        fb.quant_act_weight(A[i], W, ue8m0=ue8m0, qx=qa, sx=sa, qw=qw, sw=sw)
        if sync:
            torch.cuda.synchronize()
        gemm(qa, sa, qw, sw, C=C)

    got = [torch.empty((4096, 2112), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    for i in range(n):
        pair(i, got[i], sync=False)
    torch.cuda.synchronize()
    assert fb.get_device_error() == 0
    for i in range(n):
        ref = torch.empty_like(got[i])
        pair(i, ref, sync=True)
        torch.cuda.synchronize()
        assert torch.equal(got[i], ref), f"iteration {i} differs from the synchronised run"
    assert not torch.equal(got[0], got[1])
    rows = sample_rows(4096, 32, seed=9, must=(0, 4095))
    Wh = np.concatenate([d["Wq"], d["Wkv"]])
    if ue8m0:
        oqa, osa = orc.quant_1x128_rows_pow2(d["A"])
        oqw, osw = orc.quant_128x128_pow2(Wh)
        ref = orc.gemm_exact_sum(oqa, osa, oqw, osw, 0, rows=rows)
    else:
        oqa, osa = orc.quant_1x128_rows(d["A"])
        oqw, osw = orc.quant_128x128(Wh)
        ref = orc.gemm_blockscaled(oqa, osa, oqw, osw, 0, rows=rows)
    assert_gemm_close(host_bits(got[0][torch.from_numpy(rows).cuda()]), orc.bf16_round(ref), "back to back")
