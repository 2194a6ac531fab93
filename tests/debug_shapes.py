"""Small odd shapes through every kernel family of the bounds-checked library
(run by tests/test_gpu_debug.py in a child process with FP8BS_LIBRARY=debug):
after each family the library's bounds-check record must be clear, and the
results must still match the oracle (quantisers bit for bit, GEMMs within the
tolerance of tests/gpu_util.py).  Prints one line per family and "debug ok"."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402
from tests.gpu_util import assert_gemm_close, dev, host_bits  # noqa: E402


def main():
    assert os.environ.get("FP8BS_LIBRARY") == "debug"
    import fp8_fine_grained_27_b300 as fb
    from fp8_fine_grained_27_b300 import binding
    assert binding.lib().fp8bs_debug_build() == 1
    oracle.build()

    def clear(what):
        torch.cuda.synchronize()
        site = fb.debug_site()
        assert site == 0, f"{what}: bounds check {site} failed"
        assert fb.get_device_error() == 0, what
        print(f"{what}: no bounds violation", flush=True)

    # quantisers and the dense GEMM: M = 1, 127, 129; N = 576 (a partial block) and 72
    for M, N, K in [(1, 576, 256), (127, 72, 384), (129, 576, 128), (300, 136, 640)]:
        a = synth.fill_bf16(synth.OUTLIER, synth.key(90, M), (M, K), 1.0, 0.01, 50.0, k2=synth.key(91, M))
        w = synth.fill_bf16(synth.NORMAL, synth.key(92, N), (N, K), 0.02)
        qa, sa = fb.quant_1x128(dev(a))
        qb, sb = fb.quant_128x128(dev(w))
        oqa, osa = oracle.quant_1x128_rows(a)
        oqb, osb = oracle.quant_128x128(w)
        assert np.array_equal(qa.cpu().numpy(), oqa) and np.array_equal(qb.cpu().numpy(), oqb)
        for tn in (0, 128, 192, 256):
            fb.set_gemm_tile_n(tn)
            for od in (torch.bfloat16, torch.float32):
                C = fb.gemm_blockscaled(qa, sa, qb, sb, 0, out_dtype=od)
                torch.cuda.synchronize()
                ref = oracle.gemm_blockscaled(oqa, osa, oqb, osb, 0)
                assert_gemm_close(host_bits(C), oracle.bf16_round(ref) if od == torch.bfloat16 else ref,
                                  f"{M}x{N}x{K} tile {tn}")
        fb.set_gemm_tile_n(0)
        clear(f"dense {M}x{N}x{K}")

    # FP32 output over more tiles than CTAs: the last round shared out by K chunks
    a = synth.fill_bf16(synth.NORMAL, synth.key(100, 1), (2560 - 40, 384), 1.0)
    w = synth.fill_bf16(synth.NORMAL, synth.key(102, 1), (2048 - 24, 384), 0.02)
    qa, sa = fb.quant_1x128(dev(a))
    qb, sb = fb.quant_128x128(dev(w))
    for tn in (0, 128):
        fb.set_gemm_tile_n(tn)
        C = fb.gemm_blockscaled(qa, sa, qb, sb, 0, out_dtype=torch.float32)
        torch.cuda.synchronize()
        ref = oracle.gemm_blockscaled(*oracle.quant_1x128_rows(a), *oracle.quant_128x128(w), 0)
        assert_gemm_close(host_bits(C), ref, f"split last round, tile {tn}")
    fb.set_gemm_tile_n(0)
    clear("dense FP32, last round split by K")

    # Dgrad (transposed weight quantiser) and Wgrad (token-wise quantiser, per-row scales)
    d = synth.dgrad(T=129, Cout=256, Cin=128)
    qdy, sdy = fb.quant_1x128(dev(d["dY"]))
    _, _, qwt, swt = fb.quant_128x128_t(dev(d["W"]))
    fb.gemm_blockscaled(qdy, sdy, qwt, swt, 0)
    clear("dgrad 129x128x256")
    for Cout, Cin, T in [(128, 8, 128), (384, 264, 384), (200, 264, 256)]:  # 200: a short last row tile
        w = synth.wgrad(T=T, Cout=Cout, Cin=Cin)
        qd, sd = fb.quant_1x128(dev(w["dY"]), along=1)
        qx, sx = fb.quant_1x128(dev(w["X"]), along=1)
        for tn in (0, 128, 192, 256):
            fb.set_gemm_tile_n(tn)
            dW = fb.gemm_blockscaled(qd, sd, qx, sx, 1, out_dtype=torch.float32)
            torch.cuda.synchronize()
            oqd, osd = oracle.quant_1x128_cols(w["dY"])
            oqx, osx = oracle.quant_1x128_cols(w["X"])
            assert_gemm_close(host_bits(dW), oracle.gemm_blockscaled(oqd, osd, oqx, osx, 1), f"wgrad {Cout}x{Cin}")
        fb.set_gemm_tile_n(0)
        clear(f"wgrad {Cout}x{Cin}x{T}")

    # grouped GEMM with empty and ragged experts, and the MoE chain
    sizes = [0, 5, 0, 128, 129, 1, 0, 31]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M, N, K = int(offs[-1]) + 3, 136, 256
    a = synth.fill_bf16(synth.NORMAL, synth.key(93, 0), (M, K), 1.0)
    w = synth.fill_bf16(synth.NORMAL, synth.key(94, 0), (len(sizes), N, K), 0.02)
    qa, sa = fb.quant_1x128(dev(a))
    qb = torch.empty((len(sizes), N, K), dtype=torch.uint8, device="cuda")
    sb = torch.empty((len(sizes), 2, K // 128), dtype=torch.float32, device="cuda")
    wd = dev(w)
    for e in range(len(sizes)):
        fb.quant_128x128(wd[e], q=qb[e], s=sb[e])
    for tn in (0, 128, 256):
        fb.set_gemm_tile_n(tn)
        fb.grouped_gemm_moe(qa, sa, qb, sb, torch.from_numpy(offs).cuda())
    fb.set_gemm_tile_n(0)
    clear("grouped, empty experts")
    T, D, E, k, Nh = 100, 256, 8, 2, 128
    x = synth.fill_bf16(synth.NORMAL, synth.key(95, 0), (T, D), 1.0)
    cent = synth.fill_f32(synth.NORMAL, synth.key(96, 0), (E, D), 1.0 / np.sqrt(D))
    bias = synth.fill_f32(synth.NORMAL, synth.key(97, 0), (E,), 0.5)
    wu = synth.fill_bf16(synth.NORMAL, synth.key(98, 0), (E, 2 * Nh, D), 0.05)
    wdn = synth.fill_bf16(synth.NORMAL, synth.key(99, 0), (E, D, Nh), 0.05)
    qwu, swu = fb.quant_128x128(dev(wu.reshape(-1, D)))
    qwd, swd = fb.quant_128x128(dev(wdn.reshape(-1, Nh)))
    qwu, swu = qwu.view(E, 2 * Nh, D), swu.view(E, 2 * Nh // 128, D // 128)
    qwd, swd = qwd.view(E, D, Nh), swd.view(E, D // 128, Nh // 128)
    xd = dev(x)
    r = fb.moe_route(xd, torch.from_numpy(np.ascontiguousarray(cent.T)).cuda(), torch.from_numpy(bias).cuda(), k)
    qg, sg = fb.quant_1x128_gather(xd, r["token_of_row"])
    h, sh = fb.grouped_gemm_moe_swiglu(qg, sg, qwu, swu, r["offsets"])
    Y = fb.grouped_gemm_moe(h, sh, qwd, swd, r["offsets"])
    fb.moe_combine(Y, r["row_of"], r["gate"])
    clear("moe chain")

    # UE8M0 variant on a ragged shape
    a = synth.fill_bf16(synth.NORMAL, synth.key(100, 0), (129, 256), 1.0)
    w = synth.fill_bf16(synth.NORMAL, synth.key(101, 0), (576, 256), 0.02)
    pa, psa = fb.quant_1x128_ue8m0(dev(a))
    pb, psb = fb.quant_128x128_ue8m0(dev(w))
    for od in (torch.bfloat16, torch.float32):
        fb.gemm_ue8m0(pa, psa, pb, psb, out_dtype=od)
    clear("ue8m0 129x576x256")
    print("debug ok", flush=True)


if __name__ == "__main__":
    main()
