"""Timing of the CPU oracle on the benchmark workloads (test infrastructure: the
oracle is the reference arm of the benchmark, timed on the host's cores).

For each workload: the quantisers' rate (GB/s of the algorithmic bytes, BF16
read + code write + scale write) over a bounded sample of the operand, the
GEMM's rate on a sample of output rows (every column, the full K), and the full
GEMM's time extrapolated from that rate (labelled as extrapolated: the oracle
computes every output row the same way, so its time is proportional to the
rows).  Workload 1 is timed in full, with all threads and with one.  Prints one
JSON object.

    python -m oracle.timing [--quick]
"""
from __future__ import annotations

import argparse
import json
import time

import numpy as np


def _rate(fn, reps=1):
    fn()  # first call: table set-up, page-in
    t0 = time.perf_counter()
    for _ in range(reps):
        fn()
    return (time.perf_counter() - t0) / reps


def main():
    import oracle
    import synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--quick", action="store_true", help="smaller samples (a CPU check of the script)")
    args = ap.parse_args()
    oracle.build()
    rows = 4 if args.quick else 32
    out = {"threads": oracle.nthreads(), "workloads": {}}

    # 1 tiny: in full, all threads and one thread
    d = synth.tiny()
    qa, sa = oracle.quant_1x128_rows(d["A"])
    qb, sb = oracle.quant_128x128(d["B"])
    gf = 2.0 * 128 * 256 * 512
    t_all = _rate(lambda: oracle.gemm_blockscaled(qa, sa, qb, sb, 0), reps=5)
    t_one = _rate(lambda: oracle.gemm_blockscaled(qa, sa, qb, sb, 0, threads=1), reps=5)
    tq = _rate(lambda: (oracle.quant_1x128_rows(d["A"]), oracle.quant_128x128(d["B"])), reps=5)
    out["workloads"]["tiny 128x256x512"] = {
        "gemm_gflops": round(gf / t_all / 1e9, 3), "gemm_gflops_1_thread": round(gf / t_one / 1e9, 3),
        "quant_gbs": round((128 * 512 * (3 + 4 / 128) + 256 * 512 * (3 + 4 / 16384)) / tq / 1e9, 3),
        "gemm_ms": round(t_all * 1e3, 3), "gemm_ms_1_thread": round(t_one * 1e3, 3)}

    def dense(name, A, Ws, M, K, b_mode=0, colwise=False):
        """A: the activation operand; Ws: weights; quantiser and sampled-row GEMM rates."""
        if colwise:
            qa, sa = oracle.quant_1x128_cols(A)
            ta = _rate(lambda: oracle.quant_1x128_cols(A))
        else:
            qa, sa = oracle.quant_1x128_rows(A)
            ta = _rate(lambda: oracle.quant_1x128_rows(A))
        qbytes = A.size * (3 + 4 / 128)
        tw, wbytes, gf_full, t_rows = 0.0, 0.0, 0.0, 0.0
        sample = np.linspace(0, qa.shape[0] - 1, rows).astype(np.int64)
        for W in Ws:
            if colwise:
                qb, sb = oracle.quant_1x128_cols(W)
                tw += _rate(lambda: oracle.quant_1x128_cols(W))
                wbytes += W.size * (3 + 4 / 128)
            else:
                qb, sb = oracle.quant_128x128(W)
                tw += _rate(lambda: oracle.quant_128x128(W))
                wbytes += W.size * (3 + 4 / 16384)
            t_rows += _rate(lambda: oracle.gemm_blockscaled(qa, sa, qb, sb, b_mode, rows=sample))
            gf_full += 2.0 * qa.shape[0] * qb.shape[0] * qa.shape[1]
        per_row = t_rows / rows
        out["workloads"][name] = {
            "quant_gbs": round((qbytes + wbytes) / (ta + tw) / 1e9, 3),
            "gemm_gflops_sampled_rows": round(gf_full / qa.shape[0] / per_row / 1e9, 3),
            "gemm_rows_sampled": rows, "gemm_ms_per_row": round(per_row * 1e3, 3),
            "gemm_full_s_extrapolated": round(per_row * qa.shape[0], 1)}

    d = synth.mla()
    dense("mla 4096x(1536+576)x7168", d["A"], [d["Wq"], d["Wkv"]], 4096, 7168)
    d = synth.ffn()
    dense("ffn 16384x18432x7168", d["A"], [d["B"]], 16384, 7168)
    d = synth.wgrad()
    dense("wgrad 2048x7168x16384 (FP32 out)", d["dY"], [d["X"]], 2048, 16384, b_mode=1, colwise=True)
    print(json.dumps(out, indent=1))


if __name__ == "__main__":
    main()
