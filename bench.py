#!/usr/bin/env python3
"""Benchmark: fine-grained FP8 (E4M3) quantise + block-scaled GEMM steps on B300.

One step = one pass of the whole hot path over one batch of the workload:
  ffn   (default) A 16384x7168 (Student-t), B 18432x7168: quantise both
        (one launch), one GEMM 16384x18432x7168 with BF16 output.  The
        largest dense GEMM of the pages' model, and the primary GEMM number.
  mla   A 4096x7168 BF16 -> 1x128 quantise; W_q 1536x7168 and
        W_kv 576x7168 stored stacked as one 2112x7168 weight (1536 is a
        multiple of 128, so no 128x128 block straddles the two) -> one
        128x128 quantise and one GEMM whose column slices [0,1536) and
        [1536,2112) are the q and kv latents (BF16 out).
  wgrad dY 16384x2048, X 16384x7168: token-wise 1x128 quantise (transposed
        codes), dW = dY^T X with FP32 output.
  dgrad dY 16384x18432, W 18432x7168: dY 1x128 and W's transposed 128x128
        quantisation, dX = dY W (BF16 out).
  moe   4096 tokens routed top-8 over 256 experts (32768 rows): quantise the
        grouped rows, up grouped GEMM (N=4096, K=7168) with pre-quantised
        expert weights.
  moe_chain  the whole routed-expert layer: routing (FP32 logits, top-8,
        grouping), gather-quantise, up GEMM with fused SwiGLU + quantise,
        down GEMM, combine (--tokens, --experts size it).
  mla_ue8m0, ffn_ue8m0  the mla / ffn steps in the power-of-two (UE8M0)
        scale variant on the tensor cores' block-scaled MMA.
In the mla/ffn steps one launch quantises both the activation and the weight.
Inputs are seeded synthetic tensors (synth/), resident in HBM before timing.
L2 is flushed before every timed step, outside the step's CUDA events: a 256 MB
write, then a 256 MB read that evicts the dirty lines the write left
(--flush-mode write keeps only the write).  The warm-up runs back to back
(a few steps queued ahead of the GPU, no synchronisation per step) for at
least --min-warmup-s and goes straight into the timed steps, so the GPU is
under steady load when timing starts; the clock sampler runs from before the
warm-up.  Prints one JSON line (rank 0).

--impl reference times the CPU oracle (oracle/) on a bounded sample of the
same workload instead: the method's plain restatement on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


PROFILES = os.path.join(ROOT, "profiles")
# workload -> (ncu summary under profiles/, sources whose hash it records)
GEMM_PROFILE = {"mla": ("gemm_kernel_mla_4096x2112x7168.md", ["gemm.cuh", "ptx.cuh"]),
                "ffn": ("gemm_kernel_ffn_16384x18432x7168.md", ["gemm.cuh", "ptx.cuh"]),
                "dgrad": ("gemm_kernel_dgrad_16384x7168x18432.md", ["gemm.cuh", "ptx.cuh"]),
                "wgrad": ("gemm_kernel_wgrad_2048x7168x16384.md", ["gemm.cuh", "ptx.cuh"]),
                "mla_ue8m0": ("mx_gemm_kernel_mla_ue8m0.md", ["mx.cuh", "ptx.cuh"]),
                "ffn_ue8m0": ("mx_gemm_kernel_ffn_ue8m0.md", ["mx.cuh", "ptx.cuh"])}


def kernel_source_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "fp8_fine_grained_27_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per GEMM launch from the committed ncu summary of this
    workload, or None if there is none or the kernel source changed since."""
    entry = GEMM_PROFILE.get(workload)
    if not entry:
        return None
    name, sources = entry
    try:
        text = open(os.path.join(PROFILES, name)).read()
    except OSError:
        return None
    fields = dict(l.split(":", 1) for l in text.splitlines() if l.startswith(("kernel_source_sha256_16:", "traffic_bytes_per_launch:")))
    if fields.get("kernel_source_sha256_16", "").split()[0:1] != [kernel_source_hash(sources)]:
        return None
    return int(fields["traffic_bytes_per_launch"].split()[0])


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return dict(FALLBACK), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0, t1):
        """Median SM clock, maximum and active throttle reasons of the samples
        taken between wall times t0 and t1 (all samples if none fall inside)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = [l for (ts, l) in self.lines if t0 - 0.05 <= ts <= t1 + 0.05] or [l for _, l in self.lines]
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in rows:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ------------------------------------------------------------------ workloads
# tokens and experts of the moe_chain layer (--tokens / --experts; a smaller layer is for
# profiling captures that must fit in a few GB)
MOE_CHAIN = {"tokens": 4096, "experts": 256}


def workload_desc(name):
    return {
        "mla": {"workload": "mla_down_proj", "M": 4096, "K": 7168, "N": [1536, 576],
                "gemms": "2 (q 1536 + kv 576, one launch over the stacked 2112-row weight)",
                "quant": "A 1x128, [W_q; W_kv] 128x128", "out": "bf16"},
        "ffn": {"workload": "dense_ffn", "M": 16384, "K": 7168, "N": [18432],
                "gemms": 1, "quant": "A 1x128, B 128x128", "out": "bf16"},
        "ffn_ue8m0": {"workload": "dense_ffn_ue8m0_variant", "M": 16384, "K": 7168, "N": [18432], "gemms": 1,
                      "quant": "A 1x128, B 128x128, power-of-two (UE8M0) scales",
                      "gemm": "tcgen05 kind::mxf8f6f4 block-scaled MMA (no promotion pass)", "out": "bf16"},
        "mla_ue8m0": {"workload": "mla_down_proj_ue8m0_variant", "M": 4096, "K": 7168, "N": [1536, 576],
                      "gemms": "1 (stacked 2112-row weight)",
                      "quant": "A 1x128, [W_q; W_kv] 128x128, power-of-two (UE8M0) scales",
                      "gemm": "tcgen05 kind::mxf8f6f4 block-scaled MMA (no promotion pass)", "out": "bf16"},
        "wgrad": {"workload": "wgrad", "M": 2048, "K": 16384, "N": [7168],
                  "gemms": 1, "quant": "dY, X 1x128 along tokens (transposed)", "out": "fp32"},
        "dgrad": {"workload": "dgrad_ffn", "M": 16384, "K": 18432, "N": [7168], "gemms": 1,
                  "quant": "dY 1x128, W 128x128 written transposed (codes + scales)", "out": "bf16"},
        "moe_chain": {"workload": "moe_layer_forward", "M": 8 * MOE_CHAIN["tokens"], "K": [7168, 2048],
                      "N": [4096, 7168], "tokens": MOE_CHAIN["tokens"], "experts": MOE_CHAIN["experts"], "topk": 8,
                      "gemms": "2 grouped (up 2x2048 with fused SwiGLU + 1x128 quantise; down 7168)",
                      "quant": "gathered token rows 1x128 (weights pre-quantised)",
                      "other": "routing (FP32 logits, top-8, grouping), combine", "out": "bf16"},
        "moe": {"workload": "moe_grouped_up", "M": 32768, "K": 7168, "N": [4096], "experts": 256,
                "topk": 8, "gemms": 1, "quant": "grouped rows 1x128 (weights pre-quantised)", "out": "bf16"},
        "tiny": {"workload": "tiny", "M": 128, "K": 512, "N": [256], "gemms": 1,
                 "quant": "A 1x128, B 128x128", "out": "bf16"},
    }[name]


METRIC = "block-scaled FP8 GEMM TFLOPS (% of B300 FP8 peak); quantize GB/s (% HBM)"


def bench_config(args, world):
    """The `config` object of both arms' lines (same keys, same values)."""
    if world == 1:
        par = "single GPU"
    elif args.workload == "wgrad":
        par = f"data parallel x{world}: each rank's 16384 tokens, FP32 dW partials reduce-scattered"
    else:
        par = f"replicas x{world}"
    return {**workload_desc(args.workload),
            "l2": f"flushed ({args.flush_mb} MB {args.flush_mode}) before every step",
            "parallelism": par}


# kernels of this library one labelled call launches (fp8_moe_route: logits, selection,
# grouping; the data-parallel reduce-scatter is the collective library's, none of ours)
KERNELS_PER_CALL = {"route": 3, "reduce_scatter": 0}


def gemm_flops(name):
    d = workload_desc(name)
    if name == "moe_chain":
        return sum(2.0 * d["M"] * n * k for n, k in zip(d["N"], d["K"]))
    return sum(2.0 * d["M"] * n * d["K"] for n in d["N"])


def quant_bytes(name):
    """Algorithmic HBM bytes of the step's quantisation: BF16 read + code
    write + 4-byte scale per 128 elements (1x128) or per 128x128 block."""
    d = workload_desc(name)
    if name in ("mla", "ffn", "tiny", "mla_ue8m0", "ffn_ue8m0"):
        ea = d["M"] * d["K"]
        ew = sum(d["N"]) * d["K"]
        return ea * (3 + 4 / 128) + ew * (3 + 4 / (128 * 128))
    if name == "wgrad":
        e = d["K"] * (d["M"] + d["N"][0])
        return e * (3 + 4 / 128)
    if name == "dgrad":
        return d["M"] * d["K"] * (3 + 4 / 128) + d["K"] * d["N"][0] * (3 + 4 / (128 * 128))
    if name == "moe":
        return d["M"] * d["K"] * (3 + 4 / 128)
    if name == "moe_chain":
        return d["M"] * d["K"][0] * (3 + 4 / 128)
    raise KeyError(name)


class Step:
    """Device buffers and the launch sequence of one step.  Every launch goes
    through the C ABI (fp8_fine_grained_27_b300.binding)."""

    def __init__(self, name, fb, torch, seed=0, rank=0):
        import synth
        self.name, self.fb, self.torch = name, fb, torch
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).cuda()  # noqa: E731
        self.kernels = []  # (label, kind) per launch, in order
        if name in ("mla", "tiny", "mla_ue8m0"):
            d = synth.mla(seed=seed) if name != "tiny" else synth.tiny(seed=seed)
            self.host = {"A": d["A"], "W": [np.concatenate([d["Wq"], d["Wkv"]])] if name != "tiny" else [d["B"]]}
        elif name in ("ffn", "ffn_ue8m0"):
            d = synth.ffn(seed=seed)
            self.host = {"A": d["A"], "W": [d["B"]]}
        elif name == "wgrad":
            d = synth.wgrad(seed=seed)
            self.host = {"dY": d["dY"], "X": d["X"]}
        elif name == "dgrad":
            d = synth.dgrad(seed=seed)
            self.host = {"dY": d["dY"], "W": d["W"]}
        elif name == "moe_chain":
            cent, bias = synth.moe_router(seed=seed, E=MOE_CHAIN["experts"])
            self.host = {"X": synth.moe_tokens(seed=seed, T=MOE_CHAIN["tokens"]), "cent": cent, "bias": bias}
        elif name == "moe":
            tok = synth.moe_tokens(seed=seed)
            offs, token_of_row = synth.moe_route(tok, seed=seed)
            self.host = {"A": np.ascontiguousarray(tok[token_of_row]), "offs": offs}
        self.d = {}
        if name in ("mla", "tiny", "ffn", "mla_ue8m0", "ffn_ue8m0"):
            self.d["A"] = dev(self.host["A"])
            self.d["W"] = [dev(w) for w in self.host["W"]]
            M, K = self.host["A"].shape
            self.d["qa"] = torch.empty((M, K), dtype=torch.uint8, device="cuda")
            self.d["sa"] = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
            self.d["qw"] = [torch.empty_like(w, dtype=torch.uint8) for w in self.d["W"]]
            self.d["sw"] = [torch.empty(((w.shape[0] + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
                            for w in self.d["W"]]
            self.d["C"] = [torch.empty((M, w.shape[0]), dtype=torch.bfloat16, device="cuda") for w in self.d["W"]]
        elif name == "wgrad":
            self.d["dY"], self.d["X"] = dev(self.host["dY"]), dev(self.host["X"])
            T, Co = self.host["dY"].shape
            Ci = self.host["X"].shape[1]
            self.d["qdy"] = torch.empty((Co, T), dtype=torch.uint8, device="cuda")
            self.d["sdy"] = torch.empty((T // 128, Co), dtype=torch.float32, device="cuda")
            self.d["qx"] = torch.empty((Ci, T), dtype=torch.uint8, device="cuda")
            self.d["sx"] = torch.empty((T // 128, Ci), dtype=torch.float32, device="cuda")
            self.d["C"] = [torch.empty((Co, Ci), dtype=torch.float32, device="cuda")]
        elif name == "dgrad":
            self.d["dY"], self.d["W"] = dev(self.host["dY"]), dev(self.host["W"])
            T, Co = self.host["dY"].shape
            Ci = self.host["W"].shape[1]
            self.d["qdy"] = torch.empty((T, Co), dtype=torch.uint8, device="cuda")
            self.d["sdy"] = torch.empty((Co // 128, T), dtype=torch.float32, device="cuda")
            self.d["qwt"] = torch.empty((Ci, Co), dtype=torch.uint8, device="cuda")
            self.d["swt"] = torch.empty((Ci // 128, (Co + 127) // 128), dtype=torch.float32, device="cuda")
            self.d["C"] = [torch.empty((T, Ci), dtype=torch.bfloat16, device="cuda")]
        elif name == "moe_chain":
            T, D = self.host["X"].shape
            E, k, Nh = MOE_CHAIN["experts"], 8, 2048
            R = T * k
            self.d["X"] = dev(self.host["X"])
            self.d["cent"] = torch.from_numpy(np.ascontiguousarray(self.host["cent"].T)).cuda()  # k-major
            self.d["bias"] = torch.from_numpy(self.host["bias"]).cuda()
            self.d["route"] = {
                "logits": torch.empty((T, E), dtype=torch.float32, device="cuda"),
                "expert_idx": torch.empty((T, k), dtype=torch.int32, device="cuda"),
                "gate": torch.empty((T, k), dtype=torch.float32, device="cuda"),
                "offsets": torch.empty(E + 1, dtype=torch.int32, device="cuda"),
                "token_of_row": torch.empty(R, dtype=torch.int32, device="cuda"),
                "row_of": torch.empty((T, k), dtype=torch.int32, device="cuda")}
            self.d["ws"] = torch.empty(max(fb.lib().fp8_moe_route_workspace_size(E), 256), dtype=torch.uint8,
                                       device="cuda")
            self.d["qa"] = torch.empty((R, D), dtype=torch.uint8, device="cuda")
            self.d["sa"] = torch.empty((D // 128, R), dtype=torch.float32, device="cuda")
            self.d["h"] = torch.empty((R, Nh), dtype=torch.uint8, device="cuda")
            self.d["sh"] = torch.empty((Nh // 128, R), dtype=torch.float32, device="cuda")
            self.d["Y"] = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")
            self.d["qwu"] = torch.empty((E, 2 * Nh, D), dtype=torch.uint8, device="cuda")
            self.d["swu"] = torch.empty((E, 2 * Nh // 128, D // 128), dtype=torch.float32, device="cuda")
            self.d["qwd"] = torch.empty((E, D, Nh), dtype=torch.uint8, device="cuda")
            self.d["swd"] = torch.empty((E, D // 128, Nh // 128), dtype=torch.float32, device="cuda")
            for e0 in range(0, E, 16):  # expert weights: quantised once, outside the step
                w = dev(synth.moe_weights("up", e0, e0 + 16, seed=seed))
                fb.quant_128x128(w.view(-1, D), q=self.d["qwu"][e0:e0 + 16].view(-1, D),
                                 s=self.d["swu"][e0:e0 + 16].view(-1, D // 128))
                w = dev(synth.moe_weights("down", e0, e0 + 16, seed=seed))
                fb.quant_128x128(w.view(-1, Nh), q=self.d["qwd"][e0:e0 + 16].view(-1, Nh),
                                 s=self.d["swd"][e0:e0 + 16].view(-1, Nh // 128))
                del w
            self.d["C"] = [torch.empty((T, D), dtype=torch.bfloat16, device="cuda")]
        elif name == "moe":
            self.d["A"] = dev(self.host["A"])
            M, K = self.host["A"].shape
            G, N = 256, 4096
            self.d["qa"] = torch.empty((M, K), dtype=torch.uint8, device="cuda")
            self.d["sa"] = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
            self.d["qb"] = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
            self.d["sb"] = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda")
            for e0 in range(0, G, 16):  # expert weights: quantised once, outside the step
                w = dev(synth.moe_weights("up", e0, e0 + 16, seed=seed))
                fb.quant_128x128(w.reshape(16 * N, K), q=self.d["qb"][e0:e0 + 16].view(16 * N, K),
                                 s=self.d["sb"][e0:e0 + 16].view(16 * N // 128, K // 128))
                del w
            self.d["offs"] = torch.from_numpy(self.host["offs"].astype(np.int32)).cuda()
            self.d["C"] = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda")]
        torch.cuda.synchronize()

    def launches(self):
        """Return [(label, callable)] for one step."""
        fb, d = self.fb, self.d
        if self.name in ("mla_ue8m0", "ffn_ue8m0"):
            # one launch quantises the activation and the (stacked) weight
            L = [("quant_act_weight_ue8m0", lambda: fb.quant_act_weight(d["A"], d["W"][0], ue8m0=True, qx=d["qa"],
                                                                        sx=d["sa"], qw=d["qw"][0], sw=d["sw"][0]))]
            for i in range(len(d["W"])):
                L.append(("gemm_ue8m0", lambda i=i: fb.gemm_ue8m0(d["qa"], d["sa"], d["qw"][i], d["sw"][i],
                                                                  C=d["C"][i])))
            return L
        if self.name in ("mla", "tiny", "ffn"):
            # one launch quantises the activation and the (stacked) weight
            L = [("quant_act_weight", lambda: fb.quant_act_weight(d["A"], d["W"][0], qx=d["qa"], sx=d["sa"],
                                                                  qw=d["qw"][0], sw=d["sw"][0]))]
            for i in range(len(d["W"])):
                L.append(("gemm", lambda i=i: fb.gemm_blockscaled(d["qa"], d["sa"], d["qw"][i], d["sw"][i], 0,
                                                                  C=d["C"][i])))
            return L
        if self.name == "wgrad":
            return [("quant_1x128_cols_dY", lambda: fb.quant_1x128(d["dY"], along=1, q=d["qdy"], s=d["sdy"])),
                    ("quant_1x128_cols_X", lambda: fb.quant_1x128(d["X"], along=1, q=d["qx"], s=d["sx"])),
                    ("gemm", lambda: fb.gemm_blockscaled(d["qdy"], d["sdy"], d["qx"], d["sx"], 1, C=d["C"][0]))]
        if self.name == "dgrad":
            return [("quant_1x128", lambda: fb.quant_1x128(d["dY"], q=d["qdy"], s=d["sdy"])),
                    ("quant_128x128_t", lambda: fb.quant_128x128_t(d["W"], straight=False, qt=d["qwt"], st=d["swt"])),
                    ("gemm", lambda: fb.gemm_blockscaled(d["qdy"], d["sdy"], d["qwt"], d["swt"], 0, C=d["C"][0]))]
        if self.name == "moe_chain":
            r = d["route"]
            return [("route", lambda: fb.moe_route(d["X"], d["cent"], d["bias"], 8, out=r, workspace=d["ws"])),
                    ("quant_1x128_gather", lambda: fb.quant_1x128_gather(d["X"], r["token_of_row"], q=d["qa"],
                                                                         s=d["sa"])),
                    ("gemm_up_swiglu", lambda: fb.grouped_gemm_moe_swiglu(d["qa"], d["sa"], d["qwu"], d["swu"],
                                                                          r["offsets"], Q=d["h"], s=d["sh"])),
                    ("gemm_down", lambda: fb.grouped_gemm_moe(d["h"], d["sh"], d["qwd"], d["swd"], r["offsets"],
                                                              C=d["Y"])),
                    ("combine", lambda: fb.moe_combine(d["Y"], r["row_of"], r["gate"], out=d["C"][0]))]
        if self.name == "moe":
            return [("quant_1x128", lambda: fb.quant_1x128(d["A"], q=d["qa"], s=d["sa"])),
                    ("gemm", lambda: fb.grouped_gemm_moe(d["qa"], d["sa"], d["qb"], d["sb"], d["offs"],
                                                         C=d["C"][0]))]
        raise KeyError(self.name)

    def host_inputs(self):
        """(name, host array) of this step's BF16 activations, for the end-to-end
        run.  Weights are layer parameters and stay resident in HBM, as the
        MoE workloads' experts do; the step still quantises them every time."""
        if self.name in ("mla", "tiny", "ffn", "mla_ue8m0", "ffn_ue8m0"):
            return [("A", self.host["A"])]
        if self.name == "wgrad":
            return [("dY", self.host["dY"]), ("X", self.host["X"])]
        if self.name == "dgrad":
            return [("dY", self.host["dY"])]
        if self.name == "moe_chain":
            return [("X", self.host["X"])]
        return [("A", self.host["A"])]


# ------------------------------------------------------------------ ranks
def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The slowest rank's value (the job's step time under weak scaling)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, seconds_slowest: float, world: int) -> float:
    """Whole-job throughput of `world` replicas that each process
    units_per_rank in their own time; the job ends with the slowest rank."""
    return world * units_per_rank / seconds_slowest


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world):
    import torch

    import fp8_fine_grained_27_b300 as fb
    fb.lib()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    step = Step(args.workload, fb, torch, seed=rank)
    launches = step.launches()
    if dist is not None and args.workload == "wgrad":
        # data-parallel Wgrad: each rank's tokens give an FP32 partial dW; one
        # reduce-scatter sums them and leaves each rank its rows (ZeRO-1)
        from fp8_fine_grained_27_b300 import dp
        dw_rows = torch.empty((step.d["C"][0].shape[0] // world, step.d["C"][0].shape[1]), dtype=torch.float32,
                              device="cuda")
        launches.append(("reduce_scatter", lambda: dp.reduce_scatter_rows(step.d["C"][0], out=dw_rows)))
    flush = torch.empty(args.flush_mb << 20, dtype=torch.uint8, device="cuda")
    # A write-only flush leaves L2 full of dirty lines, which the step's first
    # kernel then has to write back to HBM on top of its own traffic; reading a
    # second buffer of the same size afterwards evicts them (outside the timed
    # region) and leaves only clean lines of no use to the step.
    flush_rd = torch.ones(args.flush_mb << 18, dtype=torch.float32, device="cuda") if args.flush_mode == "write+read" else None

    def flush_l2():
        flush.zero_()
        if flush_rd is not None:
            flush_rd.sum()

    stream = torch.cuda.current_stream()

    def one_step():
        flush_l2()
        for _, f in launches:
            f()

    nk = len(launches)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    # Warm-up: W steps, then more until --min-warmup-s of wall time has passed,
    # issued back to back.  At most QUEUE steps are in flight ahead of the
    # host (it waits on the event of an earlier step, not on the device), so
    # the wall time tracks the GPU's and the GPU never idles between steps.
    # The timed steps follow straight after (the barrier and synchronisation
    # around them are the only gap), so they run under the same steady load.
    QUEUE = 4
    inflight = []
    n_warm = 0
    t_warm = time.time()
    while n_warm < args.warmup or (time.time() - t_warm < args.min_warmup_s and n_warm < 100000):
        one_step()
        e = torch.cuda.Event()
        e.record(stream)
        inflight.append(e)
        if len(inflight) > QUEUE:
            inflight.pop(0).synchronize()
        n_warm += 1
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    fb.gemm_clock(reset=True)
    t0 = time.time()
    # The timed region: each step's launches go out back to back, as a caller
    # issues them, with events only around the step.
    for k in range(args.steps):
        flush_l2()
        ev[k][0].record(stream)
        for _, f in launches:
            f()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t1 = time.time()
    # the SM clock the GEMM kernels ran at in the timed region (measured in the
    # kernels: the sampled board clock cannot resolve them)
    gemm_mhz, gemm_launches = fb.gemm_clock(reset=True)
    if fb.get_device_error() != 0:
        raise RuntimeError("device error during the warm-up or the timed region")
    # A second pass over the same number of steps puts events between the
    # launches, for the per-kernel split (an event between two launches keeps
    # the GEMM's set-up from overlapping the quantiser before it, so that pass
    # is not the step time).
    for k in range(args.steps):
        flush_l2()
        evk[k][0].record(stream)
        for j, (_, f) in enumerate(launches):
            f()
            evk[k][j + 1].record(stream)
    torch.cuda.synchronize()
    t2 = time.time()
    gemm_mhz_split, _ = fb.gemm_clock(reset=True)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    clocks_split = sampler.summary(t1, t2)
    clocks_warm = sampler.summary(t_warm, t0)
    if fb.get_device_error() != 0:
        raise RuntimeError("device error during the per-kernel pass")

    per_step = [ev[k][0].elapsed_time(ev[k][1]) for k in range(args.steps)]
    per_kernel = {}
    for k in range(args.steps):
        for j, (label, _) in enumerate(launches):
            per_kernel.setdefault(label, []).append(evk[k][j].elapsed_time(evk[k][j + 1]))
    ms_step = max_over_ranks(float(np.mean(per_step)), dist, "cuda")

    flops = gemm_flops(args.workload)
    qbytes = quant_bytes(args.workload)
    value = job_throughput(flops, ms_step * 1e-3, world) / 1e12
    peaks, peaks_src = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    fp8_peak_sustained = 2.0 * peaks.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"])
    # GEMM launches of one step (there may be several): their summed mean duration
    g_idx = [j for j, (l, _) in enumerate(launches) if l.startswith("gemm")]
    gemm_ms = float(np.mean([sum(evk[k][j].elapsed_time(evk[k][j + 1]) for j in g_idx) for k in range(args.steps)]))
    q_idx = [j for j, (l, _) in enumerate(launches) if l.startswith("quant")]
    quant_ms = float(np.mean([sum(evk[k][j].elapsed_time(evk[k][j + 1]) for j in q_idx) for k in range(args.steps)]))
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    quant_gbs = qbytes / (quant_ms * 1e-3) / 1e9

    e2e = run_e2e(args, step, torch, fb, launches, flops, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(args.workload, budget_s=args.cpu_budget)

    first, last = per_step[:5], per_step[-5:]
    line = {
        "metric": METRIC,
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "warmup_steps_run": n_warm, "warmup_s": round(t0 - t_warm, 3),
        "ms_per_step": round(ms_step, 5),
        "ms_per_step_median": round(float(np.median(per_step)), 5),
        # the spread of the timed steps: a ramp (first steps slower than the
        # last) would show here
        "per_step_ms": {"first5_median": round(float(np.median(first)), 5),
                        "last5_median": round(float(np.median(last)), 5),
                        "min": round(float(min(per_step)), 5), "max": round(float(max(per_step)), 5)},
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> fp32 accumulate",
        "data": "synthetic (seeded; shapes of the DeepSeek-V3 pages)",
        "config": bench_config(args, world),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                     "traffic": profiled_traffic(args.workload),
                     "traffic_note": "DRAM read+write bytes per GEMM launch, ncu (profiles/), null if the kernel changed since",
                     "peak_source": f"{peaks_src}: 2 x bf16_tflops (dense FP8 = 2 x BF16), the burst figure",
                     # the power-capped figure, for runs whose clocks show sw_power_cap
                     "peak_sustained": round(fp8_peak_sustained, 1),
                     "frac_sustained": round(achieved / fp8_peak_sustained, 4),
                     "kernel": "gemm_kernel", "kernel_ms": round(gemm_ms, 5),
                     # the SM clock inside the GEMM kernels (their own clock64 over
                     # globaltimer), and the fraction of the peak's cycles the kernel
                     # keeps busy: achieved x (max clock / that clock) / peak
                     "sm_mhz_in_kernel": round(gemm_mhz_split, 1) if gemm_mhz_split else None,
                     "sm_mhz_in_kernel_timed_region": round(gemm_mhz, 1) if gemm_mhz else None,
                     "frac_at_max_clock": (round(achieved * peaks.get("sm_max_mhz", 2032.0) / gemm_mhz_split / fp8_peak, 4)
                                           if gemm_mhz_split else None)},
        "quant": {"achieved_gbs": round(quant_gbs, 1), "peak_gbs": peaks["hbm_gbs"],
                  "frac": round(quant_gbs / peaks["hbm_gbs"], 4), "kernel_ms": round(quant_ms, 5),
                  "bytes_per_step": int(qbytes)},
        "per_kernel_ms": {l: round(float(np.mean(v)), 5) for l, v in per_kernel.items()},
        "per_kernel_note": "second pass of the same steps with an event between launches",
        "e2e": e2e,
        "gpu_launches": sum(KERNELS_PER_CALL.get(l, 1) for l, _ in launches) * args.steps,
        "clocks": clocks,
        # the same sampler over the warm-up and over the per-kernel pass, and
        # the step time in SM clock cycles at the timed region's median clock
        "clocks_bins": {"warmup": clocks_warm, "per_kernel_pass": clocks_split,
                        "step_kcycles_at_median_mhz": (round(ms_step * clocks["sm_mhz"], 1)
                                                       if clocks.get("sm_mhz") else None)},
        "wall_s_timed_region": round(t1 - t0, 3),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_e2e(args, step, torch, fb, launches, flops, world, dist):
    """Same metric through the public API with host buffers: pinned H2D of the
    step's BF16 inputs, the step's launches, D2H of the outputs, per step."""
    pinned = [(n, torch.from_numpy(np.ascontiguousarray(a)).pin_memory()) for n, a in step.host_inputs()]
    outs = step.d["C"]
    out_host = [torch.empty(c.shape, dtype=c.dtype).pin_memory() for c in outs]
    # each uploaded activation lands in the device buffer of the same name
    targets = {name: step.d[name] for name, _ in pinned}
    h2d = sum(p.numel() * p.element_size() for _, p in pinned)
    d2h = sum(o.numel() * o.element_size() for o in out_host)
    n = max(3, min(args.e2e_steps, args.steps))
    # The read-back of step i runs on a side stream while step i+1's inputs go
    # up and its launches run on the launch stream (the link is full duplex).
    # The outputs alternate between two device buffers, so step i+1 does not
    # wait for step i's read-back, only for step i-1's, which used the same
    # buffer.  Every step still uploads its inputs and reads back its result.
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    out_sets = [outs, [torch.empty_like(o) for o in outs]]
    read_back = [None, None]  # the last read-back of each output set

    def one_step(k):
        for name, p in pinned:
            targets[name].view(torch.int16).copy_(p.view(torch.int16), non_blocking=True)
        if read_back[k % 2] is not None:
            main.wait_event(read_back[k % 2])
        step.d["C"] = out_sets[k % 2]
        for _, f in launches:
            f()
        computed = torch.cuda.Event()
        computed.record(main)
        side.wait_event(computed)
        with torch.cuda.stream(side):
            for o, h in zip(out_sets[k % 2], out_host):
                h.copy_(o, non_blocking=True)
        done = torch.cuda.Event()
        done.record(side)
        read_back[k % 2] = done

    for k in range(2):
        one_step(k)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for k in range(n):
        one_step(k)
    torch.cuda.synchronize()
    dt = max_over_ranks((time.perf_counter() - t0) / n, dist, "cuda")
    step.d["C"] = outs
    return {"value": round(job_throughput(flops, dt, world) / 1e12, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n, "ms_per_step": round(dt * 1e3, 4)}


# ------------------------------------------------------------------ oracle arm
def oracle_sample(workload, seed=0):
    """A bounded sample of one step for the CPU oracle: (work fn, flops, description)."""
    import oracle
    import synth
    oracle.build()
    if workload in ("mla", "tiny"):
        d = synth.mla(seed=seed) if workload == "mla" else synth.tiny(seed=seed)
        Ws = [d["Wq"], d["Wkv"]] if workload == "mla" else [d["B"]]
        rows = 32 if workload == "mla" else 128
        A = np.ascontiguousarray(d["A"][:rows])

        def work():
            qa, sa = oracle.quant_1x128_rows(A)
            for W in Ws:
                qb, sb = oracle.quant_128x128(W)
                oracle.gemm_blockscaled(qa, sa, qb, sb, 0)
        flops = sum(2.0 * rows * W.shape[0] * W.shape[1] for W in Ws)
        return work, flops, f"{rows} of {d['A'].shape[0]} rows of A (quantise + both GEMMs) plus full weight quantisation"
    if workload in ("mla_ue8m0", "ffn_ue8m0"):
        d = synth.ffn(seed=seed, M=16, N=2048) if workload == "ffn_ue8m0" else synth.mla(seed=seed)
        A = np.ascontiguousarray(d["A"][:16])
        Ws = [d["B"]] if workload == "ffn_ue8m0" else [d["Wq"], d["Wkv"]]

        def work():
            qa, sa = oracle.quant_1x128_rows_pow2(A)
            for W in Ws:
                qb, sb = oracle.quant_128x128_pow2(W)
                oracle.gemm_exact_sum(qa, sa, qb, sb, 0)
        flops = sum(2.0 * 16 * W.shape[0] * W.shape[1] for W in Ws)
        return work, flops, "16 rows of A (power-of-two quantisation + exact-sum GEMM) against the full weights"
    if workload == "ffn":
        d = synth.ffn(seed=seed, M=16, N=18432)
        A, B = d["A"], d["B"][:2048]

        def work():
            qa, sa = oracle.quant_1x128_rows(A)
            qb, sb = oracle.quant_128x128(B)
            oracle.gemm_blockscaled(qa, sa, qb, sb, 0)
        return work, 2.0 * 16 * 2048 * 7168, "16 rows x 2048 columns of the 16384x18432x7168 GEMM, with their quantisation"
    if workload == "wgrad":
        d = synth.wgrad(seed=seed)
        dY, X = d["dY"][:, :16], d["X"][:, :512]
        dY, X = np.ascontiguousarray(dY), np.ascontiguousarray(X)

        def work():
            qd, sd = oracle.quant_1x128_cols(dY)
            qx, sx = oracle.quant_1x128_cols(X)
            oracle.gemm_blockscaled(qd, sd, qx, sx, 1)
        return work, 2.0 * 16 * 512 * 16384, "16 x 512 outputs of dW (K = 16384 tokens), with their token-wise quantisation"
    if workload == "dgrad":
        d = synth.dgrad(seed=seed, T=16)
        dY, W = d["dY"], np.ascontiguousarray(d["W"][:, :2048])

        def work():
            qd, sd = oracle.quant_1x128_rows(dY)
            _, _, qwt, swt = oracle.quant_128x128_t(W)
            oracle.gemm_blockscaled(qd, sd, qwt, swt, 0)
        return work, 2.0 * 16 * 2048 * 18432, "16 rows x 2048 columns of dX (K = 18432), with their quantisation"
    if workload == "moe_chain":
        tok = synth.moe_tokens(seed=seed)[:1]
        cent, bias = synth.moe_router(seed=seed)

        def work():
            l = oracle.route_logits(tok, cent)
            sel, gate = oracle.route_select(l, bias, 8)
            ys = []
            for t in range(tok.shape[0]):
                qa, sa = oracle.quant_1x128_rows(np.ascontiguousarray(np.repeat(tok[t:t + 1], 8, axis=0)))
                for j, e in enumerate(sel[t]):
                    qu, su = oracle.quant_128x128(synth.moe_weights("up", int(e), int(e) + 1, seed=seed)[0])
                    h, sh = oracle.swiglu_quant(oracle.gemm_blockscaled(qa[j:j + 1], sa[:, j:j + 1], qu, su, 0))
                    qd, sd = oracle.quant_128x128(synth.moe_weights("down", int(e), int(e) + 1, seed=seed)[0])
                    ys.append(oracle.bf16_round(oracle.gemm_blockscaled(h, sh, qd, sd, 0)))
            oracle.moe_combine(np.concatenate(ys), np.arange(len(ys), dtype=np.int32).reshape(-1, 8), gate)
        flops = 1 * 8 * (2.0 * 4096 * 7168 + 2.0 * 7168 * 2048)
        return work, flops, ("1 of 4096 tokens through the layer (routing over all 256 experts, each token's "
                             "8 experts' weight quantisation, up GEMM + SwiGLU, down GEMM, combine)")
    if workload == "moe":
        tok = synth.moe_tokens(seed=seed, T=64)
        W = synth.moe_weights("up", 0, 1, seed=seed)[0][:1024]

        def work():
            qa, sa = oracle.quant_1x128_rows(tok)
            qb, sb = oracle.quant_128x128(W)
            oracle.gemm_blockscaled(qa, sa, qb, sb, 0)
        return work, 2.0 * 64 * 1024 * 7168, "64 rows x 1024 columns of one expert's up GEMM, with quantisation"
    raise KeyError(workload)


def run_cpu_baseline(workload, budget_s=20.0):
    import oracle
    work, flops, desc = oracle_sample(workload)
    work()  # first call builds tables
    reps, t = 0, 0.0
    t0 = time.perf_counter()
    while True:
        work()
        reps += 1
        t = time.perf_counter() - t0
        if t > budget_s or reps >= 50:
            break
    return {"value": round(flops * reps / t / 1e12, 8), "unit": "TFLOP/s", "cores": oracle.nthreads(),
            "kind": "oracle", "sample": desc, "reps": reps, "seconds": round(t, 2)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    work, flops, desc = oracle_sample(args.workload)
    import oracle
    for _ in range(args.warmup):
        work()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        work()
        times.append(time.perf_counter() - t0)
    ms = float(np.mean(times)) * 1e3
    value = flops / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 8), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 codes, f64 chunk sums, f32 promotion", "data": "synthetic (seeded)",
        "config": bench_config(args, world),
        "cpu_baseline": {"value": round(value, 8), "unit": "TFLOP/s", "cores": oracle.nthreads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default="ffn", choices=["mla", "ffn", "wgrad", "dgrad", "moe", "moe_chain", "tiny",
                                                        "mla_ue8m0", "ffn_ue8m0"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="keep warming up (back to back) until this long has passed")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush-mb", type=int, default=256, help="L2 flush buffer (> 126 MB L2)")
    ap.add_argument("--flush-mode", choices=("write", "write+read"), default="write+read",
                    help="L2 flush: a write, or a write followed by a read of a second buffer")
    ap.add_argument("--tokens", type=int, default=4096, help="moe_chain: tokens per step")
    ap.add_argument("--experts", type=int, default=256, help="moe_chain: routed experts (a multiple of 16)")
    args = ap.parse_args()
    if args.experts % 16 != 0 or not 16 <= args.experts <= 1024 or args.tokens < 1:
        ap.error("--experts must be a multiple of 16 in 16..1024 and --tokens positive")
    MOE_CHAIN.update(tokens=args.tokens, experts=args.experts)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", args.gpus))
    if args.impl == "reference":
        args.steps = args.steps or 5
        args.warmup = args.warmup if args.warmup is not None else 1
        run_reference(args, rank, world)
        return
    default_steps = {"mla": 10000, "tiny": 10000, "ffn": 200, "wgrad": 1000, "dgrad": 200, "moe": 300,
                     "moe_chain": 200, "mla_ue8m0": 10000, "ffn_ue8m0": 200}[args.workload]
    args.steps = args.steps or default_steps
    args.warmup = max(3, args.warmup if args.warmup is not None else 20)
    run_ours(args, rank, world)


if __name__ == "__main__":
    main()
