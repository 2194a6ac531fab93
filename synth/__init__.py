"""Seeded synthetic inputs for the FP8 block-scaled GEMM workloads.

This module serves both sides of every parity check (the CUDA library and
the CPU oracle) and holds none of the quantisation or GEMM arithmetic: it
draws counter-based random numbers (``synth.c``), rounds them to BF16 input
tensors and, for the MoE workload, forms the expert groups from routing
scores.

Workloads (shapes from the DeepSeek-V3 pages: MLA q latent 1536, KV latent
512 + RoPE key 64, 256 routed experts, top-8, expert width 2048; hidden size
7168):
  1 tiny   A 128x512 ~N(0,1), 1% of entries x50; B 256x512 ~N(0,0.02)
  2 mla    A 4096x7168 ~N(0,1); W_q 1536x7168, W_kv 576x7168 ~N(0,0.02)
  3 moe    tokens 4096x7168 ~N(0,1) routed top-8 of 256 experts (sigmoid
           affinity plus per-expert bias ~N(0,0.5)) -> 32768 grouped rows;
           up W [256][4096][7168], down input 32768x2048 ~N(0,1),
           down W [256][7168][2048], weights ~N(0,0.02)
  4 wgrad  dY 16384x2048, X 16384x7168 ~N(0,1e-2)
  5 ffn    A 16384x7168 Student-t(df=3); B 18432x7168 ~N(0,0.02)

Every tensor has its own stream key, key = mix64(seed ^ (workload << 8) ^ tensor).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off",
                               "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        L.syn_mix64.argtypes = [u64]
        L.syn_mix64.restype = u64
        L.syn_u64.argtypes = [u64, u64]
        L.syn_u64.restype = u64
        L.syn_uniform.argtypes = [u64, u64]
        L.syn_uniform.restype = ctypes.c_double
        L.syn_normal.argtypes = [u64, u64]
        L.syn_normal.restype = ctypes.c_double
        L.syn_fill.argtypes = [ctypes.c_int, u64, u64, u64, i64, ctypes.c_double,
                               ctypes.c_double, ctypes.c_double, vp, vp, ctypes.c_int]
        L.syn_fill.restype = None
        L.syn_route_logits.argtypes = [vp, vp, i64, i64, i64, vp, ctypes.c_int]
        L.syn_route_logits.restype = None
        _lib = L
    return _lib


def _threads():
    return max(1, os.cpu_count() or 1)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def key(workload: int, tensor: int, seed: int = 0) -> int:
    return int(lib().syn_mix64((seed ^ (workload << 8) ^ tensor) & (2**64 - 1)))


NORMAL, OUTLIER, STUDENT_T = 0, 1, 2


def fill_bf16(kind: int, k: int, shape, sigma: float = 1.0, p: float = 0.0,
              factor: float = 1.0, k2: int = 0, start: int = 0, out=None) -> np.ndarray:
    """BF16 bit patterns (uint16) of the given distribution, elements start.."""
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    lib().syn_fill(kind, k, k2, start, n, sigma, p, factor, _p(out), None, _threads())
    return out


def fill_f32(kind: int, k: int, shape, sigma: float = 1.0, p: float = 0.0,
             factor: float = 1.0, k2: int = 0, start: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(shape, np.float32)
    lib().syn_fill(kind, k, k2, start, n, sigma, p, factor, None, _p(out), _threads())
    return out


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.uint32) << 16).view(np.float32)


# --- workloads --------------------------------------------------------------

WORKLOADS = {1: "tiny", 2: "mla", 3: "moe", 4: "wgrad", 5: "ffn", 6: "dgrad"}


def tiny(seed: int = 0, M: int = 128, N: int = 256, K: int = 512):
    """Workload 1: A [M,K] ~N(0,1) with 1% of entries times 50, B [N,K] ~N(0,0.02)."""
    A = fill_bf16(OUTLIER, key(1, 0, seed), (M, K), 1.0, 0.01, 50.0, k2=key(1, 1, seed))
    B = fill_bf16(NORMAL, key(1, 2, seed), (N, K), 0.02)
    return {"A": A, "B": B}


def mla(seed: int = 0, M: int = 4096, K: int = 7168, Nq: int = 1536, Nkv: int = 576):
    """Workload 2: MLA down-projections (q latent 1536; KV latent 512 + RoPE key 64)."""
    A = fill_bf16(NORMAL, key(2, 0, seed), (M, K), 1.0)
    Wq = fill_bf16(NORMAL, key(2, 1, seed), (Nq, K), 0.02)
    Wkv = fill_bf16(NORMAL, key(2, 2, seed), (Nkv, K), 0.02)
    return {"A": A, "Wq": Wq, "Wkv": Wkv}


def wgrad(seed: int = 0, T: int = 16384, Cout: int = 2048, Cin: int = 7168):
    """Workload 4: dW = dY^T X, both operands tiled 1x128 along tokens."""
    dY = fill_bf16(NORMAL, key(4, 0, seed), (T, Cout), 1e-2)
    X = fill_bf16(NORMAL, key(4, 1, seed), (T, Cin), 1e-2)
    return {"dY": dY, "X": X}


def ffn(seed: int = 0, M: int = 16384, N: int = 18432, K: int = 7168):
    """Workload 5: heavy-tailed activations (Student-t, df=3) against ~N(0,0.02) weights."""
    A = fill_bf16(STUDENT_T, key(5, 0, seed), (M, K), 1.0, 3.0, k2=key(5, 1, seed))
    B = fill_bf16(NORMAL, key(5, 2, seed), (N, K), 0.02)
    return {"A": A, "B": B}


# MoE (workload 3) ------------------------------------------------------------

def dgrad(seed: int = 0, T: int = 16384, Cout: int = 18432, Cin: int = 7168):
    """Workload 6: the data gradient of the large FFN layer, dX [T, Cin] = dY W, with
    dY [T, Cout] ~N(0, 1e-2) and the FFN weight W [Cout, Cin] ~N(0, 0.02) (the same stream
    as workload 5's B when the sizes match)."""
    dY = fill_bf16(NORMAL, key(6, 0, seed), (T, Cout), 1e-2)
    W = fill_bf16(NORMAL, key(5, 2, seed), (Cout, Cin), 0.02)
    return {"dY": dY, "W": W}


def moe_tokens(seed: int = 0, T: int = 4096, D: int = 7168):
    return fill_bf16(NORMAL, key(3, 0, seed), (T, D), 1.0)


def moe_route(tokens_bf16: np.ndarray, E: int = 256, topk: int = 8, seed: int = 0):
    """Group rows by expert the way the aux-loss-free router selects them
    (DeepSeek-V3 report, §4): sigmoid affinity s = sigmoid(u . e_i) to centroid
    e_i ~ N(0, 1/D), top-k on s + b_i with b_i ~ N(0, 0.5), ties to the lower
    expert index.  Returns (offsets int32 [E+1], token index per grouped row
    int64 [T*topk]); rows are sorted by (expert, token)."""
    T, D = tokens_bf16.shape
    cent = fill_f32(NORMAL, key(3, 1, seed), (E, D), 1.0 / np.sqrt(D))
    bias = fill_f32(NORMAL, key(3, 2, seed), (E,), 0.5).astype(np.float64)
    logits = np.empty((T, E), np.float64)
    tok = np.ascontiguousarray(tokens_bf16)
    lib().syn_route_logits(_p(tok), _p(cent), T, D, E, _p(logits), _threads())
    s = 1.0 / (1.0 + np.exp(-logits))
    score = s + bias[None, :]
    order = np.argsort(-score, axis=1, kind="stable")[:, :topk]
    experts = order.reshape(-1)
    tokens = np.repeat(np.arange(T, dtype=np.int64), topk)
    perm = np.lexsort((tokens, experts))
    counts = np.bincount(experts, minlength=E)
    offsets = np.zeros(E + 1, np.int64)
    np.cumsum(counts, out=offsets[1:])
    return offsets.astype(np.int32), tokens[perm]


def moe_router(seed: int = 0, E: int = 256, D: int = 7168):
    """Router inputs of workload 3: expert centroids f32 [E, D] ~N(0, 1/D) and selection
    biases f32 [E] ~N(0, 0.5) (the streams moe_route draws from)."""
    cent = fill_f32(NORMAL, key(3, 1, seed), (E, D), 1.0 / np.sqrt(D))
    bias = fill_f32(NORMAL, key(3, 2, seed), (E,), 0.5)
    return cent, bias


def moe_weights(which: str, e_lo: int, e_hi: int, seed: int = 0,
                N: int | None = None, K: int | None = None) -> np.ndarray:
    """Expert weights e_lo..e_hi-1 of the up (N=4096, K=7168) or down
    (N=7168, K=2048) projection, BF16 [e_hi-e_lo, N, K]; any expert range is
    drawn on demand from the same stream."""
    if which == "up":
        N, K, t = (N or 4096), (K or 7168), 3
    else:
        N, K, t = (N or 7168), (K or 2048), 4
    n = N * K
    out = np.empty((e_hi - e_lo, N, K), np.uint16)
    fill_bf16(NORMAL, key(3, t, seed), out.shape, 0.02, start=e_lo * n, out=out)
    return out


def moe_down_input(seed: int = 0, R: int = 32768, K: int = 2048):
    return fill_bf16(NORMAL, key(3, 5, seed), (R, K), 1.0)
