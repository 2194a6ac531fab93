"""CPU oracle for fine-grained FP8 (E4M3) quantisation and the block-scaled GEMM.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark load it; the product path never does.  The arithmetic lives
in ``oracle.c`` (plain C99, built with no fast-math and no FP contraction);
this module only marshals numpy arrays into it.  Nothing here is shared with
the CUDA library.

Sources: "DeepSeek-V3 技术报告：从 671B MoE 到低成本训练系统" (xutianle.me)
§6 (FP8 GEMMs for Fprop/Dgrad/Wgrad, outputs in BF16 or FP32), §6.1 (1x128
activation tiles, 128x128 weight blocks, online scales), §6.2 (FP32 promotion
after every 128 FP8 products), §2 and §4 (the MoE layer: sigmoid routing with
a selection bias, top-8 of 256 experts, SwiGLU experts).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against the format definition, torch's independent float8_e4m3fn
conversion, exact rational brute force and closed-form identities.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
          "-shared", "-pthread", "-D_POSIX_C_SOURCE=200809L"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_bf16_rne.argtypes = [ctypes.c_float]
        L.orc_bf16_rne.restype = ctypes.c_uint16
        L.orc_tile_scale.argtypes = [ctypes.c_float]
        L.orc_tile_scale.restype = ctypes.c_float
        for fn in (L.orc_quant_1x128_rows, L.orc_quant_1x128_cols, L.orc_quant_128x128):
            fn.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, i32]
            fn.restype = None
        L.orc_gemm_blockscaled.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32,
                                           i64, i64, vp, i64, vp, i32]
        L.orc_gemm_blockscaled.restype = None
        L.orc_bf16_round_buffer.argtypes = [vp, vp, i64]
        L.orc_bf16_round_buffer.restype = None
        L.orc_e4m3_encode_buffer.argtypes = [vp, vp, i64, i32]
        L.orc_e4m3_encode_buffer.restype = None
        L.orc_e4m3_encode_patterns.argtypes = [ctypes.c_uint64, i64, vp, i32]
        L.orc_e4m3_encode_patterns.restype = None
        L.orc_pow2_exponent.argtypes = [ctypes.c_float]
        L.orc_pow2_exponent.restype = i32
        for fn in (L.orc_quant_1x128_rows_pow2, L.orc_quant_128x128_pow2):
            fn.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, i32]
            fn.restype = None
        L.orc_gemm_exact_sum.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32, i64, i64, vp, i64, vp, i32]
        L.orc_gemm_exact_sum.restype = None
        L.orc_route_logits.argtypes = [vp, i64, i64, i64, vp, i64, i64, vp, i32]
        L.orc_route_logits.restype = None
        L.orc_route_select.argtypes = [vp, i64, i64, vp, i32, vp, vp]
        L.orc_route_select.restype = None
        L.orc_route_gates.argtypes = [vp, i64, i64, vp, i32, vp]
        L.orc_route_gates.restype = None
        L.orc_route_permute.argtypes = [vp, i64, i32, i64, vp, vp, vp]
        L.orc_route_permute.restype = None
        L.orc_swiglu_quant.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, i32]
        L.orc_swiglu_quant.restype = None
        L.orc_moe_combine.argtypes = [vp, i64, i64, vp, vp, i64, i32, vp, i64, i32]
        L.orc_moe_combine.restype = None
        _lib = L
    return _lib


def nthreads() -> int:
    return max(1, os.cpu_count() or 1)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return np.ascontiguousarray(a)


# --- format ---------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e4m3_encode(y: float) -> int:
    return int(lib().orc_e4m3_encode(float(np.float32(y))))


def e4m3_encode_array(x: np.ndarray, threads: int | None = None) -> np.ndarray:
    x = _c(x.astype(np.float32, copy=False), np.float32)
    q = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_buffer(_p(x), _p(q), x.size, threads or nthreads())
    return q


def e4m3_encode_patterns(lo: int, n: int, threads: int | None = None) -> np.ndarray:
    """Encode the FP32 values whose bit patterns are lo, lo+1, ..., lo+n-1."""
    q = np.empty(n, np.uint8)
    lib().orc_e4m3_encode_patterns(lo, n, _p(q), threads or nthreads())
    return q


def decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def tile_scale(amax: float) -> float:
    return float(lib().orc_tile_scale(float(np.float32(amax))))


def bf16_round(x: np.ndarray) -> np.ndarray:
    x = _c(x.astype(np.float32, copy=False), np.float32)
    y = np.empty(x.shape, np.uint16)
    lib().orc_bf16_round_buffer(_p(x), _p(y), x.size)
    return y


# --- quantisers -------------------------------------------------------------

def quant_1x128_rows(x_bf16: np.ndarray, threads: int | None = None):
    """x_bf16: uint16 [M, K].  Returns codes uint8 [M, K], scales f32 [K/128, M]."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    lib().orc_quant_1x128_rows(_p(x), M, K, K, _p(q), K, _p(s), M, threads or nthreads())
    return q, s


def quant_1x128_cols(x_bf16: np.ndarray, threads: int | None = None):
    """x_bf16: uint16 [T, C]; tiles of 128 tokens per channel.
    Returns codes uint8 [C, T] (tokens contiguous) and scales f32 [T/128, C]."""
    x = _c(x_bf16, np.uint16)
    T, C = x.shape
    assert T % 128 == 0
    q = np.empty((C, T), np.uint8)
    s = np.empty((T // 128, C), np.float32)
    lib().orc_quant_1x128_cols(_p(x), T, C, C, _p(q), T, _p(s), C, threads or nthreads())
    return q, s


def quant_128x128(w_bf16: np.ndarray, threads: int | None = None):
    """w_bf16: uint16 [N, K].  Returns codes uint8 [N, K], scales f32 [ceil(N/128), K/128]."""
    w = _c(w_bf16, np.uint16)
    N, K = w.shape
    assert K % 128 == 0
    q = np.empty((N, K), np.uint8)
    s = np.empty(((N + 127) // 128, K // 128), np.float32)
    lib().orc_quant_128x128(_p(w), N, K, K, _p(q), K, _p(s), K // 128, threads or nthreads())
    return q, s


def quant_128x128_t(w_bf16: np.ndarray, threads: int | None = None):
    """128x128 block quantisation of w [N, K] and its transposed form (V3 report §6: the Dgrad GEMM
    takes the FP8 weights; §6.1: 128x128 blocks).  A block of w^T holds the same elements as the
    block of w it comes from, so its amax, scale and codes are the same: the transposed
    quantisation is the transpose of the codes and of the block-scale grid.
    Returns q [N, K], s [ceil(N/128), K/128], qt [K, N], st [K/128, ceil(N/128)]."""
    q, s = quant_128x128(w_bf16, threads)
    return q, s, np.ascontiguousarray(q.T), np.ascontiguousarray(s.T)


# --- GEMM -------------------------------------------------------------------

def gemm_blockscaled(A: np.ndarray, sa: np.ndarray, B: np.ndarray, sb: np.ndarray,
                     b_mode: int = 0, rows=None, threads: int | None = None) -> np.ndarray:
    """FP32 accumulators of C = A * B^T with per-chunk FP32 promotion.

    A: codes [M, K]; sa: [K/128, M]; B: codes [N, K];
    sb: [ceil(N/128), K/128] (b_mode 0) or [K/128, N] (b_mode 1).
    rows: optional list of row indices of A; returns f32 [len(rows), N]."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2 and K % 128 == 0
    assert sa.shape == (K // 128, M)
    if b_mode == 0:
        assert sb.shape == ((N + 127) // 128, K // 128)
    else:
        assert sb.shape == (K // 128, N)
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = _c(np.asarray(rows, dtype=np.int64), np.int64)
    out = np.empty((rows.size, N), np.float32)
    lib().orc_gemm_blockscaled(_p(A), K, _p(sa), M, _p(B), K, _p(sb), sb.shape[1], b_mode,
                               N, K, _p(rows), rows.size, _p(out), threads or nthreads())
    return out


def gemm_blockscaled_bf16(A, sa, B, sb, b_mode=0, rows=None, threads=None) -> np.ndarray:
    """As gemm_blockscaled, rounded to BF16 bits (uint16)."""
    return bf16_round(gemm_blockscaled(A, sa, B, sb, b_mode, rows, threads))


def grouped_gemm(A: np.ndarray, sa: np.ndarray, B: np.ndarray, sb: np.ndarray,
                 offsets: np.ndarray, rows=None, threads: int | None = None) -> np.ndarray:
    """Grouped (MoE) GEMM: rows offsets[e]..offsets[e+1]-1 of A use expert e's
    weights B[e] ([G, N, K]) and block scales sb[e] ([G, ceil(N/128), K/128]).
    Returns FP32 accumulators for the requested rows (default: all), [len(rows), N]."""
    offsets = np.asarray(offsets, dtype=np.int64)
    G, N, K = B.shape
    M = A.shape[0]
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, N), np.float32)
    expert_of = np.searchsorted(offsets, rows, side="right") - 1
    for e in np.unique(expert_of):
        sel = np.nonzero(expert_of == e)[0]
        out[sel] = gemm_blockscaled(A, sa, B[e], sb[e], 0, rows[sel], threads)
    return out


# --- the MoE chain (V3 report §2 DeepSeekMoE, §4 aux-loss-free routing) ----

def route_logits(x_bf16: np.ndarray, centroids: np.ndarray, threads: int | None = None) -> np.ndarray:
    """Affinity logits l[t, e] = u_t . c_e in double (exact products, a double sum:
    within D * 2^-53 * sum|u c| of the exact value).  x_bf16: uint16 [T, D];
    centroids: f32 [E, D].  Returns f64 [T, E]."""
    x = _c(x_bf16, np.uint16)
    c = _c(centroids, np.float32)
    T, D = x.shape
    E = c.shape[0]
    out = np.empty((T, E), np.float64)
    lib().orc_route_logits(_p(x), T, D, D, _p(c), D, E, _p(out), threads or nthreads())
    return out


def route_select(logits: np.ndarray, bias: np.ndarray, topk: int):
    """Top-k experts per token by sigmoid(l) + b (double; ties to the lower index), listed in
    increasing expert order, with gates s_e / sum of the chosen s.  logits: [T, E] (taken as
    double).  Returns (sel int32 [T, k], gate f32 [T, k])."""
    l = _c(logits, np.float64)
    b = _c(bias, np.float32)
    T, E = l.shape
    assert 0 < topk <= E
    sel = np.empty((T, topk), np.int32)
    gate = np.empty((T, topk), np.float32)
    lib().orc_route_select(_p(l), T, E, _p(b), topk, _p(sel), _p(gate))
    return sel, gate


def route_gates(logits: np.ndarray, sel: np.ndarray):
    """Gates of a given selection sel int32 [T, k]: s_e / sum of the chosen s (double, in
    the listed order), rounded to f32.  logits: [T, E] (taken as double)."""
    l = _c(logits, np.float64)
    sl = _c(sel, np.int32)
    T, E = l.shape
    k = sl.shape[1]
    gate = np.empty((T, k), np.float32)
    lib().orc_route_gates(_p(l), T, E, _p(sl), k, _p(gate))
    return gate


def route_permute(sel: np.ndarray, E: int):
    """Rows grouped by expert, tokens in increasing order within an expert.  Returns
    (offsets int32 [E+1], token_of_row int32 [T*k], row_of int32 [T, k])."""
    sel = _c(sel, np.int32)
    T, k = sel.shape
    offsets = np.empty(E + 1, np.int32)
    tor = np.empty(T * k, np.int32)
    row_of = np.empty((T, k), np.int32)
    lib().orc_route_permute(_p(sel), T, k, E, _p(offsets), _p(tor), _p(row_of))
    return offsets, tor, row_of


def swiglu_quant(acc: np.ndarray, threads: int | None = None):
    """SwiGLU of up-projection accumulators acc f32 [R, 2*Nh] (gate | up) and its 1x128
    quantisation.  Returns codes uint8 [R, Nh] and scales f32 [Nh/128, R]."""
    a = _c(acc, np.float32)
    R, N2 = a.shape
    Nh = N2 // 2
    assert N2 == 2 * Nh and Nh % 128 == 0
    q = np.empty((R, Nh), np.uint8)
    s = np.empty((Nh // 128, R), np.float32)
    lib().orc_swiglu_quant(_p(a), R, Nh, N2, _p(q), Nh, _p(s), R, threads or nthreads())
    return q, s


def moe_combine(Y_bf16: np.ndarray, row_of: np.ndarray, gate: np.ndarray,
                threads: int | None = None) -> np.ndarray:
    """y[t] = sum_j gate[t, j] * Y[row_of[t, j]] (FP32 fused multiply-adds in j order, then
    BF16).  Y_bf16: uint16 [R, N].  Returns uint16 [T, N]."""
    Y = _c(Y_bf16, np.uint16)
    row_of = _c(row_of, np.int32)
    gate = _c(gate, np.float32)
    T, k = row_of.shape
    N = Y.shape[1]
    out = np.empty((T, N), np.uint16)
    lib().orc_moe_combine(_p(Y), N, N, _p(row_of), _p(gate), T, k, _p(out), N, threads or nthreads())
    return out


# --- power-of-two (UE8M0) scales --------------------------------------------

def token_shards(T: int, world: int):
    """Token boundaries of `world` data-parallel ranks: contiguous ranges of whole
    128-token tiles, rank r holding tiles [floor(r n / world), floor((r+1) n / world))
    of the n = T / 128 tiles.  Returns [(t0, t1)] per rank."""
    assert T % 128 == 0 and world >= 1
    n = T // 128
    return [(128 * (r * n // world), 128 * ((r + 1) * n // world)) for r in range(world)]


def wgrad_dp(dY_bf16: np.ndarray, X_bf16: np.ndarray, world: int, threads: int | None = None):
    """Data-parallel Wgrad over `world` ranks ([V3-report] §7: ZeRO-1 data parallelism
    over the batch; §6: the Wgrad GEMM in FP8 with FP32 output).  Each rank's shard of
    tokens (token_shards) gives dW_r = dY_r^T X_r by the single-rank rule (token-wise
    1x128 tiles, FP32 promotion every 128 tokens, gemm_blockscaled in row-scale mode);
    the ranks' partials are then summed in FP32 in rank order:
    dW = ((dW_0 + dW_1) + dW_2) + ...  Returns (dW f32 [Cout, Cin], [dW_r])."""
    dY = _c(dY_bf16, np.uint16)
    X = _c(X_bf16, np.uint16)
    assert dY.shape[0] == X.shape[0]
    parts = []
    for t0, t1 in token_shards(dY.shape[0], world):
        qd, sd = quant_1x128_cols(dY[t0:t1], threads)
        qx, sx = quant_1x128_cols(X[t0:t1], threads)
        parts.append(gemm_blockscaled(qd, sd, qx, sx, 1, threads=threads))
    acc = parts[0].copy()
    for part in parts[1:]:
        acc = np.add(acc, part, dtype=np.float32)
    return acc, parts


def pow2_exponent(amax: float) -> int:
    """e of the tile scale 2^e: the smallest integer with amax <= 448 * 2^e (e >= -127; 0 for amax 0)."""
    return int(lib().orc_pow2_exponent(float(amax)))


def quant_1x128_rows_pow2(x_bf16: np.ndarray, threads: int | None = None):
    """1x128 tiles with power-of-two scales: codes uint8 [M, K], scales f32 [K/128, M] (each 2^e)."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    lib().orc_quant_1x128_rows_pow2(_p(x), M, K, K, _p(q), K, _p(s), M, threads or nthreads())
    return q, s


def quant_128x128_pow2(w_bf16: np.ndarray, threads: int | None = None):
    """128x128 blocks with power-of-two scales: codes uint8 [N, K], scales f32 [ceil(N/128), K/128]."""
    w = _c(w_bf16, np.uint16)
    N, K = w.shape
    assert K % 128 == 0
    q = np.empty((N, K), np.uint8)
    s = np.empty(((N + 127) // 128, K // 128), np.float32)
    lib().orc_quant_128x128_pow2(_p(w), N, K, K, _p(q), K, _p(s), K // 128, threads or nthreads())
    return q, s


def gemm_exact_sum(A, sa, B, sb, b_mode: int = 0, rows=None, threads: int | None = None) -> np.ndarray:
    """fl32 of the double sum over all K of the scaled code products (layouts as gemm_blockscaled)."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    M, K = A.shape
    N = B.shape[0]
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, N), np.float32)
    lib().orc_gemm_exact_sum(_p(A), K, _p(sa), M, _p(B), K, _p(sb), sb.shape[1], b_mode,
                             N, K, _p(rows), rows.size, _p(out), threads or nthreads())
    return out
