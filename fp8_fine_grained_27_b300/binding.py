"""ctypes binding of libfp8bs (argument marshalling only).

Each function takes torch CUDA tensors, allocates missing outputs with torch
(device memory is the caller's), and calls the C entry point of the same
name on the current torch stream.  All arithmetic happens in the library's
kernels; a non-zero status raises :class:`Fp8bsError`.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# FP8BS_LIBRARY=debug selects the bounds-checked build (libfp8bs_debug.so)
LIB_PATH = os.path.join(_HERE, "libfp8bs_debug.so" if os.environ.get("FP8BS_LIBRARY") == "debug" else "libfp8bs.so")

OK, EINVAL, EALIGN, EARCH, ECUDA, ETIMEOUT = 0, -1, -2, -3, -4, -5

# every symbol include/fp8bs.h declares
EXPORTS = (
    "fp8_quant_1x128", "fp8_quant_128x128", "fp8_quant_128x128_t", "fp8_quant_1x128_ue8m0",
    "fp8_quant_128x128_ue8m0", "fp8_quant_act_weight", "fp8_gemm_ue8m0", "fp8_gemm_blockscaled",
    "fp8_grouped_gemm_moe", "fp8_moe_route_workspace_size", "fp8_moe_route", "fp8_moe_route_noalloc",
    "fp8_quant_1x128_gather", "fp8_grouped_gemm_moe_swiglu", "fp8_moe_combine", "fp8bs_e4m3_encode", "fp8bs_status_string",
    "fp8bs_get_device_error",
    "fp8bs_selftest_timeout", "fp8bs_selftest_division", "fp8bs_set_gemm_tile_n",
    "fp8bs_set_gemm_split_last_round", "fp8bs_version", "fp8bs_debug_build", "fp8bs_debug_site", "fp8bs_gemm_clock",
)


class Fp8bsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {lib().fp8bs_status_string(status).decode()} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libfp8bs.so (built in-tree by __graft_entry__.build or build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run fp8_fine_grained_27_b300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.fp8_quant_1x128.argtypes = [vp, i64, i64, i64, i32, vp, i64, vp, i64, vp]
        L.fp8_quant_128x128.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp]
        L.fp8_quant_1x128_ue8m0.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp]
        L.fp8_quant_128x128_ue8m0.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp]
        L.fp8_quant_act_weight.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, i64, i64, vp, i64, vp, i64,
                                           i32, vp]
        L.fp8_gemm_ue8m0.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32, i64, i64, i64, vp]
        L.fp8_quant_128x128_t.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp]
        L.fp8_gemm_blockscaled.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32, vp, i64, i32, i64, i64, i64, vp]
        L.fp8_grouped_gemm_moe.argtypes = [vp, i64, vp, i64, vp, vp, vp, i32, i64, vp, i64, i32, i64, i64, vp]
        L.fp8_moe_route_workspace_size.argtypes = [i32]
        L.fp8_moe_route_workspace_size.restype = i64
        L.fp8_moe_route.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, i64, vp]
        L.fp8_moe_route_noalloc.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.fp8_quant_1x128_gather.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp]
        L.fp8_grouped_gemm_moe_swiglu.argtypes = [vp, i64, vp, i64, vp, vp, vp, i32, i64, vp, i64, vp, i64, i64,
                                                  i64, vp]
        L.fp8_moe_combine.argtypes = [vp, i64, i64, vp, vp, i64, i32, i64, vp, i64, vp]
        L.fp8bs_e4m3_encode.argtypes = [vp, vp, i64, vp]
        L.fp8bs_status_string.argtypes = [i32]
        L.fp8bs_status_string.restype = ctypes.c_char_p
        L.fp8bs_get_device_error.argtypes = [vp]
        L.fp8bs_selftest_timeout.argtypes = [i64, vp]
        L.fp8bs_selftest_division.argtypes = [vp, vp]
        L.fp8bs_set_gemm_tile_n.argtypes = [i32]
        L.fp8bs_set_gemm_split_last_round.argtypes = [i32]
        L.fp8bs_debug_build.argtypes = []
        L.fp8bs_debug_site.argtypes = [vp]
        L.fp8bs_gemm_clock.argtypes = [vp, vp, i32, vp]
        L.fp8bs_version.restype = ctypes.c_char_p
        for name in ("fp8_quant_1x128", "fp8_quant_128x128", "fp8_quant_128x128_t", "fp8_quant_1x128_ue8m0",
                     "fp8_quant_128x128_ue8m0", "fp8_quant_act_weight", "fp8_gemm_ue8m0", "fp8_gemm_blockscaled",
                     "fp8_grouped_gemm_moe", "fp8_moe_route", "fp8_moe_route_noalloc", "fp8_quant_1x128_gather",
                     "fp8_grouped_gemm_moe_swiglu", "fp8_moe_combine", "fp8bs_e4m3_encode", "fp8bs_get_device_error",
                     "fp8bs_selftest_timeout", "fp8bs_selftest_division", "fp8bs_set_gemm_tile_n",
                     "fp8bs_set_gemm_split_last_round", "fp8bs_debug_build", "fp8bs_debug_site", "fp8bs_gemm_clock"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check(fn, rc):
    if rc != OK:
        raise Fp8bsError(fn, rc)


def _ld(t: torch.Tensor) -> int:
    assert t.dim() == 2 and t.stride(1) == 1, "row-major matrix with unit column stride expected"
    return t.stride(0)


def quant_1x128(x: torch.Tensor, along: int = 0, q=None, s=None, stream=None):
    """1x128 tile quantisation of BF16 x [M, K].
    along=0: q [M, K] codes, s [K/128, M];  along=1: q [K, M] codes, s [M/128, K]."""
    M, K = x.shape
    if along == 0:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
        s = torch.empty((K // 128, M), dtype=torch.float32, device=x.device) if s is None else s
    else:
        q = torch.empty((K, M), dtype=torch.uint8, device=x.device) if q is None else q
        s = torch.empty((M // 128, K), dtype=torch.float32, device=x.device) if s is None else s
    _check("fp8_quant_1x128", lib().fp8_quant_1x128(_ptr(x), M, K, _ld(x), along, _ptr(q), _ld(q),
                                                    _ptr(s), _ld(s), _stream(stream)))
    return q, s


def quant_128x128(w: torch.Tensor, q=None, s=None, stream=None):
    """128x128 block quantisation of BF16 w [N, K]: q [N, K], s [ceil(N/128), K/128]."""
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q is None else q
    s = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=w.device) if s is None else s
    _check("fp8_quant_128x128", lib().fp8_quant_128x128(_ptr(w), N, K, _ld(w), _ptr(q), _ld(q),
                                                        _ptr(s), _ld(s), _stream(stream)))
    return q, s


def quant_act_weight(x: torch.Tensor, w: torch.Tensor, ue8m0: bool = False, qx=None, sx=None, qw=None, sw=None,
                     stream=None):
    """x [M, Kx] in 1x128 tiles and w [N, Kw] in 128x128 blocks, one launch.
    Returns (qx [M, Kx], sx [Kx/128, M], qw [N, Kw], sw [ceil(N/128), Kw/128])."""
    M, Kx = x.shape
    N, Kw = w.shape
    qx = torch.empty((M, Kx), dtype=torch.uint8, device=x.device) if qx is None else qx
    sx = torch.empty((Kx // 128, M), dtype=torch.float32, device=x.device) if sx is None else sx
    qw = torch.empty((N, Kw), dtype=torch.uint8, device=w.device) if qw is None else qw
    sw = torch.empty(((N + 127) // 128, Kw // 128), dtype=torch.float32, device=w.device) if sw is None else sw
    _check("fp8_quant_act_weight", lib().fp8_quant_act_weight(
        _ptr(x), M, Kx, _ld(x), _ptr(qx), _ld(qx), _ptr(sx), _ld(sx), _ptr(w), N, Kw, _ld(w), _ptr(qw), _ld(qw),
        _ptr(sw), _ld(sw), 1 if ue8m0 else 0, _stream(stream)))
    return qx, sx, qw, sw


def quant_1x128_ue8m0(x: torch.Tensor, q=None, s=None, stream=None):
    """1x128 tiles with power-of-two scales: q [M, K], s [K/128, M] (FP32 powers of two)."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
    s = torch.empty((K // 128, M), dtype=torch.float32, device=x.device) if s is None else s
    _check("fp8_quant_1x128_ue8m0", lib().fp8_quant_1x128_ue8m0(_ptr(x), M, K, _ld(x), _ptr(q), _ld(q), _ptr(s),
                                                                _ld(s), _stream(stream)))
    return q, s


def quant_128x128_ue8m0(w: torch.Tensor, q=None, s=None, stream=None):
    """128x128 blocks with power-of-two scales: q [N, K], s [ceil(N/128), K/128]."""
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q is None else q
    s = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=w.device) if s is None else s
    _check("fp8_quant_128x128_ue8m0", lib().fp8_quant_128x128_ue8m0(_ptr(w), N, K, _ld(w), _ptr(q), _ld(q),
                                                                    _ptr(s), _ld(s), _stream(stream)))
    return q, s


def quant_128x128_t(w: torch.Tensor, straight: bool = True, q=None, s=None, qt=None, st=None, stream=None):
    """128x128 block quantisation of BF16 w [N, K] with transposed outputs:
    qt [K, N] codes and st [K/128, ceil(N/128)] scales (the quantisation of w^T), plus, when
    straight, q [N, K] and s [ceil(N/128), K/128] as quant_128x128 writes them.
    Returns (q, s, qt, st); q and s are None when not straight."""
    N, K = w.shape
    nb = (N + 127) // 128
    if straight:
        q = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q is None else q
        s = torch.empty((nb, K // 128), dtype=torch.float32, device=w.device) if s is None else s
    else:
        q = s = None
    qt = torch.empty((K, N), dtype=torch.uint8, device=w.device) if qt is None else qt
    st = torch.empty((K // 128, nb), dtype=torch.float32, device=w.device) if st is None else st
    _check("fp8_quant_128x128_t", lib().fp8_quant_128x128_t(
        _ptr(w), N, K, _ld(w), _ptr(q), _ld(q) if q is not None else 0, _ptr(s), _ld(s) if s is not None else 0,
        _ptr(qt), _ld(qt), _ptr(st), _ld(st), _stream(stream)))
    return q, s, qt, st


def gemm_blockscaled(A, sa, B, sb, b_scale_mode: int = 0, out_dtype=torch.bfloat16, C=None, stream=None):
    """C = A * B^T with fine-grained scales (FP32 promotion every 128 K)."""
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype, device=A.device)
    od = 0 if C.dtype == torch.bfloat16 else 1
    _check("fp8_gemm_blockscaled", lib().fp8_gemm_blockscaled(
        _ptr(A), _ld(A), _ptr(sa), _ld(sa), _ptr(B), _ld(B), _ptr(sb), _ld(sb), b_scale_mode,
        _ptr(C), _ld(C), od, M, N, K, _stream(stream)))
    return C


def gemm_ue8m0(A, sa, B, sb, out_dtype=torch.bfloat16, C=None, stream=None):
    """C = A * B^T with power-of-two scales applied by the tensor cores' block scaling."""
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype, device=A.device)
    od = 0 if C.dtype == torch.bfloat16 else 1
    _check("fp8_gemm_ue8m0", lib().fp8_gemm_ue8m0(
        _ptr(A), _ld(A), _ptr(sa), _ld(sa), _ptr(B), _ld(B), _ptr(sb), _ld(sb), _ptr(C), _ld(C), od, M, N, K,
        _stream(stream)))
    return C


def grouped_gemm_moe(A, sa, B, sb, offsets, out_dtype=torch.bfloat16, C=None, stream=None):
    """Per-expert GEMMs: A [M_total, K] codes (expert-sorted), B [G, N, K], sb [G, ceil(N/128), K/128],
    offsets int32 [G+1] on the device."""
    M, K = A.shape
    G, N, K2 = B.shape
    assert K == K2 and B.is_contiguous() and sb.is_contiguous() and offsets.dtype == torch.int32
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype, device=A.device)
    od = 0 if C.dtype == torch.bfloat16 else 1
    _check("fp8_grouped_gemm_moe", lib().fp8_grouped_gemm_moe(
        _ptr(A), _ld(A), _ptr(sa), _ld(sa), _ptr(B), _ptr(sb), _ptr(offsets), G, M,
        _ptr(C), _ld(C), od, N, K, _stream(stream)))
    return C


def e4m3_encode(x: torch.Tensor, q=None, stream=None):
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if q is None else q
    _check("fp8bs_e4m3_encode", lib().fp8bs_e4m3_encode(_ptr(x), _ptr(q), x.numel(), _stream(stream)))
    return q


def set_gemm_tile_n(bn: int) -> None:
    """GEMM output tile width: 128, 192, 256, or 0 for automatic."""
    _check("fp8bs_set_gemm_tile_n", lib().fp8bs_set_gemm_tile_n(bn))


def set_gemm_split_last_round(on: bool) -> None:
    """FP32-output GEMMs: share the last round's tiles out by K chunks (True,
    the default; bit-identical results) or run whole tiles only (False)."""
    _check("fp8bs_set_gemm_split_last_round", lib().fp8bs_set_gemm_split_last_round(1 if on else 0))


def get_device_error(stream=None) -> int:
    return lib().fp8bs_get_device_error(_stream(stream))


def moe_route(x: torch.Tensor, centroids_t: torch.Tensor, bias: torch.Tensor, topk: int, out=None,
              workspace=None, stream=None):
    """Routing of BF16 tokens x [T, D] over E experts (centroids k-major f32 [D, E], bias f32 [E]).
    Returns a dict of device tensors: logits [T, E], expert_idx [T, k], gate [T, k],
    offsets [E+1], token_of_row [T*k], row_of [T, k] (int32 / f32)."""
    T, D = x.shape
    E = centroids_t.shape[1]
    centroids = centroids_t
    dev = x.device
    o = out if out is not None else {
        "logits": torch.empty((T, E), dtype=torch.float32, device=dev),
        "expert_idx": torch.empty((T, topk), dtype=torch.int32, device=dev),
        "gate": torch.empty((T, topk), dtype=torch.float32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "token_of_row": torch.empty(T * topk, dtype=torch.int32, device=dev),
        "row_of": torch.empty((T, topk), dtype=torch.int32, device=dev),
    }
    nbytes = lib().fp8_moe_route_workspace_size(E)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    _check("fp8_moe_route", lib().fp8_moe_route(
        _ptr(x), T, D, _ld(x), _ptr(centroids), _ld(centroids), _ptr(bias), E, topk,
        _ptr(o["logits"]), _ptr(o["expert_idx"]), _ptr(o["gate"]), _ptr(o["offsets"]),
        _ptr(o["token_of_row"]), _ptr(o["row_of"]), _ptr(workspace), workspace.numel(), _stream(stream)))
    return o


def moe_route_noalloc(x: torch.Tensor, centroids_t: torch.Tensor, bias: torch.Tensor, topk: int, out=None,
                      stream=None):
    """moe_route without a workspace argument (the library's static device scratch)."""
    T, D = x.shape
    E = centroids_t.shape[1]
    dev = x.device
    o = out if out is not None else {
        "logits": torch.empty((T, E), dtype=torch.float32, device=dev),
        "expert_idx": torch.empty((T, topk), dtype=torch.int32, device=dev),
        "gate": torch.empty((T, topk), dtype=torch.float32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "token_of_row": torch.empty(T * topk, dtype=torch.int32, device=dev),
        "row_of": torch.empty((T, topk), dtype=torch.int32, device=dev),
    }
    _check("fp8_moe_route_noalloc", lib().fp8_moe_route_noalloc(
        _ptr(x), T, D, _ld(x), _ptr(centroids_t), _ld(centroids_t), _ptr(bias), E, topk,
        _ptr(o["logits"]), _ptr(o["expert_idx"]), _ptr(o["gate"]), _ptr(o["offsets"]),
        _ptr(o["token_of_row"]), _ptr(o["row_of"]), _stream(stream)))
    return o


def quant_1x128_gather(x: torch.Tensor, row_map: torch.Tensor, q=None, s=None, stream=None):
    """1x128 quantisation of the rows x[row_map[r]]: q [R, K], s [K/128, R]."""
    T, K = x.shape
    R = row_map.numel()
    q = torch.empty((R, K), dtype=torch.uint8, device=x.device) if q is None else q
    s = torch.empty((K // 128, R), dtype=torch.float32, device=x.device) if s is None else s
    _check("fp8_quant_1x128_gather", lib().fp8_quant_1x128_gather(
        _ptr(x), T, K, _ld(x), _ptr(row_map), R, _ptr(q), _ld(q), _ptr(s), _ld(s), _stream(stream)))
    return q, s


def grouped_gemm_moe_swiglu(A, sa, B, sb, offsets, Q=None, s=None, stream=None):
    """Up projection [G, 2*Nh, K] (gate rows, then up rows) with SwiGLU + 1x128 quantisation
    fused: returns codes Q [M_total, Nh] and scales s [Nh/128, M_total]."""
    M, K = A.shape
    G, N2, _ = B.shape
    Nh = N2 // 2
    Q = torch.empty((M, Nh), dtype=torch.uint8, device=A.device) if Q is None else Q
    s = torch.empty((Nh // 128, M), dtype=torch.float32, device=A.device) if s is None else s
    _check("fp8_grouped_gemm_moe_swiglu", lib().fp8_grouped_gemm_moe_swiglu(
        _ptr(A), _ld(A), _ptr(sa), _ld(sa), _ptr(B), _ptr(sb), _ptr(offsets), G, M, _ptr(Q), _ld(Q),
        _ptr(s), _ld(s), Nh, K, _stream(stream)))
    return Q, s


def moe_combine(Y: torch.Tensor, row_of: torch.Tensor, gate: torch.Tensor, out=None, stream=None):
    """out[t] = sum_j gate[t, j] * Y[row_of[t, j]] (BF16)."""
    R, N = Y.shape
    T, k = row_of.shape
    out = torch.empty((T, N), dtype=torch.bfloat16, device=Y.device) if out is None else out
    _check("fp8_moe_combine", lib().fp8_moe_combine(
        _ptr(Y), _ld(Y), R, _ptr(row_of), _ptr(gate), T, k, N, _ptr(out), _ld(out), _stream(stream)))
    return out


def selftest_division(stream=None):
    """(code mismatches, quotient mismatches) of the fast quotient against the
    IEEE divide over every BF16 (amax, x) pair with |x| <= amax."""
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    _check("fp8bs_selftest_division", lib().fp8bs_selftest_division(_ptr(out), _stream(stream)))
    code, quot = out.tolist()
    return code, quot


def selftest_timeout(timeout_ns: int, stream=None):
    _check("fp8bs_selftest_timeout", lib().fp8bs_selftest_timeout(timeout_ns, _stream(stream)))


def debug_site(stream=None) -> int:
    """First failed bounds check since the last read (0: none; always 0 in the release build)."""
    rc = lib().fp8bs_debug_site(_stream(stream))
    if rc < 0:
        raise Fp8bsError("fp8bs_debug_site", rc)
    return rc


def gemm_clock(reset: bool = False, stream=None):
    """(mean SM MHz the GEMM kernels ran at, launches counted) since the last reset."""
    mhz, n = ctypes.c_double(0.0), ctypes.c_longlong(0)
    _check("fp8bs_gemm_clock", lib().fp8bs_gemm_clock(ctypes.byref(mhz), ctypes.byref(n), 1 if reset else 0,
                                                     _stream(stream)))
    return mhz.value, n.value
