"""Shared helpers for the GPU parity tests: upload seeded inputs, fetch results,
and compare GEMM outputs with the oracle's under the stated tolerance.

GEMM tolerance (BF16 or FP32 outputs against the oracle's outputs rounded the
same way): relative Frobenius error <= 1e-3 over the compared rows, and every
element within 2e-2 x that row's max |C|.  The tensor cores sum each
128-product chunk in their own order, so a few BF16 results land one ulp
(2^-8 relative) away from the oracle's; the bound leaves room for that and
for nothing larger.
"""
import numpy as np
import torch

REL_FRO = 1e-3
ROW_MAX = 2e-2


def dev(a: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm_errors(got: np.ndarray, ref: np.ndarray):
    """got/ref: BF16 bits (uint16) or float32, same shape [rows, N]."""
    g = bf16_bits_to_f64(got) if got.dtype == np.uint16 else got.astype(np.float64)
    r = bf16_bits_to_f64(ref) if ref.dtype == np.uint16 else ref.astype(np.float64)
    fro = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
    rowmax = np.abs(r).max(axis=1, keepdims=True)
    worst = (np.abs(g - r) / np.maximum(rowmax, 1e-300)).max()
    return fro, worst


def assert_gemm_close(got, ref, what=""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got.astype(np.float64) if got.dtype != np.uint16 else bf16_bits_to_f64(got)).all(), what
    fro, worst = gemm_errors(got, ref)
    assert fro <= REL_FRO and worst <= ROW_MAX, f"{what}: rel_fro={fro:.3e} max_row_rel={worst:.3e}"
    return fro, worst


def sample_rows(M: int, n: int, seed: int, must=()):
    rng = np.random.default_rng(seed)
    rows = set(int(r) for r in must if 0 <= r < M)
    rows.update(int(r) for r in rng.choice(M, size=min(n, M), replace=False))
    return np.array(sorted(rows), dtype=np.int64)


GUARD_ROWS = 3


def canary_output(M: int, N: int, dtype, device="cuda"):
    """An output view C [M, N] inside a NaN-filled buffer with a padded row
    pitch and guard rows above and below.  Returns (C, buf, rows, cols): the
    GEMM must write exactly buf[rows, cols] and nothing else."""
    esize = 2 if dtype == torch.bfloat16 else 4
    per16 = 16 // esize
    ld = (N + per16 - 1) // per16 * per16 + 2 * per16  # padded pitch, still a multiple of 16 bytes
    buf = torch.full((M + 2 * GUARD_ROWS, ld), float("nan"), dtype=dtype, device=device)
    C = buf[GUARD_ROWS:GUARD_ROWS + M, :N]
    return C, buf, slice(GUARD_ROWS, GUARD_ROWS + M), slice(0, N)


def assert_canaries_untouched(buf: torch.Tensor, rows: slice, cols: slice, what=""):
    """Every element of buf outside [rows, cols] still holds the NaN it was filled with."""
    mask = torch.ones(buf.shape, dtype=torch.bool, device=buf.device)
    mask[rows, cols] = False
    outside = buf[mask]
    assert torch.isnan(outside.float()).all(), f"{what}: the GEMM wrote outside C"
