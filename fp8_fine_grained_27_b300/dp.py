"""Data-parallel Wgrad across ranks: the tokens (the Wgrad GEMM's K) are split
between data-parallel ranks, each rank forms an FP32 partial dW from its own
tokens with the library's kernels, and one reduce-scatter sums the partials
and leaves each rank its share of dW's rows.

"DeepSeek-V3 技术报告" §7: training shards the batch across data-parallel
ranks with ZeRO-1 (each rank owns a slice of the optimizer state, so the
gradient is reduce-scattered, not all-reduced); §6: the Wgrad GEMM runs in
FP8 with an FP32 result.

Summation.  A token shard is a run of whole 128-token tiles, so every 1x128
tile of the single-rank quantisation lies in one shard and is quantised the
same way.  Each rank's partial promotes its own tiles in token order; the
partials are then added across ranks in FP32.  With two ranks that sum is
exact-commutative and equals the reference's rank-order sum bit for bit; with
more ranks the collective's own order may differ from rank order by FP32
rounding of the additions.  The result differs from the single-rank dW only by
the order of the FP32 additions across the shard boundaries.

Only argument marshalling and the collective live here: the quantisers and
the GEMM are the C-ABI kernels (binding.py), the reduce-scatter is
torch.distributed's (NCCL on GPUs).
"""
from __future__ import annotations

import torch

from . import binding


def token_shard(T: int, world: int, rank: int) -> tuple[int, int]:
    """Tokens [t0, t1) of `rank`: contiguous whole 128-token tiles, rank r taking
    tiles floor(r n / world) .. floor((r+1) n / world) - 1 of the n = T / 128."""
    if T % 128 != 0 or world < 1 or not 0 <= rank < world:
        raise ValueError("T must be a multiple of 128 and 0 <= rank < world")
    n = T // 128
    return 128 * (rank * n // world), 128 * ((rank + 1) * n // world)


def wgrad_local(dY: torch.Tensor, X: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """This rank's FP32 partial dW_r = dY_r^T X_r from its tokens: dY [T_r, Cout] and
    X [T_r, Cin] BF16, each quantised 1x128 along the tokens, then the Wgrad GEMM
    (per-row scales of both operands, FP32 out).  Returns [Cout, Cin] f32."""
    qdy, sdy = binding.quant_1x128(dY, along=1, stream=stream)
    qx, sx = binding.quant_1x128(X, along=1, stream=stream)
    return binding.gemm_blockscaled(qdy, sdy, qx, sx, 1, out_dtype=torch.float32, C=out, stream=stream)


def reduce_scatter_rows(partial: torch.Tensor, group=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Sum the ranks' partials [Cout, Cin] and return this rank's rows of the sum:
    rows rank * Cout / world .. (rank + 1) * Cout / world - 1 (Cout divisible by world)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    cout = partial.shape[0]
    if cout % world != 0:
        raise ValueError("the rows of dW must split evenly across the ranks")
    if out is None:
        out = torch.empty((cout // world, partial.shape[1]), dtype=partial.dtype, device=partial.device)
    dist.reduce_scatter_tensor(out, partial.contiguous(), op=dist.ReduceOp.SUM, group=group)
    return out


def wgrad_dp(dY: torch.Tensor, X: torch.Tensor, group=None) -> torch.Tensor:
    """This rank's rows of dW = sum over ranks of dY_r^T X_r (its tokens' dY and X)."""
    return reduce_scatter_rows(wgrad_local(dY, X), group)
