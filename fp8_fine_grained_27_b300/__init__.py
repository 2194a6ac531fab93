"""Fine-grained FP8 (E4M3) block-scaled GEMM for B300 (sm_103a).

The compute lives in ``libfp8bs.so`` (hand-written CUDA: tile quantisers and
tcgen05 GEMMs, C ABI in ``include/fp8bs.h``); :mod:`.binding` marshals torch
tensors into it.  There is no CPU path: if the library is missing the import
of the binding fails.
"""
from .binding import (  # noqa: F401
    Fp8bsError,
    e4m3_encode,
    debug_site,
    gemm_blockscaled,
    gemm_clock,
    gemm_ue8m0,
    get_device_error,
    grouped_gemm_moe,
    grouped_gemm_moe_swiglu,
    lib,
    moe_combine,
    moe_route,
    moe_route_noalloc,
    quant_1x128,
    quant_1x128_gather,
    quant_1x128_ue8m0,
    quant_128x128,
    quant_act_weight,
    quant_128x128_ue8m0,
    quant_128x128_t,
    selftest_division,
    selftest_timeout,
    set_gemm_split_last_round,
    set_gemm_tile_n,
)
