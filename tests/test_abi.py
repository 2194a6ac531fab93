"""The C-ABI library builds for sm_103a, loads, and exports every symbol its header declares.
No compute calls here (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


@pytest.fixture(scope="module")
def libpath():
    from fp8_fine_grained_27_b300 import build
    return build.build()


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("fp8_quant_1x128", "fp8_quant_128x128", "fp8_gemm_blockscaled", "fp8_grouped_gemm_moe"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    L = ctypes.CDLL(libpath)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_lists_every_declared_symbol():
    from fp8_fine_grained_27_b300 import binding
    assert sorted(binding.EXPORTS) == declared_functions()


def test_status_strings_and_argument_errors(libpath):
    """Argument validation returns before touching the device."""
    from fp8_fine_grained_27_b300 import binding as b
    L = b.lib()
    assert L.fp8bs_status_string(0) == b"ok"
    assert b"aligned" in L.fp8bs_status_string(-2)
    vp = ctypes.c_void_p
    # negative sizes, bad mode, K not a multiple of 128, unaligned pointers
    assert L.fp8_quant_1x128(vp(16), -1, 128, 128, 0, vp(16), 128, vp(16), 1, None) == b.EINVAL
    assert L.fp8_quant_1x128(vp(16), 4, 128, 128, 2, vp(16), 128, vp(16), 4, None) == b.EINVAL
    assert L.fp8_quant_1x128(vp(18), 4, 128, 128, 0, vp(16), 128, vp(16), 4, None) == b.EALIGN
    assert L.fp8_quant_128x128(vp(16), 4, 100, 128, vp(16), 128, vp(16), 1, None) == b.EINVAL
    # transposed block quantiser: N % 16, q without s, unaligned transposed pitch
    assert L.fp8_quant_128x128_t(vp(16), 24, 128, 128, None, 0, None, 0, vp(16), 32, vp(16), 1,
                                 None) == b.EINVAL
    assert L.fp8_quant_128x128_t(vp(16), 32, 128, 128, vp(16), 128, None, 0, vp(16), 32, vp(16), 1,
                                 None) == b.EINVAL
    assert L.fp8_quant_128x128_t(vp(16), 32, 128, 128, None, 0, None, 0, vp(16), 40, vp(16), 1,
                                 None) == b.EALIGN
    assert L.fp8_quant_128x128_t(None, 0, 128, 128, None, 0, None, 0, None, 0, None, 0, None) == b.OK
    assert L.fp8_gemm_blockscaled(vp(16), 128, vp(16), 4, vp(16), 128, vp(16), 1, 0, vp(16), 8, 0,
                                  4, 8, 100, None) == b.EINVAL
    assert L.fp8_gemm_blockscaled(vp(16), 128, vp(16), 4, vp(16), 128, vp(16), 1, 2, vp(16), 8, 0,
                                  4, 8, 128, None) == b.EINVAL
    assert L.fp8_gemm_blockscaled(vp(16), 128, vp(16), 4, vp(16), 128, vp(16), 1, 0, vp(16), 12, 0,
                                  4, 12, 128, None) == b.EINVAL  # N % 8
    assert L.fp8_gemm_blockscaled(vp(17), 128, vp(16), 4, vp(16), 128, vp(16), 1, 0, vp(16), 8, 0,
                                  4, 8, 128, None) == b.EALIGN
    assert L.fp8_grouped_gemm_moe(vp(16), 128, vp(16), 4, vp(16), vp(16), vp(16), 0, 4, vp(16), 8, 0,
                                  8, 128, None) == b.EINVAL  # G = 0
    assert L.fp8bs_selftest_timeout(0, None) == b.EINVAL
    # process-wide switches take only their documented values
    assert L.fp8bs_set_gemm_tile_n(96) == b.EINVAL
    assert L.fp8bs_set_gemm_split_last_round(2) == b.EINVAL
    assert L.fp8bs_set_gemm_split_last_round(0) == b.OK
    assert L.fp8bs_set_gemm_split_last_round(1) == b.OK
    # sizes past the 32-bit tile indexing are refused before any launch
    big = 1 << 31
    assert L.fp8_gemm_blockscaled(vp(16), 128, vp(16), big, vp(16), 128, vp(16), 1, 0, vp(16), 8, 0,
                                  big, 8, 128, None) == b.EINVAL
    assert L.fp8_gemm_ue8m0(vp(16), 128, vp(16), 4, vp(16), big, vp(16), 1, vp(16), big, 0,
                            4, big, 128, None) == b.EINVAL
    assert L.fp8_quant_1x128(vp(16), big + 1, 128, 128, 0, vp(16), 128, vp(16), big + 1, None) == b.EINVAL
    assert L.fp8_quant_128x128(vp(16), big + 1, 128, 128, vp(16), 128, vp(16), 1, None) == b.EINVAL
    # empty problems are a successful no-op
    assert L.fp8_gemm_blockscaled(None, 128, None, 4, None, 128, None, 1, 0, None, 8, 0,
                                  0, 8, 128, None) == b.OK


def test_empty_problems_return_before_any_launch(libpath):
    """Empty inputs are a successful no-op and argument errors are caught without a device:
    these calls never reach the GPU."""
    from fp8_fine_grained_27_b300 import binding as b
    L = b.lib()
    vp = ctypes.c_void_p
    assert L.fp8_quant_1x128(None, 0, 128, 128, 0, None, 128, None, 1, None) == b.OK
    assert L.fp8_quant_1x128(None, 4, 0, 128, 1, None, 128, None, 1, None) == b.OK
    assert L.fp8_quant_128x128(None, 0, 128, 128, None, 128, None, 1, None) == b.OK
    assert L.fp8_quant_1x128_ue8m0(None, 0, 128, 128, None, 128, None, 1, None) == b.OK
    assert L.fp8_quant_128x128_ue8m0(None, 4, 0, 128, None, 128, None, 1, None) == b.OK
    assert L.fp8_quant_act_weight(None, 0, 128, 128, None, 128, None, 1, None, 0, 128, 128, None, 128, None, 1,
                                  0, None) == b.OK
    assert L.fp8_quant_act_weight(None, 0, 128, 128, None, 128, None, 1, None, 0, 128, 128, None, 128, None, 1,
                                  2, None) == b.EINVAL  # unknown scale rule
    assert L.fp8_quant_1x128_gather(None, 10, 128, 128, None, 0, None, 128, None, 1, None) == b.OK
    assert L.fp8_gemm_ue8m0(None, 128, None, 4, None, 128, None, 1, None, 8, 0, 0, 8, 128, None) == b.OK
    assert L.fp8_grouped_gemm_moe_swiglu(vp(16), 128, vp(16), 4, vp(16), vp(16), vp(16), 1, 0, vp(16), 128,
                                         vp(16), 4, 128, 128, None) == b.OK
    assert L.fp8_grouped_gemm_moe_swiglu(vp(16), 128, vp(16), 4, vp(16), vp(16), vp(16), 1, 4, vp(16), 128,
                                         vp(16), 4, 100, 128, None) == b.EINVAL  # Nh % 128
    assert L.fp8_moe_combine(None, 8, 0, None, None, 0, 2, 8, None, 8, None) == b.OK
    assert L.fp8_moe_combine(vp(16), 8, 4, vp(16), vp(16), 2, 0, 8, vp(16), 8, None) == b.EINVAL  # topk 0
    # routing: expert count not a multiple of 4, top-k above the expert count, D not a multiple of 32
    ws = vp(256)
    assert L.fp8_moe_route(vp(16), 4, 64, 64, vp(16), 8, vp(16), 6, 2, vp(16), vp(16), vp(16), vp(16), vp(16),
                           vp(16), ws, 256, None) == b.EINVAL
    assert L.fp8_moe_route(vp(16), 4, 64, 64, vp(16), 8, vp(16), 8, 9, vp(16), vp(16), vp(16), vp(16), vp(16),
                           vp(16), ws, 256, None) == b.EINVAL
    assert L.fp8_moe_route(vp(16), 4, 48, 64, vp(16), 8, vp(16), 8, 2, vp(16), vp(16), vp(16), vp(16), vp(16),
                           vp(16), ws, 256, None) == b.EINVAL
    assert L.fp8_moe_route(vp(16), 4, 64, 64, vp(16), 8, vp(16), 8, 2, vp(16), vp(16), vp(16), vp(16), vp(16),
                           vp(16), ws, 16, None) == b.EINVAL  # workspace too small
