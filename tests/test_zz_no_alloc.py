"""The allocation-free routing entry point (fp8_moe_route_noalloc) against the workspace
entry point (fp8_moe_route): identical results on two consecutive calls with different
inputs (the second call reuses the library's scratch), no device memory allocated by the
call itself (outputs allocated beforehand, the C entry point called directly), and an
expert count whose workspace would not fit is refused before any launch."""
import ctypes

import numpy as np
import pytest
import torch

import synth


def test_noalloc_refuses_oversize_before_launch():
    from fp8_fine_grained_27_b300 import binding as b
    L = b.lib()
    vp = ctypes.c_void_p
    # E = 1028 needs more than the 4 KB static scratch (and exceeds the expert limit)
    assert L.fp8_moe_route_noalloc(vp(16), 4, 64, 64, vp(16), 1028, vp(16), 1028, 2, vp(16), vp(16), vp(16),
                                   vp(16), vp(16), vp(16), None) == b.EINVAL
    assert L.fp8_moe_route_workspace_size(1028) == -1
    assert L.fp8_moe_route_workspace_size(1024) <= 4096


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_on_two_calls():
    import fp8_fine_grained_27_b300 as fb
    assert torch.cuda.is_available()
    for call, (T, D, E, k) in enumerate([(300, 512, 64, 6), (1000, 1024, 256, 8)]):
        x = synth.fill_bf16(synth.NORMAL, synth.key(60, call), (T, D), 1.0)
        cent = synth.fill_f32(synth.NORMAL, synth.key(61, call), (E, D), 1.0 / np.sqrt(D))
        bias = synth.fill_f32(synth.NORMAL, synth.key(62, call), (E,), 0.5)
        xd = torch.from_numpy(x).view(torch.bfloat16).cuda()
        cd = torch.from_numpy(np.ascontiguousarray(cent.T)).cuda()
        bd = torch.from_numpy(bias).cuda()
        ref = fb.moe_route(xd, cd, bd, k)
        got = fb.moe_route_noalloc(xd, cd, bd, k)
        torch.cuda.synchronize()
        for name in ref:
            assert torch.equal(ref[name], got[name]), (call, name)


@pytest.mark.gpu
def test_noalloc_call_allocates_no_device_memory():
    """With its outputs allocated beforehand, a (warm) call of the C entry point
    changes neither torch's allocator total nor the device's free memory."""
    import fp8_fine_grained_27_b300 as fb
    from fp8_fine_grained_27_b300 import binding as b
    assert torch.cuda.is_available()
    T, D, E, k = 512, 512, 128, 8
    x = synth.fill_bf16(synth.NORMAL, synth.key(63, 0), (T, D), 1.0)
    cent = synth.fill_f32(synth.NORMAL, synth.key(64, 0), (E, D), 1.0 / np.sqrt(D))
    bias = synth.fill_f32(synth.NORMAL, synth.key(65, 0), (E,), 0.5)
    xd = torch.from_numpy(x).view(torch.bfloat16).cuda()
    cd = torch.from_numpy(np.ascontiguousarray(cent.T)).cuda()
    bd = torch.from_numpy(bias).cuda()
    out = fb.moe_route_noalloc(xd, cd, bd, k)  # first call: the library's one-time set-up
    torch.cuda.synchronize()
    L = b.lib()

    def call():
        rc = L.fp8_moe_route_noalloc(
            xd.data_ptr(), T, D, D, cd.data_ptr(), E, bd.data_ptr(), E, k, out["logits"].data_ptr(),
            out["expert_idx"].data_ptr(), out["gate"].data_ptr(), out["offsets"].data_ptr(),
            out["token_of_row"].data_ptr(), out["row_of"].data_ptr(), None)
        assert rc == b.OK, rc

    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    call()
    call()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    ref = fb.moe_route(xd, cd, bd, k)
    torch.cuda.synchronize()
    for name in ref:
        assert torch.equal(ref[name], out[name]), name
