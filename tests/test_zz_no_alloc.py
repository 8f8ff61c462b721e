"""The chunked scan entry point that allocates no device memory.

Callers that cannot allocate device memory during the call -- a framework that
owns every byte of device memory and passes in only the call's tensors, or host
code on a fixed memory budget that must not touch the allocator -- use
mamba_selective_scan_fwd_noalloc, whose scratch is a static device array inside
the library.  These tests call it through the C ABI and compare it with the
regular chunked scan.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import selective_state_space_148_b300 as m
from selective_state_space_148_b300 import inputs
from helpers import TOL_STATE, TOL_Y, assert_close, dev_inputs, f32_dev, to_host_f64

FAKE = 256  # never dereferenced: the calls below are rejected before anything is launched


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = m.lib()
    # 1 x 4096 channels x 16 states x 64 chunks of 32 steps needs 16.8 MB > 16 MiB
    st = lib.mamba_selective_scan_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 1, FAKE, None, None,
                                              1, 4096, 64 * 32, 16, m.MAMBA_BF16, 32, None)
    assert st == -11
    assert "scratch" in m.status_string(st)
    assert lib.mamba_selective_scan_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 1, FAKE, None, None,
                                                1, 4, 64, 16, m.MAMBA_BF16, 0, None) == -2      # chunk_len >= 1
    assert lib.mamba_selective_scan_fwd_noalloc(None, FAKE, FAKE, FAKE, FAKE, None, None, None, 1, FAKE, None, None,
                                                1, 4, 64, 16, m.MAMBA_BF16, 32, None) == -1


@pytest.mark.gpu
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_noalloc_matches_chunked_entry_point_on_two_calls(io):
    import torch
    chunk_len = 256
    for call, seed in enumerate((41, 42)):          # two calls in a row, different inputs each time
        x = inputs.make_scan_inputs(2, 40, 16, 3000, io=io, seed=seed)
        t = dev_inputs(x)
        h0 = f32_dev(np.random.default_rng(seed).normal(0, 0.3, (2, 40, 16)).astype(np.float32)) if call else None
        y_ref = torch.empty_like(t["u"])
        h_ref = torch.empty((2, 40, 16), dtype=torch.float32, device="cuda")
        m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], 1,
                                      y_ref, h_ref, h0=h0, chunk_len=chunk_len)
        y = torch.full_like(t["u"], float("nan"))
        h = torch.full((2, 40, 16), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        st = m.lib().mamba_selective_scan_fwd_noalloc(
            t["u"].data_ptr(), t["delta"].data_ptr(), t["A"].data_ptr(), t["B"].data_ptr(), t["C"].data_ptr(),
            t["D"].data_ptr(), t["z"].data_ptr(), t["delta_bias"].data_ptr(), 1, y.data_ptr(), h.data_ptr(),
            None if h0 is None else h0.data_ptr(), 2, 40, 3000, 16, m.MAMBA_BF16 if io == "bf16" else m.MAMBA_F32,
            chunk_len, torch.cuda.current_stream().cuda_stream)
        assert st == 0, m.status_string(st)
        torch.cuda.synchronize()
        if call:
            # after the first call (which looks up the array's address and may load the kernels), a call
            # changes neither torch's allocation count nor the device's free memory
            assert (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]) == before
        assert_close(to_host_f64(y), to_host_f64(y_ref), TOL_Y[io], f"call {call} y")
        assert_close(h.cpu().numpy(), h_ref.cpu().numpy(), TOL_STATE, f"call {call} last_state")
