"""Every output element of the full-size workloads against the float64 oracle.

The scan workloads (the 130M- and 2.8B-shaped layers, the 2.8B layer with
d_state 64, the 1M-step DNA sequence) run through the C ABI in the launch
configuration the benchmark times (automatic plan: the direct scan, or the
chunked scan for the DNA sequence).  The oracle computes every channel; the DNA
sequence is checked in channel blocks so that host memory stays bounded.  The
decode workload runs 1000 chained steps over the whole [256, 5120, 16] state;
the oracle keeps its own float64 chain over every row and is never
re-synchronised to the GPU: y is compared in full at every step, the state in
full after the last one.  Each test prints its largest error ratio
max |gpu - oracle| / (1 + |oracle|).
"""
import concurrent.futures as cf

import numpy as np
import pytest

import oracle
import selective_state_space_148_b300 as m
from selective_state_space_148_b300 import inputs
from helpers import TOL_STATE, TOL_STATE_CHAIN, TOL_Y, assert_close, dev_inputs, f32_dev, to_dev, to_host_f64

pytestmark = pytest.mark.gpu


def run_workload_on_gpu(x):
    import torch
    Bsz, Dch, L, N = x.shape
    t = dev_inputs(x)
    y = torch.empty_like(t["u"])
    h = torch.empty((Bsz, Dch, N), dtype=torch.float32, device="cuda")
    m.mamba_selective_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], 1, y, h)
    torch.cuda.synchronize()
    assert m.mamba_device_error() == 0
    del t
    return y, h


@pytest.mark.parametrize("name", ["mamba130m_b8_d1536_n16_l2048_bf16", "mamba2p8b_b4_d5120_n16_l4096_bf16",
                                  "mamba2p8b_b4_d5120_n64_l4096_bf16"])
def test_layer_every_element(name):
    x = inputs.make_workload(name)
    Bsz, Dch, L, N = x.shape
    y, h = run_workload_on_gpu(x)
    yg = to_host_f64(y)
    hg = h.cpu().numpy().astype(np.float64)
    del y, h
    yr, hr = oracle.selective_scan(x.f64("u"), x.f64("delta"), x.f64("A"), x.f64("B"), x.f64("C"), x.f64("D"),
                                   x.f64("z"), x.f64("delta_bias"))
    ey = assert_close(yg, yr, TOL_Y["bf16"], f"{name} y")
    eh = assert_close(hg, hr, TOL_STATE, f"{name} last_state")
    print(f"{name}: every element, max err ratio y {ey:.3g} (tol {TOL_Y['bf16']}), "
          f"last_state {eh:.3g} (tol {TOL_STATE})")


@pytest.mark.parametrize("flags", [0x1, 0x3])
def test_layer_with_flags_every_element(flags):
    """The 130M-shaped layer with the exact zero-order hold, forwards and in reverse time."""
    import torch
    name = "mamba130m_b8_d1536_n16_l2048_bf16"
    x = inputs.make_workload(name)
    Bsz, Dch, L, N = x.shape
    t = dev_inputs(x)
    y = torch.empty_like(t["u"])
    h = torch.empty((Bsz, Dch, N), dtype=torch.float32, device="cuda")
    m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], 1,
                                  y, h, flags=flags)
    torch.cuda.synchronize()
    assert m.mamba_device_error() == 0
    yr, hr = oracle.selective_scan(x.f64("u"), x.f64("delta"), x.f64("A"), x.f64("B"), x.f64("C"), x.f64("D"),
                                   x.f64("z"), x.f64("delta_bias"), disc=1, reverse=bool(flags & 0x2))
    ey = assert_close(to_host_f64(y), yr, TOL_Y["bf16"], f"{name} flags={flags} y")
    eh = assert_close(h.cpu().numpy().astype(np.float64), hr, TOL_STATE, f"{name} flags={flags} last_state")
    print(f"{name} flags={flags}: every element, max err ratio y {ey:.3g}, last_state {eh:.3g}")


def test_dna_sequence_every_element_in_channel_blocks():
    import torch
    name = "dna_b1_d1536_n16_l1048576_bf16"
    x = inputs.make_workload(name)
    Bsz, Dch, L, N = x.shape
    assert m.mamba_scan_workspace_size(Bsz, Dch, L, N) > 0     # the automatic plan takes the chunked scan
    y, h = run_workload_on_gpu(x)
    ybits = y.view(torch.int16).cpu().numpy().view(np.uint16)
    hg = h.cpu().numpy().astype(np.float64)
    del y, h
    torch.cuda.empty_cache()
    Bf, Cf = x.f64("B"), x.f64("C")
    ey = eh = 0.0
    blk = 96
    for lo in range(0, Dch, blk):
        hi = min(Dch, lo + blk)
        sl = lambda a: inputs.to_f64(a[:, lo:hi], x.io)
        yr, hr = oracle.selective_scan(sl(x.u), sl(x.delta), x.A[lo:hi].astype(np.float64), Bf, Cf,
                                       x.D[lo:hi].astype(np.float64), sl(x.z), x.delta_bias[lo:hi].astype(np.float64))
        ey = max(ey, assert_close(inputs.to_f64(ybits[:, lo:hi], "bf16"), yr, TOL_Y["bf16"], f"{name} y [{lo}:{hi}]"))
        eh = max(eh, assert_close(hg[:, lo:hi], hr, TOL_STATE, f"{name} last_state [{lo}:{hi}]"))
    print(f"{name}: every element, max err ratio y {ey:.3g} (tol {TOL_Y['bf16']}), last_state {eh:.3g} "
          f"(tol {TOL_STATE})")


def test_decode_1000_steps_every_element():
    import torch
    cfg = inputs.DECODE_WORKLOAD
    Bsz, Dch, N, io, seed, steps = cfg["batch"], cfg["dim"], cfg["dstate"], cfg["io"], cfg["seed"], cfg["steps"]
    A, D, bias, _ = inputs.channel_params(Dch, N, seed)
    st0 = inputs.make_decode_state(Bsz, Dch, N, seed)
    state = f32_dev(st0)
    Ad, Dd, bd = f32_dev(A), f32_dev(D), f32_dev(bias)
    A64, D64, b64 = A.astype(np.float64), D.astype(np.float64), bias.astype(np.float64)
    ref = np.ascontiguousarray(st0.astype(np.float64))
    y = torch.empty((Bsz, Dch), dtype=torch.bfloat16, device="cuda")
    gen = lambda k: inputs.make_decode_step(Bsz, Dch, N, seed, k, io)
    worst_y = 0.0
    with cf.ThreadPoolExecutor(1) as ex:      # draws the next step's inputs while this step is checked
        nxt = ex.submit(gen, 0)
        for k in range(steps):
            s = nxt.result()
            if k + 1 < steps:
                nxt = ex.submit(gen, k + 1)
            u, dl, z, B, C = (to_dev(getattr(s, n), io) for n in ("u", "delta", "z", "B", "C"))
            m.mamba_state_update(state, u, dl, Ad, B, C, Dd, z, bd, 1, y)
            yr = oracle.state_update_inplace(ref, s.f64("u"), s.f64("delta"), A64, s.f64("B"), s.f64("C"), D64,
                                             s.f64("z"), b64)
            worst_y = max(worst_y, assert_close(to_host_f64(y), yr, TOL_Y[io], f"step {k} y"))
    torch.cuda.synchronize()
    assert m.mamba_device_error() == 0
    es = assert_close(state.cpu().numpy().astype(np.float64), ref, TOL_STATE_CHAIN, "state after 1000 steps")
    print(f"decode {cfg['name']}: {steps} chained steps, every element, max err ratio y {worst_y:.3g} "
          f"(tol {TOL_Y[io]}), state {es:.3g} (tol {TOL_STATE_CHAIN})")
