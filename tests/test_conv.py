"""The convolution branch: depthwise causal conv1d (width 4) + SiLU, alone and fused into the scan.

CPU tests check argument validation through the C ABI; GPU tests compare with the
float64 oracle (the scan of the oracle's convolution output).
"""
import numpy as np
import pytest

import oracle
import selective_state_space_148_b300 as m
from selective_state_space_148_b300 import inputs
from helpers import TOL_STATE, TOL_Y, assert_close, dev_inputs, f32_dev, to_host_f64

FAKE = 256  # never dereferenced: rejected before any launch


def test_conv_validation():
    L = m.lib()
    f = lambda **kw: L.mamba_causal_conv1d_silu(kw.get("x", FAKE), kw.get("w", FAKE), None, 1, kw.get("u", FAKE),
                                                kw.get("B", 1), 4, kw.get("L", 8), kw.get("dtype", 1), None)
    assert f(x=None) == -1 and f(w=None) == -1 and f(u=None) == -1
    assert f(B=0) == -2 and f(L=0) == -2
    assert f(dtype=5) == -4
    g = lambda **kw: L.mamba_selective_scan_fwd_conv(kw.get("x", FAKE), kw.get("w", FAKE), None, FAKE, FAKE, FAKE,
                                                     FAKE, None, FAKE, None, 1, FAKE, None, 1, 4, 8,
                                                     kw.get("N", 16), 1, None)
    assert g(x=None) == -1 and g(w=None) == -1
    assert g(N=65) == -3


def conv_inputs(Bsz, Dch, N, L, io, seed):
    x = inputs.make_scan_inputs(Bsz, Dch, N, L, io=io, seed=seed)   # x.u serves as the conv input
    w, b = inputs.conv_params(Dch, seed)
    return x, w, b


def oracle_conv_scan(x, w, b, with_z=True, u_stored=False):
    """Oracle scan of u = SiLU(conv(x)).  u_stored: u is rounded to the storage type first, as the two-step
    path does when it writes u to memory before the scan reads it (the fused kernel keeps u in fp32)."""
    u = oracle.causal_conv1d(x.f64("u"), w.astype(np.float64), b.astype(np.float64))
    if u_stored and x.io == "bf16":
        u = inputs.to_f64(inputs.f32_to_bf16_bits(u.astype(np.float32)), "bf16")
    return oracle.selective_scan(u, x.f64("delta"), x.f64("A"), x.f64("B"), x.f64("C"), x.f64("D"),
                                 x.f64("z") if with_z else None, x.f64("delta_bias"))


@pytest.mark.gpu
@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("L", [1, 3, 8, 9, 256, 300, 1000])
@pytest.mark.parametrize("silu", [True, False])
def test_conv_standalone(io, L, silu):
    import torch
    x, w, b = conv_inputs(2, 37, 4, L, io, seed=60 + L)
    t = dev_inputs(x)
    u = torch.empty_like(t["u"])
    for bias in (b, None):
        m.mamba_causal_conv1d_silu(t["u"], f32_dev(w), None if bias is None else f32_dev(bias), silu, u)
        torch.cuda.synchronize()
        ref = oracle.causal_conv1d(x.f64("u"), w.astype(np.float64), None if bias is None else bias.astype(np.float64),
                                   silu=silu)
        assert_close(to_host_f64(u), ref, TOL_Y[io], f"conv {io} L={L} silu={silu}")


@pytest.mark.gpu
def test_conv_standalone_unaligned_view():
    import torch
    x, w, b = conv_inputs(1, 5, 4, 64, "bf16", seed=70)
    t = dev_inputs(x)
    big = torch.empty(t["u"].numel() + 1, dtype=t["u"].dtype, device="cuda")
    big[1:].copy_(t["u"].reshape(-1))
    xv = big[1:].view(t["u"].shape)
    u = torch.empty_like(xv)
    m.mamba_causal_conv1d_silu(xv, f32_dev(w), f32_dev(b), True, u)
    torch.cuda.synchronize()
    assert_close(to_host_f64(u), oracle.causal_conv1d(x.f64("u"), w.astype(np.float64), b.astype(np.float64)),
                 TOL_Y["bf16"], "conv unaligned")


@pytest.mark.gpu
@pytest.mark.parametrize("shape,io,with_z,fused", [
    ((2, 45, 16, 256), "bf16", True, True),      # fused tensor-memory kernel
    ((2, 45, 12, 72), "bf16", True, True),       # fused, N < 16
    ((1, 13, 16, 4096), "bf16", True, True),     # fused, chunked (halo across chunk boundaries)
    ((2, 45, 16, 256), "bf16", False, False),    # no gate: convolution then scan
    ((2, 21, 32, 128), "bf16", True, False),     # N > 16: convolution then scan
    ((2, 21, 16, 130), "bf16", True, False),     # unaligned rows: convolution then scan
    ((1, 9, 16, 200), "f32", True, False),       # fp32: convolution then scan
])
def test_conv_fed_scan(shape, io, with_z, fused):
    import torch
    Bsz, Dch, N, L = shape
    x, w, b = conv_inputs(Bsz, Dch, N, L, io, seed=80 + N + L)
    t = dev_inputs(x)
    y = torch.empty_like(t["u"])
    last = torch.empty((Bsz, Dch, N), dtype=torch.float32, device="cuda")
    m.mamba_selective_scan_fwd_conv(t["u"], f32_dev(w), f32_dev(b), t["delta"], t["A"], t["B"], t["C"], t["D"],
                                    t["z"] if with_z else None, t["delta_bias"], 1, y, last)
    torch.cuda.synchronize()
    assert m.mamba_device_error() == 0
    yr, hr = oracle_conv_scan(x, w, b, with_z, u_stored=not fused)
    assert_close(to_host_f64(y), yr, TOL_Y[io], f"conv-fed scan {shape} {io} y")
    eh = assert_close(last.cpu().numpy().astype(np.float64), hr, TOL_STATE, f"conv-fed scan {shape} {io} last_state")
    print(f"conv-fed scan {shape} {io} {'fused' if fused else 'two-step'}: last_state err ratio {eh:.3g}")


@pytest.mark.gpu
def test_fused_path_allocates_nothing(monkeypatch):
    """The fused kernel needs no temporary: with the allocation made to fail on the host, the fused
    case still runs while the two-step case (no gate) reports MAMBA_ERR_ALLOC."""
    import torch
    x, w, b = conv_inputs(2, 45, 16, 256, "bf16", seed=90)
    t = dev_inputs(x)
    y = torch.empty_like(t["u"])
    monkeypatch.setenv("MAMBA_FAULT_INJECT", "alloc")
    m.mamba_selective_scan_fwd_conv(t["u"], f32_dev(w), f32_dev(b), t["delta"], t["A"], t["B"], t["C"], t["D"],
                                    t["z"], t["delta_bias"], 1, y, None)
    torch.cuda.synchronize()
    yr, _ = oracle_conv_scan(x, w, b)
    assert_close(to_host_f64(y), yr, TOL_Y["bf16"], "fused under injected allocation failure")
    with pytest.raises(m.MambaError) as e:
        m.mamba_selective_scan_fwd_conv(t["u"], f32_dev(w), f32_dev(b), t["delta"], t["A"], t["B"], t["C"],
                                        t["D"], None, t["delta_bias"], 1, y, None)
    assert e.value.status == -5
