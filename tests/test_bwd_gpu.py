"""Backward pass of the scan on the GPU against the float64 oracle's chain rule.

The oracle backward is itself pinned by central differences of the forward
oracle (tests/test_oracle_pins.py).  Per-element outputs (du, ddelta, dz) are
compared elementwise; the fp32 sums (dA, dB, dC, dD, ddelta_bias) add up many
terms of both signs, so they are compared against the scale of the tensor:
max |gpu - ref| <= tol * (1 + max |ref|).
"""
import numpy as np
import pytest

import oracle
import selective_state_space_148_b300 as m
from selective_state_space_148_b300 import inputs
from helpers import TOL_Y, assert_close, dev_inputs, to_host_f64

pytestmark = pytest.mark.gpu

TOL_SUM = {"f32": 2e-4, "bf16": 2e-3}


def run_bwd(x, dy, with_z=True, softplus=True):
    import torch
    t = dev_inputs(x)
    Bsz, Dch, L, N = x.shape
    dyd = dev_inputs(inputs.ScanInputs(io=x.io, u=dy, delta=dy, z=None, B=x.B, C=x.C, A=x.A, D=x.D,
                                       delta_bias=x.delta_bias))["u"]
    du, ddelta = torch.empty_like(t["u"]), torch.empty_like(t["u"])
    dz = torch.empty_like(t["u"]) if with_z else None
    f32 = dict(dtype=torch.float32, device="cuda")
    dA, dB, dC = torch.empty((Dch, N), **f32), torch.empty((Bsz, N, L), **f32), torch.empty((Bsz, N, L), **f32)
    dD, dbias = torch.empty(Dch, **f32), torch.empty(Dch, **f32)
    m.mamba_selective_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"] if with_z else None,
                               t["delta_bias"], softplus, dyd, du, ddelta, dA, dB, dC, dD, dz, dbias)
    torch.cuda.synchronize()
    out = dict(du=to_host_f64(du), ddelta=to_host_f64(ddelta), dA=dA.cpu().numpy().astype(np.float64),
               dB=dB.cpu().numpy().astype(np.float64), dC=dC.cpu().numpy().astype(np.float64),
               dD=dD.cpu().numpy().astype(np.float64), ddelta_bias=dbias.cpu().numpy().astype(np.float64))
    out["dz"] = to_host_f64(dz) if with_z else None
    return out


def ref_bwd(x, dy, with_z=True, softplus=True):
    return oracle.selective_scan_bwd(x.f64("u"), x.f64("delta"), x.f64("A"), x.f64("B"), x.f64("C"),
                                     inputs.to_f64(dy, x.io), x.f64("D"), x.f64("z") if with_z else None,
                                     x.f64("delta_bias"), softplus_flag=softplus)


def check_bwd(x, tag, with_z=True, softplus=True, seed=0):
    r = np.random.default_rng(seed)
    dy = inputs._store(r.standard_normal(x.u.shape).astype(np.float32), x.io)
    g = run_bwd(x, dy, with_z, softplus)
    ref = ref_bwd(x, dy, with_z, softplus)
    for k in ("du", "ddelta") + (("dz",) if with_z else ()):
        assert_close(g[k], ref[k], TOL_Y[x.io], f"{tag} {k}")
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        err = np.abs(g[k] - ref[k]).max()
        scale = 1.0 + np.abs(ref[k]).max()
        assert np.all(np.isfinite(g[k])), f"{tag} {k}: non-finite"
        assert err <= TOL_SUM[x.io] * scale, f"{tag} {k}: max err {err:.3g} vs scale {scale:.3g}"


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 4, 16, 17, 33, 64])
def test_backward_state_sizes(io, N):
    x = inputs.make_scan_inputs(2, 37, N, 100, io=io, seed=100 + N)
    check_bwd(x, f"bwd N={N} {io}", seed=N)


@pytest.mark.parametrize("L", [1, 7, 8, 9, 257])
def test_backward_lengths(L):
    x = inputs.make_scan_inputs(1, 40, 16, L, io="f32", seed=200 + L)
    check_bwd(x, f"bwd L={L}", seed=L)


@pytest.mark.parametrize("variant", ["no_gate", "no_softplus"])
def test_backward_variants(variant):
    x = inputs.make_scan_inputs(2, 19, 16, 120, io="f32", seed=300)
    if variant == "no_softplus":
        x.delta_bias = (x.delta_bias * 0 + 2.0).astype(np.float32)   # Delta = Delta_raw + bias stays positive
    check_bwd(x, variant, with_z=variant != "no_gate", softplus=variant != "no_softplus", seed=3)


def test_backward_long_rows():
    """Rows of the 130M-shaped layer's length (L = 2048, bf16) over 96 channels, every output against the oracle."""
    x = inputs.make_scan_inputs(1, 96, 16, 2048, io="bf16", seed=400)
    check_bwd(x, "bwd L=2048 D=96", seed=4)


def test_backward_full_130m_layer_every_element():
    """The whole 130M-shaped layer (B8 D1536 N16 L2048, bf16), in the launch configuration the benchmark
    times: every du, ddelta, dz element and every dA, dB, dC, dD, ddelta_bias sum against the oracle."""
    x = inputs.make_workload("mamba130m_b8_d1536_n16_l2048_bf16")
    check_bwd(x, "bwd 130M layer", seed=5)
    assert m.mamba_device_error() == 0

