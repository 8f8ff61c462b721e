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


def run_bwd(x, dy, with_z=True, softplus=True, train=False):
    """The backward on the GPU: mamba_selective_scan_bwd, or (train) mamba_selective_scan_fwd_save followed by
    mamba_selective_scan_bwd_from_ckpt, whose forward outputs are checked against the oracle here too."""
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
    zz = t["z"] if with_z else None
    if train:
        y = torch.empty_like(t["u"])
        ck = torch.empty(m.mamba_scan_bwd_ckpt_size(Bsz, Dch, L, N) // 4, dtype=torch.float32, device="cuda")
        m.mamba_selective_scan_fwd_save(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], zz, t["delta_bias"],
                                        softplus, y, None, ck)
        m.mamba_selective_scan_bwd_from_ckpt(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], zz, t["delta_bias"],
                                             softplus, dyd, ck, du, ddelta, dA, dB, dC, dD, dz, dbias)
        torch.cuda.synchronize()
        yr, _ = oracle.selective_scan(x.f64("u"), x.f64("delta"), x.f64("A"), x.f64("B"), x.f64("C"), x.f64("D"),
                                      x.f64("z") if with_z else None, x.f64("delta_bias"), softplus_flag=softplus)
        assert_close(to_host_f64(y), yr, TOL_Y[x.io], "training pair forward y")
        del ck
    else:
        m.mamba_selective_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], zz, t["delta_bias"], softplus,
                                   dyd, du, ddelta, dA, dB, dC, dD, dz, dbias)
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


def check_bwd(x, tag, with_z=True, softplus=True, seed=0, train=False):
    r = np.random.default_rng(seed)
    dy = inputs._store(r.standard_normal(x.u.shape).astype(np.float32), x.io)
    g = run_bwd(x, dy, with_z, softplus, train)
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


@pytest.mark.parametrize("path", ["self_checkpointed", "training_pair"])
def test_backward_full_130m_layer_every_element(path):
    """The whole 130M-shaped layer (B8 D1536 N16 L2048, bf16), in the launch configuration the benchmark
    times: every du, ddelta, dz element and every dA, dB, dC, dD, ddelta_bias sum against the oracle -- the
    backward that takes its own checkpoints, and the forward-with-checkpoints / backward-from-checkpoints
    pair (whose forward outputs are checked too)."""
    x = inputs.make_workload("mamba130m_b8_d1536_n16_l2048_bf16")
    check_bwd(x, f"bwd 130M layer ({path})", seed=5, train=path == "training_pair")
    assert m.mamba_device_error() == 0


# ----------------------------------------------------------------------------- the training pair

def ckpt_geometry(N):
    ns = 4 if N <= 16 else 8 if N <= 32 else 16
    return 64 // ns, 4 * ns          # steps between checkpoints, padded states


@pytest.mark.parametrize("io,N,L", [("bf16", 12, 200), ("bf16", 16, 200), ("bf16", 32, 200), ("bf16", 64, 200),
                                    ("f32", 16, 200), ("bf16", 4, 200), ("f32", 24, 200), ("bf16", 16, 199),
                                    ("bf16", 16, 16), ("bf16", 64, 3)])
def test_training_pair_checkpoints_and_gradients(io, N, L):
    """The training pair's checkpoints and gradients against the oracle (training_pair_checks)."""
    training_pair_checks(io, N, L)


@pytest.mark.parametrize("N", [16, 32, 64])
def test_training_pair_lean_form(N, monkeypatch):
    """The same checks with MAMBA_TM_LEAN=1: the lean form of the tensor-memory kernel (12..18 compute warps,
    its checkpoint-writing instantiation) serves the forward."""
    monkeypatch.setenv("MAMBA_TM_LEAN", "1")
    training_pair_checks("bf16", N, 200)


def training_pair_checks(io, N, L):
    """mamba_selective_scan_fwd_save writes y, last_state and, for every k >= 1, the state before step k * c
    (c = 16, 8, 4 for N <= 16, 32, 64): each checkpoint is compared with the oracle's last_state over the
    first k * c steps, and the padding states past N must be zero.  mamba_selective_scan_bwd_from_ckpt then
    gives the oracle's gradients.  Aligned rows with 8 < N <= 64 (fp32: N <= 16) take the tensor-memory
    kernel's checkpoint writes; N = 4, fp32 N = 24 and the odd length 199 take the scan followed by the
    checkpoint sweep; L = 16 and L = 3 have a single checkpoint chunk."""
    import torch
    x = inputs.make_scan_inputs(2, 37, N, L, io=io, seed=600 + N + L)
    Bsz, Dch, _, _ = x.shape
    c, P = ckpt_geometry(N)
    K = -(-L // c)
    t = dev_inputs(x)
    y = torch.empty_like(t["u"])
    last = torch.empty((Bsz, Dch, N), dtype=torch.float32, device="cuda")
    assert m.mamba_scan_bwd_ckpt_size(Bsz, Dch, L, N) == Bsz * Dch * K * P * 4
    ck = torch.full((Bsz, Dch, K, P), float("nan"), dtype=torch.float32, device="cuda")
    m.mamba_selective_scan_fwd_save(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], 1,
                                    y, last, ck)
    torch.cuda.synchronize()
    assert m.mamba_device_error() == 0
    yr, hr = oracle.selective_scan(x.f64("u"), x.f64("delta"), x.f64("A"), x.f64("B"), x.f64("C"), x.f64("D"),
                                   x.f64("z"), x.f64("delta_bias"))
    assert_close(to_host_f64(y), yr, TOL_Y[io], "fwd_save y")
    assert_close(last.cpu().numpy().astype(np.float64), hr, 1e-4, "fwd_save last_state")
    ckh = ck.cpu().numpy().astype(np.float64)
    for k in range(1, K):
        tk = k * c
        _, hk = oracle.selective_scan(x.f64("u")[:, :, :tk], x.f64("delta")[:, :, :tk], x.f64("A"),
                                      x.f64("B")[:, :, :tk], x.f64("C")[:, :, :tk], x.f64("D"), x.f64("z")[:, :, :tk],
                                      x.f64("delta_bias"))
        assert_close(ckh[:, :, k, :N], hk, 1e-4, f"checkpoint {k} (state before step {tk})")
        assert np.all(ckh[:, :, k, N:] == 0), f"checkpoint {k}: padding states"
    check_bwd(x, f"training pair N={N} {io} L={L}", seed=N + L, train=True)

