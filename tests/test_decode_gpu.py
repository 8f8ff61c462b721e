"""Parity of the CUDA decode step (mamba_state_update) with the float64 oracle,
over chains of steps in which the oracle keeps its own state and is never
re-synchronised to the GPU's."""
import numpy as np
import pytest

import oracle
import selective_state_space_148_b300 as m
from selective_state_space_148_b300 import inputs
from helpers import TOL_STATE, TOL_STATE_CHAIN, TOL_Y, assert_close, f32_dev, to_dev, to_host_f64

pytestmark = pytest.mark.gpu


def chain(Bsz, Dch, N, steps, io, seed, sample=None, with_z=True, with_D=True):
    import torch
    A, D, bias, _ = inputs.channel_params(Dch, N, seed)
    st0 = inputs.make_decode_state(Bsz, Dch, N, seed)
    state = f32_dev(st0)
    Ad, Dd, bd = f32_dev(A), f32_dev(D), f32_dev(bias)
    if sample is None:
        sample = [(b, d) for b in range(Bsz) for d in range(Dch)]
    sb = np.array([b for b, _ in sample])
    sd = np.array([d for _, d in sample])
    ref_state = st0[sb, sd].astype(np.float64)[None]          # [1, S, N]: one "batch" of sampled channels
    worst_y = 0.0
    for k in range(steps):
        s = inputs.make_decode_step(Bsz, Dch, N, seed, k, io)
        u, dl, z, B, C = (to_dev(getattr(s, n), io) for n in ("u", "delta", "z", "B", "C"))
        y = torch.empty_like(u)
        m.mamba_state_update(state, u, dl, Ad, B, C, Dd if with_D else None, z if with_z else None, bd, 1, y)
        # oracle on the sampled channels, each one its own (b, d) problem
        su, sdl, sz = (inputs.to_f64(getattr(s, n)[sb, sd], io) for n in ("u", "delta", "z"))
        sB, sC = (inputs.to_f64(getattr(s, n)[sb], io) for n in ("B", "C"))
        yr = np.empty(len(sample))
        new = np.empty_like(ref_state)
        for j, (b, d) in enumerate(sample):
            yy, hh = oracle.state_update(ref_state[:, j:j + 1], su[j].reshape(1, 1), sdl[j].reshape(1, 1),
                                         A[d:d + 1].astype(np.float64), sB[j:j + 1], sC[j:j + 1],
                                         D[d:d + 1].astype(np.float64) if with_D else None,
                                         sz[j].reshape(1, 1) if with_z else None, bias[d:d + 1].astype(np.float64))
            yr[j] = yy[0, 0]
            new[:, j] = hh[:, 0]
        ref_state = new
        yg = to_host_f64(y)[sb, sd]
        worst_y = max(worst_y, assert_close(yg, yr, TOL_Y[io], f"step {k} y"))
    torch.cuda.synchronize()
    hg = state.cpu().numpy().astype(np.float64)[sb, sd]
    es = assert_close(hg, ref_state[0], TOL_STATE_CHAIN if steps > 100 else TOL_STATE, "final state")
    return worst_y, es


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_small_chain(io):
    ey, es = chain(4, 64, 16, 50, io, seed=31)
    print(f"decode small {io}: y {ey:.3g} state {es:.3g}")


@pytest.mark.parametrize("N", [1, 3, 5, 8, 16, 17, 32, 64])
def test_decode_state_sizes(N):
    chain(3, 17, N, 12, "bf16", seed=32)


def test_decode_optional_inputs():
    chain(2, 33, 16, 10, "bf16", seed=33, with_z=False, with_D=False)


def test_scan_then_step_equals_longer_scan():
    """scan over t < L, then one decode step for token L, matches the oracle scan over L + 1 tokens."""
    import torch
    x = inputs.make_scan_inputs(2, 40, 16, 129, io="f32", seed=34)
    yr, hr = oracle.selective_scan(x.f64("u"), x.f64("delta"), x.f64("A"), x.f64("B"), x.f64("C"), x.f64("D"),
                                   x.f64("z"), x.f64("delta_bias"))
    L = 128
    dev = lambda a: f32_dev(np.ascontiguousarray(a))
    u, dl, z, B, C = (dev(getattr(x, n)[..., :L]) for n in ("u", "delta", "z", "B", "C"))
    y = torch.empty_like(u)
    h = torch.empty((2, 40, 16), dtype=torch.float32, device="cuda")
    m.mamba_selective_scan_fwd(u, dl, f32_dev(x.A), B, C, f32_dev(x.D), z, f32_dev(x.delta_bias), 1, y, h)
    yl = torch.empty((2, 40), dtype=torch.float32, device="cuda")
    m.mamba_state_update(h, dev(x.u[..., L]), dev(x.delta[..., L]), f32_dev(x.A), dev(x.B[..., L]),
                         dev(x.C[..., L]), f32_dev(x.D), dev(x.z[..., L]), f32_dev(x.delta_bias), 1, yl)
    torch.cuda.synchronize()
    assert_close(to_host_f64(y), yr[..., :L], TOL_Y["f32"], "scan part")
    assert_close(to_host_f64(yl), yr[..., L], TOL_Y["f32"], "step token")
    assert_close(h.cpu().numpy(), hr, TOL_STATE, "state after step")
