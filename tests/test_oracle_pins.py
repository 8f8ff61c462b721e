"""Pins for the float64 oracle: closed forms, brute force and invariants.

The pages print no numeric worked example, so the oracle is tied to things the
method text fixes by itself:
  * the LTI special case equals the convolution with K = (C B_bar, C A_bar B_bar, ...)
    (Mamba tutorial, freeguideonline, section 2.3);
  * A = 0, Delta = 1 makes the state a running sum;
  * brute-force unrolling of the recurrence on L <= 8
    h_t = sum_{s<=t} (prod_{s<r<=t} A_bar_r) B_bar_s u_s;
  * the geometric series for constant inputs;
  * the exact zero-order hold (section 2.2) agrees with integrating the
    continuous system x' = A x + B u (section 2.1) over each step;
  * hand-worked cases in tests/golden/hand_worked.json;
  * invariants: linearity, causality, C = 0, z = 0, chunking, scan/step, reverse.
Each check would fail on a dropped term, a wrong sign or index, or a
transposed operand in the oracle.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.integrate import solve_ivp
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def rand_case(rng, Bsz, Dch, L, N, a_range=(-2.0, -0.05)):
    return dict(
        u=rng.standard_normal((Bsz, Dch, L)),
        delta=rng.normal(0.0, 0.5, (Bsz, Dch, L)),
        A=rng.uniform(a_range[0], a_range[1], (Dch, N)),
        B=rng.standard_normal((Bsz, N, L)),
        C=rng.standard_normal((Bsz, N, L)),
        D=rng.standard_normal(Dch),
        z=rng.standard_normal((Bsz, Dch, L)),
        delta_bias=rng.uniform(-3.0, 0.0, Dch),
    )


def softplus_lib(x):
    return np.logaddexp(0.0, x)


# --------------------------------------------------------------------------- hand-worked cases

@pytest.mark.parametrize("case", json.load(open(GOLDEN))["scan"], ids=lambda c: c["name"])
def test_hand_worked_scan(case):
    L, N = case["L"], case["N"]
    u = np.array(case["u"], dtype=float).reshape(1, 1, L)
    delta = np.array(case["delta"], dtype=float).reshape(1, 1, L)
    A = np.array(case["A"], dtype=float).reshape(1, N)
    B = np.array(case["B"], dtype=float).reshape(1, N, L)
    C = np.array(case["C"], dtype=float).reshape(1, N, L)
    z = None if case["z"] is None else np.array(case["z"], dtype=float).reshape(1, 1, L)
    y, last = oracle.selective_scan(u, delta, A, B, C, D=np.array([case["D"]]), z=z,
                                    delta_bias=np.array([case["bias"]]), softplus_flag=case["softplus"],
                                    disc=case["zoh"])
    np.testing.assert_allclose(y.ravel(), case["y"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(last.ravel(), case["last"], rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["step"], ids=lambda c: c["name"])
def test_hand_worked_step(case):
    N = case["N"]
    y, st = oracle.state_update(np.array(case["state"]).reshape(1, 1, N), np.array([[case["u"]]]),
                                np.array([[case["delta"]]]), np.array(case["A"]).reshape(1, N),
                                np.array(case["B"]).reshape(1, N), np.array(case["C"]).reshape(1, N),
                                D=np.array([case["D"]]), z=None, delta_bias=np.array([case["bias"]]),
                                softplus_flag=case["softplus"])
    np.testing.assert_allclose(y.ravel(), [case["y"]], rtol=1e-14)
    np.testing.assert_allclose(st.ravel(), case["new_state"], rtol=1e-14)


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("gate", [False, True])
def test_lti_equals_convolution(gate):
    """Delta, B, C constant in t: y = u * K + D u with K_k = sum_n C_n A_bar_n^k Delta B_n."""
    rng = np.random.default_rng(11)
    Bsz, Dch, L, N = 2, 3, 256, 4
    A = rng.uniform(-2.0, -0.01, (Dch, N))
    draw = rng.normal(0.0, 0.5, Dch)                 # one Delta_raw per channel, constant in t
    bias = rng.uniform(-4.0, 0.0, Dch)
    Bn = rng.standard_normal((Bsz, N))
    Cn = rng.standard_normal((Bsz, N))
    D = rng.standard_normal(Dch)
    u = rng.standard_normal((Bsz, Dch, L))
    z = rng.standard_normal((Bsz, Dch, L)) if gate else None
    delta = np.broadcast_to(draw[None, :, None], (Bsz, Dch, L))
    Bt = np.broadcast_to(Bn[:, :, None], (Bsz, N, L))
    Ct = np.broadcast_to(Cn[:, :, None], (Bsz, N, L))
    y, _ = oracle.selective_scan(u, delta, A, Bt, Ct, D=D, z=z, delta_bias=bias, softplus_flag=True)
    k = np.arange(L)
    for b in range(Bsz):
        for d in range(Dch):
            dt = softplus_lib(draw[d] + bias[d])
            # materialised kernel: K_k = sum_n C_n * exp(k * dt * A_n) * dt * B_n  (A_bar^k in closed form)
            K = (Cn[b][None, :] * np.exp(np.outer(k, dt * A[d])) * dt * Bn[b][None, :]).sum(axis=1)
            ref = np.convolve(u[b, d], K)[:L] + D[d] * u[b, d]
            if gate:
                ref = ref * z[b, d] * expit(z[b, d])
            scale = np.abs(ref).max()
            assert np.abs(y[b, d] - ref).max() <= 1e-12 * scale


def test_running_sum():
    """A = 0, Delta = 1 (softplus off), B = C = 1, D = 0: y_t = N * sum_{s<=t} u_s, exactly for integers."""
    rng = np.random.default_rng(12)
    Bsz, Dch, L, N = 2, 5, 300, 7
    u = rng.integers(-50, 50, (Bsz, Dch, L)).astype(float)
    y, last = oracle.selective_scan(u, np.ones((Bsz, Dch, L)), np.zeros((Dch, N)), np.ones((Bsz, N, L)),
                                    np.ones((Bsz, N, L)), D=np.zeros(Dch), z=None, delta_bias=np.zeros(Dch),
                                    softplus_flag=False)
    assert np.array_equal(y, N * np.cumsum(u, axis=-1))
    assert np.array_equal(last, np.broadcast_to(np.cumsum(u, axis=-1)[..., -1:], (Bsz, Dch, N)))


@pytest.mark.parametrize("t_len", [1, 2, 5, 8])
def test_geometric_closed_form(t_len):
    """N = 1, u = 1, constant Delta and A, B = C = 1, D = 0: y_t = Delta (1 - a^{t+1}) / (1 - a), a = e^{Delta A}."""
    dt, a = 0.37, -0.8
    y, _ = oracle.selective_scan(np.ones((1, 1, t_len)), np.full((1, 1, t_len), dt), np.array([[a]]),
                                 np.ones((1, 1, t_len)), np.ones((1, 1, t_len)), D=None, z=None, delta_bias=None,
                                 softplus_flag=False)
    abar = math.exp(dt * a)
    ref = [dt * (1 - abar ** (t + 1)) / (1 - abar) for t in range(t_len)]
    np.testing.assert_allclose(y.ravel(), ref, rtol=1e-14)


def brute_force(c, softplus_flag=True, gate=True, h0=None, reverse=False, zoh=False):
    """Unrolled sum over source steps s with explicit products of A_bar over the steps in between."""
    u, A, B, C, D = c["u"], c["A"], c["B"], c["C"], c["D"]
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    dt = c["delta"] + c["delta_bias"][None, :, None]
    if softplus_flag:
        dt = softplus_lib(dt)
    order = list(range(L))[::-1] if reverse else list(range(L))
    y = np.zeros((Bsz, Dch, L))
    last = np.zeros((Bsz, Dch, N))
    for b in range(Bsz):
        for d in range(Dch):
            abar = np.exp(dt[b, d][:, None] * A[d][None, :])             # [L, N]
            if zoh:
                wB = (abar - 1.0) / A[d][None, :] * B[b].T               # [L, N]
            else:
                wB = dt[b, d][:, None] * B[b].T
            for i, t in enumerate(order):
                h = np.zeros(N)
                for j in range(i + 1):                                   # source step s = order[j]
                    s = order[j]
                    prod = np.ones(N)
                    for r in order[j + 1:i + 1]:
                        prod = prod * abar[r]
                    h = h + prod * wB[s] * u[b, d, s]
                if h0 is not None:
                    prod = np.ones(N)
                    for r in order[:i + 1]:
                        prod = prod * abar[r]
                    h = h + prod * h0[b, d]
                yt = (C[b][:, t] * h).sum() + D[d] * u[b, d, t]
                if gate:
                    zt = c["z"][b, d, t]
                    yt *= zt * expit(zt)
                y[b, d, t] = yt
                if i == L - 1:
                    last[b, d] = h
    return y, last


@pytest.mark.parametrize("L", [1, 3, 8])
@pytest.mark.parametrize("variant", ["plain", "no_softplus", "h0", "reverse", "zoh", "no_gate"])
def test_bruteforce_unroll(L, variant):
    rng = np.random.default_rng(100 + L)
    c = rand_case(rng, 2, 3, L, 4)
    sp = variant != "no_softplus"
    gate = variant != "no_gate"
    h0 = rng.standard_normal((2, 3, 4)) if variant == "h0" else None
    rev = variant == "reverse"
    zoh = variant == "zoh"
    y, last = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], D=c["D"],
                                    z=c["z"] if gate else None, delta_bias=c["delta_bias"], softplus_flag=sp,
                                    h0=h0, disc=oracle.DISC_ZOH if zoh else oracle.DISC_SIMPLE, reverse=rev)
    yr, lr = brute_force(c, softplus_flag=sp, gate=gate, h0=h0, reverse=rev, zoh=zoh)
    np.testing.assert_allclose(y, yr, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(last, lr, rtol=1e-12, atol=1e-13)


def test_zoh_matches_continuous_system():
    """Exact ZOH: h_t is the solution of x' = A x + B_t u_t after a step of length Delta_t from h_{t-1}."""
    rng = np.random.default_rng(13)
    L, N = 6, 3
    A = rng.uniform(-2.0, -0.2, (1, N))
    dts = rng.uniform(0.05, 0.9, L)
    B = rng.standard_normal((1, N, L))
    u = rng.standard_normal((1, 1, L))
    C = np.zeros((1, N, L))
    _, last_all = None, None
    x = np.zeros(N)
    for t in range(L):
        sol = solve_ivp(lambda _s, xx: A[0] * xx + B[0, :, t] * u[0, 0, t], (0.0, dts[t]), x, rtol=1e-12,
                        atol=1e-14, method="DOP853")
        x = sol.y[:, -1]
        _, h = oracle.selective_scan(u[:, :, :t + 1], dts[None, None, :t + 1], A, B[:, :, :t + 1],
                                     C[:, :, :t + 1], softplus_flag=False, disc=oracle.DISC_ZOH)
        np.testing.assert_allclose(h.ravel(), x, rtol=1e-9, atol=1e-11)


def test_zoh_steady_state():
    """Constant input under exact ZOH settles at the continuous fixed point x* = -B u / A."""
    N, L = 3, 4000
    A = np.array([[-0.5, -1.0, -3.0]])
    Bv = np.array([0.7, -1.2, 2.0])
    _, h = oracle.selective_scan(np.full((1, 1, L), 1.5), np.full((1, 1, L), 0.05), A,
                                 np.broadcast_to(Bv[None, :, None], (1, N, L)), np.zeros((1, N, L)),
                                 softplus_flag=False, disc=oracle.DISC_ZOH)
    np.testing.assert_allclose(h.ravel(), -Bv * 1.5 / A[0], rtol=1e-10)


def test_zoh_limit_a_zero():
    """With A = 0 the ZOH weight reduces to Delta * B (the limit of (e^{Delta A} - 1)/A)."""
    rng = np.random.default_rng(14)
    c = rand_case(rng, 1, 2, 9, 3)
    c["A"][:] = 0.0
    y1, l1 = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"],
                                   disc=oracle.DISC_ZOH)
    y2, l2 = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"],
                                   disc=oracle.DISC_SIMPLE)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(l1, l2)


def test_softplus_special_values():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-16, abs=0)
    assert oracle.softplus(50.0) == pytest.approx(50.0, rel=1e-15)
    assert oracle.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-14)
    for x in (-3.0, -0.5, 0.25, 4.0):
        assert oracle.softplus(x) == pytest.approx(float(softplus_lib(x)), rel=1e-15)


# --------------------------------------------------------------------------- invariants

def test_linearity_in_u():
    rng = np.random.default_rng(15)
    c = rand_case(rng, 2, 3, 64, 5)
    u2 = rng.standard_normal(c["u"].shape)
    f = lambda uu: oracle.selective_scan(uu, c["delta"], c["A"], c["B"], c["C"], c["D"], None, c["delta_bias"])
    y1, h1 = f(c["u"])
    y2, h2 = f(u2)
    y3, h3 = f(2.5 * c["u"] - 0.75 * u2)
    np.testing.assert_allclose(y3, 2.5 * y1 - 0.75 * y2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h3, 2.5 * h1 - 0.75 * h2, rtol=1e-12, atol=1e-12)


def test_causality():
    rng = np.random.default_rng(16)
    c = rand_case(rng, 1, 2, 40, 4)
    y1, _ = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"])
    for t0 in (0, 17, 39):
        u = c["u"].copy()
        u[0, 1, t0] += 3.0
        y2, _ = oracle.selective_scan(u, c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"])
        np.testing.assert_array_equal(y2[0, 1, :t0], y1[0, 1, :t0])
        np.testing.assert_array_equal(y2[0, 0], y1[0, 0])                  # other channel untouched
        assert np.abs(y2[0, 1, t0:] - y1[0, 1, t0:]).max() > 0


def test_c_zero_and_z_zero():
    rng = np.random.default_rng(17)
    c = rand_case(rng, 2, 3, 30, 4)
    y, _ = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], np.zeros_like(c["C"]), c["D"], c["z"],
                                 c["delta_bias"])
    np.testing.assert_allclose(y, c["D"][None, :, None] * c["u"] * c["z"] * expit(c["z"]), rtol=1e-14)
    y, _ = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], np.zeros_like(c["z"]),
                                 c["delta_bias"])
    assert np.all(y == 0.0)


@pytest.mark.parametrize("k", [1, 13, 63])
def test_chunk_consistency(k):
    """scan[0, L) == scan[0, k) followed by scan[k, L) started from its last state."""
    rng = np.random.default_rng(18)
    c = rand_case(rng, 2, 2, 64, 4)
    full_y, full_h = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"],
                                           c["delta_bias"])
    sl = lambda a, lo, hi: a[..., lo:hi]
    y1, h1 = oracle.selective_scan(*(sl(c[n], 0, k) for n in ("u", "delta")), c["A"],
                                   *(sl(c[n], 0, k) for n in ("B", "C")), c["D"], sl(c["z"], 0, k),
                                   c["delta_bias"])
    y2, h2 = oracle.selective_scan(*(sl(c[n], k, 64) for n in ("u", "delta")), c["A"],
                                   *(sl(c[n], k, 64) for n in ("B", "C")), c["D"], sl(c["z"], k, 64),
                                   c["delta_bias"], h0=h1)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=-1), full_y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h2, full_h, rtol=1e-13, atol=1e-14)


def test_scan_equals_repeated_step():
    rng = np.random.default_rng(19)
    c = rand_case(rng, 2, 3, 20, 4)
    y, h = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"])
    st = np.zeros((2, 3, 4))
    for t in range(20):
        yt, st = oracle.state_update(st, c["u"][..., t], c["delta"][..., t], c["A"], c["B"][..., t],
                                     c["C"][..., t], c["D"], c["z"][..., t], c["delta_bias"])
        np.testing.assert_allclose(yt, y[..., t], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(st, h, rtol=1e-14, atol=1e-15)


def test_reverse_is_flipped_forward():
    rng = np.random.default_rng(20)
    c = rand_case(rng, 2, 3, 33, 4)
    yr, hr = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"],
                                   reverse=True)
    f = {n: np.ascontiguousarray(c[n][..., ::-1]) for n in ("u", "delta", "B", "C", "z")}
    yf, hf = oracle.selective_scan(f["u"], f["delta"], c["A"], f["B"], f["C"], c["D"], f["z"], c["delta_bias"])
    np.testing.assert_array_equal(yr, yf[..., ::-1])
    np.testing.assert_array_equal(hr, hf)


def test_channels_independent_and_broadcast():
    """B and C are shared by every channel of a batch; A, D, bias belong to a channel."""
    rng = np.random.default_rng(21)
    c = rand_case(rng, 2, 4, 16, 3)
    y, h = oracle.selective_scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"])
    for b in range(2):
        for d in range(4):
            y1, h1 = oracle.selective_scan(c["u"][b:b + 1, d:d + 1], c["delta"][b:b + 1, d:d + 1],
                                           c["A"][d:d + 1], c["B"][b:b + 1], c["C"][b:b + 1], c["D"][d:d + 1],
                                           c["z"][b:b + 1, d:d + 1], c["delta_bias"][d:d + 1])
            np.testing.assert_array_equal(y1[0, 0], y[b, d])
            np.testing.assert_array_equal(h1[0, 0], h[b, d])


# ----------------------------------------------------------------------------- causal conv1d + SiLU (the branch feeding the scan)
# ai.xwebgame.com summary, "running it in PyTorch" block: Conv1d(d_inner, d_inner, kernel_size=4,
# groups=d_inner, padding=3), first L outputs, then SiLU.

def _conv_case(seed, Bsz=2, Dch=5, L=23, W=4):
    r = np.random.default_rng(seed)
    return r.normal(size=(Bsz, Dch, L)), r.normal(size=(Dch, W)), r.normal(size=Dch)


def test_conv_identity_tap_is_the_input():
    x, w, _ = _conv_case(0)
    w[:] = 0.0
    w[:, 3] = 1.0                      # the tap on x_t itself
    assert np.array_equal(oracle.causal_conv1d(x, w, None, silu=False), x)


def test_conv_shift_tap_delays_by_one_with_zero_padding():
    x, w, _ = _conv_case(1)
    w[:] = 0.0
    w[:, 2] = 1.0                      # the tap on x_{t-1}
    u = oracle.causal_conv1d(x, w, None, silu=False)
    assert np.array_equal(u[..., 1:], x[..., :-1])
    assert np.all(u[..., 0] == 0.0)


def test_conv_matches_numpy_convolution():
    """pre_t = b + sum_k w_k x_{t-3+k} is the first L terms of the full convolution with the reversed taps."""
    x, w, b = _conv_case(2)
    u = oracle.causal_conv1d(x, w, b, silu=False)
    ref = np.stack([[np.convolve(x[i, d], w[d][::-1])[:x.shape[2]] + b[d] for d in range(x.shape[1])]
                    for i in range(x.shape[0])])
    np.testing.assert_allclose(u, ref, rtol=0, atol=1e-13)


def test_conv_is_causal_with_a_width_four_window():
    x, w, b = _conv_case(3)
    u0 = oracle.causal_conv1d(x, w, b)
    x2 = x.copy()
    x2[1, 2, 10] += 1.0
    u1 = oracle.causal_conv1d(x2, w, b)
    changed = np.argwhere(u1 != u0)
    assert {tuple(c) for c in changed} == {(1, 2, t) for t in range(10, 14)}


def test_conv_silu_values():
    """SiLU(0) = 0, SiLU(1) = 1/(1+e^-1) = 0.7310585786300049, SiLU(-1) = -0.2689414213699951."""
    x = np.array([[[0.0, 1.0, -1.0]]])
    w = np.array([[0.0, 0.0, 0.0, 1.0]])
    u = oracle.causal_conv1d(x, w, None, silu=True)
    np.testing.assert_allclose(u[0, 0], [0.0, 0.7310585786300049, -0.2689414213699951], rtol=0, atol=1e-15)


def test_conv_then_scan_composes_with_the_scan_oracle():
    """The fused path's reference is the scan of u = SiLU(conv(x)): with the identity tap and no bias
    it reduces to the scan of SiLU(x)."""
    r = np.random.default_rng(4)
    Bsz, Dch, L, N = 1, 3, 17, 4
    x = r.normal(size=(Bsz, Dch, L))
    w = np.zeros((Dch, 4))
    w[:, 3] = 1.0
    delta, A = r.normal(size=(Bsz, Dch, L)) - 2, -np.tile(np.arange(1.0, N + 1), (Dch, 1))
    B, C = r.normal(size=(Bsz, N, L)), r.normal(size=(Bsz, N, L))
    u = oracle.causal_conv1d(x, w, None)
    y1, h1 = oracle.selective_scan(u, delta, A, B, C)
    y2, h2 = oracle.selective_scan(x / (1 + np.exp(-x)), delta, A, B, C)
    np.testing.assert_allclose(y1, y2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(h1, h2, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- backward (chain rule of the forward scan)

def _bwd_case(seed, Bsz=2, Dch=2, N=3, L=6):
    r = np.random.default_rng(seed)
    return dict(u=r.normal(size=(Bsz, Dch, L)), delta=r.normal(size=(Bsz, Dch, L)) - 1.0,
                A=-r.uniform(0.5, 2.0, size=(Dch, N)), B=r.normal(size=(Bsz, N, L)), C=r.normal(size=(Bsz, N, L)),
                D=r.normal(size=Dch), z=r.normal(size=(Bsz, Dch, L)), delta_bias=0.1 * r.normal(size=Dch),
                dy=r.normal(size=(Bsz, Dch, L)))


@pytest.mark.parametrize("gate,softplus", [(True, True), (False, True), (True, False)])
def test_backward_matches_central_differences(gate, softplus):
    """Every gradient of sum(dy * y) against central differences of the forward oracle (step 1e-6)."""
    c = _bwd_case(7)
    if not softplus:
        c["delta"] = np.abs(c["delta"]) + 0.1          # Delta = Delta_raw + bias stays positive
    z = c["z"] if gate else None
    g = oracle.selective_scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], c["dy"], c["D"], z,
                                  c["delta_bias"], softplus_flag=softplus)

    def loss(**kw):
        a = {k: c[k] for k in ("u", "delta", "A", "B", "C", "D", "delta_bias")}
        a["z"] = z
        a.update(kw)
        y, _ = oracle.selective_scan(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["delta_bias"],
                                     softplus_flag=softplus)
        return float((c["dy"] * y).sum())

    eps = 1e-6
    names = [("u", "du"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC"), ("D", "dD"),
             ("delta_bias", "ddelta_bias")] + ([("z", "dz")] if gate else [])
    for name, key in names:
        arr = c[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            fd[idx] = (loss(**{name: p}) - loss(**{name: m})) / (2 * eps)
        np.testing.assert_allclose(g[key], fd, rtol=1e-6, atol=1e-8, err_msg=key)
    if not gate:
        assert g["dz"] is None


def test_backward_running_sum_closed_form():
    """A = 0, Delta = 1 (softplus off), B = C = 1, D = 0, no gate: h_t[n] = sum_{s<=t} u_s and
    y_t = N sum_{s<=t} u_s.  With dy = 1 at the last step only: du_s = N for every s, dB_{s,n} = u_s
    (dh = 1 at every step) and dC is h_{L-1} = sum u at the last step, 0 elsewhere."""
    Bsz, Dch, N, L = 1, 1, 4, 7
    u = np.arange(1.0, L + 1).reshape(1, 1, L)
    dy = np.zeros((1, 1, L))
    dy[0, 0, -1] = 1.0
    g = oracle.selective_scan_bwd(u, np.ones((1, 1, L)), np.zeros((1, N)), np.ones((1, N, L)), np.ones((1, N, L)), dy,
                                  np.zeros(1), None, np.zeros(1), softplus_flag=False)
    np.testing.assert_array_equal(g["du"], np.full((1, 1, L), float(N)))
    np.testing.assert_array_equal(g["dB"], np.broadcast_to(u[:, :1, :], (1, N, L)))   # dh = 1 at every step
    expect_dC = np.zeros((1, N, L))
    expect_dC[0, :, -1] = u.sum()                                                    # h_{L-1} = sum u
    np.testing.assert_array_equal(g["dC"], expect_dC)
