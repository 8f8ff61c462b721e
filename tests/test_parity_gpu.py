"""Parity of the CUDA selective scan (through the C ABI) with the float64 oracle.

Small and mid sizes, element by element on every output (the full-size
workloads are in test_full_size_gpu.py).  Every call is followed by a check
that no bounded device-side wait of the kernels gave up.
"""
import numpy as np
import pytest

import oracle
import selective_state_space_148_b300 as m
from selective_state_space_148_b300 import inputs
from helpers import TOL_STATE, TOL_Y, assert_close, dev_inputs, f32_dev, to_host_f64

pytestmark = pytest.mark.gpu


def run_gpu(x, softplus=True, with_z=True, with_D=True, with_bias=True, h0=None, chunk_len=0, flags=0,
            want_last=True):
    import torch
    t = dev_inputs(x)
    y = torch.empty_like(t["u"])
    last = torch.empty((x.shape[0], x.shape[1], x.shape[3]), dtype=torch.float32, device="cuda") if want_last else None
    h0d = f32_dev(h0)
    if h0 is None and chunk_len == 0 and flags == 0:
        m.mamba_selective_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"] if with_D else None,
                                   t["z"] if with_z else None, t["delta_bias"] if with_bias else None, softplus, y,
                                   last)
    else:
        m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"] if with_D else None,
                                      t["z"] if with_z else None, t["delta_bias"] if with_bias else None, softplus,
                                      y, last, h0=h0d, flags=flags, chunk_len=chunk_len)
    torch.cuda.synchronize()
    assert m.mamba_device_error() == 0
    return to_host_f64(y), (last.cpu().numpy().astype(np.float64) if want_last else None)


def run_oracle(x, softplus=True, with_z=True, with_D=True, with_bias=True, h0=None, disc=0, reverse=False):
    return oracle.selective_scan(x.f64("u"), x.f64("delta"), x.f64("A"), x.f64("B"), x.f64("C"),
                                 x.f64("D") if with_D else None, x.f64("z") if with_z else None,
                                 x.f64("delta_bias") if with_bias else None, softplus_flag=softplus, h0=h0,
                                 disc=disc, reverse=reverse)


def check(x, tag, **kw):
    okw = {k: v for k, v in kw.items() if k in ("softplus", "with_z", "with_D", "with_bias", "h0")}
    yg, hg = run_gpu(x, **kw)
    yr, hr = run_oracle(x, **okw)
    ey = assert_close(yg, yr, TOL_Y[x.io], f"{tag} y")
    eh = assert_close(hg, hr, TOL_STATE, f"{tag} last_state")
    return ey, eh


# ----------------------------------------------------------------------------- workloads, whole outputs

def test_tiny_fp32_workload():
    x = inputs.make_workload("tiny_b1_d64_n16_l256_f32")
    ey, eh = check(x, "tiny")
    print(f"tiny fp32: max y err ratio {ey:.3g}, state {eh:.3g}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 7, 8, 9, 31, 33, 63, 65, 257, 1000])
def test_lengths(io, L):
    x = inputs.make_scan_inputs(2, 37, 16, L, io=io, seed=7)
    check(x, f"L={L} {io}")


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 12, 16, 17, 24, 32, 33, 48, 64])
def test_state_sizes(N):
    x = inputs.make_scan_inputs(2, 19, N, 130, io="bf16", seed=8)
    check(x, f"N={N}")
    x = inputs.make_scan_inputs(1, 9, N, 77, io="f32", seed=9)
    check(x, f"N={N} f32")


@pytest.mark.parametrize("variant", ["no_softplus", "no_z", "no_D", "no_bias", "nothing_optional"])
def test_optional_inputs(variant):
    x = inputs.make_scan_inputs(2, 40, 16, 200, io="bf16", seed=10)
    kw = dict(softplus=variant != "no_softplus", with_z=variant not in ("no_z", "nothing_optional"),
              with_D=variant not in ("no_D", "nothing_optional"), with_bias=variant not in ("no_bias", "nothing_optional"))
    if variant == "no_softplus":
        # Delta = Delta_raw + bias must stay positive for a decaying state: shift the raw values up
        x.delta_bias = (x.delta_bias * 0 + 2.0).astype(np.float32)
    check(x, variant, **kw)


def test_no_last_state():
    x = inputs.make_scan_inputs(2, 20, 16, 100, io="bf16", seed=11)
    yg, _ = run_gpu(x, want_last=False)
    yr, _ = run_oracle(x)
    assert_close(yg, yr, TOL_Y["bf16"], "y without last_state")


def test_mid_bf16_several_tiles():
    x = inputs.make_scan_inputs(3, 100, 16, 1000, io="bf16", seed=12)
    ey, eh = check(x, "mid bf16")
    print(f"mid bf16: y err ratio {ey:.3g}, state {eh:.3g}")


def test_initial_state_direct():
    x = inputs.make_scan_inputs(2, 33, 16, 150, io="f32", seed=13)
    h0 = np.random.default_rng(1).normal(0, 0.5, (2, 33, 16)).astype(np.float32).astype(np.float64)
    check(x, "h0 direct", h0=h0, chunk_len=-1)


# ----------------------------------------------------------------------------- chunked scan

@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("chunk_len", [32, 64, 96, 160, 1024])
def test_chunked_forced(io, chunk_len):
    x = inputs.make_scan_inputs(2, 24, 16, 999, io=io, seed=14)
    check(x, f"chunked {chunk_len} {io}", chunk_len=chunk_len)


@pytest.mark.parametrize("N", [4, 16, 33, 64])
def test_chunked_state_sizes(N):
    x = inputs.make_scan_inputs(1, 20, N, 700, io="bf16", seed=15)
    check(x, f"chunked N={N}", chunk_len=64)


def test_chunked_with_initial_state():
    x = inputs.make_scan_inputs(2, 24, 16, 500, io="f32", seed=16)
    h0 = np.random.default_rng(2).normal(0, 0.5, (2, 24, 16)).astype(np.float32).astype(np.float64)
    check(x, "chunked h0", h0=h0, chunk_len=64)


def test_chunked_equals_direct_bits_close():
    """Forced chunked scans agree with the direct scan for several chunk counts."""
    x = inputs.make_scan_inputs(1, 64, 16, 4096, io="bf16", seed=17)
    y0, h0 = run_gpu(x, chunk_len=-1)
    for cl in (32, 128, 1000, 4096):
        y1, h1 = run_gpu(x, chunk_len=cl)
        assert_close(y1, y0, TOL_Y["bf16"], f"chunk {cl} vs direct y")
        assert_close(h1, h0, TOL_STATE, f"chunk {cl} vs direct state")


def test_automatic_choice_uses_chunks_for_long_thin_problems():
    # one channel block and a long sequence: the automatic plan cuts it into chunks
    assert m.mamba_scan_workspace_size(1, 16, 1 << 16, 16, 0, m.MAMBA_BF16) > 0
    # a wide problem stays direct
    assert m.mamba_scan_workspace_size(8, 1536, 2048, 16, 0, m.MAMBA_BF16) == 0
    x = inputs.make_scan_inputs(1, 16, 16, 1 << 14, io="bf16", seed=18)
    check(x, "auto chunked")


# ----------------------------------------------------------------------------- memory safety and errors

def test_guard_regions_untouched():
    """Outputs written through views inside larger buffers: the guard elements keep their sentinel."""
    import torch
    x = inputs.make_scan_inputs(2, 21, 16, 77, io="bf16", seed=19)
    t = dev_inputs(x)
    G = 64
    ybuf = torch.full((2 * 21 * 77 + 2 * G,), -12345.0, dtype=torch.float32, device="cuda").to(torch.bfloat16)
    sentinel = float(ybuf[0].float())          # -12345 rounded to bf16
    hbuf = torch.full((2 * 21 * 16 + 2 * G,), -777.0, dtype=torch.float32, device="cuda")
    y = ybuf[G:G + 2 * 21 * 77].view(2, 21, 77)
    h = hbuf[G:G + 2 * 21 * 16].view(2, 21, 16)
    m.mamba_selective_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], 1, y, h)
    torch.cuda.synchronize()
    assert torch.all(ybuf[:G].float() == sentinel) and torch.all(ybuf[-G:].float() == sentinel)
    assert torch.all(hbuf[:G] == -777.0) and torch.all(hbuf[-G:] == -777.0)
    yr, hr = run_oracle(x)
    assert_close(to_host_f64(y), yr, TOL_Y["bf16"], "guarded y")
    assert_close(h.cpu().numpy(), hr, TOL_STATE, "guarded state")


def test_misaligned_pointers_take_scalar_path():
    import torch
    x = inputs.make_scan_inputs(2, 18, 16, 64, io="bf16", seed=20)
    t = dev_inputs(x)
    off = {}
    for k in ("u", "delta", "z", "B", "C"):   # copy into a buffer shifted by one element
        buf = torch.empty(t[k].numel() + 1, dtype=t[k].dtype, device="cuda")
        buf[1:].copy_(t[k].reshape(-1))
        off[k] = buf[1:].view(t[k].shape)
    y = torch.empty(t["u"].numel() + 1, dtype=torch.bfloat16, device="cuda")[1:].view(t["u"].shape)
    h = torch.empty((2, 18, 16), dtype=torch.float32, device="cuda")
    m.mamba_selective_scan_fwd(off["u"], off["delta"], t["A"], off["B"], off["C"], t["D"], off["z"],
                               t["delta_bias"], 1, y, h)
    torch.cuda.synchronize()
    yr, hr = run_oracle(x)
    assert_close(to_host_f64(y), yr, TOL_Y["bf16"], "misaligned y")
    assert_close(h.cpu().numpy(), hr, TOL_STATE, "misaligned state")


def test_caller_workspace_and_errors(monkeypatch):
    import torch
    x = inputs.make_scan_inputs(1, 16, 16, 2048, io="bf16", seed=21)
    t = dev_inputs(x)
    need = m.mamba_scan_workspace_size(1, 16, 2048, 16, 128, m.MAMBA_BF16)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(t["u"])
    h = torch.empty((1, 16, 16), dtype=torch.float32, device="cuda")
    m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], 1, y,
                                  h, chunk_len=128, workspace=ws, workspace_bytes=need)
    torch.cuda.synchronize()
    yr, hr = run_oracle(x)
    assert_close(to_host_f64(y), yr, TOL_Y["bf16"], "caller workspace y")
    with pytest.raises(m.MambaError) as ei:
        m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                                      1, y, h, chunk_len=128, workspace=ws, workspace_bytes=need - 4)
    assert ei.value.status == -9
    monkeypatch.setenv("MAMBA_FAULT_INJECT", "alloc")
    with pytest.raises(m.MambaError) as ei:
        m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                                      1, y, h, chunk_len=128)
    assert ei.value.status == -5
    # the direct path allocates nothing and is unaffected
    m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], 1, y,
                                  h, chunk_len=-1)
    torch.cuda.synchronize()
    assert_close(to_host_f64(y), yr, TOL_Y["bf16"], "direct y under injected allocation failure")


# ----------------------------------------------------------------------------- flags: exact ZOH, reverse scan

FLAG_CASES = {  # name -> (flags, oracle disc, oracle reverse)
    "zoh": (0x1, 1, False),
    "reverse": (0x2, 0, True),
    "zoh_reverse": (0x3, 1, True),
}


@pytest.mark.parametrize("case", sorted(FLAG_CASES))
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4, 16, 33, 64])
def test_flags_direct(case, io, N):
    flags, disc, rev = FLAG_CASES[case]
    x = inputs.make_scan_inputs(2, 21, N, 300, io=io, seed=20 + N)
    h0 = np.random.default_rng(N).normal(0, 0.3, (2, 21, N)).astype(np.float32)
    for h in (None, h0):
        yg, hg = run_gpu(x, h0=h, flags=flags, chunk_len=-1)
        yr, hr = run_oracle(x, h0=None if h is None else h.astype(np.float64), disc=disc, reverse=rev)
        assert_close(yg, yr, TOL_Y[io], f"{case} N={N} {io} y")
        assert_close(hg, hr, TOL_STATE, f"{case} N={N} {io} last_state")


@pytest.mark.parametrize("case", sorted(FLAG_CASES))
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_flags_chunked(case, io):
    flags, disc, rev = FLAG_CASES[case]
    x = inputs.make_scan_inputs(1, 13, 16, 1000, io=io, seed=31)
    h0 = np.random.default_rng(5).normal(0, 0.3, (1, 13, 16)).astype(np.float32)
    yg, hg = run_gpu(x, h0=h0, flags=flags, chunk_len=128)
    yr, hr = run_oracle(x, h0=h0.astype(np.float64), disc=disc, reverse=rev)
    assert_close(yg, yr, TOL_Y[io], f"chunked {case} {io} y")
    assert_close(hg, hr, TOL_STATE, f"chunked {case} {io} last_state")


def test_zoh_with_a_zero_state():
    """A state with A = 0 takes the limit Delta * B of the ZOH weight."""
    x = inputs.make_scan_inputs(1, 9, 16, 200, io="f32", seed=33)
    x.A = x.A.copy()
    x.A[:, 3] = 0.0
    x.A[4, :] = 0.0
    yg, hg = run_gpu(x, flags=0x1, chunk_len=-1)
    yr, hr = run_oracle(x, disc=1)
    assert_close(yg, yr, TOL_Y["f32"], "zoh A=0 y")
    assert_close(hg, hr, TOL_STATE, "zoh A=0 last_state")


def test_flags_unaligned_and_ragged():
    """Flagged calls take scalar loads everywhere: odd L and offset views."""
    import torch
    x = inputs.make_scan_inputs(2, 11, 16, 97, io="bf16", seed=34)
    t = dev_inputs(x)
    big = {k: torch.empty(v.numel() + 1, dtype=v.dtype, device="cuda") for k, v in t.items() if k in ("u", "delta", "z")}
    for k, v in big.items():
        v[1:].copy_(t[k].reshape(-1))
        t[k] = v[1:].view(t[k].shape)
    y = torch.empty_like(t["u"])
    last = torch.empty((2, 11, 16), dtype=torch.float32, device="cuda")
    m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], 1,
                                  y, last, flags=0x3, chunk_len=-1)
    torch.cuda.synchronize()
    yr, hr = run_oracle(x, disc=1, reverse=True)
    assert_close(to_host_f64(y), yr, TOL_Y["bf16"], "flags unaligned y")
    assert_close(last.cpu().numpy().astype(np.float64), hr, TOL_STATE, "flags unaligned last_state")


# ----------------------------------------------------------------------------- tensor-memory kernel, N up to 64

@pytest.mark.parametrize("N", [9, 12, 16, 17, 20, 32, 33, 40, 64])
@pytest.mark.parametrize("L", [72, 256])
def test_aligned_state_sizes(N, L):
    """16-byte aligned rows (the tensor-memory kernel for bf16, 8 < N <= 64): direct, no gate, and chunked with h0."""
    x = inputs.make_scan_inputs(2, 45, N, L, io="bf16", seed=50 + N)
    check(x, f"aligned N={N} L={L}")
    check(x, f"aligned N={N} L={L} no z", with_z=False)
    h0 = np.random.default_rng(N).normal(0, 0.3, (2, 45, N)).astype(np.float32)
    yg, hg = run_gpu(x, h0=h0, chunk_len=64)
    yr, hr = run_oracle(x, h0=h0.astype(np.float64))
    assert_close(yg, yr, TOL_Y["bf16"], f"aligned chunked N={N} L={L} y")
    assert_close(hg, hr, TOL_STATE, f"aligned chunked N={N} L={L} last_state")


# ----------------------------------------------------------------------------- bounded waits: the abort path

def test_bounded_wait_gives_up_and_reports_timeout(monkeypatch):
    """With its pipeline waits capped at zero polls (the MAMBA_TEST_WAIT_POLLS hook), the tensor-memory
    kernel gives up at its first wait for an input tile, takes the abort path (it still drains its own
    copies and MMAs before freeing tensor memory) and the device error word reports the timeout; the
    next call without the hook runs normally and matches the oracle."""
    import torch
    x = inputs.make_scan_inputs(2, 45, 16, 256, io="bf16", seed=95)   # aligned bf16, N = 16: tensor-memory kernel
    assert m.mamba_device_error() == 0
    monkeypatch.setenv("MAMBA_TEST_WAIT_POLLS", "0")
    t = dev_inputs(x)
    y = torch.empty_like(t["u"])
    last = torch.empty((2, 45, 16), dtype=torch.float32, device="cuda")
    for chunk_len in (-1, 64):                 # the direct scan, then both kernels of the chunked scan
        m.mamba_selective_scan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                                      1, y, last, chunk_len=chunk_len)
        torch.cuda.synchronize()
        assert m.mamba_device_error() == m.STATUS_CODE["MAMBA_ERR_DEVICE_TIMEOUT"]
        assert m.mamba_device_error() == 0     # read and cleared
    monkeypatch.delenv("MAMBA_TEST_WAIT_POLLS")
    ey, eh = check(x, "after an aborted call")
    print(f"after the aborted calls: y err ratio {ey:.3g}, state {eh:.3g}")


# ----------------------------------------------------------------------------- flags on the tensor-memory kernel

@pytest.mark.parametrize("case", sorted(FLAG_CASES))
@pytest.mark.parametrize("io,N", [("bf16", 12), ("bf16", 16), ("bf16", 32), ("bf16", 64), ("f32", 16)])
@pytest.mark.parametrize("L", [256, 1000])
def test_flags_tensor_memory_path(case, io, N, L):
    """16-byte aligned rows (L a multiple of 8): the flagged tensor-memory kernel, direct and chunked, with
    and without h0; L = 1000 ends in a partial 32-step tile."""
    flags, disc, rev = FLAG_CASES[case]
    x = inputs.make_scan_inputs(2, 40, N, L, io=io, seed=100 + N + L)
    h0 = np.random.default_rng(N + L).normal(0, 0.3, (2, 40, N)).astype(np.float32)
    for h, chunk_len in ((None, -1), (h0, -1), (h0, 128)):
        yg, hg = run_gpu(x, h0=h, flags=flags, chunk_len=chunk_len)
        yr, hr = run_oracle(x, h0=None if h is None else h.astype(np.float64), disc=disc, reverse=rev)
        assert_close(yg, yr, TOL_Y[io], f"{case} N={N} L={L} {io} chunk={chunk_len} y")
        assert_close(hg, hr, TOL_STATE, f"{case} N={N} L={L} {io} chunk={chunk_len} last_state")


# ----------------------------------------------------------------------------- decay-truncated chunked scan

@pytest.mark.parametrize("regime", ["fast_decay", "slow_decay", "no_softplus", "growing_state"])
@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("scheme", ["truncated", "two-pass"])
def test_chunked_scan_correction_regimes(regime, io, scheme, monkeypatch):
    """The decay-truncated chunked scan (the default) corrects each chunk's y for its entering state and
    stops where that contribution has decayed below fp32 resolution: a stop after a few tiles (dt near
    1), no stop within a 1024-step chunk (dt near 1e-3, the smallest step of the workloads), and the
    cases where the decay is not guaranteed monotone (softplus off; a positive A) and the correction must
    run to the end of every chunk.  The two-pass scan (MAMBA_CHUNKED_SCAN=two-pass) on the same inputs.
    With and without h0."""
    if scheme == "two-pass":
        monkeypatch.setenv("MAMBA_CHUNKED_SCAN", "two-pass")
    else:
        monkeypatch.delenv("MAMBA_CHUNKED_SCAN", raising=False)
    x = inputs.make_scan_inputs(1, 40, 16, 6144, io=io, seed=120)
    softplus = regime != "no_softplus"
    if regime == "fast_decay":
        x.delta_bias = np.full(40, 1.0, dtype=np.float32)        # dt = softplus(1 + N(0, 0.5)) ~ 1.3
    elif regime == "slow_decay":
        x.delta_bias = np.full(40, -6.9, dtype=np.float32)       # dt ~ 1e-3
    elif regime == "no_softplus":
        x.delta_bias = np.full(40, 2.0, dtype=np.float32)        # Delta = raw + 2 > 0 in practice
    else:
        x.A = x.A.copy()
        x.A[:, 0] = 0.02                                         # one growing state per channel
    h0 = np.random.default_rng(3).normal(0, 0.3, (1, 40, 16)).astype(np.float32)
    for h in (None, h0):
        yg, hg = run_gpu(x, softplus=softplus, h0=h, chunk_len=1024)
        yr, hr = run_oracle(x, softplus=softplus, h0=None if h is None else h.astype(np.float64))
        assert_close(yg, yr, TOL_Y[io], f"{regime} {io} h0={h is not None} y")
        assert_close(hg, hr, TOL_STATE, f"{regime} {io} last_state")


# ----------------------------------------------------------------------------- lean form: 12..18 compute warps

@pytest.mark.parametrize("N", [12, 16, 32, 64])
@pytest.mark.parametrize("with_z", [True, False])
def test_lean_form_forced(N, with_z, monkeypatch):
    """MAMBA_TM_LEAN=1 puts every plain, aligned, direct bf16 scan on the lean form of the tensor-memory
    kernel (one step pair's TMEM columns at a time, 12..18 compute warps per CTA): ragged channel tiles,
    a ragged time tail, every element against the oracle."""
    monkeypatch.setenv("MAMBA_TM_LEAN", "1")
    x = inputs.make_scan_inputs(2, 300, N, 1000, io="bf16", seed=60 + N)
    check(x, f"lean N={N} z={with_z}", with_z=with_z)
    # softplus off: Delta = Delta_raw + bias must stay positive for a decaying state
    x.delta_bias = (x.delta_bias * 0 + 2.0).astype(np.float32)
    check(x, f"lean N={N} z={with_z} no softplus, no D", with_z=with_z, softplus=False, with_D=False)


@pytest.mark.parametrize("N,Dch", [(16, 21000), (32, 10600), (64, 5300)])
def test_lean_form_widest_cta_chosen_automatically(N, Dch):
    """Channel counts for which only the widest lean CTA (18 compute warps) fits the batch in one wave of
    148 SMs, where the regular 8..11-warp CTAs need two: the automatic choice takes the lean form at
    W = 18, 19 warps per CTA, 5 on some SM sub-partitions (ragged last CTA, ragged time tail; 16-byte
    aligned rows, so the tensor-memory kernel serves it)."""
    x = inputs.make_scan_inputs(1, Dch, N, 200, io="bf16", seed=70 + N)
    check(x, f"lean widest N={N} Dch={Dch}")
