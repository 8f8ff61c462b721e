"""Seeded synthetic inputs for the selective scan and the decode step.

This module only draws random numbers and rounds them to the storage type; it
holds none of the scan's arithmetic.  Both the CUDA path and the float64
oracle read the arrays it returns, so the two sides see bit-identical inputs.

Recipe (the same for every workload):
  * every tensor row has its own stream: numpy PCG64 seeded with
    SeedSequence([seed, tag, *row]); a row is (b, d) for u / Delta_raw / z,
    (b, n) for B / C, and one stream each for dt, D, the DNA embedding table
    and the DNA symbol sequence.  Any row can therefore be regenerated alone.
  * u, z, B, C ~ N(0, 1); Delta_raw ~ N(0, 0.5) (standard deviation 0.5);
    D ~ N(0, 1) in fp32; A[d, n] = -(n + 1) in fp32 (n counted from 0).
  * dt[d] = exp(U[ln 1e-3, ln 1e-1]); delta_bias[d] = softplus^-1(dt[d]) =
    dt + log(-expm1(-dt)), evaluated in float64 and stored in fp32.
  * draws are made in float32 and, for bf16 workloads, rounded once to bf16
    with round-to-nearest-even.
  * DNA-shaped u: a table E in {+1, -1}^(4 x Dch) and i.i.d. uniform symbols
    s_t in {0, 1, 2, 3}; u[0, d, t] = E[s_t, d].
  * decode: the fp32 state ~ N(0, 0.1) (standard deviation 0.1); each step k
    draws its own u, Delta_raw, z [Bsz, Dch] and B, C [Bsz, N] with k in the
    stream key.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

TAG_DT, TAG_D, TAG_U, TAG_DELTA, TAG_Z, TAG_B, TAG_C, TAG_STATE, TAG_EMBED, TAG_SYMBOLS, TAG_CONV_W, TAG_CONV_B = range(12)

# Named workloads: (batch, d_inner, d_state, seq_len, io dtype, seed, u kind).
WORKLOADS = {
    # tiny scan, fp32 everywhere
    "tiny_b1_d64_n16_l256_f32": dict(batch=1, dim=64, dstate=16, seqlen=256, io="f32", seed=0, u_kind="normal"),
    # one Mamba-130M-shaped layer
    "mamba130m_b8_d1536_n16_l2048_bf16": dict(batch=8, dim=1536, dstate=16, seqlen=2048, io="bf16", seed=1,
                                              u_kind="normal"),
    # one Mamba-2.8B-shaped layer, and its d_state 64 variant
    "mamba2p8b_b4_d5120_n16_l4096_bf16": dict(batch=4, dim=5120, dstate=16, seqlen=4096, io="bf16", seed=2,
                                              u_kind="normal"),
    "mamba2p8b_b4_d5120_n64_l4096_bf16": dict(batch=4, dim=5120, dstate=64, seqlen=4096, io="bf16", seed=2,
                                              u_kind="normal"),
    # one DNA-length sequence
    "dna_b1_d1536_n16_l1048576_bf16": dict(batch=1, dim=1536, dstate=16, seqlen=1 << 20, io="bf16", seed=3,
                                           u_kind="dna"),
}
DECODE_WORKLOAD = dict(name="decode_b256_d5120_n16_bf16", batch=256, dim=5120, dstate=16, io="bf16", seed=4,
                       steps=1000)

_POOL_WORKERS = max(1, min(16, os.cpu_count() or 1))


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value in a synthetic input")
    b = x.view(np.uint32)
    r = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _store(x32: np.ndarray, io: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if io == "bf16" else np.ascontiguousarray(x32, dtype=np.float32)


def to_f64(stored: np.ndarray, io: str) -> np.ndarray:
    """Exact float64 widening of a stored (bf16 bits or fp32) array."""
    return (bf16_bits_to_f32(stored) if io == "bf16" else stored).astype(np.float64)


def _normal_rows(seed: int, tag: int, rows, n: int, std: float, io: str, out: np.ndarray) -> None:
    """Fill out[i, :] with row rows[i]'s stream (float32 draws, then storage rounding)."""
    def work(lo, hi):
        buf = np.empty((hi - lo, n), dtype=np.float32)
        for i in range(lo, hi):
            r = rows[i]
            key = (seed, tag) + (tuple(r) if isinstance(r, tuple) else (r,))
            _rng(*key).standard_normal(n, dtype=np.float32, out=buf[i - lo])
        if std != 1.0:
            buf *= np.float32(std)
        out[lo:hi] = _store(buf, io)
    nrows = len(rows)
    if nrows * n < (1 << 20) or _POOL_WORKERS == 1:
        work(0, nrows)
        return
    step = max(1, min(max(1, (1 << 22) // n), (nrows + 4 * _POOL_WORKERS - 1) // (4 * _POOL_WORKERS)))
    with _cf.ThreadPoolExecutor(_POOL_WORKERS) as ex:
        list(ex.map(lambda lo: work(lo, min(nrows, lo + step)), range(0, nrows, step)))


def channel_params(dim: int, dstate: int, seed: int):
    """A [D, N], D [D], delta_bias [D] (all fp32) and dt [D] (float64)."""
    dt = np.exp(_rng(seed, TAG_DT).uniform(np.log(1e-3), np.log(1e-1), size=dim))
    bias = (dt + np.log(-np.expm1(-dt))).astype(np.float32)
    D = _rng(seed, TAG_D).standard_normal(dim, dtype=np.float32)
    A = np.broadcast_to(-(np.arange(dstate, dtype=np.float32) + 1.0), (dim, dstate)).copy()
    return A, D, bias, dt


def conv_params(dim: int, seed: int, width: int = 4):
    """Depthwise causal conv taps [D, width] ~ N(0, 0.5) and bias [D] ~ N(0, 0.1), fp32.

    The pages give no initialisation for the convolution branch; these keep SiLU(conv(x)) of
    unit-scale x at the scale of the scan's u."""
    w = (0.5 * _rng(seed, TAG_CONV_W).standard_normal((dim, width))).astype(np.float32)
    b = (0.1 * _rng(seed, TAG_CONV_B).standard_normal(dim)).astype(np.float32)
    return w, b


@dataclasses.dataclass
class ScanInputs:
    io: str                 # "f32" or "bf16": storage type of u, delta, z, B, C (and y)
    u: np.ndarray           # [Bsz, Dch, L]   uint16 bf16 bits or float32
    delta: np.ndarray       # [Bsz, Dch, L]   Delta_raw
    z: np.ndarray | None    # [Bsz, Dch, L]
    B: np.ndarray           # [Bsz, N, L]
    C: np.ndarray           # [Bsz, N, L]
    A: np.ndarray           # [Dch, N] float32
    D: np.ndarray           # [Dch] float32
    delta_bias: np.ndarray  # [Dch] float32

    @property
    def shape(self):
        Bsz, Dch, L = self.u.shape
        return Bsz, Dch, L, self.A.shape[1]

    def f64(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        if a is None:
            return None
        if name in ("A", "D", "delta_bias"):
            return a.astype(np.float64)
        return to_f64(a, self.io)


def make_scan_inputs(batch: int, dim: int, dstate: int, seqlen: int, io: str = "bf16", seed: int = 0,
                     u_kind: str = "normal", with_z: bool = True) -> ScanInputs:
    if io not in ("f32", "bf16"):
        raise ValueError(io)
    sdt = np.uint16 if io == "bf16" else np.float32
    A, D, bias, _ = channel_params(dim, dstate, seed)
    ch_rows = [(b, d) for b in range(batch) for d in range(dim)]
    st_rows = [(b, n) for b in range(batch) for n in range(dstate)]

    u = np.empty((batch * dim, seqlen), dtype=sdt)
    if u_kind == "normal":
        _normal_rows(seed, TAG_U, ch_rows, seqlen, 1.0, io, u)
    elif u_kind == "dna":
        if batch != 1:
            raise ValueError("the DNA-shaped input is a single sequence")
        E = np.where(_rng(seed, TAG_EMBED).integers(0, 2, size=(4, dim)) == 1, 1.0, -1.0).astype(np.float32)
        sym = _rng(seed, TAG_SYMBOLS).integers(0, 4, size=seqlen)
        for d in range(dim):
            u[d] = _store(E[sym, d], io)
    else:
        raise ValueError(u_kind)
    delta = np.empty((batch * dim, seqlen), dtype=sdt)
    _normal_rows(seed, TAG_DELTA, ch_rows, seqlen, 0.5, io, delta)
    z = None
    if with_z:
        z = np.empty((batch * dim, seqlen), dtype=sdt)
        _normal_rows(seed, TAG_Z, ch_rows, seqlen, 1.0, io, z)
    Bm = np.empty((batch * dstate, seqlen), dtype=sdt)
    _normal_rows(seed, TAG_B, st_rows, seqlen, 1.0, io, Bm)
    Cm = np.empty((batch * dstate, seqlen), dtype=sdt)
    _normal_rows(seed, TAG_C, st_rows, seqlen, 1.0, io, Cm)
    sh = (batch, dim, seqlen)
    return ScanInputs(io=io, u=u.reshape(sh), delta=delta.reshape(sh), z=None if z is None else z.reshape(sh),
                      B=Bm.reshape(batch, dstate, seqlen), C=Cm.reshape(batch, dstate, seqlen), A=A, D=D,
                      delta_bias=bias)


def make_workload(name: str, **over) -> ScanInputs:
    cfg = dict(WORKLOADS[name])
    cfg.update(over)
    return make_scan_inputs(cfg["batch"], cfg["dim"], cfg["dstate"], cfg["seqlen"], cfg["io"], cfg["seed"],
                            cfg.get("u_kind", "normal"), cfg.get("with_z", True))


@dataclasses.dataclass
class DecodeStep:
    io: str
    u: np.ndarray       # [Bsz, Dch]
    delta: np.ndarray   # [Bsz, Dch]
    z: np.ndarray       # [Bsz, Dch]
    B: np.ndarray       # [Bsz, N]
    C: np.ndarray       # [Bsz, N]

    def f64(self, name):
        return to_f64(getattr(self, name), self.io)


def make_decode_state(batch: int, dim: int, dstate: int, seed: int) -> np.ndarray:
    st = np.empty((batch, dim * dstate), dtype=np.float32)
    _normal_rows(seed, TAG_STATE, list(range(batch)), dim * dstate, 0.1, "f32", st)
    return st.reshape(batch, dim, dstate)


def make_decode_step(batch: int, dim: int, dstate: int, seed: int, step: int, io: str = "bf16") -> DecodeStep:
    sdt = np.uint16 if io == "bf16" else np.float32
    out = {}
    for name, tag, n, std in (("u", TAG_U, dim, 1.0), ("delta", TAG_DELTA, dim, 0.5), ("z", TAG_Z, dim, 1.0),
                              ("B", TAG_B, dstate, 1.0), ("C", TAG_C, dstate, 1.0)):
        a = np.empty((batch, n), dtype=sdt)
        _normal_rows(seed, tag, [(step, b) for b in range(batch)], n, std, io, a)
        out[name] = a
    return DecodeStep(io=io, **out)
