"""float64 CPU oracle for the selective scan (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never does: it shares no code with this module.

The arithmetic lives in ``oracle.c`` (plain sequential loops in double
precision); this module only compiles it with gcc and marshals numpy arrays.
Every array is widened to float64 before the call, so the oracle sees exactly
the values (bf16- or fp32-rounded) that the GPU path reads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

DISC_SIMPLE = 0
DISC_ZOH = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.oracle_softplus.restype = ctypes.c_double
        lib.oracle_softplus.argtypes = [ctypes.c_double]
        lib.oracle_selective_scan.restype = None
        lib.oracle_selective_scan.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ci, ci, ci, dp, dp, dp,
                                              i64, i64, i64, i64]
        lib.oracle_state_update.restype = None
        lib.oracle_state_update.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, ci, ci, dp, i64, i64, i64]
        lib.oracle_selective_scan_bwd.restype = None
        lib.oracle_selective_scan_bwd.argtypes = [dp] * 8 + [ci] + [dp] * 10 + [i64] * 4
        lib.oracle_causal_conv1d.restype = None
        lib.oracle_causal_conv1d.argtypes = [dp, dp, dp, ci, dp, i64, i64, i64, i64]
        lib.oracle_num_threads.restype = ci
        lib.oracle_set_num_threads.argtypes = [ci]
        _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def softplus(x: float) -> float:
    return _load().oracle_softplus(float(x))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus_flag=True,
                   h0=None, disc=DISC_SIMPLE, reverse=False):
    """y[b,d,t], last_state[b,d,n] of the selective scan, in float64.

    Shapes: u, delta, z: [Bsz, Dch, L]; B, C: [Bsz, N, L]; A: [Dch, N];
    D, delta_bias: [Dch]; h0: [Bsz, Dch, N].
    """
    u, delta, A, B, C = (_f64(x) for x in (u, delta, A, B, C))
    D, z, delta_bias, h0 = (_f64(x) for x in (D, z, delta_bias, h0))
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    if N > 4096:
        raise ValueError("oracle supports N <= 4096")
    assert delta.shape == u.shape and B.shape == (Bsz, N, L) and C.shape == (Bsz, N, L)
    assert A.shape == (Dch, N)
    assert z is None or z.shape == u.shape
    assert D is None or D.shape == (Dch,)
    assert delta_bias is None or delta_bias.shape == (Dch,)
    assert h0 is None or h0.shape == (Bsz, Dch, N)
    y = np.empty((Bsz, Dch, L), dtype=np.float64)
    last = np.empty((Bsz, Dch, N), dtype=np.float64)
    _load().oracle_selective_scan(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                  _ptr(delta_bias), int(bool(softplus_flag)), int(disc), int(bool(reverse)),
                                  _ptr(h0), _ptr(y), _ptr(last), Bsz, Dch, L, N)
    return y, last


def state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus_flag=True,
                 disc=DISC_SIMPLE):
    """One recurrent step.  Returns (y[b,d], new_state[b,d,n]); the input is not modified.

    Shapes: state: [Bsz, Dch, N]; u, delta, z: [Bsz, Dch]; B, C: [Bsz, N];
    A: [Dch, N]; D, delta_bias: [Dch].
    """
    st = _f64(state).copy()
    u, delta, A, B, C = (_f64(x) for x in (u, delta, A, B, C))
    D, z, delta_bias = (_f64(x) for x in (D, z, delta_bias))
    Bsz, Dch, N = st.shape
    if N > 4096:
        raise ValueError("oracle supports N <= 4096")
    assert u.shape == (Bsz, Dch) and delta.shape == (Bsz, Dch)
    assert B.shape == (Bsz, N) and C.shape == (Bsz, N) and A.shape == (Dch, N)
    y = np.empty((Bsz, Dch), dtype=np.float64)
    _load().oracle_state_update(_ptr(st), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _ptr(z), _ptr(delta_bias), int(bool(softplus_flag)), int(disc), _ptr(y),
                                Bsz, Dch, N)
    return y, st


def state_update_inplace(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus_flag=True,
                         disc=DISC_SIMPLE):
    """The step of ``state_update`` applied to ``state`` itself (a C-contiguous float64 array, overwritten
    with the new state); returns y[b,d].  For long chains over large states, where copying the state at
    every step would dominate."""
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64 and state.flags.c_contiguous):
        raise TypeError("state must be a C-contiguous float64 array")
    u, delta, A, B, C = (_f64(x) for x in (u, delta, A, B, C))
    D, z, delta_bias = (_f64(x) for x in (D, z, delta_bias))
    Bsz, Dch, N = state.shape
    if N > 4096:
        raise ValueError("oracle supports N <= 4096")
    assert u.shape == (Bsz, Dch) and delta.shape == (Bsz, Dch)
    assert B.shape == (Bsz, N) and C.shape == (Bsz, N) and A.shape == (Dch, N)
    y = np.empty((Bsz, Dch), dtype=np.float64)
    _load().oracle_state_update(_ptr(state), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _ptr(z), _ptr(delta_bias), int(bool(softplus_flag)), int(disc), _ptr(y),
                                Bsz, Dch, N)
    return y


def causal_conv1d(x, w, bias=None, silu=True):
    """Depthwise causal convolution (width W = w.shape[1]) of x [Bsz, Dch, L], then SiLU.

    pre_t = bias_d + sum_k w[d, k] x_{t-(W-1)+k} with x_s = 0 for s < 0 (the pages' Conv1d with
    groups = d_inner, padding = W - 1, first L outputs), u = SiLU(pre) when silu is true.
    """
    x = _f64(x)
    Bsz, Dch, L = x.shape
    w = _f64(w)
    assert w.shape[0] == Dch
    b = None if bias is None else _f64(bias)
    u = np.empty_like(x)
    _load().oracle_causal_conv1d(_ptr(x), _ptr(w), _ptr(b), int(bool(silu)), _ptr(u), Bsz * Dch, Dch, L, w.shape[1])
    return u


def selective_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus_flag=True):
    """Gradients of sum(dy * y) for the forward scan (simple discretisation, forward time, zero h0).

    Returns a dict with du, ddelta [Bsz, Dch, L]; dA [Dch, N]; dB, dC [Bsz, N, L]; dD, ddelta_bias [Dch];
    dz [Bsz, Dch, L] (None without a gate)."""
    u, delta, A, B, C, dy = (_f64(a) for a in (u, delta, A, B, C, dy))
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    D = None if D is None else _f64(D)
    z = None if z is None else _f64(z)
    bias = None if delta_bias is None else _f64(delta_bias)
    out = dict(du=np.empty_like(u), ddelta=np.empty_like(u), dA=np.empty((Dch, N)), dB=np.empty((Bsz, N, L)),
               dC=np.empty((Bsz, N, L)), dD=np.empty(Dch), dz=np.empty_like(u) if z is not None else None,
               ddelta_bias=np.empty(Dch))
    work = np.empty((L + 1) * N + 2 * L + N)
    _load().oracle_selective_scan_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(bias),
                                      int(bool(softplus_flag)), _ptr(dy), _ptr(out["du"]), _ptr(out["ddelta"]),
                                      _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                                      _ptr(out["dz"]), _ptr(out["ddelta_bias"]), _ptr(work), Bsz, Dch, L, N)
    return out
