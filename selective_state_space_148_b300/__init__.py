"""B300-native (sm_103a) selective scan for Mamba: Python binding of libmambascan.so.

The binding marshals arguments only: every step of the scan runs in the CUDA
kernels behind the C ABI declared in ``include/mamba_scan.h``.  PyTorch is used
for device memory and streams.  There is no CPU fallback: if the library is
missing or no GPU is present the calls raise.

Functions with the C names take torch tensors that the caller allocated and
mirror the C signatures; ``selective_scan_fwd`` and ``state_update`` are small
conveniences that allocate the outputs.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmambascan.so")

MAMBA_F32 = 0
MAMBA_BF16 = 1
MAMBA_FLAG_ZOH = 0x1
MAMBA_FLAG_REVERSE = 0x2

STATUS = {
    0: "MAMBA_OK", -1: "MAMBA_ERR_NULL_ARG", -2: "MAMBA_ERR_BAD_SHAPE", -3: "MAMBA_ERR_UNSUPPORTED_N",
    -4: "MAMBA_ERR_BAD_DTYPE", -5: "MAMBA_ERR_ALLOC", -6: "MAMBA_ERR_LAUNCH", -7: "MAMBA_ERR_DEVICE_TIMEOUT",
    -8: "MAMBA_ERR_BAD_FLAGS", -9: "MAMBA_ERR_WORKSPACE", -10: "MAMBA_ERR_DEVICE", -11: "MAMBA_ERR_SCRATCH_LIMIT",
}
STATUS_CODE = {name: code for code, name in STATUS.items()}
NOALLOC_SCRATCH_BYTES = 16 << 20

_lib = None


class MambaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")


def lib() -> ctypes.CDLL:
    """Load libmambascan.so from the package directory (built by build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m selective_state_space_148_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, ci, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        L.mamba_selective_scan_fwd.restype = ci
        L.mamba_selective_scan_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, vp, vp, i64, i64, i64, i64, ci, vp]
        L.mamba_selective_scan_fwd_ex.restype = ci
        L.mamba_selective_scan_fwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, vp, vp, vp, i64, i64, i64, i64,
                                                  ci, ci, i64, vp, sz, vp]
        L.mamba_selective_scan_fwd_noalloc.restype = ci
        L.mamba_selective_scan_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, vp, vp, vp, i64, i64, i64,
                                                       i64, ci, i64, vp]
        L.mamba_scan_workspace_size.restype = sz
        L.mamba_scan_workspace_size.argtypes = [i64, i64, i64, i64, i64, ci]
        L.mamba_state_update.restype = ci
        L.mamba_state_update.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, vp, i64, i64, i64, ci, vp]
        L.mamba_status_string.restype = ctypes.c_char_p
        L.mamba_status_string.argtypes = [ci]
        L.mamba_device_error.restype = ci
        L.mamba_device_error.argtypes = []
        L.mamba_causal_conv1d_silu.restype = ci
        L.mamba_causal_conv1d_silu.argtypes = [vp, vp, vp, ci, vp, i64, i64, i64, ci, vp]
        L.mamba_selective_scan_fwd_conv.restype = ci
        L.mamba_selective_scan_fwd_conv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, vp, vp, i64, i64,
                                                    i64, i64, ci, vp]
        L.mamba_selective_scan_bwd.restype = ci
        L.mamba_selective_scan_bwd.argtypes = [vp] * 8 + [ci] + [vp] * 9 + [i64] * 4 + [ci, vp]
        L.mamba_scan_bwd_ckpt_size.restype = sz
        L.mamba_scan_bwd_ckpt_size.argtypes = [i64] * 4
        L.mamba_selective_scan_fwd_save.restype = ci
        L.mamba_selective_scan_fwd_save.argtypes = [vp] * 8 + [ci] + [vp] * 3 + [i64] * 4 + [ci, vp]
        L.mamba_selective_scan_bwd_from_ckpt.restype = ci
        L.mamba_selective_scan_bwd_from_ckpt.argtypes = [vp] * 8 + [ci] + [vp] * 10 + [i64] * 4 + [ci, vp]
        L.mamba_bench_ex2.restype = ci
        L.mamba_bench_ex2.argtypes = [vp, vp, i64, ci, ci, vp]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mamba_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return MAMBA_F32
    if t.dtype == torch.bfloat16:
        return MAMBA_BF16
    raise TypeError(f"unsupported storage dtype {t.dtype}; use float32 or bfloat16")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MambaError(status, where)


# ----------------------------------------------------------------------------- C-named calls

def mamba_selective_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, stream=None):
    """Selective scan (zero initial state).  Shapes: u, delta, z, y [Bsz, Dch, L]; B, C [Bsz, N, L];
    A [Dch, N] fp32; D, delta_bias [Dch] fp32; last_state [Bsz, Dch, N] fp32 or None."""
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    st = lib().mamba_selective_scan_fwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                        _ptr(delta_bias), int(bool(softplus_flag)), _ptr(y), _ptr(last_state),
                                        Bsz, Dch, L, N, _dtype_code(u), _stream(stream))
    _check(st, "mamba_selective_scan_fwd")


def mamba_selective_scan_fwd_ex(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, h0=None,
                                flags=0, chunk_len=0, workspace=None, workspace_bytes=0, stream=None):
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    st = lib().mamba_selective_scan_fwd_ex(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                           _ptr(delta_bias), int(bool(softplus_flag)), _ptr(y), _ptr(last_state),
                                           _ptr(h0), Bsz, Dch, L, N, _dtype_code(u), int(flags), int(chunk_len),
                                           _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "mamba_selective_scan_fwd_ex")


def mamba_selective_scan_fwd_noalloc(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, h0=None,
                                     chunk_len=256, stream=None):
    """Chunked scan whose scratch is the library's static device array (no device allocation)."""
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    st = lib().mamba_selective_scan_fwd_noalloc(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                                _ptr(delta_bias), int(bool(softplus_flag)), _ptr(y), _ptr(last_state),
                                                _ptr(h0), Bsz, Dch, L, N, _dtype_code(u), int(chunk_len),
                                                _stream(stream))
    _check(st, "mamba_selective_scan_fwd_noalloc")


def mamba_causal_conv1d_silu(x, conv_w, conv_bias, silu_flag, u, stream=None):
    """u = SiLU(conv_bias + depthwise causal width-4 convolution of x).  x, u [Bsz, Dch, L];
    conv_w [Dch, 4] fp32; conv_bias [Dch] fp32 or None."""
    Bsz, Dch, L = x.shape
    st = lib().mamba_causal_conv1d_silu(_ptr(x), _ptr(conv_w), _ptr(conv_bias), int(bool(silu_flag)), _ptr(u),
                                        Bsz, Dch, L, _dtype_code(x), _stream(stream))
    _check(st, "mamba_causal_conv1d_silu")


def mamba_selective_scan_fwd_conv(x, conv_w, conv_bias, delta, A, B, C, D, z, delta_bias, softplus_flag, y,
                                  last_state, stream=None):
    """Selective scan of u = SiLU(causal conv(x)) (the convolution branch fused into the scan)."""
    Bsz, Dch, L = x.shape
    N = A.shape[1]
    st = lib().mamba_selective_scan_fwd_conv(_ptr(x), _ptr(conv_w), _ptr(conv_bias), _ptr(delta), _ptr(A), _ptr(B),
                                             _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(softplus_flag)),
                                             _ptr(y), _ptr(last_state), Bsz, Dch, L, N, _dtype_code(x),
                                             _stream(stream))
    _check(st, "mamba_selective_scan_fwd_conv")


def mamba_selective_scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta, dA, dB, dC, dD, dz,
                             ddelta_bias, stream=None):
    """Gradients of sum(dy * y) of the forward scan (zero initial state).  du, ddelta, dz like u; dA [Dch, N],
    dB, dC [Bsz, N, L], dD, ddelta_bias [Dch] fp32 (written from zero)."""
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    st = lib().mamba_selective_scan_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                        _ptr(delta_bias), int(bool(softplus_flag)), _ptr(dy), _ptr(du), _ptr(ddelta),
                                        _ptr(dA), _ptr(dB), _ptr(dC), _ptr(dD), _ptr(dz), _ptr(ddelta_bias),
                                        Bsz, Dch, L, N, _dtype_code(u), _stream(stream))
    _check(st, "mamba_selective_scan_bwd")


def mamba_scan_bwd_ckpt_size(Bsz, Dch, L, N) -> int:
    """Bytes of the checkpoint buffer of mamba_selective_scan_fwd_save / mamba_selective_scan_bwd_from_ckpt."""
    n = lib().mamba_scan_bwd_ckpt_size(int(Bsz), int(Dch), int(L), int(N))
    if n == 0:
        raise MambaError(-2, "mamba_scan_bwd_ckpt_size")
    return int(n)


def mamba_selective_scan_fwd_save(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, ckpt,
                                  stream=None):
    """The direct forward scan that also writes the backward pass's checkpoints into ckpt (fp32, at least
    mamba_scan_bwd_ckpt_size bytes)."""
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    st = lib().mamba_selective_scan_fwd_save(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                             _ptr(delta_bias), int(bool(softplus_flag)), _ptr(y), _ptr(last_state),
                                             _ptr(ckpt), Bsz, Dch, L, N, _dtype_code(u), _stream(stream))
    _check(st, "mamba_selective_scan_fwd_save")


def mamba_selective_scan_bwd_from_ckpt(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, ckpt, du, ddelta, dA,
                                       dB, dC, dD, dz, ddelta_bias, stream=None):
    """mamba_selective_scan_bwd starting from the checkpoints mamba_selective_scan_fwd_save wrote."""
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    st = lib().mamba_selective_scan_bwd_from_ckpt(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                                  _ptr(delta_bias), int(bool(softplus_flag)), _ptr(dy), _ptr(ckpt),
                                                  _ptr(du), _ptr(ddelta), _ptr(dA), _ptr(dB), _ptr(dC), _ptr(dD),
                                                  _ptr(dz), _ptr(ddelta_bias), Bsz, Dch, L, N, _dtype_code(u),
                                                  _stream(stream))
    _check(st, "mamba_selective_scan_bwd_from_ckpt")


def mamba_scan_workspace_size(Bsz, Dch, L, N, chunk_len=0, dtype=MAMBA_BF16) -> int:
    n = lib().mamba_scan_workspace_size(int(Bsz), int(Dch), int(L), int(N), int(chunk_len), int(dtype))
    if n == ctypes.c_size_t(-1).value:
        raise MambaError(-2, "mamba_scan_workspace_size")
    return int(n)


def mamba_state_update(state, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, stream=None):
    """One recurrent step, state [Bsz, Dch, N] fp32 updated in place; u, delta, z, y [Bsz, Dch]; B, C [Bsz, N]."""
    Bsz, Dch, N = state.shape
    st = lib().mamba_state_update(_ptr(state), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                  _ptr(delta_bias), int(bool(softplus_flag)), _ptr(y), Bsz, Dch, N,
                                  _dtype_code(u), _stream(stream))
    _check(st, "mamba_state_update")


def mamba_device_error() -> int:
    """Read and clear the device error word (MAMBA_OK or MAMBA_ERR_DEVICE_TIMEOUT)."""
    return lib().mamba_device_error()


def mamba_bench_ex2(cycles, sink, iters, blocks, threads, stream=None):
    st = lib().mamba_bench_ex2(_ptr(cycles), _ptr(sink), int(iters), int(blocks), int(threads), _stream(stream))
    _check(st, "mamba_bench_ex2")


# ----------------------------------------------------------------------------- conveniences

def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None,
                       return_last_state=True, flags=0, chunk_len=0, stream=None):
    """Allocate y (and last_state) and run the scan; returns (y, last_state or None)."""
    import torch
    y = torch.empty_like(u)
    last = None
    if return_last_state:
        last = torch.empty((u.shape[0], u.shape[1], A.shape[1]), dtype=torch.float32, device=u.device)
    if h0 is None and flags == 0 and chunk_len == 0:
        mamba_selective_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, y, last, stream=stream)
    else:
        mamba_selective_scan_fwd_ex(u, delta, A, B, C, D, z, delta_bias, softplus, y, last, h0=h0, flags=flags,
                                    chunk_len=chunk_len, stream=stream)
    return y, last


def state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, stream=None):
    """Advance `state` in place by one token; returns y [Bsz, Dch]."""
    import torch
    y = torch.empty_like(u)
    mamba_state_update(state, u, delta, A, B, C, D, z, delta_bias, softplus, y, stream=stream)
    return y
