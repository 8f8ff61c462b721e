"""The C-ABI library: it loads, exports every declared entry point, and rejects
bad arguments on the host with the documented status codes (no GPU needed:
every call here returns before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest

import selective_state_space_148_b300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for mt in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(mamba_\w+)\s*\(", src, flags=re.M):
            names.add(mt.group(1))
    return sorted(names)


def test_library_builds_and_loads():
    from selective_state_space_148_b300 import build
    build.build()
    assert os.path.exists(m.LIB_PATH)
    m.lib()


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert {"mamba_selective_scan_fwd", "mamba_selective_scan_fwd_ex", "mamba_state_update",
            "mamba_status_string", "mamba_scan_workspace_size", "mamba_bench_ex2"} <= set(names)
    lib = ctypes.CDLL(m.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    for code in m.STATUS:
        s = m.status_string(code)
        assert s and s != "unknown status"
    assert m.status_string(12345) == "unknown status"


FAKE = 256  # a non-NULL pointer value that is never dereferenced: every call below fails validation first


def scan(**kw):
    args = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, sp=1, y=FAKE, last=None,
                Bsz=1, Dch=4, L=8, N=16, dtype=m.MAMBA_BF16)
    args.update(kw)
    return m.lib().mamba_selective_scan_fwd(args["u"], args["delta"], args["A"], args["B"], args["C"], args["D"],
                                            args["z"], args["bias"], args["sp"], args["y"], args["last"],
                                            args["Bsz"], args["Dch"], args["L"], args["N"], args["dtype"], None)


@pytest.mark.parametrize("field", ["u", "delta", "A", "B", "C", "y"])
def test_null_required_pointer(field):
    assert scan(**{field: None}) == -1


@pytest.mark.parametrize("kw,code", [
    (dict(Bsz=0), -2), (dict(Dch=0), -2), (dict(L=0), -2), (dict(N=0), -2), (dict(L=-5), -2),
    (dict(N=65), -3), (dict(N=1000), -3), (dict(dtype=2), -4), (dict(dtype=-1), -4),
    (dict(Bsz=70000), -2), (dict(Dch=1 << 41), -2), (dict(L=1 << 30, Dch=1 << 20), -2),
])
def test_bad_sizes(kw, code):
    assert scan(**kw) == code


def test_bad_flags_and_workspace_size():
    L = m.lib()
    st = L.mamba_selective_scan_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 1, FAKE, None, None,
                                       1, 4, 8, 16, m.MAMBA_BF16, 0x80, 0, None, 0, None)
    assert st == -8
    assert L.mamba_scan_workspace_size(0, 4, 8, 16, 0, 1) == ctypes.c_size_t(-1).value
    assert L.mamba_scan_workspace_size(1, 4, 8, 99, 0, 1) == ctypes.c_size_t(-1).value
    # forced direct scan needs no workspace, whatever the device
    assert L.mamba_scan_workspace_size(1, 4, 1 << 20, 16, -1, 1) == 0


def test_state_update_validation():
    L = m.lib()
    f = lambda **kw: L.mamba_state_update(kw.get("state", FAKE), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                                          1, kw.get("y", FAKE), kw.get("Bsz", 2), 4, kw.get("N", 16),
                                          kw.get("dtype", 1), None)
    assert f(state=None) == -1
    assert f(y=None) == -1
    assert f(Bsz=0) == -2
    assert f(N=65) == -3
    assert f(dtype=7) == -4


def test_bench_validation():
    L = m.lib()
    assert L.mamba_bench_ex2(None, FAKE, 10, 1, 32, None) == -1
    assert L.mamba_bench_ex2(FAKE, FAKE, 0, 1, 32, None) == -2
    assert L.mamba_bench_ex2(FAKE, FAKE, 10, 1, 2048, None) == -2


def test_training_pair_host_checks():
    """Checkpoint buffer sizes and the host-side argument checks of the forward-with-checkpoints and
    backward-from-checkpoints entry points (no GPU: every call fails validation first)."""
    L = m.lib()
    # Bsz * Dch * ceil(L / c) * P * 4 bytes with (c, P) = (16, 16), (8, 32), (4, 64) for N <= 16, 32, 64
    assert L.mamba_scan_bwd_ckpt_size(8, 1536, 2048, 16) == 8 * 1536 * 128 * 16 * 4
    assert L.mamba_scan_bwd_ckpt_size(2, 3, 17, 32) == 2 * 3 * 3 * 32 * 4
    assert L.mamba_scan_bwd_ckpt_size(1, 1, 5, 64) == 1 * 1 * 2 * 64 * 4
    assert L.mamba_scan_bwd_ckpt_size(1, 1, 5, 65) == 0
    assert L.mamba_scan_bwd_ckpt_size(0, 1, 5, 16) == 0

    def fwd(ck, N=16, dt=m.MAMBA_BF16, y=FAKE):
        return L.mamba_selective_scan_fwd_save(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 1, y, None, ck, 1, 4, 64,
                                               N, dt, None)

    def bwd(ck, N=16):
        return L.mamba_selective_scan_bwd_from_ckpt(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 1, FAKE, ck, FAKE,
                                                    FAKE, FAKE, FAKE, FAKE, None, None, None, 1, 4, 64, N,
                                                    m.MAMBA_BF16, None)

    assert fwd(None) == m.STATUS_CODE["MAMBA_ERR_NULL_ARG"]
    assert fwd(FAKE, y=None) == m.STATUS_CODE["MAMBA_ERR_NULL_ARG"]
    assert fwd(FAKE + 4) == m.STATUS_CODE["MAMBA_ERR_BAD_SHAPE"]        # checkpoints must be 16-byte aligned
    assert fwd(FAKE, N=65) == m.STATUS_CODE["MAMBA_ERR_UNSUPPORTED_N"]
    assert fwd(FAKE, dt=7) == m.STATUS_CODE["MAMBA_ERR_BAD_DTYPE"]
    assert bwd(None) == m.STATUS_CODE["MAMBA_ERR_NULL_ARG"]
    assert bwd(FAKE + 4) == m.STATUS_CODE["MAMBA_ERR_BAD_SHAPE"]
    assert bwd(FAKE, N=0) == m.STATUS_CODE["MAMBA_ERR_BAD_SHAPE"]
