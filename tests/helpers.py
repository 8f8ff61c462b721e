"""Shared test helpers: host <-> device conversion of the generator's arrays and
the tolerance check.  No scan arithmetic here."""
import numpy as np

from selective_state_space_148_b300 import inputs

# Tolerances (elementwise, |gpu - oracle| <= tol * (1 + |oracle|)):
TOL_Y = {"f32": 1e-4, "bf16": 2e-2}   # y for fp32 / bf16 storage
TOL_STATE = 1e-4                      # fp32 last_state of a scan
TOL_STATE_CHAIN = 1e-3                # fp32 state after a long chain of decode steps


def to_dev(arr, io, device="cuda"):
    """Generator array (bf16 bits or fp32) -> torch tensor on the GPU with the storage dtype."""
    import torch
    if arr is None:
        return None
    if io == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


def f32_dev(arr, device="cuda"):
    import torch
    if arr is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


def to_host_f64(t):
    """GPU tensor (fp32 or bf16) -> float64 numpy array, exact."""
    import torch
    if t.dtype == torch.bfloat16:
        return inputs.to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    return t.float().cpu().numpy().astype(np.float64)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


def assert_close(got, ref, tol, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max |err|/(1+|ref|) = {e:.3g} > {tol}"
    return e


def dev_inputs(x: "inputs.ScanInputs"):
    """All scan inputs of a ScanInputs on the GPU."""
    return dict(u=to_dev(x.u, x.io), delta=to_dev(x.delta, x.io), z=to_dev(x.z, x.io), B=to_dev(x.B, x.io),
                C=to_dev(x.C, x.io), A=f32_dev(x.A), D=f32_dev(x.D), delta_bias=f32_dev(x.delta_bias))
