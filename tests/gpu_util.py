"""Helpers of the GPU tests: move a synthetic workload to the device, run the library
through its binding, compare with the oracle."""

from __future__ import annotations

import numpy as np

import synth

# max |delta| bounds on out and lse by input type (the method's stated tolerances)
TOL = {"f32": (1e-4, 1e-4), "bf16": (2e-2, 1e-2), "f16": (5e-3, 5e-3)}


def torch_dtype(dt):
    import torch

    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dt]


def to_device(arr: np.ndarray, dt: str, dev="cuda"):
    import torch

    if dt == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(dev).view(torch.bfloat16)
    if dt == "f16":
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float16)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(dev)


def out_to_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def device_inputs(wl):
    import torch

    return (to_device(wl.qkv, wl.dtype), to_device(wl.cos, wl.dtype), to_device(wl.sin, wl.dtype),
            torch.from_numpy(wl.cu.astype(np.int64).astype(np.int32)).cuda())


def run(pk, wl, window=None, inputs=None):
    """(out, lse) as float64 numpy arrays; checks the device status word."""
    import torch

    window = wl.window if window is None else window
    qkv, cos, sin, cu = inputs or device_inputs(wl)
    out, lse = pk.attend(qkv, cos, sin, cu, wl.H, window, wl.scale)
    torch.cuda.synchronize()
    st = pk.last_status()
    assert st == 0, f"device status {st}: {pk.status_string(st)}"
    return out_to_f64(out), lse.cpu().numpy().astype(np.float64)


def max_err(a, b) -> float:
    return float(np.max(np.abs(a - b))) if a.size else 0.0
