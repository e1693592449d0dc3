"""pk_attend_backward against the oracle's fp64 gradient (oracle_attend_backward), on the
forward's own out and lse: element types, windows, scales of both signs, groups of short
sequences and pieces of long ones (several records adding to the same keys)."""

import numpy as np
import pytest

import synth
from gpu_util import device_inputs, out_to_f64, to_device

pytestmark = pytest.mark.gpu

# max |delta| / max |reference| by input type, about four times the largest seen. fp32: the
# forward's out and lse are exact to fp32 rounding (seen 6e-7). 16-bit: the forward's lse comes
# from q', k' rounded to the input type and its out is rounded too, so P and D carry those
# errors, and dqkv is rounded once more (seen 4.6e-3 in bf16, 8.6e-4 in fp16).
REL = {"f32": 1e-5, "bf16": 1.5e-2, "f16": 3e-3}

CASES = [
    ("pieces", [300, 129, 5, 0, 64], 0, 0.125),
    ("pieces_w", [300, 129, 5, 0, 64], 7, 0.125),
    ("groups", [3, 9, 1, 0, 17, 30, 2, 11], 2, 0.125),
    ("neg_scale", [200, 40], 0, -0.2),
]


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_backward_parity(pk, orc, dt, case):
    import torch

    name, lens, window, scale = case
    H = 2
    wl = synth.make_lens_workload(name, lens, dt, H=H, window=window, seed=len(lens) + window, scale=scale)
    qkv, cos, sin, cu = device_inputs(wl)
    out, lse = pk.attend(qkv, cos, sin, cu, H, window, scale)
    rng = np.random.default_rng(3)
    dout_np = synth.to_storage(rng.standard_normal((wl.T, H * 64)).astype(np.float32), dt)
    dout = to_device(dout_np, dt)
    dqkv = pk.attend_backward(qkv, cos, sin, cu, H, window, scale, out, lse, dout)
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    got = out_to_f64(dqkv)
    want = orc.attend_backward(wl.qkv, wl.cos, wl.sin, wl.cu, H, window, scale, dout_np, dtype=dt)
    assert np.all(np.isfinite(got))
    for part, nm in ((0, "dq"), (1, "dk"), (2, "dv")):
        a = slice(part * H * 64, (part + 1) * H * 64)
        err = float(np.max(np.abs(got[:, a] - want[:, a])))
        ref = float(np.max(np.abs(want[:, a])))
        assert err <= REL[dt] * max(ref, 1e-3), f"{nm}: max|delta| {err:.3e}, max|ref| {ref:.3e}"


def test_backward_global_config_full_size(pk, orc):
    """The encoder-base global layer (64 sequences of 32..512 tokens, H = 12, bf16) at full size:
    every element of dq, dk, dv against the fp64 gradient."""
    import torch

    wl = synth.make_config("global")
    H = wl.H
    qkv, cos, sin, cu = device_inputs(wl)
    out, lse = pk.attend(qkv, cos, sin, cu, H, 0, wl.scale)
    rng = np.random.default_rng(11)
    dout_np = synth.to_storage(rng.standard_normal((wl.T, H * 64)).astype(np.float32), "bf16")
    dout = to_device(dout_np, "bf16")
    dqkv = pk.attend_backward(qkv, cos, sin, cu, H, 0, wl.scale, out, lse, dout)
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    got = out_to_f64(dqkv)
    want = orc.attend_backward(wl.qkv, wl.cos, wl.sin, wl.cu, H, 0, wl.scale, dout_np, dtype="bf16")
    assert np.all(np.isfinite(got))
    for part, nm in ((0, "dq"), (1, "dk"), (2, "dv")):
        a = slice(part * H * 64, (part + 1) * H * 64)
        err = float(np.max(np.abs(got[:, a] - want[:, a])))
        ref = float(np.max(np.abs(want[:, a])))
        assert err <= REL["bf16"] * max(ref, 1e-3), f"{nm}: max|delta| {err:.3e}, max|ref| {ref:.3e}"
