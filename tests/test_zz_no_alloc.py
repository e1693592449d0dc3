"""pk_attend_noalloc, the entry point for callers that cannot allocate device memory (a
process with a fixed memory plan, a plugin whose enqueue step may not allocate, an
application whose own pool owns the device): it must give what pk_attend gives, call after
call, while using only the scratch area compiled into the library.

This file is collected last on purpose: the first call on a device does a one-time set-up,
and the test must hold both in a fresh process and after every other test has run.
"""

import ctypes

import numpy as np
import pytest

import synth
from gpu_util import device_inputs

pytestmark = pytest.mark.gpu

CASES = [
    ("bf16_global", [300, 5, 129, 64, 1, 700], "bf16", 3, 0),
    ("f16_window", [40, 1, 16, 200, 3, 9], "f16", 2, 4),
    ("f32_small", [37, 64, 150], "f32", 2, 0),
]


def _call(lib, pk, wl, inputs, out, lse, status, stream):
    qkv, cos, sin, cu = inputs
    return lib.pk_attend_noalloc(pk.dtype_code(qkv), qkv.data_ptr(), cos.data_ptr(), sin.data_ptr(), cu.data_ptr(),
                                 wl.S, wl.T, wl.H, wl.window, ctypes.c_float(wl.scale), out.data_ptr(), lse.data_ptr(),
                                 status.data_ptr(), stream)


def _same_as_pk_attend(pk, wl, calls=2):
    """Runs pk_attend once and pk_attend_noalloc `calls` times on the same inputs; the two run
    the same scheduler and attention kernels, so their outputs must be identical bit for bit."""
    import torch

    lib = pk.load()
    inputs = device_inputs(wl)
    ref_o, ref_l = pk.attend(*inputs, wl.H, wl.window, wl.scale)    # the allocating entry point
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    stream = pk._stream_handle(None)
    for call in range(calls):
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = _call(lib, pk, wl, inputs, out, lse, status, stream)
        assert rc == 0, pk.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        assert torch.equal(out, ref_o), f"call {call}: out differs from pk_attend's"
        assert torch.equal(lse, ref_l), f"call {call}: lse differs from pk_attend's"


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_noalloc_matches_pk_attend_on_two_calls(pk, case):
    name, lens, dtype, H, w = case
    wl = synth.make_lens_workload(name, lens, dtype, H=H, window=w, seed=7)
    _same_as_pk_attend(pk, wl)


def test_noalloc_near_its_token_limit(pk):
    """Short sequences (1 to 16 tokens) and a window, packed to a few tokens under the
    static scratch's limit: the most tile records and scheduler slots the scratch must hold."""
    rng = np.random.default_rng(11)
    total = pk.NOALLOC_MAX_T - 5
    lens = rng.integers(1, 17, size=total // 4)
    cut = int(np.searchsorted(np.cumsum(lens), total))
    lens = lens[:cut + 1].copy()
    lens[-1] -= int(lens.sum()) - total
    lens = lens[lens > 0]
    wl = synth.make_lens_workload("near_limit", lens, "bf16", H=2, window=4, seed=3, P=16)
    assert wl.T == total
    _same_as_pk_attend(pk, wl, calls=1)


def test_noalloc_allocates_no_device_memory(pk):
    """After a first call has done the per-device set-up, a call leaves the free device
    memory exactly as it was."""
    import torch

    wl = synth.make_lens_workload("mem", [300, 5, 129, 64], "bf16", H=2, window=0, seed=9)
    lib = pk.load()
    inputs = device_inputs(wl)
    out = torch.empty((wl.T, wl.H * 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.H, wl.T), dtype=torch.float32, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    stream = pk._stream_handle(None)
    assert _call(lib, pk, wl, inputs, out, lse, status, stream) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call(lib, pk, wl, inputs, out, lse, status, stream) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert int(status.item()) == 0
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_noalloc_rejects_too_large_and_reports_bad_cu(pk):
    import torch

    lib = pk.load()
    stream = pk._stream_handle(None)
    p = ctypes.c_void_p(0x1000)
    # beyond the static scratch capacity: rejected before anything is launched
    rc = lib.pk_attend_noalloc(1, p, p, p, p, 1, pk.NOALLOC_MAX_T + 1, 1, 0, ctypes.c_float(0.125), p, p,
                               ctypes.c_void_p(0), stream)
    assert rc == 9 and "PK_NOALLOC_MAX_T" in pk.status_string(rc)
    # a malformed cu is reported through the status pointer of the call that saw it
    wl = synth.make_lens_workload("bad", [10, 20], "bf16", H=1, window=0, seed=1)
    qkv, cos, sin, _ = device_inputs(wl)
    cu = torch.tensor([0, 25, 20], dtype=torch.int32, device="cuda")
    out = torch.empty((wl.T, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, wl.T), dtype=torch.float32, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    rc = lib.pk_attend_noalloc(1, qkv.data_ptr(), cos.data_ptr(), sin.data_ptr(), cu.data_ptr(), 2, wl.T, 1, 0,
                               ctypes.c_float(0.125), out.data_ptr(), lse.data_ptr(), status.data_ptr(), stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 5   # PK_ERR_BAD_CU
