"""The tuned forward entry point and every candidate it times (GPU): each kernel against the
oracle element by element, the cache keeping one pick per key, and the capture rule."""

import numpy as np
import pytest

import synth
from gpu_util import TOL, device_inputs, max_err, out_to_f64

pytestmark = pytest.mark.gpu

SHAPES = [
    ("mixed_w0", [300, 5, 129, 64, 1, 700, 256, 33], "bf16", 3, 0),
    ("mixed_f16_w0", [130, 1, 64, 65, 257, 9], "f16", 2, 0),
    ("window_70", [900, 40, 300], "bf16", 2, 70),
    ("window_4", [7, 1, 16, 3, 200, 12], "f16", 3, 4),
    ("f32_w0", [37, 64, 150], "f32", 2, 0),
    ("f32_w70_long", [1200, 300, 5], "f32", 2, 70),
]


def _tuned(pk, wl, inputs):
    import torch

    out, lse = pk.attend(*inputs, wl.H, wl.window, wl.scale, tuned=True, max_len=int(wl.lens.max()))
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    return out, lse


@pytest.mark.parametrize("shape", SHAPES, ids=lambda c: c[0])
def test_tuned_matches_oracle_and_keeps_its_pick(pk, orc, shape):
    import torch

    name, lens, dtype, H, w = shape
    wl = synth.make_lens_workload(name, lens, dtype, H=H, window=w, seed=len(lens))
    pk.pk_tune_clear()
    dt = pk.dtype_code(device_inputs(wl)[0])
    assert pk.pk_tune_pick(dt, H, w, wl.T, int(wl.lens.max())) == -1
    inputs = device_inputs(wl)
    o1, l1 = _tuned(pk, wl, inputs)
    pick = pk.pk_tune_pick(dt, H, w, wl.T, int(wl.lens.max()))
    if 1 <= w <= 16:
        assert pick == 0
    elif dtype == "f32":
        assert pick in (1, 5)
    else:
        assert pick in (2, 3, 4)
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, H, w, wl.scale, dtype)
    to, tl = TOL[dtype]
    assert max_err(out_to_f64(o1), want_o) <= to
    assert max_err(l1.cpu().numpy().astype(np.float64), want_l) <= tl
    # later calls with the key run the kept kernel: the same result, bit for bit
    o2, l2 = _tuned(pk, wl, inputs)
    assert pk.pk_tune_pick(dt, H, w, wl.T, int(wl.lens.max())) == pick
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("kernel", ["tc", "tc_single", "q4"])
@pytest.mark.parametrize("shape", [s for s in SHAPES if s[2] != "f32" and not 1 <= s[4] <= 16], ids=lambda c: c[0])
def test_every_tensor_core_candidate_matches_oracle(pk, orc, monkeypatch, kernel, shape):
    name, lens, dtype, H, w = shape
    wl = synth.make_lens_workload(name, lens, dtype, H=H, window=w, seed=len(lens) + 1)
    monkeypatch.setenv("PK_ATTN", kernel)
    import torch

    out, lse = pk.attend(*device_inputs(wl), H, w, wl.scale)
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, H, w, wl.scale, dtype)
    to, tl = TOL[dtype]
    assert max_err(out_to_f64(out), want_o) <= to
    assert max_err(lse.cpu().numpy().astype(np.float64), want_l) <= tl


def test_untuned_key_is_not_tuned_under_capture(pk):
    """A first call of a key with several candidates would have to wait for the stream: under
    capture it is refused; once tuned outside, the same call is captured and replays."""
    import torch

    wl = synth.make_lens_workload("cap", [200, 7, 129], "bf16", H=2, window=0, seed=21)
    qkv, cos, sin, cu = device_inputs(wl)
    out = torch.zeros((wl.T, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, wl.T), dtype=torch.float32, device="cuda")
    pk.pk_tune_clear()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pk.attend(qkv, cos, sin, cu, 2, 0, wl.scale, out=out, lse=lse, stream=s)  # the workspace exists
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        with pytest.raises(pk.PKError) as err:
            pk.attend(qkv, cos, sin, cu, 2, 0, wl.scale, out=out, lse=lse, stream=s, tuned=True, max_len=200)
    assert err.value.code == 10
    ref_o, ref_l = pk.attend(qkv, cos, sin, cu, 2, 0, wl.scale, tuned=True, max_len=200, stream=s)
    torch.cuda.synchronize()
    out.zero_()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        pk.attend(qkv, cos, sin, cu, 2, 0, wl.scale, out=out, lse=lse, stream=s, tuned=True, max_len=200)
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
