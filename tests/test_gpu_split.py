"""fp32 inputs on the tensor cores (PK_KERNEL_SPLIT, GPU): every element against the fp64
oracle at the fp32 tolerance, for ragged and grouped sequences, empty sequences, windows
beyond the narrow band, every kind of scale, and the global layer's shapes at full size
with fp32 storage; plus the dispatch rules around it."""

import numpy as np
import pytest

import synth
from gpu_util import TOL, device_inputs, max_err, out_to_f64

pytestmark = pytest.mark.gpu

CASES = [
    # name, lengths, heads, window, scale
    ("groups_w0", [1, 5, 16, 33, 7, 64, 129, 3, 200], 3, 0, None),
    ("long_w0", [1000, 130, 257], 2, 0, None),
    ("empty_seqs", [0, 50, 0, 0, 129, 0], 2, 0, None),
    ("window_17", [300, 17, 18, 2], 2, 17, None),
    ("window_70", [900, 40, 300], 2, 70, None),
    ("window_300", [700, 20], 1, 300, None),
    ("neg_scale", [200, 77, 129], 2, 0, -0.125),
    ("small_scale", [260, 3, 129], 2, 0, 0.05),
    ("zero_scale", [140, 9], 1, 0, 0.0),
]


def _check(pk, orc, wl):
    import torch

    out, lse = pk.attend(*device_inputs(wl), wl.H, wl.window, wl.scale)
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, wl.window, wl.scale, "f32")
    to, tl = TOL["f32"]
    eo = max_err(out_to_f64(out), want_o)
    el = max_err(lse.cpu().numpy().astype(np.float64), want_l)
    assert eo <= to and el <= tl, (wl.name, eo, el)
    return eo, el


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_split_matches_oracle(pk, orc, monkeypatch, case):
    name, lens, H, w, scale = case
    monkeypatch.setenv("PK_ATTN", "split")
    assert pk.pk_forward_kernel(pk.PK_F32, w) == 5
    wl = synth.make_lens_workload(name, lens, "f32", H=H, window=w, seed=len(lens) + 3, scale=scale)
    _check(pk, orc, wl)


def test_split_tiny_configuration(pk, orc, monkeypatch):
    monkeypatch.setenv("PK_ATTN", "split")
    _check(pk, orc, synth.make_config("tiny"))


def test_split_global_shapes_full_size(pk, orc, monkeypatch):
    """The global layer's lengths, heads and tables (T about 17k, H = 12) with fp32 storage."""
    monkeypatch.setenv("PK_ATTN", "split")
    g = synth.make_config("global")
    wl = synth.make_lens_workload("global_f32", g.lens, "f32", H=g.H, window=0, base=g.base, seed=11)
    _check(pk, orc, wl)


def test_split_is_not_used_for_a_16_bit_output_or_narrow_windows(pk, orc, monkeypatch):
    """pk_attend_mixed (fp32 storage, 16-bit output) and windows of 1..16 keep their own
    kernels under PK_ATTN=split, and match the oracle."""
    import torch

    monkeypatch.setenv("PK_ATTN", "split")
    assert pk.pk_forward_kernel(pk.PK_F32, 4) == 0
    wl = synth.make_lens_workload("mixed_out", [130, 7, 64], "f32", H=2, window=0, seed=9)
    qkv, cos, sin, cu = device_inputs(wl)
    out, lse = pk.attend(qkv, cos, sin, cu, wl.H, wl.window, wl.scale, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, wl.window, wl.scale, "f32")
    assert max_err(out.float().cpu().numpy().astype(np.float64), want_o) <= 2e-2
    assert max_err(lse.cpu().numpy().astype(np.float64), want_l) <= 1e-4
