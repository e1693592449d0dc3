"""The narrow-window kernel (windows 1..16, `pk_attend_band_kernel`) against the oracle, element by
element (GPU): every instance (largest window 4, 8 and 16) for every storage type, both signs of
the scale, sequences shorter than the window, sequences crossing the 32-token blocks the kernel
stages, empty sequences, and a token count that is not a multiple of 32."""

import numpy as np
import pytest

import synth
from gpu_util import TOL, max_err, run

pytestmark = pytest.mark.gpu

# lengths: shorter than every window, exactly one block, blocks plus a ragged tail, empties
LENS = [1, 2, 0, 5, 31, 32, 33, 0, 17, 64, 65, 3, 100, 7, 0, 129, 9]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("window", [1, 3, 4, 5, 8, 9, 12, 16])
def test_band_matches_oracle(pk, orc, dtype, window):
    wl = synth.make_lens_workload(f"band_w{window}", LENS, dtype, H=3, window=window, seed=100 + window)
    code = {"f32": pk.PK_F32, "bf16": pk.PK_BF16, "f16": pk.PK_F16}[dtype]
    assert pk.KERNELS[pk.pk_forward_kernel(code, window)] == "band"
    got_o, got_l = run(pk, wl)
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, window, wl.scale, wl.dtype)
    to, tl = TOL[dtype]
    eo, el = max_err(got_o, want_o), max_err(got_l, want_l)
    assert eo <= to and el <= tl, f"w={window} {dtype}: max|dout| {eo:.3e} (<= {to}), max|dlse| {el:.3e} (<= {tl})"


@pytest.mark.parametrize("scale", [-0.3, 0.05, 1.0])
@pytest.mark.parametrize("window", [2, 7, 16])
def test_band_scales(pk, orc, scale, window):
    wl = synth.make_lens_workload("band_scale", LENS, "f16", H=2, window=window, seed=7, scale=scale)
    got_o, got_l = run(pk, wl)
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, window, wl.scale, wl.dtype)
    to, tl = TOL["f16"]
    eo, el = max_err(got_o, want_o), max_err(got_l, want_l)
    assert eo <= to and el <= tl, f"w={window} scale {scale}: max|dout| {eo:.3e}, max|dlse| {el:.3e}"


def test_band_many_heads_and_a_long_sequence(pk, orc):
    # heads beyond one CTA's group of four, a sequence far longer than the window
    lens = [3000, 11, 0, 40]
    wl = synth.make_lens_workload("band_heads", lens, "bf16", H=7, window=6, seed=21)
    got_o, got_l = run(pk, wl)
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, wl.window, wl.scale, wl.dtype)
    to, tl = TOL["bf16"]
    assert max_err(got_o, want_o) <= to and max_err(got_l, want_l) <= tl
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_l))
