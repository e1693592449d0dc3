"""The oracle reproduces the stored fixture (regression; inputs from packed.rs mod tests)."""

import numpy as np
import pytest

import synth
from golden_io import read_fixture


@pytest.mark.parametrize("window", [0, 8, 64])
def test_oracle_matches_golden(orc, window):
    wl = synth.p1_fixture("bf16", window)
    out, lse = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, window, wl.scale, "bf16")
    g_lse, g_out = read_fixture(window)
    np.testing.assert_allclose(lse, g_lse, rtol=1e-14, atol=1e-14)
    for a, row in g_out.items():
        np.testing.assert_allclose(out[a], row, rtol=1e-14, atol=1e-14)
