"""pk_attend_mixed: fp32 inputs and arithmetic with a 16-bit output (kime's FP32-qkv,
half-output attention variant) against the oracle, and against the fp32 path's own output
rounded to the 16-bit type (the same fp32 values, one rounding: bit for bit)."""

import numpy as np
import pytest

import synth
from gpu_util import device_inputs, max_err, out_to_f64

pytestmark = pytest.mark.gpu

# half an ulp of the output type, relative
REL = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def _torch_dt(name):
    import torch

    return {"f16": torch.float16, "bf16": torch.bfloat16}[name]


@pytest.mark.parametrize("odt", ["f16", "bf16"])
@pytest.mark.parametrize("window", [0, 5, 100])
@pytest.mark.parametrize("lens", [[37, 0, 129, 1, 300], [64] * 9 + [250]], ids=["ragged", "even"])
def test_mixed_parity(pk, orc, odt, window, lens):
    import torch

    wl = synth.make_lens_workload("mixed", lens, "f32", H=3, window=window, seed=len(lens) + window)
    qkv, cos, sin, cu = device_inputs(wl)
    out, lse = pk.attend(qkv, cos, sin, cu, wl.H, window, wl.scale, out_dtype=_torch_dt(odt))
    ref_out, ref_lse = pk.attend(qkv, cos, sin, cu, wl.H, window, wl.scale)  # fp32 out, same arithmetic
    torch.cuda.synchronize()
    assert out.dtype == _torch_dt(odt) and pk.last_status() == 0
    # one rounding of the fp32 path's values
    assert torch.equal(out, ref_out.to(_torch_dt(odt)))
    assert torch.equal(lse, ref_lse)
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, window, wl.scale, "f32")
    got_o = out_to_f64(out)
    assert np.all(np.abs(got_o - want_o) <= 1e-4 + REL[odt] * np.abs(want_o))
    assert max_err(lse.cpu().numpy().astype(np.float64), want_l) <= 1e-4


def test_mixed_rejects_other_inputs(pk):
    import torch

    wl = synth.make_lens_workload("mixed", [10], "bf16", H=1, window=0, seed=1)
    qkv, cos, sin, cu = device_inputs(wl)
    with pytest.raises(TypeError):
        pk.attend(qkv, cos, sin, cu, 1, 0, wl.scale, out_dtype=torch.float16)
    # the C entry point checks the output type
    p = qkv.data_ptr()
    assert pk.pk_attend_mixed(7, p, p, p, cu.data_ptr(), 1, 10, 1, 0, 0.125, p, p, None) == 1
