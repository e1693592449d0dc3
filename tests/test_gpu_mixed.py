"""pk_attend_mixed: fp32 inputs and arithmetic with a 16-bit output (kime's FP32-qkv,
half-output attention variant) against the oracle, and against the fp32 path's own output
rounded to the 16-bit type (the same fp32 values, one rounding: bit for bit); and
pk_attend_mixed_ops: fp32 storage with 16-bit tensor-core operands against the oracle and
against the 16-bit path on the same values."""

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


# ------------------------------------------------------------------------------------------
# pk_attend_mixed_ops: fp32 storage, 16-bit tensor-core operands, fp32 out (the pages' attend
# with f32 storage and f16 operands)

TOL16 = {"f16": (5e-3, 5e-3), "bf16": (2e-2, 1e-2)}


@pytest.mark.parametrize("op", ["f16", "bf16"])
@pytest.mark.parametrize("window", [0, 70])
@pytest.mark.parametrize("lens", [[37, 0, 129, 1, 300, 20, 5], [512, 130, 64]], ids=["ragged", "long"])
def test_mixed_ops_parity(pk, orc, op, window, lens):
    import torch

    wl = synth.make_lens_workload("mops", lens, "f32", H=3, window=window, seed=len(lens) + window + 3)
    qkv, cos, sin, cu = device_inputs(wl)
    out, lse = pk.attend_mixed_ops(qkv, cos, sin, cu, wl.H, window, wl.scale, _torch_dt(op))
    torch.cuda.synchronize()
    assert out.dtype == torch.float32 and pk.last_status() == 0
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, window, wl.scale, "f32")
    to, tl = TOL16[op]
    assert max_err(out_to_f64(out), want_o) <= to
    assert max_err(lse.cpu().numpy().astype(np.float64), want_l) <= tl


@pytest.mark.parametrize("op", ["f16", "bf16"])
@pytest.mark.parametrize("scale", [0.125, -0.05])
def test_mixed_ops_equals_the_16bit_path(pk, op, scale):
    """fp32 inputs holding op-type values: the same rotated operands as the op-type path, so
    the same scores, probabilities and sums -- out equal before its rounding, lse equal."""
    import torch

    wl16 = synth.make_lens_workload("m16", [300, 5, 129, 64, 1, 700], op, H=2, window=0, seed=17)
    q16, c16, s16, cu = device_inputs(wl16)
    ref_o, ref_l = pk.attend(q16, c16, s16, cu, wl16.H, 0, scale)
    out, lse = pk.attend_mixed_ops(q16.float(), c16.float(), s16.float(), cu, wl16.H, 0, scale, _torch_dt(op))
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    assert torch.equal(out.to(_torch_dt(op)), ref_o)
    assert torch.equal(lse, ref_l)


def test_mixed_ops_rejects_other_operand_types(pk):
    wl = synth.make_lens_workload("mops", [10], "f32", H=1, window=0, seed=1)
    qkv, cos, sin, cu = device_inputs(wl)
    p = qkv.data_ptr()
    assert pk.pk_attend_mixed_ops(0, p, p, p, cu.data_ptr(), 1, 10, 1, 0, 0.125, p, p, None) == 1
