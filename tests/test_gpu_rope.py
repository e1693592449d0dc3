"""The standalone rotation (pk_rope) against the oracle's oracle_rope_qkv, element by element:
every layout (halves, interleaved pairs), partial dims, both directions, in place and out of
place, the three element types; the device error for a position past the tables."""

import numpy as np
import pytest

import synth
from gpu_util import out_to_f64, to_device

pytestmark = pytest.mark.gpu

# one rounding of an fp32 result to the element type: half an ulp, relative
REL = {"f32": 2e-6, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def _case(dt, lens, H, dims, seed, P=None):
    rng = np.random.default_rng(seed)
    cu = synth.cu_from_lens(lens)
    T = int(cu[-1])
    qkv = synth.to_storage(rng.standard_normal((T, 3 * H * 64)).astype(np.float32), dt)
    P = P or max(1, int(max(lens)) if len(lens) else 1)
    c, s = synth.rope_tables_dims(P, dims, 10000.0)
    return cu, qkv, synth.to_storage(c, dt), synth.to_storage(s, dt)


def _run(pk, dt, cu, qkv, c, s, H, dims, trad, inv, in_place=False, status=None):
    import torch

    x = to_device(qkv, dt)
    cu_d = torch.from_numpy(cu.astype(np.int64).astype(np.int32)).cuda()
    out = x if in_place else None
    y = pk.rope(x, to_device(c, dt), to_device(s, dt), cu_d, H, dims, trad, inv, out=out, status=status)
    torch.cuda.synchronize()
    return out_to_f64(y)


def _check(got, want, dt):
    # half an ulp of the element type, plus the fp32 arithmetic's own rounding (a few units of
    # 2^-24 of inputs of magnitude below 8)
    err = np.abs(got - want)
    bound = REL[dt] * np.abs(want) + 2e-6
    assert np.all(err <= bound), (float(err.max()), float((err - bound).max()))


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("dims", [64, 32, 6, 2])
@pytest.mark.parametrize("trad", [False, True])
@pytest.mark.parametrize("inv", [False, True])
def test_rope_parity(pk, orc, dt, dims, trad, inv):
    lens = [37, 0, 129, 1, 300, 0, 0, 64]
    H = 3
    cu, qkv, c, s = _case(dt, lens, H, dims, seed=dims + 7 * trad + 13 * inv)
    want = orc.rope_qkv(qkv, c, s, cu, H, dims, trad, inv, dtype=dt, table_dtype=dt)
    got = _run(pk, dt, cu, qkv, c, s, H, dims, trad, inv)
    _check(got, want, dt)
    # v and the features past dims come through unchanged
    T = int(cu[-1])
    x64 = synth.to_f64(qkv, dt).reshape(T, 3 * H, 64)
    g = got.reshape(T, 3 * H, 64)
    assert np.array_equal(g[:, 2 * H:], x64[:, 2 * H:])
    assert np.array_equal(g[:, :2 * H, dims:], x64[:, :2 * H, dims:])


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_rope_in_place_and_round_trip(pk, orc, dt):
    import torch

    lens = [200, 3, 0, 77]
    H = 2
    cu, qkv, c, s = _case(dt, lens, H, 64, seed=5)
    x = to_device(qkv, dt)
    cu_d = torch.from_numpy(cu.astype(np.int64).astype(np.int32)).cuda()
    cd, sd = to_device(c, dt), to_device(s, dt)
    y = pk.rope(x, cd, sd, cu_d, H, 64, False, False, out=x)  # in place
    torch.cuda.synchronize()
    assert y.data_ptr() == x.data_ptr()
    want = orc.rope_qkv(qkv, c, s, cu, H, 64, False, False, dtype=dt, table_dtype=dt)
    _check(out_to_f64(x), want, dt)
    # back again: the inverse of the rounded forward result, within two roundings
    back = out_to_f64(pk.rope(x, cd, sd, cu_d, H, 64, False, True))
    x64 = synth.to_f64(qkv, dt)
    assert np.all(np.abs(back - x64) <= 4 * REL[dt] * (np.abs(x64) + 1.0))


def test_rope_full_size(pk, orc):
    """The short-sequence workload's shape (T = 65536, H = 12, 7676 sequences), every element."""
    wl = synth.make_config("short")
    c, s = synth.rope_tables_dims(int(wl.lens.max()), 64, 10000.0)
    c, s = synth.to_storage(c, "f16"), synth.to_storage(s, "f16")
    want = orc.rope_qkv(wl.qkv, c, s, wl.cu, wl.H, 64, False, False, dtype="f16", table_dtype="f16")
    got = _run(pk, "f16", wl.cu, wl.qkv, c, s, wl.H, 64, False, False)
    _check(got, want, "f16")


def test_rope_position_past_tables_is_reported(pk, orc):
    """Tables shorter than a sequence: PK_ERR_BAD_CU in the status word, the other tokens right."""
    import torch

    lens = [10, 40, 5]
    H = 1
    cu, qkv, c, s = _case("bf16", lens, H, 64, seed=9, P=40)
    c_short, s_short = c[:20], s[:20]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(pk, "bf16", cu, qkv, c_short, s_short, H, 64, False, False, status=status)
    assert int(status.item()) == 5  # PK_ERR_BAD_CU
    want = orc.rope_qkv(qkv, c, s, cu, H, 64, False, False, dtype="bf16", table_dtype="bf16")
    T = int(cu[-1])
    seq = np.searchsorted(cu, np.arange(T), side="right") - 1
    pos = np.arange(T) - cu[seq]
    ok = pos < 20
    _check(got[ok], want[ok], "bf16")
