"""The CUDA path against the oracle, element by element (GPU)."""

import numpy as np
import pytest

import oracle_pins
import synth
from golden_io import read_fixture
from gpu_util import TOL, device_inputs, max_err, run

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------------------------------
# schedule: bit-exact against the oracle's records


def _sched_cases():
    cases = list(oracle_pins.schedule_cases())
    for i, name in enumerate(synth.CONFIG_NAMES):
        lens = synth.config_lens(name, np.random.default_rng(i))
        w = {"tiny": 0, "global": 0, "local": 64, "long": 0, "short": 4}[name]
        cases.append((name, synth.cu_from_lens(lens), w))
        cases.append((name + "_w7", synth.cu_from_lens(lens), 7))
    # adversarial: long runs of empty sequences, lengths around every boundary
    cases.append(("empties", synth.cu_from_lens([0] * 300 + [5] + [0] * 300 + [130] + [0] * 10), 0))
    lens = []
    for L in (0, 1, 15, 16, 17, 63, 64, 65, 66, 127, 128, 129, 191, 192, 193, 255, 256, 257, 8192):
        lens += [L, 1, L]
    cases.append(("boundaries", synth.cu_from_lens(lens), 0))
    cases.append(("boundaries_w", synth.cu_from_lens(lens), 100))
    # more sequences than the scheduler stages in shared memory (cu read from global memory),
    # over enough windows for a cluster of scheduler blocks, with 128-member groups
    rng = np.random.default_rng(77)
    cases.append(("many_tiny", synth.cu_from_lens(rng.integers(0, 4, size=60000)), 0))
    cases.append(("many_tiny_mixed", synth.cu_from_lens(
        np.where(rng.random(52000) < 0.01, rng.integers(65, 600, size=52000), rng.integers(0, 3, size=52000))), 3))
    # enough windows that the scheduler's record slots live in the workspace, not in shared memory
    cases.append(("many_windows", synth.cu_from_lens(
        np.where(rng.random(3000) < 0.3, rng.integers(65, 500, size=3000), rng.integers(0, 30, size=3000))), 0))
    return cases


@pytest.mark.parametrize("case", _sched_cases(), ids=lambda c: c[0])
def test_schedule_bit_exact(pk, orc, case):
    import torch

    name, cu, w = case
    T = int(cu[-1])
    want = orc.schedule(cu, w)
    got = pk.schedule(torch.from_numpy(cu.astype(np.int64).astype(np.int32)).cuda(), T, w)
    got = got.cpu().numpy().view(np.uint32)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.array_equal(got, want)
    assert not oracle_pins.schedule_failures(got, cu, w)


# ------------------------------------------------------------------------------------------
# element-wise parity at sizes the oracle finishes in seconds


def _check(pk, orc, wl, window=None):
    window = wl.window if window is None else window
    got_o, got_l = run(pk, wl, window)
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, window, wl.scale, wl.dtype)
    to, tl = TOL[wl.dtype]
    eo, el = max_err(got_o, want_o), max_err(got_l, want_l)
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_l))
    assert eo <= to and el <= tl, f"{wl.name} w={window}: max|dout| {eo:.3e} (<= {to}), max|dlse| {el:.3e} (<= {tl})"
    return eo, el


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("window", [0, 8, 64])
def test_packed_rs_fixture(pk, orc, dtype, window):
    """The packed.rs test inputs (LENS 5, 40, 1, 33, 70; HEADS 2), windows None / 8 / 64."""
    _check(pk, orc, synth.p1_fixture(dtype, window))


@pytest.mark.parametrize("window", [0, 8, 64])
def test_packed_rs_fixture_golden(pk, window):
    wl = synth.p1_fixture("bf16", window)
    got_o, got_l = run(pk, wl)
    g_lse, g_out = read_fixture(window)
    assert max_err(got_l, g_lse) <= TOL["bf16"][1]
    for a, row in g_out.items():
        assert max_err(got_o[a], row) <= TOL["bf16"][0]


def test_tiny_config(pk, orc):
    _check(pk, orc, synth.make_config("tiny"))


RAGGED = [
    ("crossing", [300, 129, 1, 128, 127, 257], 0),
    ("crossing_w1", [300, 129, 1, 128, 127, 257], 1),
    ("crossing_w70", [300, 129, 1, 128, 127, 257], 70),
    ("shorts", [1, 2, 3, 16, 64, 65, 5, 9, 33, 1, 1, 64, 63, 7], 0),
    ("shorts_w4", [1, 2, 3, 16, 64, 65, 5, 9, 33, 1, 1, 64, 63, 7], 4),
    ("empties", [0, 0, 40, 0, 200, 0, 0, 3, 0], 0),
    ("single", [1], 0),
    ("one_long", [1000], 0),
    ("one_long_w200", [1000], 200),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", RAGGED, ids=lambda c: c[0])
def test_ragged(pk, orc, dtype, case):
    name, lens, w = case
    wl = synth.make_lens_workload(name, lens, dtype, H=3, window=w, seed=len(lens), base=10000.0)
    _check(pk, orc, wl)


@pytest.mark.parametrize("H", [1, 16])
def test_heads(pk, orc, H):
    wl = synth.make_lens_workload("heads", [90, 200, 17], "bf16", H=H, window=0, seed=H)
    _check(pk, orc, wl)


def test_max_length_sequence(pk, orc):
    """One sequence of 8192 tokens (the longest of the measured configurations): every element."""
    wl = synth.make_lens_workload("max", [8192], "bf16", H=2, window=0, seed=5)
    got_o, got_l = run(pk, wl)
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, 2, 0, wl.scale, "bf16")
    assert max_err(got_o, want_o) <= TOL["bf16"][0]
    assert max_err(got_l, want_l) <= TOL["bf16"][1]


def test_deterministic(pk):
    wl = synth.make_lens_workload("det", [300, 5, 129, 64], "bf16", H=4, window=0, seed=3)
    inputs = device_inputs(wl)
    o1, l1 = run(pk, wl, inputs=inputs)
    o2, l2 = run(pk, wl, inputs=inputs)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ------------------------------------------------------------------------------------------
# paths of the tensor-core kernel that the workloads above do not reach


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("scale", [1.0, 0.05, -0.125, 0.0])
def test_scales(pk, orc, dtype, scale):
    """A positive scale is applied to the scores in the softmax, any other multiplies q. The
    inputs' spread is chosen so that the scaled scores keep unit spread (as at scale 1/8 with
    unit inputs): the rotated q and k are rounded to the input type for the tensor cores, and
    larger scores would carry that rounding past the stated tolerances at any scale."""
    sigma = (1.0 / (8.0 * abs(scale))) ** 0.5 if scale != 0.0 else 1.0
    wl = synth.make_lens_workload("scale", [130, 40, 5, 260], dtype, H=2, window=0, seed=11, scale=scale,
                                  sigma=sigma)
    _check(pk, orc, wl)


@pytest.mark.parametrize("window", [0, 2])
def test_group_with_many_members(pk, orc, window):
    """A group of short sequences with more member offsets than the kernel stages in shared
    memory (a group takes any number of empty sequences): rows find their sequence in cu."""
    lens = [3] + [0] * 100 + [5] + [0] * 50 + [7, 2] + [0] * 20 + [40, 200]
    wl = synth.make_lens_workload("members", lens, "bf16", H=2, window=window, seed=12)
    sched = orc.schedule(wl.cu, window)
    assert int(sched[:, 5].max()) > 130  # nseq of the group: past the staged offsets
    _check(pk, orc, wl)


@pytest.mark.parametrize("lens", [[129], [129, 129], [127, 300, 5], [640, 64, 640]], ids=str)
def test_pairs(pk, orc, lens):
    """Odd and even record counts, pieces sharing a key stream, a stream that ends mid-pair."""
    for window in (0, 100):
        wl = synth.make_lens_workload("pairs", lens, "bf16", H=3, window=window, seed=len(lens))
        _check(pk, orc, wl)
