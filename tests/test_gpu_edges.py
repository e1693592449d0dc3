"""Edge cases, stray-write canaries, device-detected errors and streams (GPU)."""

import numpy as np
import pytest

import synth
from gpu_util import TOL, device_inputs, max_err, out_to_f64, run, to_device

pytestmark = pytest.mark.gpu

SENT = -12345.0


def _padded(torch, T, H, dtype, pad=7):
    """out and lse views with `pad` extra sentinel-filled rows / entries after them."""
    out_buf = torch.full(((T + pad) * H * 64,), SENT, dtype=dtype, device="cuda")
    lse_buf = torch.full((H * T + pad,), SENT, dtype=torch.float32, device="cuda")
    return out_buf, lse_buf, out_buf[: T * H * 64].view(T, H * 64), lse_buf[: H * T].view(H, T)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_no_stray_writes(pk, orc, dtype):
    import torch

    wl = synth.make_lens_workload("canary", [3, 130, 64, 1, 70], dtype, H=2, window=0, seed=1)
    qkv, cos, sin, cu = device_inputs(wl)
    td = qkv.dtype
    out_buf, lse_buf, out, lse = _padded(torch, wl.T, wl.H, td)
    pk.attend(qkv, cos, sin, cu, wl.H, 0, wl.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert pk.last_status() == 0
    assert torch.all(out_buf[wl.T * wl.H * 64:] == SENT)
    assert torch.all(lse_buf[wl.H * wl.T:] == SENT)
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, 0, wl.scale, dtype)
    to, tl = TOL[dtype]
    assert max_err(out_to_f64(out), want_o) <= to
    assert max_err(lse.cpu().numpy().astype(np.float64), want_l) <= tl


@pytest.mark.parametrize("bad", ["first_not_zero", "decreasing", "last_not_T"])
def test_malformed_cu_sets_status(pk, bad):
    import torch

    wl = synth.make_lens_workload("bad", [10, 20, 30], "bf16", H=1, window=0, seed=2)
    qkv, cos, sin, _ = device_inputs(wl)
    cu = wl.cu.astype(np.int64).copy()
    if bad == "first_not_zero":
        cu[0] = 1
    elif bad == "decreasing":
        cu[1], cu[2] = cu[2], cu[1]
    else:
        cu[-1] -= 1
    cu_d = torch.from_numpy(cu.astype(np.int32)).cuda()
    out_buf, lse_buf, out, lse = _padded(torch, wl.T, wl.H, torch.bfloat16, pad=0)
    # (max_len given: the binding's own table check would otherwise refuse the bad cu first)
    pk.attend(qkv, cos, sin, cu_d, wl.H, 0, wl.scale, out=out, lse=lse,
              max_len=int(wl.lens.max()))   # returns: error is on the device
    assert pk.last_status() == 5   # PK_ERR_BAD_CU
    assert pk.last_status() == 0   # cleared by the read
    assert torch.all(out_buf == SENT) and torch.all(lse_buf == SENT)   # nothing written
    with pytest.raises(pk.PKError):
        pk.schedule(cu_d, wl.T, 0)


def test_empty_batch(pk):
    import torch

    qkv = torch.empty((0, 3 * 64), dtype=torch.bfloat16, device="cuda")
    cos = torch.zeros((1, 32), dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros((1,), dtype=torch.int32, device="cuda")
    out, lse = pk.attend(qkv, cos, cos, cu, 1, 0, 0.125)
    assert out.shape == (0, 64) and lse.shape == (1, 0)
    assert pk.last_status() == 0


def test_misaligned_pointer_rejected(pk):
    import torch

    wl = synth.make_lens_workload("align", [8], "bf16", H=1, window=0, seed=0)
    _, cos, sin, cu = device_inputs(wl)
    flat = torch.zeros(wl.T * 192 + 1, dtype=torch.bfloat16, device="cuda")
    qkv = flat[1:].view(wl.T, 192)
    with pytest.raises(pk.PKError) as e:
        pk.attend(qkv, cos, sin, cu, 1, 0, 0.125)
    assert e.value.code == 2


def test_side_streams(pk, orc):
    """Calls on two non-default streams at once each get their own workspace."""
    import torch

    a = synth.make_lens_workload("sa", [200, 3, 77], "bf16", H=2, window=0, seed=11)
    b = synth.make_lens_workload("sb", [5, 300, 64, 9], "bf16", H=2, window=16, seed=12)
    ia, ib = device_inputs(a), device_inputs(b)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    res = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            oa = pk.attend(*ia, a.H, a.window, a.scale, stream=s1)
        with torch.cuda.stream(s2):
            ob = pk.attend(*ib, b.H, b.window, b.scale, stream=s2)
        res.append((oa, ob))
    torch.cuda.synchronize()
    assert pk.last_status(s1) == 0 and pk.last_status(s2) == 0
    wa = orc.attend(a.qkv, a.cos, a.sin, a.cu, a.H, a.window, a.scale, "bf16")
    wb = orc.attend(b.qkv, b.cos, b.sin, b.cu, b.H, b.window, b.scale, "bf16")
    for (oa, ob) in res:
        assert max_err(out_to_f64(oa[0]), wa[0]) <= TOL["bf16"][0]
        assert max_err(out_to_f64(ob[0]), wb[0]) <= TOL["bf16"][0]


def test_window_zero_equals_large_window(pk):
    wl = synth.make_lens_workload("wz", [100, 300, 7], "bf16", H=2, window=0, seed=4)
    inputs = device_inputs(wl)
    o0, l0 = run(pk, wl, 0, inputs)
    o1, l1 = run(pk, wl, 299, inputs)
    o2, l2 = run(pk, wl, 100000, inputs)
    # the same keys are visible; the key ranges of windowed pieces are the same here too
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    assert np.array_equal(o0, o2) and np.array_equal(l0, l2)


def test_constant_values(pk):
    """v constant over each sequence's keys gives out = that constant (P rows sum to l)."""
    wl = synth.make_lens_workload("const", [50, 200, 1, 129], "f16", H=2, window=5, seed=6)
    qkv = wl.qkv.copy()
    rng = np.random.default_rng(3)
    want = np.zeros((wl.T, wl.H * 64))
    for s in range(wl.S):
        a, b = int(wl.cu[s]), int(wl.cu[s + 1])
        for h in range(wl.H):
            c = rng.standard_normal(64).astype(np.float16)
            qkv[a:b, (2 * wl.H + h) * 64:(2 * wl.H + h + 1) * 64] = c
            want[a:b, h * 64:(h + 1) * 64] = c.astype(np.float64)
    wl.qkv = qkv
    o, _ = run(pk, wl)
    assert max_err(o, want) <= TOL["f16"][0]


_STALL_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"]); sys.path.insert(0, os.path.join(os.environ["ROOT"], "tests"))
import numpy as np, torch
import rope_cu_tile_gb300 as pk
import synth
from gpu_util import device_inputs, out_to_f64
from oracle import get
pk.load()
wl = synth.make_lens_workload("stall", [300, 40, 129], "bf16", H=2, window=0, seed=9)
qkv, cos, sin, cu = device_inputs(wl)
os.environ["PK_DEBUG_SKIP_ARRIVE"] = "1"
pk.attend(qkv, cos, sin, cu, wl.H, 0, wl.scale)
torch.cuda.synchronize()
stalled = pk.last_status()
del os.environ["PK_DEBUG_SKIP_ARRIVE"]
out, lse = pk.attend(qkv, cos, sin, cu, wl.H, 0, wl.scale)
torch.cuda.synchronize()
after = pk.last_status()
want_o, want_l = get().attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, 0, wl.scale, "bf16")
eo = float(np.max(np.abs(out_to_f64(out) - want_o)))
el = float(np.max(np.abs(lse.cpu().numpy().astype(np.float64) - want_l)))
print(json.dumps({"stalled": stalled, "after": after, "eo": eo, "el": el}))
"""


def test_withheld_hand_off_times_out_and_the_context_stays_usable():
    """A producer that withholds its first work-item hand-off (test hook): every consumer's
    bounded wait runs out, the call ends with PK_ERR_TIMEOUT in the status word, and the next
    call on the same context is correct. Nothing traps, faults or hangs."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, ROOT=root, PK_TIMEOUT_MS="100")
    env.pop("PK_DEBUG_SKIP_ARRIVE", None)
    p = subprocess.run([sys.executable, "-c", _STALL_SCRIPT], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-3000:]
    r = json.loads(p.stdout.strip().splitlines()[-1])
    assert r["stalled"] == 6, r  # PK_ERR_TIMEOUT
    assert r["after"] == 0, r
    assert r["eo"] <= TOL["bf16"][0] and r["el"] <= TOL["bf16"][1], r


def test_cuda_graph_capture(pk, orc):
    """After a first call has set up the stream's workspace, a call captured in a CUDA graph
    (both kernels, the attention kernel's programmatic launch included) replays correctly."""
    import torch

    wl = synth.make_lens_workload("graph", [200, 7, 129, 64], "bf16", H=2, window=0, seed=13)
    qkv, cos, sin, cu = device_inputs(wl)
    s = torch.cuda.Stream()
    out = torch.empty((wl.T, wl.H * 64), dtype=qkv.dtype, device="cuda")
    lse = torch.empty((wl.H, wl.T), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        pk.attend(qkv, cos, sin, cu, wl.H, 0, wl.scale, out=out, lse=lse, stream=s)
    torch.cuda.synchronize()
    out.fill_(0)
    lse.fill_(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pk.attend(qkv, cos, sin, cu, wl.H, 0, wl.scale, out=out, lse=lse, stream=s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert pk.last_status(s) == 0
    want_o, want_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, 0, wl.scale, "bf16")
    assert max_err(out_to_f64(out), want_o) <= TOL["bf16"][0]
    assert max_err(lse.cpu().numpy().astype(np.float64), want_l) <= TOL["bf16"][1]


def test_capture_that_would_allocate_is_refused(pk):
    """A captured call whose stream has no workspace yet returns PK_ERR_CAPTURE and launches
    nothing; the capture itself stays valid and replays the rest of its work."""
    import torch

    wl = synth.make_lens_workload("graph-fresh", [130, 5], "bf16", H=1, window=0, seed=14)
    qkv, cos, sin, cu = device_inputs(wl)
    out = torch.full((wl.T, wl.H * 64), 7.0, dtype=qkv.dtype, device="cuda")
    lse = torch.zeros((wl.H, wl.T), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    pk.release()  # no stream has a workspace now
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lse.fill_(3.0)
        with pytest.raises(pk.PKError) as err:
            pk.attend(qkv, cos, sin, cu, wl.H, 0, wl.scale, out=out, lse=lse, stream=s)
    assert err.value.code == 10  # PK_ERR_CAPTURE
    g.replay()
    torch.cuda.synchronize()
    assert bool((lse == 3.0).all()) and bool((out == 7.0).all())
