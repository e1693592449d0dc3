"""The C-ABI library: every symbol include/pk.h declares is exported, and host-side argument
checks answer without touching a GPU (no compute call runs here)."""

import ctypes
import os
import re

import pytest

import rope_cu_tile_gb300 as pk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        with open(os.path.join(ROOT, "include", h)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(pk_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from rope_cu_tile_gb300 import build

    build.build()
    return pk.load()


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(pk.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(11):
        assert pk.status_string(code) != "unknown status"
    assert pk.status_string(99) == "unknown status"
    assert lib.pk_version() >= 100


def test_argument_checks_need_no_gpu(lib):
    # rejected before any CUDA call: negative sizes, H < 1, null pointers, misalignment
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)
    null = ctypes.c_void_p(0)
    args = dict(qkv=p, cos=p, sin=p, cu=p, S=1, T=5, H=2, window=0, scale=0.125, out=p, lse=p, stream=null)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return pk.pk_attend(a["qkv"], a["cos"], a["sin"], a["cu"], a["S"], a["T"], a["H"], a["window"],
                            a["scale"], a["out"], a["lse"], a["stream"])

    assert call(S=-1) == 1
    assert call(T=-1) == 1
    assert call(H=0) == 1
    assert call(H=100000) == 1
    assert call(window=-3) == 1
    assert call(S=0) == 1            # T > 0 with no sequences
    assert call(qkv=null) == 1
    assert call(lse=null) == 1
    assert call(qkv=odd) == 2
    assert call(out=odd) == 2
    assert call(T=0, S=0, qkv=null, cos=null, sin=null, cu=null, out=null, lse=null) == 0  # nothing to do
    assert pk.pk_attend_dt(7, p, p, p, p, 1, 5, 2, 0, 0.125, p, p, null) == 1
    assert lib.pk_schedule_capacity(0) == 1
    assert lib.pk_schedule_capacity(64) == 4
    assert lib.pk_schedule_capacity(65) == 7


def test_rope_argument_checks_need_no_gpu(lib):
    # pk_rope rejects bad arguments before any CUDA call
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)
    null = ctypes.c_void_p(0)
    args = dict(dtype=1, x=p, y=p, cos=p, sin=p, P=16, cu=p, S=1, T=5, H=2, dims=64, trad=0, inv=0,
                status=null, stream=null)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return pk.pk_rope(a["dtype"], a["x"], a["y"], a["cos"], a["sin"], a["P"], a["cu"], a["S"], a["T"],
                          a["H"], a["dims"], a["trad"], a["inv"], a["status"], a["stream"])

    assert call(dtype=7) == 1
    assert call(dims=0) == 1
    assert call(dims=7) == 1         # odd
    assert call(dims=66) == 1        # more than the head
    assert call(H=0) == 1
    assert call(S=-1) == 1
    assert call(S=0) == 1            # T > 0 with no sequences
    assert call(P=0) == 1
    assert call(x=null) == 1
    assert call(cos=null) == 1
    assert call(x=odd) == 2          # a 16-bit word is 4 bytes
    assert call(dtype=0, y=ctypes.c_void_p(0x1004)) == 2  # fp32 words are 8 bytes
    assert call(T=0, S=0, x=null, y=null, cos=null, sin=null, cu=null) == 0  # nothing to do


def test_schedule_capacity_matches_oracle(lib, orc):
    for T in (0, 1, 63, 64, 65, 131072, 10**9):
        assert lib.pk_schedule_capacity(T) == orc.schedule_cap(T)


def test_backward_mixed_noalloc_argument_checks_need_no_gpu(lib):
    # rejected before any CUDA call, like pk_attend's
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)
    null = ctypes.c_void_p(0)

    def bwd(**kw):
        a = dict(dtype=1, qkv=p, cos=p, sin=p, cu=p, S=1, T=5, H=2, window=0, scale=0.125, out=p, lse=p,
                 dout=p, dqkv=p, stream=null)
        a.update(kw)
        return pk.pk_attend_backward(a["dtype"], a["qkv"], a["cos"], a["sin"], a["cu"], a["S"], a["T"], a["H"],
                                     a["window"], a["scale"], a["out"], a["lse"], a["dout"], a["dqkv"],
                                     a["stream"])

    assert bwd(dtype=7) == 1
    assert bwd(H=0) == 1
    assert bwd(dout=null) == 1
    assert bwd(dqkv=null) == 1
    assert bwd(dout=odd) == 2
    assert bwd(dqkv=odd) == 2
    assert bwd(qkv=odd) == 2
    assert bwd(T=0, S=0, qkv=null, cos=null, sin=null, cu=null, out=null, lse=null, dout=null, dqkv=null) == 0

    assert pk.pk_attend_mixed(7, p, p, p, p, 1, 5, 2, 0, 0.125, p, p, null) == 1       # out type
    assert pk.pk_attend_mixed(2, odd, p, p, p, 1, 5, 2, 0, 0.125, p, p, null) == 2     # qkv alignment

    def noalloc(**kw):
        a = dict(dtype=1, qkv=p, cos=p, sin=p, cu=p, S=1, T=5, H=2, window=0, scale=0.125, out=p, lse=p,
                 status=null, stream=null)
        a.update(kw)
        return pk.pk_attend_noalloc(a["dtype"], a["qkv"], a["cos"], a["sin"], a["cu"], a["S"], a["T"], a["H"],
                                    a["window"], a["scale"], a["out"], a["lse"], a["status"], a["stream"])

    assert noalloc(dtype=7) == 1
    assert noalloc(T=(1 << 20) + 1) == 9   # PK_ERR_TOO_LARGE past PK_NOALLOC_MAX_T
    assert noalloc(cu=null) == 1
    assert noalloc(status=odd) == 2
    assert noalloc(T=0, S=0, qkv=null, cos=null, sin=null, cu=null, out=null, lse=null) == 0
