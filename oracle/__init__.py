"""fp64 CPU oracle for packed RoPE attention: TEST INFRASTRUCTURE ONLY.

Only the tests, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg may import
this package. The product path (the CUDA library and its binding) never does.

The arithmetic lives in `oracle.c` (plain C, fp64); this module compiles it with gcc and
marshals numpy arrays to it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DT_CODES = {"f64": 0, "f32": 1, "bf16": 2, "f16": 3}
REC = 8  # uint32 fields per tile record


def compile_oracle(out_path: str = _LIB, mutant: int = 0) -> str:
    """Compile oracle.c into a shared library (mutant > 0 plants a known mistake)."""
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", out_path, _SRC, "-lpthread", "-lm"]
    if mutant:
        cmd.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    subprocess.run(cmd, check=True)
    return out_path


def build() -> str:
    if (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_oracle(_LIB)
    return _LIB


class Oracle:
    """ctypes front of one compiled oracle library."""

    def __init__(self, path: str | None = None):
        self.lib = ctypes.CDLL(path or build())
        L = self.lib
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oracle_attend.argtypes = [vp, i32, vp, vp, i32, vp, i32, i64, i32, i32, dbl, vp, vp, i32]
        L.oracle_attend.restype = i32
        L.oracle_attend_rows.argtypes = [vp, i32, vp, vp, i32, vp, i32, i64, i32, i32, dbl,
                                         vp, vp, i64, vp, vp, i32]
        L.oracle_attend_rows.restype = i32
        L.oracle_rope.argtypes = [vp, i32, i64, vp, vp, i32, vp]
        L.oracle_rope.restype = None
        L.oracle_rope_qkv.argtypes = [vp, i32, vp, vp, i32, i64, vp, i32, i64, i32, i32, i32, i32, vp]
        L.oracle_rope_qkv.restype = i32
        L.oracle_attend_backward.argtypes = [vp, i32, vp, vp, i32, vp, i32, i64, i32, i32, dbl, vp, i32, vp]
        L.oracle_attend_backward.restype = i32
        L.oracle_schedule.argtypes = [vp, i32, i64, i32, vp, i64, ctypes.POINTER(i64)]
        L.oracle_schedule.restype = i32
        L.oracle_schedule_cap.argtypes = [i64]
        L.oracle_schedule_cap.restype = i64
        L.oracle_threads.argtypes = []
        L.oracle_threads.restype = i32

    @staticmethod
    def _arr(a, dtype):
        a = np.ascontiguousarray(a)
        code = DT_CODES[dtype]
        if dtype in ("bf16", "f16"):
            a = np.ascontiguousarray(a).view(np.uint16)
        elif dtype == "f32":
            a = a.astype(np.float32, copy=False)
        else:
            a = a.astype(np.float64, copy=False)
        return a, code

    def threads(self) -> int:
        return int(self.lib.oracle_threads())

    def attend(self, qkv, cos, sin, cu, H: int, window: int, scale: float, dtype: str,
               table_dtype: str | None = None, nthreads: int = 0):
        """out [T, H*64] and lse [H, T] in float64."""
        table_dtype = table_dtype or dtype
        q, dq = self._arr(qkv, dtype)
        c, dc = self._arr(cos, table_dtype)
        s, _ = self._arr(sin, table_dtype)
        cu = np.ascontiguousarray(cu, dtype=np.uint32)
        S = cu.shape[0] - 1
        T = int(cu[-1]) if S >= 0 else 0
        out = np.zeros((T, H * 64), dtype=np.float64)
        lse = np.zeros((H, T), dtype=np.float64)
        rc = self.lib.oracle_attend(q.ctypes.data, dq, c.ctypes.data, s.ctypes.data, dc,
                                    cu.ctypes.data, S, T, H, window, float(scale),
                                    out.ctypes.data, lse.ctypes.data, nthreads)
        if rc != 0:
            raise ValueError(f"oracle_attend failed ({rc})")
        return out, lse

    def attend_rows(self, qkv, cos, sin, cu, H: int, window: int, scale: float, dtype: str,
                    tokens, heads, table_dtype: str | None = None, nthreads: int = 0):
        """out rows [n, 64] and lse [n] for the given (token, head) pairs, in float64."""
        table_dtype = table_dtype or dtype
        q, dq = self._arr(qkv, dtype)
        c, dc = self._arr(cos, table_dtype)
        s, _ = self._arr(sin, table_dtype)
        cu = np.ascontiguousarray(cu, dtype=np.uint32)
        S = cu.shape[0] - 1
        T = int(cu[-1])
        tok = np.ascontiguousarray(tokens, dtype=np.int64)
        hd = np.ascontiguousarray(heads, dtype=np.int32)
        n = tok.shape[0]
        out = np.zeros((n, 64), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        rc = self.lib.oracle_attend_rows(q.ctypes.data, dq, c.ctypes.data, s.ctypes.data, dc,
                                         cu.ctypes.data, S, T, H, window, float(scale),
                                         tok.ctypes.data, hd.ctypes.data, n,
                                         out.ctypes.data, lse.ctypes.data, nthreads)
        if rc != 0:
            raise ValueError(f"oracle_attend_rows failed ({rc})")
        return out, lse

    def rope(self, x, pos: int, cos, sin, dtype: str = "f64", table_dtype: str = "f64"):
        xa, dx = self._arr(np.asarray(x).reshape(64), dtype)
        c, dc = self._arr(cos, table_dtype)
        s, _ = self._arr(sin, table_dtype)
        y = np.zeros(64, dtype=np.float64)
        self.lib.oracle_rope(xa.ctypes.data, dx, int(pos), c.ctypes.data, s.ctypes.data, dc,
                             y.ctypes.data)
        return y

    def rope_qkv(self, qkv, cos, sin, cu, H: int, dims: int, traditional: bool, inverse: bool,
                 dtype: str = "f64", table_dtype: str = "f64"):
        """The standalone rotation of every q and k head vector of qkv [T, 3 H 64] (v copied),
        f64 [T, 3 H 64]; tables cos/sin [P, dims / 2]."""
        cu = np.ascontiguousarray(cu, dtype=np.uint32)
        S = cu.shape[0] - 1
        T = int(cu[-1])
        xa, dx = self._arr(np.asarray(qkv).reshape(T, 3 * H * 64) if T else np.zeros((0, 3 * H * 64)), dtype)
        c, dc = self._arr(cos, table_dtype)
        s, _ = self._arr(sin, table_dtype)
        P = int(np.asarray(cos).shape[0])
        y = np.zeros((T, 3 * H * 64), dtype=np.float64)
        rc = self.lib.oracle_rope_qkv(xa.ctypes.data, dx, c.ctypes.data, s.ctypes.data, dc, P,
                                      cu.ctypes.data, S, T, H, int(dims), int(bool(traditional)),
                                      int(bool(inverse)), y.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_rope_qkv: bad arguments")
        return y

    def attend_backward(self, qkv, cos, sin, cu, H: int, window: int, scale: float, dout, dtype: str = "f64",
                        table_dtype: str | None = None, dout_dtype: str | None = None):
        """dqkv [T, 3 H 64] in f64: the gradient of sum(dout * out) with respect to qkv."""
        cu = np.ascontiguousarray(cu, dtype=np.uint32)
        S = cu.shape[0] - 1
        T = int(cu[-1])
        q, dq_ = self._arr(qkv, dtype)
        c, dc = self._arr(cos, table_dtype or dtype)
        s, _ = self._arr(sin, table_dtype or dtype)
        g, dg = self._arr(dout, dout_dtype or dtype)
        y = np.zeros((T, 3 * H * 64), dtype=np.float64)
        rc = self.lib.oracle_attend_backward(q.ctypes.data, dq_, c.ctypes.data, s.ctypes.data, dc, cu.ctypes.data,
                                             S, T, H, window, float(scale), g.ctypes.data, dg, y.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle_attend_backward -> {rc}")
        return y

    def schedule(self, cu, window: int):
        """Tile records [NT, 8] uint32 (q0, rows, k0, nk, seq, nseq, kind, ktiles)."""
        cu = np.ascontiguousarray(cu, dtype=np.uint32)
        S = cu.shape[0] - 1
        T = int(cu[-1])
        cap = int(self.lib.oracle_schedule_cap(T))
        tiles = np.zeros((cap, REC), dtype=np.uint32)
        nt = ctypes.c_int64(0)
        rc = self.lib.oracle_schedule(cu.ctypes.data, S, T, window, tiles.ctypes.data, cap,
                                      ctypes.byref(nt))
        if rc != 0:
            raise ValueError("oracle_schedule: malformed cu")
        if nt.value > cap:
            raise RuntimeError("schedule cap exceeded")
        return tiles[: nt.value].copy()

    def schedule_cap(self, T: int) -> int:
        return int(self.lib.oracle_schedule_cap(T))


_default: Oracle | None = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
