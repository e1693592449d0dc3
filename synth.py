"""Seeded synthetic inputs for packed RoPE attention.

This module is the only code shared by the CUDA path's callers (tests, bench) and the
oracle's callers. It draws sequence lengths, the packed qkv projection and the rotary
tables; it holds none of the attention arithmetic (no rotation, no scores, no softmax).

Workloads follow the five configurations the method is measured on (tiny, encoder-base
global layer, encoder-base local layer, long packed batch, short-sequence stress), plus
the fixture of the packed.rs test module (hanzo-kernel 0.2.42, `mod tests`: `rnd`,
`tables`, `LENS`, `HEADS`).

Storage conventions (packed.rs module doc, "qkv [T, 3·H·D]" ... "cos, sin [P, D/2]"):
  qkv  [T, 3*H*64]  q block | k block | v block, head h at columns h*64 of each block
  cos, sin [P, 32]  indexed by position within a sequence
  cu   [S+1] uint32 first token of each sequence, cu[S] = T

bf16 arrays are carried as uint16 bit patterns (numpy has no bfloat16); fp16 as
numpy.float16; fp32 as numpy.float32.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

D = 64
HALF = D // 2

DTYPES = ("f32", "bf16", "f16")


# ----------------------------------------------------------------------------------------
# rounding helpers (storage only)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32/float64 values -> storage array of `dtype` ('f32', 'bf16' as uint16 bits, 'f16')."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    if dtype == "f16":
        return np.ascontiguousarray(x, dtype=np.float16)
    raise ValueError(dtype)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array -> float64, exactly."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def elem_size(dtype: str) -> int:
    return 4 if dtype == "f32" else 2


# ----------------------------------------------------------------------------------------
# rotary tables


def rope_tables(p: int, base: float) -> tuple[np.ndarray, np.ndarray]:
    """cos/sin [p, 32] in float64: angle(pos, t) = pos * base^(-2t/64).

    The table recipe of packed.rs `mod tests` fn `tables` (angle in f64, then rounded to the
    storage type by the caller) and of plan.rs fn `rope_tables` (base 160000 for the
    global-layer configurations).
    """
    pos = np.arange(p, dtype=np.float64)[:, None]
    t = np.arange(HALF, dtype=np.float64)[None, :]
    ang = pos / np.power(base, 2.0 * t / D)
    return np.cos(ang), np.sin(ang)


def rope_tables_dims(p: int, dims: int, base: float) -> tuple[np.ndarray, np.ndarray]:
    """cos/sin [p, dims/2] in float64 for a rotation of the first `dims` features:
    angle(pos, j) = pos * base^(-2j/dims) (the rope op's default frequencies)."""
    pos = np.arange(p, dtype=np.float64)[:, None]
    j = np.arange(dims // 2, dtype=np.float64)[None, :]
    ang = pos / np.power(base, 2.0 * j / dims)
    return np.cos(ang), np.sin(ang)


# ----------------------------------------------------------------------------------------
# workloads


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str            # 'f32' | 'bf16' | 'f16'
    H: int
    window: int           # 0: every key of the sequence; w > 0: |i - j| <= w
    scale: float
    base: float
    lens: np.ndarray      # int64 [S]
    cu: np.ndarray        # uint32 [S+1]
    qkv: np.ndarray       # storage [T, 3*H*64]
    cos: np.ndarray       # storage [P, 32]
    sin: np.ndarray       # storage [P, 32]

    @property
    def S(self) -> int:
        return int(self.lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.cu[-1])

    @property
    def P(self) -> int:
        return int(self.cos.shape[0])


CONFIG_NAMES = ("tiny", "global", "local", "long", "short")

CONFIG_TEXT = {
    "tiny": "S=3 lengths 37,64,150 (T=251), H=2, fp32 qkv ~N(0,1), RoPE base 10000, scale 1/8, window 0",
    "global": "encoder-base global layer: H=12, bf16 qkv ~N(0,1), 64 sequences U{32..512}, base 160000, window 0",
    "local": "encoder-base local layer: H=12, bf16, 16 sequences U{1024..8192}, base 10000, window 64",
    "long": "long packed batch: H=16, bf16, lengths lognormal(median 256, sigma 1) clipped [1,8192] "
            "packed to T=131072, base 160000, window 0",
    "short": "short-sequence stress: H=12, fp16 qkv ~N(0,1.5), lengths U{1..16} packed to T=65536, "
             "base 10000, window 4",
}


def cu_from_lens(lens) -> np.ndarray:
    lens = np.asarray(lens, dtype=np.int64)
    cu = np.zeros(lens.shape[0] + 1, dtype=np.int64)
    np.cumsum(lens, out=cu[1:])
    if cu[-1] >= 2**32:
        raise ValueError("too many tokens for uint32 offsets")
    return cu.astype(np.uint32)


def _pack_to(draw, total: int) -> np.ndarray:
    """Draw lengths one at a time until they sum to >= total; cut the last so the sum is total."""
    out = []
    acc = 0
    while acc < total:
        L = int(draw())
        out.append(L)
        acc += L
    out[-1] -= acc - total
    if out[-1] == 0:
        out.pop()
    return np.asarray(out, dtype=np.int64)


def config_lens(name: str, rng: np.random.Generator) -> np.ndarray:
    if name == "tiny":
        return np.asarray([37, 64, 150], dtype=np.int64)
    if name == "global":
        return rng.integers(32, 512, size=64, endpoint=True).astype(np.int64)
    if name == "local":
        return rng.integers(1024, 8192, size=16, endpoint=True).astype(np.int64)
    if name == "long":
        def draw():
            return min(8192, max(1, int(round(math.exp(math.log(256.0) + rng.standard_normal())))))
        return _pack_to(draw, 131072)
    if name == "short":
        return _pack_to(lambda: rng.integers(1, 16, endpoint=True), 65536)
    raise ValueError(name)


_PARAMS = {
    # name: (dtype, H, window, base, sigma)
    "tiny": ("f32", 2, 0, 10000.0, 1.0),
    "global": ("bf16", 12, 0, 160000.0, 1.0),
    "local": ("bf16", 12, 64, 10000.0, 1.0),
    "long": ("bf16", 16, 0, 160000.0, 1.0),
    "short": ("f16", 12, 4, 10000.0, 1.5),
}


def make_lens_workload(name: str, lens, dtype: str, H: int, window: int, base: float = 10000.0,
                       sigma: float = 1.0, seed: int = 0, scale: float | None = None,
                       P: int | None = None) -> Workload:
    """A workload with given lengths: qkv ~ N(0, sigma) rounded to `dtype`, tables of P rows."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    cu = cu_from_lens(lens)
    T = int(cu[-1])
    x = rng.standard_normal((T, 3 * H * D), dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    qkv = to_storage(x, dtype)
    if P is None:
        P = max(1, int(lens.max()) if lens.size else 1)
    c, s = rope_tables(P, base)
    return Workload(name=name, dtype=dtype, H=H, window=window,
                    scale=(1.0 / math.sqrt(D)) if scale is None else scale, base=base,
                    lens=lens, cu=cu, qkv=qkv, cos=to_storage(c, dtype), sin=to_storage(s, dtype))


def make_config(name: str, seed: int | None = None) -> Workload:
    """One of the five measured configurations; seed defaults to the configuration's index."""
    if seed is None:
        seed = CONFIG_NAMES.index(name)
    dtype, H, window, base, sigma = _PARAMS[name]
    rng = np.random.default_rng(seed)
    lens = config_lens(name, rng)
    cu = cu_from_lens(lens)
    T = int(cu[-1])
    x = rng.standard_normal((T, 3 * H * D), dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    qkv = to_storage(x, dtype)
    del x
    c, s = rope_tables(int(lens.max()), base)
    return Workload(name=name, dtype=dtype, H=H, window=window, scale=1.0 / 8.0, base=base,
                    lens=lens, cu=cu, qkv=qkv, cos=to_storage(c, dtype), sin=to_storage(s, dtype))


# ----------------------------------------------------------------------------------------
# the packed.rs test fixture


P1_LENS = (5, 40, 1, 33, 70)
P1_HEADS = 2


def xorshift_rnd(n: int, seed: int, amp: float) -> np.ndarray:
    """packed.rs `mod tests` fn `rnd`: xorshift64 (shifts 13, 7, 17), value
    ((s mod 20001) / 10000 - 1) * amp in float32."""
    out = np.empty(n, dtype=np.float32)
    s = seed & 0xFFFFFFFFFFFFFFFF
    mask = 0xFFFFFFFFFFFFFFFF
    for i in range(n):
        s ^= (s << 13) & mask
        s ^= s >> 7
        s ^= (s << 17) & mask
        out[i] = (np.float32(s % 20001) / np.float32(10000.0) - np.float32(1.0)) * np.float32(amp)
    return out


def p1_fixture(dtype: str = "bf16", window: int = 0) -> Workload:
    """The packed.rs test inputs: LENS = [5, 40, 1, 33, 70], HEADS = 2, rnd(seed 7, amp 1),
    tables(128) with base 10000, scale 64^-0.5; rounded to `dtype`."""
    lens = np.asarray(P1_LENS, dtype=np.int64)
    cu = cu_from_lens(lens)
    T = int(cu[-1])
    x = xorshift_rnd(T * 3 * P1_HEADS * D, 7, 1.0).reshape(T, 3 * P1_HEADS * D)
    c, s = rope_tables(128, 10000.0)
    c32, s32 = c.astype(np.float32), s.astype(np.float32)
    return Workload(name="p1_fixture", dtype=dtype, H=P1_HEADS, window=window,
                    scale=float(np.float32(D) ** np.float32(-0.5)), base=10000.0, lens=lens, cu=cu,
                    qkv=to_storage(x, dtype), cos=to_storage(c32, dtype), sin=to_storage(s32, dtype))


# ----------------------------------------------------------------------------------------
# work accounting (metric definitions, not the method)


def visible_pairs(lens, window: int) -> int:
    """Number of (query, key) pairs of one head that the window lets through."""
    total = 0
    for L in np.asarray(lens, dtype=np.int64).tolist():
        if L <= 0:
            continue
        if window <= 0 or window >= L - 1:
            total += L * L
        else:
            w = window
            # row i sees min(L-1, i+w) - max(0, i-w) + 1 keys
            i = np.arange(L, dtype=np.int64)
            total += int((np.minimum(L - 1, i + w) - np.maximum(0, i - w) + 1).sum())
    return total


def algorithmic_bytes(wl: Workload) -> int:
    """qkv read once + out written + lse written + tables read + cu read."""
    e = elem_size(wl.dtype)
    T, H = wl.T, wl.H
    return T * 3 * H * D * e + T * H * D * e + 4 * H * T + 2 * wl.P * HALF * e + 4 * (wl.S + 1)
