"""Pins of the oracle against things other than itself.

Each check returns a list of failure strings (empty = pinned). They are plain functions so
that the same checks run on the oracle proper (tests/test_oracle_pins.py, which expects no
failure) and on builds of the oracle with a planted mistake (which must fail at least one).

What pins what:
  - sdpa:      packed attention is softmax attention over the packed batch with a
               block-diagonal (same sequence) and band (|i - j| <= w) mask; torch's
               scaled_dot_product_attention and logsumexp in float64 compute that directly,
               with q and k rotated here by complex multiplication.
  - rope_*:    the half-split rotation is multiplication of x[t] + i x[t+32] by c + i s;
               it keeps norms and depends only on the relative position.
  - single:    a one-token sequence returns its own v and lse = scale * q.k (angle 0).
  - uniform:   q = 0 gives equal weights: out = mean of the visible v, lse = ln(#visible).
  - consts:    v constant across keys gives out = that constant.
  - probs:     with one-hot values out holds the probabilities: rows sum to one, each
               visible p equals exp(s - lse) and lse lies in [max s, max s + ln n].
  - window:    window 0 equals a window >= max length - 1, bit for bit.
  - permute:   permuting the sequences permutes the rows, bit for bit.
  - widen:     bf16 and fp16 inputs widen exactly (same result as float64 inputs).
  - rows:      the row-at-a-time oracle equals the whole-batch one bit for bit and SDPA to
               1e-12 on every (token, head), empty sequences anywhere in the batch.
  - schedule:  the tile records partition the rows, keep every visible key of each row in
               the key range, keep that range tight, and follow the grouping rule (greedy
               packing of short sequences within 1024-token windows).
  - rope_op:   the standalone rotation reduces to the attention path's for full halves, its
               inverse undoes it, interleaved pairs are the permuted halves, untouched
               features stay, pair lengths stay, and a unit vector turns the right way.
  - backward:  the gradient equals central differences of the forward oracle, and the
               rotated key gradients of a sequence sum to zero.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import synth

D = 64


# ----------------------------------------------------------------------------------------
# independent restatements used by the pins


def complex_rotate(x: np.ndarray, cos_rows: np.ndarray, sin_rows: np.ndarray) -> np.ndarray:
    """x [..., 64] rotated as (x[:32] + i x[32:]) * (c + i s)."""
    z = x[..., :32] + 1j * x[..., 32:]
    r = z * (cos_rows + 1j * sin_rows)
    return np.concatenate([r.real, r.imag], axis=-1)


def token_seq_pos(cu: np.ndarray):
    T = int(cu[-1])
    seq = np.empty(T, dtype=np.int64)
    pos = np.empty(T, dtype=np.int64)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        seq[a:b] = s
        pos[a:b] = np.arange(b - a)
    return seq, pos


def sdpa_reference(qkv64, cos64, sin64, cu, H, window, scale):
    """out [T, H*64], lse [H, T] through torch's SDPA on the whole packed batch (float64)."""
    T = int(cu[-1])
    seq, pos = token_seq_pos(np.asarray(cu))
    same = seq[:, None] == seq[None, :]
    if window > 0:
        same &= np.abs(pos[:, None] - pos[None, :]) <= window
    mask = torch.from_numpy(same)
    out = np.zeros((T, H * D))
    lse = np.zeros((H, T))
    for h in range(H):
        q = complex_rotate(qkv64[:, h * D:(h + 1) * D], cos64[pos], sin64[pos])
        k = complex_rotate(qkv64[:, H * D + h * D:H * D + (h + 1) * D], cos64[pos], sin64[pos])
        v = qkv64[:, 2 * H * D + h * D:2 * H * D + (h + 1) * D]
        qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(a)) for a in (q, k, v))
        o = torch.nn.functional.scaled_dot_product_attention(
            qt[None, None], kt[None, None], vt[None, None], attn_mask=mask[None, None], scale=scale)
        out[:, h * D:(h + 1) * D] = o[0, 0].numpy()
        s = (qt @ kt.T) * scale
        s = s.masked_fill(~mask, -math.inf)
        lse[h] = torch.logsumexp(s, dim=-1).numpy()
    return out, lse


def _f64(wl):
    return (synth.to_f64(wl.qkv, wl.dtype), synth.to_f64(wl.cos, wl.dtype),
            synth.to_f64(wl.sin, wl.dtype))


def _rel_close(a, b, tol):
    return float(np.max(np.abs(a - b))) <= tol * max(1.0, float(np.max(np.abs(b))))


# ----------------------------------------------------------------------------------------
# pins


def pin_sdpa(orc) -> list[str]:
    fails = []
    cases = []
    for w in (0, 8, 64):
        cases.append(("p1_fixture_bf16", synth.p1_fixture("bf16", w)))
    cases.append(("p1_fixture_f32_w8", synth.p1_fixture("f32", 8)))
    cases.append(("tiny_f32", synth.make_config("tiny")))
    rng = np.random.default_rng(123)
    for k, w in enumerate((0, 1, 3, 17)):
        lens = rng.integers(0, 90, size=6)
        lens[0] = max(lens[0], 1)
        wl = synth.make_lens_workload(f"rand{k}", lens, "f16" if k % 2 else "bf16", H=3,
                                      window=w, base=500.0, sigma=1.3, seed=k)
        cases.append((f"rand{k}_w{w}", wl))
    for name, wl in cases:
        qkv64, c64, s64 = _f64(wl)
        want_o, want_l = sdpa_reference(qkv64, c64, s64, wl.cu, wl.H, wl.window, wl.scale)
        got_o, got_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, wl.window, wl.scale,
                                  wl.dtype)
        if not _rel_close(got_o, want_o, 1e-12):
            fails.append(f"sdpa out {name}: {np.max(np.abs(got_o - want_o)):.3e}")
        if not _rel_close(got_l, want_l, 1e-12):
            fails.append(f"sdpa lse {name}: {np.max(np.abs(got_l - want_l)):.3e}")
    return fails


def pin_rope(orc) -> list[str]:
    fails = []
    rng = np.random.default_rng(7)
    P = 300
    c64, s64 = synth.rope_tables(P, 10000.0)
    # arbitrary (c, s) pairs, not only unit ones: the rotation is complex multiplication
    cr = rng.standard_normal((P, 32))
    sr = rng.standard_normal((P, 32))
    for trial in range(20):
        x = rng.standard_normal(64)
        p = int(rng.integers(0, P))
        y = orc.rope(x, p, cr, sr)
        want = complex_rotate(x, cr[p], sr[p])
        if not np.allclose(y, want, rtol=0, atol=1e-13):
            fails.append(f"rope complex p={p}")
            break
        # norm kept with exact tables
        y = orc.rope(x, p, c64, s64)
        if abs(np.linalg.norm(y) - np.linalg.norm(x)) > 1e-13 * np.linalg.norm(x):
            fails.append(f"rope norm p={p}")
            break
    # relative position: rot(a, i) . rot(b, j) = rot(a, i + t) . rot(b, j + t)
    for trial in range(20):
        a, b = rng.standard_normal(64), rng.standard_normal(64)
        i, j, t = (int(v) for v in rng.integers(0, 90, size=3))
        lhs = orc.rope(a, i, c64, s64) @ orc.rope(b, j, c64, s64)
        rhs = orc.rope(a, i + t, c64, s64) @ orc.rope(b, j + t, c64, s64)
        if abs(lhs - rhs) > 1e-11 * (1 + abs(lhs)):
            fails.append(f"rope relative i={i} j={j} t={t}")
            break
    # rounded tables: |  |y|^2 - |x|^2 | <= max|c^2 + s^2 - 1| |x|^2 (+ rounding)
    cb = synth.to_storage(c64, "bf16")
    sb = synth.to_storage(s64, "bf16")
    cbf, sbf = synth.to_f64(cb, "bf16"), synth.to_f64(sb, "bf16")
    for trial in range(10):
        x = rng.standard_normal(64)
        p = int(rng.integers(0, P))
        y = orc.rope(x, p, cb, sb, "f64", "bf16")
        bound = float(np.max(np.abs(cbf[p] ** 2 + sbf[p] ** 2 - 1.0))) * float(x @ x) + 1e-12
        if abs(float(y @ y) - float(x @ x)) > bound * 1.0000001:
            fails.append(f"rope rounded-table norm p={p}")
            break
    return fails


def pin_closed_forms(orc) -> list[str]:
    fails = []
    rng = np.random.default_rng(11)
    H = 2
    scale = 0.125
    # --- single key: a sequence of length 1 returns its v; lse = scale * q.k (angle 0)
    lens = [1, 7, 1, 12, 1]
    wl = synth.make_lens_workload("single", lens, "f32", H=H, window=0, seed=3, scale=scale)
    qkv64 = synth.to_f64(wl.qkv, "f32")
    out, lse = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, H, 0, scale, "f32")
    for s, L in enumerate(lens):
        if L != 1:
            continue
        a = int(wl.cu[s])
        for h in range(H):
            q = qkv64[a, h * D:(h + 1) * D]
            k = qkv64[a, H * D + h * D:H * D + (h + 1) * D]
            v = qkv64[a, 2 * H * D + h * D:2 * H * D + (h + 1) * D]
            if not np.allclose(out[a, h * D:(h + 1) * D], v, rtol=0, atol=1e-15):
                fails.append("single-key out")
            if abs(lse[h, a] - scale * float(q @ k)) > 1e-12:
                fails.append("single-key lse")
    # --- q = 0: uniform weights over the visible keys
    for w in (0, 2, 5):
        lens = [9, 1, 14, 3]
        wl = synth.make_lens_workload("uniform", lens, "f32", H=H, window=w, seed=5, scale=scale)
        qkv = synth.to_f64(wl.qkv, "f32").copy()
        for h in range(H):
            qkv[:, h * D:(h + 1) * D] = 0.0
        out, lse = orc.attend(qkv, wl.cos, wl.sin, wl.cu, H, w, scale, "f64", "f32")
        for s, L in enumerate(lens):
            a0 = int(wl.cu[s])
            for i in range(L):
                lo = 0 if w == 0 else max(0, i - w)
                hi = L if w == 0 else min(L, i + w + 1)
                n = hi - lo
                for h in range(H):
                    v = qkv[a0 + lo:a0 + hi, 2 * H * D + h * D:2 * H * D + (h + 1) * D]
                    if not np.allclose(out[a0 + i, h * D:(h + 1) * D], v.mean(0), rtol=0,
                                       atol=1e-13):
                        fails.append(f"uniform out w={w}")
                    if abs(lse[h, a0 + i] - math.log(n)) > 1e-13:
                        fails.append(f"uniform lse w={w}")
    # --- v constant over the keys of a sequence: out = that constant
    lens = [6, 11, 2]
    wl = synth.make_lens_workload("consts", lens, "f32", H=H, window=3, seed=6, scale=scale)
    qkv = synth.to_f64(wl.qkv, "f32").copy()
    want = np.zeros((wl.T, H * D))
    for s, L in enumerate(lens):
        a, b = int(wl.cu[s]), int(wl.cu[s + 1])
        for h in range(H):
            c = rng.standard_normal(D)
            qkv[a:b, 2 * H * D + h * D:2 * H * D + (h + 1) * D] = c
            want[a:b, h * D:(h + 1) * D] = c
    out, _ = orc.attend(qkv, wl.cos, wl.sin, wl.cu, H, 3, scale, "f64", "f32")
    if not np.allclose(out, want, rtol=0, atol=1e-13):
        fails.append("constant-v out")
    return list(dict.fromkeys(fails))


def pin_probabilities(orc) -> list[str]:
    """One-hot values expose the probabilities of each row."""
    fails = []
    H = 1
    scale = 0.125
    for w in (0, 4):
        lens = [20, 1, 33, 64]
        wl = synth.make_lens_workload("probs", lens, "f32", H=H, window=w, seed=9, scale=scale)
        qkv = synth.to_f64(wl.qkv, "f32").copy()
        c64, s64 = synth.to_f64(wl.cos, "f32"), synth.to_f64(wl.sin, "f32")
        seq, pos = token_seq_pos(wl.cu)
        qkv[:, 2 * D:3 * D] = 0.0
        for a in range(wl.T):
            qkv[a, 2 * D + pos[a]] = 1.0          # v_j = e_j (in-sequence index j < 64)
        out, lse = orc.attend(qkv, wl.cos, wl.sin, wl.cu, H, w, scale, "f64", "f32")
        for s, L in enumerate(lens):
            a0 = int(wl.cu[s])
            q = complex_rotate(qkv[a0:a0 + L, 0:D], c64[:L], s64[:L])
            k = complex_rotate(qkv[a0:a0 + L, D:2 * D], c64[:L], s64[:L])
            sc = scale * (q @ k.T)
            for i in range(L):
                p = out[a0 + i, :L]
                vis = np.ones(L, bool) if w == 0 else (np.abs(np.arange(L) - i) <= w)
                if abs(p.sum() - 1.0) > 1e-12:
                    fails.append(f"probs sum w={w}")
                if np.any(np.abs(p[~vis]) > 0):
                    fails.append(f"probs masked w={w}")
                with np.errstate(over="ignore"):  # a planted mistake may push exp past the range
                    ref = np.exp(sc[i, vis] - lse[0, a0 + i])
                if not np.allclose(p[vis], ref, rtol=1e-11, atol=1e-14):
                    fails.append(f"probs exp(s-lse) w={w}")
                mx = float(sc[i, vis].max())
                if not (mx - 1e-12 <= lse[0, a0 + i] <= mx + math.log(vis.sum()) + 1e-12):
                    fails.append(f"lse bounds w={w}")
    return list(dict.fromkeys(fails))


def pin_window_and_permutation(orc) -> list[str]:
    fails = []
    lens = [13, 40, 2, 27, 1]
    wl = synth.make_lens_workload("wp", lens, "bf16", H=2, window=0, seed=21)
    o0, l0 = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, 2, 0, wl.scale, "bf16")
    o1, l1 = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, 2, max(lens) - 1, wl.scale, "bf16")
    if not (np.array_equal(o0, o1) and np.array_equal(l0, l1)):
        fails.append("window 0 != window >= max L - 1")
    o2, _ = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, 2, 1, wl.scale, "bf16")
    changed = np.any(o2 != o0, axis=1)
    seq, _ = token_seq_pos(wl.cu)
    short = np.isin(seq, [i for i, L in enumerate(lens) if L <= 2])
    if np.any(changed[short]) or not np.all(changed[~short]):
        fails.append("window 1 changes exactly the rows of sequences longer than 2")
    # permutation of the packing order
    perm = [3, 0, 4, 2, 1]
    rows = [np.arange(wl.cu[s], wl.cu[s + 1]) for s in range(len(lens))]
    new_rows = np.concatenate([rows[s] for s in perm])
    lens_p = [lens[s] for s in perm]
    cu_p = synth.cu_from_lens(lens_p)
    for w in (0, 5):
        oa, la = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, 2, w, wl.scale, "bf16")
        ob, lb = orc.attend(wl.qkv[new_rows], wl.cos, wl.sin, cu_p, 2, w, wl.scale, "bf16")
        if not (np.array_equal(ob, oa[new_rows]) and np.array_equal(lb, la[:, new_rows])):
            fails.append(f"permutation w={w}")
    return fails


def pin_widen(orc) -> list[str]:
    fails = []
    for dt in ("bf16", "f16"):
        wl = synth.make_lens_workload("widen", [9, 30], dt, H=2, window=0, seed=2, sigma=3.0)
        oa, la = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, 2, 0, wl.scale, dt)
        qkv64, c64, s64 = _f64(wl)
        if dt == "f16":
            # numpy's own float16 -> float64 conversion
            qkv64 = wl.qkv.astype(np.float64)
            c64, s64 = wl.cos.astype(np.float64), wl.sin.astype(np.float64)
        ob, lb = orc.attend(qkv64, c64, s64, wl.cu, 2, 0, wl.scale, "f64")
        if not (np.array_equal(oa, ob) and np.array_equal(la, lb)):
            fails.append(f"widen {dt}")
    # fp16 specials: subnormal and largest finite
    x = np.zeros(64, dtype=np.float16)
    x[0] = np.float16(6e-8)        # subnormal
    x[1] = np.float16(65504.0)
    x[32] = np.float16(-1.5)
    one = np.ones((1, 32), dtype=np.float16)
    zero = np.zeros((1, 32), dtype=np.float16)
    y = orc.rope(x, 0, one, zero, "f16", "f16")
    if not np.array_equal(y, x.astype(np.float64)):
        fails.append("widen f16 specials")
    return fails


# ----------------------------------------------------------------------------------------
# standalone rotation (the rope op: halves or interleaved pairs, partial dims, inverse)


def _angle_tables(P: int, h: int, rng) -> tuple[np.ndarray, np.ndarray]:
    """cos/sin [P, h] of random angles in f64 (c^2 + s^2 = 1 to rounding)."""
    th = rng.uniform(-np.pi, np.pi, size=(P, h))
    return np.cos(th), np.sin(th)


def pin_rope_op(orc) -> list[str]:
    fails = []
    rng = np.random.default_rng(11)
    H = 2
    lens = [7, 0, 12, 1]
    cu = synth.cu_from_lens(lens)
    T = int(cu[-1])
    seq, pos = token_seq_pos(cu)
    qkv = rng.standard_normal((T, 3 * H * 64))
    # (a) all 64 features in halves, forwards: the pinned rotation of the attention path
    c64, s64 = synth.rope_tables(16, 10000.0)
    y = orc.rope_qkv(qkv, c64, s64, cu, H, 64, False, False)
    for t in range(T):
        for part in range(2):
            for h in range(H):
                a = part * H * 64 + h * 64
                if not np.allclose(y[t, a:a + 64], orc.rope(qkv[t, a:a + 64], int(pos[t]), c64, s64),
                                   rtol=0, atol=1e-13):
                    fails.append("rope op: full halves differ from the attention path's rotation")
    for dims in (64, 32, 6, 2):
        h = dims // 2
        ct, st = _angle_tables(16, h, rng)
        for trad in (False, True):
            fw = orc.rope_qkv(qkv, ct, st, cu, H, dims, trad, False)
            back = orc.rope_qkv(fw, ct, st, cu, H, dims, trad, True)
            # (b) the inverse undoes the forward rotation
            if not np.allclose(back, qkv, rtol=0, atol=1e-12):
                fails.append(f"rope op: inverse(forward) != x (dims {dims}, interleaved {trad})")
            # (e) features past dims and all of v are copied exactly
            qk = fw[:, :2 * H * 64].reshape(T, 2 * H, 64)
            x_qk = qkv[:, :2 * H * 64].reshape(T, 2 * H, 64)
            if not (np.array_equal(qk[..., dims:], x_qk[..., dims:]) and
                    np.array_equal(fw[:, 2 * H * 64:], qkv[:, 2 * H * 64:])):
                fails.append(f"rope op: untouched features changed (dims {dims})")
            # (f) each pair keeps its length
            ia = np.arange(h) * 2 if trad else np.arange(h)
            ib = ia + 1 if trad else ia + h
            n0 = x_qk[..., ia] ** 2 + x_qk[..., ib] ** 2
            n1 = qk[..., ia] ** 2 + qk[..., ib] ** 2
            if not np.allclose(n0, n1, rtol=1e-12, atol=1e-12):
                fails.append(f"rope op: pair lengths changed (dims {dims}, interleaved {trad})")
        # (d) interleaved pairs = halves after moving feature 2j to j and 2j + 1 to j + h
        perm = np.arange(64)
        perm[:dims] = np.concatenate([np.arange(h) * 2, np.arange(h) * 2 + 1])
        xp = qkv.reshape(T, 3 * H, 64)[..., perm].reshape(T, -1)
        tr = orc.rope_qkv(qkv, ct, st, cu, H, dims, True, False).reshape(T, 3 * H, 64)
        hv = orc.rope_qkv(xp, ct, st, cu, H, dims, False, False).reshape(T, 3 * H, 64)
        inv_perm = np.argsort(perm)
        if not np.allclose(tr, hv[..., inv_perm], rtol=0, atol=1e-13):
            fails.append(f"rope op: interleaved pairs are not the permuted halves (dims {dims})")
    # (c) direction: the first feature of pair j turns towards the second (forwards) or away
    dims, h = 8, 4
    ct, st = _angle_tables(16, h, rng)
    for trad in (False, True):
        for j in range(h):
            a = 2 * j if trad else j
            b = a + 1 if trad else j + h
            e = np.zeros((T, 3 * H * 64))
            e[:, a] = 1.0
            fw = orc.rope_qkv(e, ct, st, cu, H, dims, trad, False)
            iv = orc.rope_qkv(e, ct, st, cu, H, dims, trad, True)
            cj, sj = ct[pos, j], st[pos, j]
            if not (np.allclose(fw[:, a], cj, atol=1e-15) and np.allclose(fw[:, b], sj, atol=1e-15) and
                    np.allclose(iv[:, a], cj, atol=1e-15) and np.allclose(iv[:, b], -sj, atol=1e-15)):
                fails.append(f"rope op: rotation direction (pair {j}, interleaved {trad})")
    return list(dict.fromkeys(fails))


# ----------------------------------------------------------------------------------------
# backward


def pin_backward(orc) -> list[str]:
    """The gradient of sum(dout * out) against central differences of the forward oracle, and
    the rows of dS summing to zero (so the rotated key gradients of a sequence sum to zero)."""
    fails = []
    rng = np.random.default_rng(21)
    H = 2
    for lens, window, scale in (([5, 0, 9], 0, 0.37), ([7, 3], 2, -0.6), ([1, 12], 4, 0.125)):
        cu = synth.cu_from_lens(lens)
        T = int(cu[-1])
        c64, s64 = synth.rope_tables(16, 10000.0)
        qkv = rng.standard_normal((T, 3 * H * 64))
        dout = rng.standard_normal((T, H * 64))
        g = orc.attend_backward(qkv, c64, s64, cu, H, window, scale, dout)

        def loss(x):
            o, _ = orc.attend(x, c64, s64, cu, H, window, scale, "f64")
            return float(np.sum(o * dout))

        h = 1e-5
        idx = rng.choice(T * 3 * H * 64, size=120, replace=False)
        for e in idx:
            xp = qkv.copy().reshape(-1)
            xm = qkv.copy().reshape(-1)
            xp[e] += h
            xm[e] -= h
            fd = (loss(xp.reshape(qkv.shape)) - loss(xm.reshape(qkv.shape))) / (2 * h)
            if abs(fd - g.reshape(-1)[e]) > 1e-6 * max(1.0, abs(fd)):
                fails.append(f"backward: d/dqkv[{e}] {g.reshape(-1)[e]:.6g} against central difference {fd:.6g}")
                break
        # sum over a sequence's keys of the rotated key gradients: zero
        seq, pos = token_seq_pos(cu)
        for sq in range(len(lens)):
            rows = np.where(seq == sq)[0]
            for hh in range(H):
                a = H * 64 + hh * 64
                tot = sum(orc.rope(g[t, a:a + 64], int(pos[t]), c64, s64) for t in rows) if len(rows) else 0
                if len(rows) and np.max(np.abs(tot)) > 1e-10 * max(1.0, np.max(np.abs(g))):
                    fails.append("backward: rotated key gradients of a sequence do not sum to zero")
    return list(dict.fromkeys(fails))


# ----------------------------------------------------------------------------------------
# schedule


BR = 128
SHORT = 64
WIN = 1024


def schedule_failures(tiles: np.ndarray, cu: np.ndarray, window: int) -> list[str]:
    """Properties that fix the schedule's records uniquely: the rows partition [0, T) in
    order; long sequences are cut at rows 0, 128, ...; short sequences are packed greedily,
    window by window (a group starts where the previous record of its window's run ended
    and stops only where the next sequence is long, belongs to another window or would
    take it past 128 rows); every key range is the hull of its rows' visible keys."""
    fails = []
    cu = np.asarray(cu, dtype=np.int64)
    S = cu.shape[0] - 1
    T = int(cu[-1])
    lens = np.diff(cu)
    t = tiles.astype(np.int64)
    q0, rows, k0, nk, seq, nseq, kind, kt = (t[:, i] for i in range(8))
    # sorted by q0, rows partition [0, T)
    if t.shape[0]:
        if np.any(np.diff(q0) <= 0):
            fails.append("q0 not increasing")
        if q0[0] != 0 or np.any(q0[1:] != (q0 + rows)[:-1]) or int((q0 + rows)[-1]) != T:
            fails.append("rows do not partition [0, T)")
    elif T != 0:
        fails.append("no tiles")
    if np.any(rows < 1) or np.any(rows > BR):
        fails.append("rows outside [1, 128]")
    if np.any(kt != (nk + 127) // 128):
        fails.append("ktiles")

    def short_in(s, w):
        return 0 <= s < S and lens[s] <= SHORT and int(cu[s]) // WIN == w

    for n in range(t.shape[0]):
        s0, ns = int(seq[n]), int(nseq[n])
        if not (0 <= s0 and s0 + ns <= S and ns >= 1):
            fails.append("member range")
            continue
        if kind[n] == 1:
            members = range(s0, s0 + ns)
            w = int(cu[s0]) // WIN
            if any(not short_in(s, w) for s in members):
                fails.append("group members")
            if int(cu[s0]) != q0[n] or int(cu[s0 + ns]) != q0[n] + rows[n]:
                fails.append("group rows")
            # greedy: the next sequence of the run would not fit ...
            s1 = s0 + ns
            if short_in(s1, w) and int(cu[s1 + 1]) - q0[n] <= BR:
                fails.append("group not maximal")
            # ... and the run's previous sequence closed the previous group
            if short_in(s0 - 1, w) and not (n > 0 and kind[n - 1] == 1 and seq[n - 1] + nseq[n - 1] == s0):
                fails.append("group does not start where the previous one ended")
        elif kind[n] == 0:
            if ns != 1 or lens[s0] <= SHORT:
                fails.append("piece of a short sequence")
            i0 = q0[n] - cu[s0]
            if i0 < 0 or i0 % BR or rows[n] != min(BR, lens[s0] - i0):
                fails.append("piece rows")
        else:
            fails.append("kind")
        if q0[n] < 0 or rows[n] < 1 or q0[n] + rows[n] > T:
            fails.append("rows outside [0, T)")
            continue
        # key range: holds every visible key, and its ends are visible to some row
        a = np.arange(q0[n], q0[n] + rows[n])
        sid = np.searchsorted(cu, a, side="right") - 1
        ss, se = cu[sid], cu[sid + 1]
        lo = ss if window == 0 else np.maximum(ss, a - window)
        hi = se if window == 0 else np.minimum(se, a + window + 1)
        if int(lo.min()) != k0[n] or int(hi.max()) != k0[n] + nk[n]:
            fails.append("key range not the hull of the visible keys")
    # every long sequence is cut entirely into pieces
    for s in range(S):
        if lens[s] > SHORT:
            m = (kind == 0) & (seq == s)
            if int(rows[m].sum()) != lens[s]:
                fails.append("long sequence not covered")
    return list(dict.fromkeys(fails))


def schedule_cases():
    rng = np.random.default_rng(99)
    cases = []
    for name in ("tiny",):
        cases.append((name, synth.make_config(name).cu, 0))
    cases.append(("p1", synth.cu_from_lens(synth.P1_LENS), 8))
    cases.append(("edges", synth.cu_from_lens([0, 1, 63, 64, 65, 127, 128, 129, 0, 0, 255, 256, 257,
                                               1, 0, 64, 64, 2]), 0))
    cases.append(("edges_w", synth.cu_from_lens([0, 1, 63, 64, 65, 127, 128, 129, 0, 0, 255, 256,
                                                  257, 1, 0, 64, 64, 2]), 3))
    cases.append(("empty_all", synth.cu_from_lens([0, 0, 0]), 0))
    cases.append(("one_token", synth.cu_from_lens([1]), 0))
    for k in range(6):
        lens = rng.integers(0, 300 if k % 2 else 40, size=int(rng.integers(1, 60)))
        cases.append((f"rand{k}", synth.cu_from_lens(lens), int(rng.choice([0, 1, 4, 64, 200]))))
    # greedy packing at exactly 128 rows, and one row over
    cases.append(("fill128", synth.cu_from_lens([64, 64, 1, 40, 40, 48, 1, 0, 127, 1]), 0))
    # several windows of dense short sequences (groups close at window ends)
    cases.append(("win_dense", synth.cu_from_lens(rng.integers(0, 20, size=400)), 0))
    cases.append(("win_dense_w", synth.cu_from_lens(rng.integers(0, 20, size=400)), 5))
    # a sequence and empty ones starting exactly at a window boundary, a short one straddling
    # the next, a long one over several windows, single-token sequences (128-member groups)
    edge = [1000, 24, 0, 0, 10, 1000, 20, 40, 3000] + [1] * 300 + [64] * 20
    cases.append(("win_edges", synth.cu_from_lens(edge), 0))
    cases.append(("win_edges_w", synth.cu_from_lens(edge), 100))
    return cases


def pin_attend_rows(orc) -> list[str]:
    """oracle_attend_rows (the row-at-a-time form, for spot checks of large outputs) finds each
    token's sequence by a search over cu; every (token, head) it returns must equal the
    whole-batch oracle bit for bit, and torch's SDPA over the packed batch to 1e-12, with
    empty sequences at the start, between others and at the end, and windows 0, 1 and 64.
    The tables have a few rows more than the longest sequence."""
    fails = []
    rng = np.random.default_rng(2024)
    layouts = [
        ("lead_empty", [0, 0, 7, 1, 30]),
        ("between_empty", [5, 0, 0, 9, 0, 1, 0, 12]),
        ("trail_empty", [17, 3, 0, 0]),
        ("all_single", [1, 1, 0, 1, 1]),
        ("mixed", [0, 70, 0, 2, 0, 0, 33, 1, 0]),
    ]
    for name, lens in layouts:
        for w in (0, 1, 64):
            wl = synth.make_lens_workload(f"{name}_w{w}", lens, "bf16", H=3, window=w, base=700.0,
                                          seed=len(lens) + w, P=max(lens) + 8)
            T = wl.T
            tok = np.repeat(np.arange(T, dtype=np.int64), wl.H)
            hd = np.tile(np.arange(wl.H, dtype=np.int32), T)
            perm = rng.permutation(tok.shape[0])
            tok, hd = tok[perm], hd[perm]
            got_o, got_l = orc.attend_rows(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, wl.window, wl.scale,
                                           wl.dtype, tok, hd)
            full_o, full_l = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, wl.window, wl.scale, wl.dtype)
            want_o = np.stack([full_o[t, h * D:(h + 1) * D] for t, h in zip(tok, hd)])
            want_l = np.array([full_l[h, t] for t, h in zip(tok, hd)])
            if not (np.array_equal(got_o, want_o) and np.array_equal(got_l, want_l)):
                fails.append(f"rows vs whole batch {name} w{w}: "
                             f"{np.max(np.abs(got_o - want_o)):.3e} / {np.max(np.abs(got_l - want_l)):.3e}")
            qkv64, c64, s64 = _f64(wl)
            ref_o, ref_l = sdpa_reference(qkv64, c64, s64, wl.cu, wl.H, wl.window, wl.scale)
            ro = np.stack([ref_o[t, h * D:(h + 1) * D] for t, h in zip(tok, hd)])
            rl = np.array([ref_l[h, t] for t, h in zip(tok, hd)])
            if not (_rel_close(got_o, ro, 1e-12) and _rel_close(got_l, rl, 1e-12)):
                fails.append(f"rows vs sdpa {name} w{w}")
    return fails


def pin_schedule(orc) -> list[str]:
    fails = []
    for name, cu, w in schedule_cases():
        tiles = orc.schedule(cu, w)
        for f in schedule_failures(tiles, cu, w):
            fails.append(f"{name}: {f}")
    return fails


ALL_PINS = (pin_sdpa, pin_rope, pin_closed_forms, pin_probabilities, pin_window_and_permutation,
            pin_widen, pin_schedule, pin_rope_op, pin_backward, pin_attend_rows)


def all_failures(orc) -> list[str]:
    out = []
    for pin in ALL_PINS:
        out += [f"{pin.__name__}: {f}" for f in pin(orc)]
    return out
