"""A discrete-event model of the hand-off protocol inside the tensor-core attention kernel
(rope_cu_tile_gb300/csrc/pk_attend_tc.cu): two MMA issuers (one per query tile X of a work
item), four softmax warps per query tile, a tensor pipe, and the mbarriers between them.

mbarriers follow the PTX rule the kernel relies on: a wait names the parity of the phase it
waits for, and it passes when the barrier's current (incomplete) phase has the other parity.
That test is only sound while the waiter is never two phases behind or ahead of the barrier, and
that is what this model checks, under random timings: every wait that passes is compared with
the event it was meant to observe (a "false pass" otherwise), and a state where every role waits
and nothing is in flight is a deadlock.

Modelled: per query tile, the S products (S = Q K^T of one key tile) and PV products in the
issuers' program order (S of tile t, then PV of tile t - 1); the softmax warps' waits and
arrivals; the tensor pipe as one queue in issue order, a commit arriving once every earlier MMA
of its thread has completed. Not modelled: the K / V rings, the Q buffers and the item hand-off,
which only add waits.

Protocols:
- one_buffer: the kernel as built. One score buffer per query tile; S(t) waits until that tile's
  softmax warps have loaded the last half of S(t - 1) (`s_consumed`).
- three_buffers: three score buffers shared by both query tiles, P written over the buffer its S
  came from, products numbered in stream order (A before B at a tile) and product n using
  buffer n % 3; S(n) waits for the PV of product n - 3 (`s_free`), for the softmax to have seen
  the tile's previous S complete (`s_taken`), and for product n - 1 to have been issued (a
  counter that only grows).
- three_buffers_unordered, three_buffers_no_taken: the same without the last two waits, or
  without `s_taken`; both are unsound and the model must find it.
"""
import random

import pytest

PROTOCOLS = ("one_buffer", "three_buffers", "three_buffers_unordered", "three_buffers_no_taken")


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0  # index of the current, incomplete phase

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.phase & 1) != parity


class Model:
    def __init__(self, protocol, items, seed):
        self.protocol = protocol
        self.items = items
        self.rng = random.Random(seed)
        self.now = 0
        self.events = []  # (time, action)
        self.pipe_free = 0
        self.last_done = {}
        self.s_done, self.pv_done_set = set(), set()
        self.taken, self.consumed, self.written = {}, {}, {}
        self.issued = 0
        b = {}
        for x in (0, 1):
            b[("s_full", x)] = Barrier(1)
            b[("s_consumed", x)] = Barrier(4)
            b[("s_taken", x)] = Barrier(4)
            b[("p_ready", x)] = Barrier(4)
            b[("pv_done", x)] = Barrier(1)
        for k in range(3):
            b[("s_free", k)] = Barrier(1)
        self.bar = b
        # products in stream order: (item, tile, query tile) -> n
        self.number = {}
        n = 0
        for i, (a1, b0, b1, ns) in enumerate(items):
            for t in range(ns):
                if t < a1:
                    self.number[(i, t, 0)] = n
                    n += 1
                if b0 <= t < b1:
                    self.number[(i, t, 1)] = n
                    n += 1

    def mma(self, who, cycles, done):
        end = max(self.now + 1, self.pipe_free) + cycles
        self.pipe_free = end
        self.last_done[who] = end
        self.events.append((end, done))

    def commit(self, who, key):
        end = max(self.last_done.get(who, 0), self.now) + 1
        self.events.append((end, self.bar[key].arrive))

    def wait(self, key, parity, observed, what):
        bar = self.bar[key]
        return ("wait", lambda: bar.passes(parity), observed, what)


def issuer(m, x):
    proto = m.protocol
    shared = proto != "one_buffer"
    ordered = proto in ("three_buffers", "three_buffers_no_taken")
    with_taken = proto == "three_buffers"
    n_s = 0  # S products of this query tile so far
    n_p = 0  # PV products
    prev = None
    for i, (a1, b0, b1, ns) in enumerate(m.items):
        lo, hi = (0, a1) if x == 0 else (b0, b1)
        for t in range(ns + 1):
            if t < ns and lo <= t < hi:
                n = m.number[(i, t, x)]
                if not shared:
                    if prev is not None:
                        yield m.wait(("s_consumed", x), (n_s - 1) & 1,
                                     lambda p=prev: m.consumed.get(p, 0) == 4, f"S{prev} read")
                else:
                    if with_taken and prev is not None:
                        yield m.wait(("s_taken", x), (n_s - 1) & 1,
                                     lambda p=prev: m.taken.get(p, 0) == 4, f"S{prev} seen")
                    if ordered:
                        yield ("wait", lambda n=n: m.issued == n, lambda: True, "turn")
                    if n >= 3:
                        yield m.wait(("s_free", n % 3), (n // 3 - 1) & 1,
                                     lambda n=n: (n - 3) in m.pv_done_set, f"PV{n - 3} done (for S{n})")
                yield ("delay", m.rng.randint(1, 30))
                m.mma(x, m.rng.randint(200, 400), lambda n=n: m.s_done.add(n))
                m.commit(x, ("s_full", x))
                if ordered:
                    m.issued = n + 1
                n_s += 1
                prev = n
            if t >= 1 and lo <= t - 1 < hi:
                n = m.number[(i, t - 1, x)]
                yield m.wait(("p_ready", x), n_p & 1, lambda n=n: m.written.get(n, 0) == 4, f"P{n} written")
                n_p += 1
                yield ("delay", m.rng.randint(1, 30))
                m.mma(x, m.rng.randint(300, 600), lambda n=n: m.pv_done_set.add(n))
                m.commit(x, ("pv_done", x))
                if shared:
                    m.commit(x, ("s_free", n % 3))


def softmax_warp(m, x):
    shared = m.protocol != "one_buffer"
    with_taken = m.protocol == "three_buffers"
    n_s = n_pv = 0

    def slow(lo, hi, p=0.05):
        return m.rng.randint(2000, 8000) if m.rng.random() < p else m.rng.randint(lo, hi)

    for i, (a1, b0, b1, ns) in enumerate(m.items):
        lo, hi = (0, a1) if x == 0 else (b0, b1)
        for j in range(lo, hi):
            n = m.number[(i, j, x)]
            yield m.wait(("s_full", x), n_s & 1, lambda n=n: n in m.s_done, f"S{n} complete")
            n_s += 1
            if with_taken:
                m.taken[n] = m.taken.get(n, 0) + 1
                m.bar[("s_taken", x)].arrive()
            yield ("delay", slow(100, 900))  # pass 1, and the load of the last half of S
            if not shared:
                m.consumed[n] = m.consumed.get(n, 0) + 1
                m.bar[("s_consumed", x)].arrive()
            if j > lo:
                p = m.number[(i, j - 1, x)]
                yield m.wait(("pv_done", x), n_pv & 1, lambda p=p: p in m.pv_done_set, f"PV{p} done")
                n_pv += 1
            yield ("delay", m.rng.randint(100, 900))  # probabilities, P written
            m.written[n] = m.written.get(n, 0) + 1
            m.bar[("p_ready", x)].arrive()
            yield ("delay", slow(1, 60, 0.02))  # until the next wait (descheduling included)
        if hi > lo:
            p = m.number[(i, hi - 1, x)]
            yield m.wait(("pv_done", x), n_pv & 1, lambda p=p: p in m.pv_done_set, f"PV{p} done (epilogue)")
            n_pv += 1
            yield ("delay", m.rng.randint(50, 300))


def simulate(protocol, items, seed):
    """None if every wait was sound and the model ran to the end, else what went wrong."""
    m = Model(protocol, items, seed)
    roles = [issuer(m, 0), issuer(m, 1)] + [softmax_warp(m, x) for x in (0, 1) for _ in range(4)]
    op = [next(r, None) for r in roles]
    wake = [None] * len(roles)
    while True:
        moved = False
        for k in m.rng.sample(range(len(roles)), len(roles)):
            while op[k] is not None:
                if op[k][0] == "delay":
                    if wake[k] is None:
                        wake[k] = m.now + op[k][1]
                    if m.now < wake[k]:
                        break
                    wake[k] = None
                else:
                    _, ready, observed, what = op[k]
                    if not ready():
                        break
                    if not observed():
                        return f"false pass at t={m.now}: {what}"
                op[k] = next(roles[k], None)
                moved = True
        if all(o is None for o in op):
            return None
        if not moved:
            future = [t for t, _ in m.events] + [w for w in wake if w is not None]
            if not future:
                waits = [o[3] for o in op if o is not None]
                return f"deadlock at t={m.now}: " + "; ".join(waits)
            m.now = max(m.now + 1, min(future))
        else:
            m.now += 1
        due = sorted((e for e in m.events if e[0] <= m.now), key=lambda e: e[0])
        m.events = [e for e in m.events if e[0] > m.now]
        for _, act in due:
            act()


def random_items(rng, k):
    """Work items as (a1, b0, b1, stream tiles): A uses stream tiles [0, a1), B uses [b0, b1)."""
    items = []
    for _ in range(k):
        u = rng.random()
        if u < 0.4:  # two pieces of one sequence, no window: one shared stream
            ns = rng.randint(1, 8)
            items.append((ns, 0, ns, ns))
        elif u < 0.6:  # shared stream with a window: A starts first, B ends last
            ns = rng.randint(2, 6)
            a1 = rng.randint(1, ns)
            items.append((a1, rng.randint(0, a1 - 1), ns, ns))
        elif u < 0.9:  # two records of different sequences: B's tiles follow A's
            a1, nb = rng.randint(1, 5), rng.randint(1, 5)
            items.append((a1, a1, a1 + nb, a1 + nb))
        else:  # A alone
            a1 = rng.randint(1, 6)
            items.append((a1, a1, a1, a1))
    return items


def failures(protocol, seeds):
    out = []
    for s in seeds:
        rng = random.Random(7919 * s + 1)
        r = simulate(protocol, random_items(rng, rng.randint(1, 12)), s)
        if r is not None:
            out.append((s, r))
    return out


@pytest.mark.parametrize("protocol", ["one_buffer", "three_buffers"])
def test_protocol_sound(protocol):
    bad = failures(protocol, range(150))
    assert not bad, bad[:3]


@pytest.mark.parametrize("protocol", ["three_buffers_unordered", "three_buffers_no_taken"])
def test_model_finds_unsound_protocols(protocol):
    # negative controls: each lacks a wait the sound protocol has, and the model must notice
    bad = failures(protocol, range(60))
    assert len(bad) >= 6, f"{protocol}: {len(bad)} of 60 runs failed"
