"""A discrete-event model of the hand-off protocol inside the tensor-core attention kernel
(rope_cu_tile_gb300/csrc/pk_attend_tc.cu), with every role of a CTA: the producer (work items,
TMA loads of Q, K and V), the four rotation warps, the two MMA issuers (one per query tile X of
a work item), the eight softmax warps (four per query tile) and the tensor pipe, joined by the
kernel's mbarriers: the item boxes, the Q buffers, the K and V rings, and the score / P / PV
hand-offs.

mbarriers follow the PTX rule the kernel relies on: a wait names the parity of the phase it
waits for, and it passes when the barrier's current (incomplete) phase has the other parity.
That test is only sound while the waiter is never two phases behind or ahead of the barrier.
Under random timings the model compares every wait that passes with the event it was meant to
observe (a "false pass" otherwise), and a state where every role waits and nothing is in flight
is a deadlock. The tensor pipe runs MMAs in issue order; a commit arrives once every earlier MMA
of its thread has completed; a TMA load arrives on its barrier after a random latency.

Score-buffer protocols:
- one_buffer: the kernel as built. One score buffer per query tile; S(t) waits until that tile's
  softmax warps have loaded the last half of S(t - 1) (`s_consumed`); an issuer sees a key tile
  outside its query tile's range after the PV of the tile before it.
- three_buffers: three score buffers shared by both query tiles, P written over the buffer its S
  came from, products numbered in stream order (A before B at a tile) and product n using
  buffer n % 3; S(n) waits for the PV of product n - 3 (`s_free`), for the softmax to have seen
  the tile's previous S complete (`s_taken`), and for product n - 1 to have been issued (a
  counter that only grows).
- three_buffers_unordered, three_buffers_no_taken: the same without the last two waits, or
  without `s_taken`; both are unsound and the model must find it.
- one_buffer_skip: one_buffer with issuers that never wait for a key or value tile outside their
  query tile's range (the issuer whose range holds the tile arrives in the other's place). A
  stage's next wait then names a phase two ahead of the one last seen, which a parity test cannot
  tell from the one before: unsound, and the model must find it.
"""
import random

import pytest

PROTOCOLS = ("one_buffer", "one_buffer_skip", "three_buffers", "three_buffers_unordered", "three_buffers_no_taken")
K_STAGES, V_STAGES = 4, 3
ITEM_CONSUMERS = 2 + 4 + 4 + 4  # issuers, rotation warps, softmax warps of A and of B


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
        self.items = items  # (a1, b0, b1, stream tiles); B is a record when b1 > b0
        self.rng = random.Random(seed)
        self.now = 0
        self.events = []  # (time, action)
        self.pipe_free = 0
        self.last_done = {}
        self.issued = 0
        self.log = {}  # event name -> count (or presence)
        bars = {}
        for mb in (0, 1):
            bars[("item_full", mb)] = Barrier(1)
            bars[("item_empty", mb)] = Barrier(ITEM_CONSUMERS)
        for x in (0, 1):
            for qb in (0, 1):
                bars[("q_full", x, qb)] = Barrier(1)
                bars[("q_ready", x, qb)] = Barrier(4)
                bars[("q_empty", x, qb)] = Barrier(1)
            bars[("s_full", x)] = Barrier(1)
            bars[("s_consumed", x)] = Barrier(4)
            bars[("s_taken", x)] = Barrier(4)
            bars[("p_ready", x)] = Barrier(4)
            bars[("pv_done", x)] = Barrier(1)
        for st in range(K_STAGES):
            bars[("k_full", st)] = Barrier(1)
            bars[("k_ready", st)] = Barrier(4)
            bars[("k_empty", st)] = Barrier(2)
        for st in range(V_STAGES):
            bars[("v_full", st)] = Barrier(1)
            bars[("v_empty", st)] = Barrier(2)
        for b in range(3):
            bars[("s_free", b)] = Barrier(1)
        self.bar = bars
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

    # --- events
    def note(self, name):
        self.log[name] = self.log.get(name, 0) + 1

    def count(self, name):
        return self.log.get(name, 0)

    def arrive(self, key, name=None):
        if name is not None:
            self.note(name)
        self.bar[key].arrive()

    def tma(self, key, name):
        def land():
            self.note(name)
            self.bar[key].arrive()
        self.events.append((self.now + self.rng.randint(300, 1500), land))

    def mma(self, who, cycles, name):
        end = max(self.now + 1, self.pipe_free) + cycles
        self.pipe_free = end
        self.last_done[who] = end
        self.events.append((end, lambda: self.note(name)))

    def commit(self, who, key, name=None):
        end = max(self.last_done.get(who, 0), self.now) + 1
        self.events.append((end, lambda: self.arrive(key, name)))

    def wait(self, key, parity, observed, what):
        bar = self.bar[key]
        return ("wait", lambda: bar.passes(parity), observed, what)

    def delay(self, lo, hi, p_slow=0.0):
        if p_slow and self.rng.random() < p_slow:
            return ("delay", self.rng.randint(2000, 8000))
        return ("delay", self.rng.randint(lo, hi))


def take_item(m, i):
    """A consumer's hand-off of item box i (None past the last item)."""
    mb = i & 1
    yield m.wait(("item_full", mb), (i >> 1) & 1, lambda: m.count(f"box{i}") == 1, f"box {i} written")
    m.arrive(("item_empty", mb), f"read{i}")


def producer(m):
    qn = [0, 0]
    kn = vn = 0
    for i in range(len(m.items) + 1):
        mb = i & 1
        yield m.wait(("item_empty", mb), ((i >> 1) & 1) ^ 1,
                     lambda i=i: i < 2 or m.count(f"read{i - 2}") == ITEM_CONSUMERS, f"box {i - 2} read")
        m.arrive(("item_full", mb), f"box{i}")
        if i == len(m.items):
            return
        a1, b0, b1, ns = m.items[i]
        for x in (0, 1) if b1 > b0 else (0,):
            q, qb = qn[x], qn[x] & 1
            yield m.wait(("q_empty", x, qb), ((q >> 1) & 1) ^ 1,
                         lambda x=x, q=q: q < 2 or m.count(f"qfree{x}.{q - 2}") == 1, f"Q{x} use {q - 2} done")
            m.tma(("q_full", x, qb), f"qland{x}.{q}")
            qn[x] += 1
        for t in range(ns + 2):  # K two tiles ahead of V
            if t < ns:
                g = kn
                yield m.wait(("k_empty", g % K_STAGES), ((g // K_STAGES) & 1) ^ 1,
                             lambda g=g: g < K_STAGES or m.count(f"kfree{g - K_STAGES}") == 2,
                             f"K{g - K_STAGES} released")
                m.tma(("k_full", g % K_STAGES), f"kland{g}")
                kn += 1
            if t >= 2:
                g = vn
                yield m.wait(("v_empty", g % V_STAGES), ((g // V_STAGES) & 1) ^ 1,
                             lambda g=g: g < V_STAGES or m.count(f"vfree{g - V_STAGES}") == 2,
                             f"V{g - V_STAGES} released")
                m.tma(("v_full", g % V_STAGES), f"vland{g}")
                vn += 1


def rotation_warp(m):
    qn = [0, 0]
    kn = 0
    for i in range(len(m.items) + 1):
        yield from take_item(m, i)
        if i == len(m.items):
            return
        a1, b0, b1, ns = m.items[i]
        jobs = [("q", 0)] + ([("q", 1)] if b1 > b0 else []) + [("k", t) for t in range(ns)]
        for kind, x in jobs:
            yield m.delay(20, 200)  # the job's table rows
            if kind == "q":
                q, qb = qn[x], qn[x] & 1
                yield m.wait(("q_full", x, qb), (q >> 1) & 1, lambda x=x, q=q: m.count(f"qland{x}.{q}") == 1,
                             f"Q{x} use {q} landed")
                yield m.delay(50, 300)
                m.arrive(("q_ready", x, qb), f"qrot{x}.{q}")
            else:
                g = kn
                yield m.wait(("k_full", g % K_STAGES), (g // K_STAGES) & 1, lambda g=g: m.count(f"kland{g}") == 1,
                             f"K{g} landed")
                yield m.delay(50, 300, 0.01)
                m.arrive(("k_ready", g % K_STAGES), f"krot{g}")
                kn += 1
        qn[0] += 1
        if b1 > b0:
            qn[1] += 1


def issuer(m, x):
    proto = m.protocol
    shared = proto not in ("one_buffer", "one_buffer_skip")
    skip = proto == "one_buffer_skip"
    ordered = proto in ("three_buffers", "three_buffers_no_taken")
    with_taken = proto == "three_buffers"
    kn = vn = qn = 0
    n_s = n_p = 0  # S and PV products of this query tile so far
    prev = None
    for i in range(len(m.items) + 1):
        yield from take_item(m, i)
        if i == len(m.items):
            return
        a1, b0, b1, ns = m.items[i]
        lo, hi = (0, a1) if x == 0 else (b0, b1)
        for t in range(ns + 1):
            own = t < ns and lo <= t < hi
            # as built, a tile outside X's range is seen after the PV of the previous tile
            late = not shared and not own
            if t < ns and not late:
                g = kn
                st = g % K_STAGES
                yield m.wait(("k_ready", st), (g // K_STAGES) & 1, lambda g=g: m.count(f"krot{g}") == 4,
                             f"K{g} rotated")
                if own:
                    n = m.number[(i, t, x)]
                    q, qb = qn, qn & 1
                    if t == lo:
                        yield m.wait(("q_ready", x, qb), (q >> 1) & 1,
                                     lambda q=q: m.count(f"qrot{x}.{q}") == 4, f"Q{x} use {q} rotated")
                    if not shared:
                        if prev is not None:
                            yield m.wait(("s_consumed", x), (n_s - 1) & 1,
                                         lambda p=prev: m.count(f"read_s{p}") == 4, f"S{prev} read")
                    else:
                        if with_taken and prev is not None:
                            yield m.wait(("s_taken", x), (n_s - 1) & 1,
                                         lambda p=prev: m.count(f"seen_s{p}") == 4, f"S{prev} seen")
                        if ordered:
                            yield ("wait", lambda n=n: m.issued == n, lambda: True, "turn")
                        if n >= 3:
                            yield m.wait(("s_free", n % 3), (n // 3 - 1) & 1,
                                         lambda n=n: m.count(f"pv{n - 3}") == 1, f"PV{n - 3} done (for S{n})")
                    yield m.delay(1, 30)
                    m.mma(x, m.rng.randint(200, 400), f"s{n}")
                    m.commit(x, ("s_full", x))
                    m.commit(x, ("k_empty", st), f"kfree{g}")
                    olo, ohi = (b0, b1) if x == 0 else (0, a1)
                    if skip and not (olo <= t < ohi):
                        m.arrive(("k_empty", st), f"kfree{g}")
                    if ordered:
                        m.issued = n + 1
                    n_s += 1
                    prev = n
                    if t + 1 == hi:
                        m.commit(x, ("q_empty", x, qb), f"qfree{x}.{q}")
                        qn += 1
                else:
                    m.arrive(("k_empty", st), f"kfree{g}")
                kn += 1
            if t >= 1 and skip and not (lo <= t - 1 < hi):
                vn += 1
            elif t >= 1:
                g = vn
                st = g % V_STAGES
                yield m.wait(("v_full", st), (g // V_STAGES) & 1, lambda g=g: m.count(f"vland{g}") == 1, f"V{g} landed")
                if lo <= t - 1 < hi:
                    n = m.number[(i, t - 1, x)]
                    yield m.wait(("p_ready", x), n_p & 1, lambda n=n: m.count(f"p{n}") == 4, f"P{n} written")
                    n_p += 1
                    yield m.delay(1, 30)
                    m.mma(x, m.rng.randint(300, 600), f"pv{n}")
                    m.commit(x, ("pv_done", x))
                    m.commit(x, ("v_empty", st), f"vfree{g}")
                    olo, ohi = (b0, b1) if x == 0 else (0, a1)
                    if skip and not (olo <= t - 1 < ohi):
                        m.arrive(("v_empty", st), f"vfree{g}")
                    if shared:
                        m.commit(x, ("s_free", n % 3))
                else:
                    m.arrive(("v_empty", st), f"vfree{g}")
                vn += 1
            if t < ns and late and skip:
                kn += 1
            elif t < ns and late:
                g = kn
                st = g % K_STAGES
                yield m.wait(("k_ready", st), (g // K_STAGES) & 1, lambda g=g: m.count(f"krot{g}") == 4,
                             f"K{g} rotated")
                m.arrive(("k_empty", st), f"kfree{g}")
                kn += 1


def softmax_warp(m, x):
    shared = m.protocol not in ("one_buffer", "one_buffer_skip")
    with_taken = m.protocol == "three_buffers"
    n_s = n_pv = 0
    for i in range(len(m.items) + 1):
        yield from take_item(m, i)
        if i == len(m.items):
            return
        a1, b0, b1, ns = m.items[i]
        lo, hi = (0, a1) if x == 0 else (b0, b1)
        for j in range(lo, hi):
            n = m.number[(i, j, x)]
            yield m.wait(("s_full", x), n_s & 1, lambda n=n: m.count(f"s{n}") == 1, f"S{n} complete")
            n_s += 1
            if with_taken:
                m.arrive(("s_taken", x), f"seen_s{n}")
            yield m.delay(100, 900, 0.05)  # pass 1, and the load of the last half of S
            if not shared:
                m.arrive(("s_consumed", x), f"read_s{n}")
            if j > lo:
                p = m.number[(i, j - 1, x)]
                yield m.wait(("pv_done", x), n_pv & 1, lambda p=p: m.count(f"pv{p}") == 1, f"PV{p} done")
                n_pv += 1
            yield m.delay(100, 900)  # probabilities, P written
            m.arrive(("p_ready", x), f"p{n}")
            yield m.delay(1, 60, 0.02)  # until the next wait (descheduling included)
        if hi > lo:
            p = m.number[(i, hi - 1, x)]
            yield m.wait(("pv_done", x), n_pv & 1, lambda p=p: m.count(f"pv{p}") == 1, f"PV{p} done (epilogue)")
            n_pv += 1
            yield m.delay(50, 300)


def simulate(protocol, items, seed):
    """None if every wait was sound and the model ran to the end, else what went wrong."""
    m = Model(protocol, items, seed)
    roles = ([producer(m)] + [rotation_warp(m) for _ in range(4)] + [issuer(m, 0), issuer(m, 1)] +
             [softmax_warp(m, x) for x in (0, 1) for _ in range(4)])
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
                waits = [o[3] for o in op if o is not None and o[0] == "wait"]
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
    bad = failures(protocol, range(120))
    assert not bad, bad[:3]


@pytest.mark.parametrize("protocol", ["three_buffers_unordered", "three_buffers_no_taken", "one_buffer_skip"])
def test_model_finds_unsound_protocols(protocol):
    # negative controls: each lacks a wait the sound protocol has, and the model must notice
    bad = failures(protocol, range(60))
    assert len(bad) >= 6, f"{protocol}: {len(bad)} of 60 runs failed"
