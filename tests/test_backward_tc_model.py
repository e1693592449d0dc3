"""A discrete-event model of the hand-off protocol of the tcgen05 backward kernel
(rope_cu_tile_gb300/csrc/pk_backward_tc.cu): the TMA producer (query chunks into two buffers in
turn, each reloaded once the products that read it have completed; the next item's K / V, into the
other of two item buffers, and first chunk loaded before the current item ends), the MMA issuer, the eight warps
of the row group (with their group barriers: a reducing barrier for each give-up decision and
the plain ones between their shared-memory writes and reads; chunk c + 1 staged right after chunk
c's probabilities), and the CTA-wide barrier between work items.

Each mbarrier wait in the kernel is bounded; a group or CTA barrier is not. The model checks,
under random timings, that (1) without faults every wait that passes saw the event it was meant
to see and the CTA runs to the end; (2) when an arrival is lost (a TMA that never lands, a commit
that never arrives), every role still ends -- no warp is left at an unbounded barrier -- and the
timeout is recorded; (3) when an arrival lands at about the wait bound, so that some warps of
the row group give up and others do not, the group still leaves together; a negative control
with per-warp decisions must hang there.
"""
import random

import pytest

TIMEOUT = 20000
NW = 8  # warps of the row group (two halves of four)


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.phase & 1) != parity


class Hang(Exception):
    pass


class Cta:
    def __init__(self, items, seed, lose=None, late=None, per_warp=False):
        self.items = items  # chunks per work item
        self.rng = random.Random(seed)
        self.now = 0
        self.events = []
        self.log = {}
        self.abort = False
        self.status = 0
        self.lose = lose  # name of the arrival to drop, or None
        self.late = late  # name of the arrival to deliver at about the wait bound
        self.per_warp = per_warp  # negative control: each warp of the row group decides alone
        self.bar = {k: Barrier(c) for k, c in (("kv_full0", 1), ("kv_full1", 1), ("kv_ready", NW), ("q_full0", 1), ("q_full1", 1),
                                               ("q_empty0", 1), ("q_empty1", 1), ("q_ready", NW),
                                               ("s_full", 1), ("p_ready", NW), ("c_done", 1), ("drain", 1))}
        self.group = {}  # named-barrier instance -> arrivals (and OR of the flags)
        self.cta = {}    # CTA barrier instance -> arrivals

    def note(self, name):
        self.log[name] = self.log.get(name, 0) + 1

    def later(self, delay, key, name):
        if name == self.late:
            delay = TIMEOUT + self.rng.randint(-1000, 1000)
        def land():
            if name == self.lose:
                return
            self.note(name)
            self.bar[key].arrive()
        self.events.append((self.now + delay, land))


def bounded(cta, key, parity, observed, what):
    """The kernel's tc_wait: gives up at once after an abort, or after TIMEOUT."""
    if cta.abort:
        return False
    t0 = cta.now
    while True:
        if cta.bar[key].passes(parity):
            if not observed():
                raise AssertionError(f"false pass at t={cta.now}: {what}")
            return True
        if cta.now - t0 > TIMEOUT:
            cta.abort = True
            cta.status = 6
            return False
        yield


def wait_bounded(cta, key, parity, observed, what, out):
    r = yield from bounded(cta, key, parity, observed, what)
    out.append(r)


def group_barrier(cta, tag, flag=False):
    """A named barrier over the row group's warps (unbounded), ORing the flags."""
    if cta.per_warp and tag[0] in ("kv", "qf", "sf", "cd"):
        return flag  # the negative control: no shared decision, no barrier
    g = cta.group.setdefault(tag, [0, False])
    g[0] += 1
    g[1] = g[1] or flag
    while cta.group[tag][0] < NW:
        yield ("blocked", f"group barrier {tag}")
    return cta.group[tag][1]


def cta_barrier(cta, tag, n=3 + NW):  # producer, issuer, the row group's warps, the idle warps
    c = cta.cta.setdefault(tag, [0])
    c[0] += 1
    while cta.cta[tag][0] < n:
        yield ("blocked", f"CTA barrier {tag}")


def producer(cta):
    """Item i's K / V go to item buffer i & 1; the next item's K / V and first chunk are loaded
    before the current item ends (only the CTA's first item is loaded at its start)."""
    n_it = n_ch = 0

    def load_chunk(g):
        if g >= 2:
            r = []
            yield from wait_bounded(cta, f"q_empty{g & 1}", ((g >> 1) - 1) & 1,
                                    lambda k=g - 2: cta.log.get(f"qe{k}", 0) == 1, f"q_empty {g - 2}", r)
            if not r[0]:
                return False
        cta.later(cta.rng.randint(300, 1500), f"q_full{g & 1}", f"q{g}")
        return True

    for i, nch in enumerate(cta.items):
        yield from cta_barrier(cta, ("item", i))
        if cta.abort:
            break
        first = i == 0
        if first:
            cta.later(cta.rng.randint(300, 1500), "kv_full0", "kv0")
        ok = True
        for c in range(0 if first else 1, nch):
            ok = yield from load_chunk(n_ch + c)
            if not ok:
                break
        if ok and i + 1 < len(cta.items):
            cta.later(cta.rng.randint(300, 1500), f"kv_full{(i + 1) & 1}", f"kv{i + 1}")
            yield from load_chunk(n_ch + nch)
        n_it += 1
        n_ch += nch
    yield from cta_barrier(cta, "end")


def issuer(cta):
    n_it = n_ch = 0
    for i, nch in enumerate(cta.items):
        yield from cta_barrier(cta, ("item", i))
        if cta.abort:
            break
        r = []
        yield from wait_bounded(cta, "kv_ready", n_it & 1, lambda k=n_it: cta.log.get(f"kr{k}", 0) == NW, "kv_ready", r)
        ok = r[0]
        for c in range(nch):
            if not ok:
                break
            ph = (n_ch + c) & 1
            r = []
            yield from wait_bounded(cta, "q_ready", ph, lambda k=n_ch + c: cta.log.get(f"qr{k}", 0) == NW, "q_ready", r)
            if not (ok := r[0]):
                break
            cta.later(cta.rng.randint(300, 700), "s_full", f"sf{n_ch + c}")
            r = []
            yield from wait_bounded(cta, "p_ready", ph, lambda k=n_ch + c: cta.log.get(f"pr{k}", 0) == NW, "p_ready", r)
            if not (ok := r[0]):
                break
            d = cta.rng.randint(800, 1600)
            cta.later(d, "c_done", f"cd{n_ch + c}")
            cta.later(d, f"q_empty{(n_ch + c) & 1}", f"qe{n_ch + c}")
        cta.later(cta.rng.randint(800, 1700), "drain", f"dr{n_it}")
        r = []
        yield from wait_bounded(cta, "drain", n_it & 1, lambda: True, "drain", r)
        n_it += 1
        n_ch += nch
    yield from cta_barrier(cta, "end")


def row_warp(cta, w):
    n_it = n_ch = 0
    for i, nch in enumerate(cta.items):
        yield from cta_barrier(cta, ("item", i))
        if cta.abort:
            break
        r = []
        yield ("delay", cta.rng.randint(1, 1500))  # warps reach their waits at different times
        yield from wait_bounded(cta, f"kv_full{n_it & 1}", (n_it >> 1) & 1, lambda k=n_it: cta.log.get(f"kv{k}", 0) == 1,
                                "kv_full", r)
        bad = yield from group_barrier(cta, ("kv", n_it), not r[0])
        if not bad:
            yield ("delay", cta.rng.randint(50, 300))
            cta.note(f"kr{n_it}")
            cta.bar["kv_ready"].arrive()
        def stage(k):
            r = []
            yield ("delay", cta.rng.randint(1, 1500))
            yield from wait_bounded(cta, f"q_full{k & 1}", (k >> 1) & 1, lambda k=k: cta.log.get(f"q{k}", 0) == 1,
                                    "q_full", r)
            if (yield from group_barrier(cta, ("qf", k), not r[0])):
                return True
            yield ("delay", cta.rng.randint(50, 300))
            yield from group_barrier(cta, ("lse", k))
            cta.note(f"qr{k}")
            cta.bar["q_ready"].arrive()
            return False
        if not bad and nch > 0:
            bad = yield from stage(n_ch)
        for c in range(nch):
            if bad:
                break
            k = n_ch + c
            ph = k & 1
            r = []
            yield ("delay", cta.rng.randint(1, 1500))
            yield from wait_bounded(cta, "s_full", ph, lambda k=k: cta.log.get(f"sf{k}", 0) == 1, "s_full", r)
            if (bad := (yield from group_barrier(cta, ("sf", k), not r[0]))):
                break
            yield ("delay", cta.rng.randint(400, 2000))
            cta.note(f"pr{k}")
            cta.bar["p_ready"].arrive()
            if c + 1 < nch:
                if (bad := (yield from stage(k + 1))):
                    break
            r = []
            yield ("delay", cta.rng.randint(1, 1500))
            yield from wait_bounded(cta, "c_done", ph, lambda k=k: cta.log.get(f"cd{k}", 0) == 1, "c_done", r)
            if (bad := (yield from group_barrier(cta, ("cd", k), not r[0]))):
                break
            yield ("delay", cta.rng.randint(100, 500))
        n_it += 1
        n_ch += nch
    yield from cta_barrier(cta, "end")


def simulate(items, seed, lose=None, late=None, per_warp=False):
    cta = Cta(items, seed, lose, late, per_warp)
    roles = [producer(cta), issuer(cta)] + [row_warp(cta, w) for w in range(NW)]
    # the idle warps (2, 3 and the non-leading lanes) only meet the CTA barriers
    def idle():
        for i in range(len(items)):
            yield from cta_barrier(cta, ("item", i))
            if cta.abort:
                break
        yield from cta_barrier(cta, "end")
    roles.append(idle())
    op = [None] * len(roles)
    wake = [None] * len(roles)
    done = [False] * len(roles)
    while True:
        moved = False
        for k in cta.rng.sample(range(len(roles)), len(roles)):
            while not done[k]:
                if op[k] is not None and op[k][0] == "delay":
                    if wake[k] is None:
                        wake[k] = cta.now + op[k][1]
                    if cta.now < wake[k]:
                        break
                    wake[k] = None
                try:
                    op[k] = next(roles[k])
                except StopIteration:
                    done[k] = True
                    moved = True
                    break
                if op[k] is None or op[k][0] == "blocked":
                    if op[k] is not None and op[k][0] == "blocked":
                        # re-check next round
                        pass
                    break
                moved = True
        if all(done):
            return cta
        if cta.now > 3_000_000:
            blocked = [o[1] for o, d in zip(op, done) if not d and o is not None and o[0] == "blocked"]
            raise Hang(f"hang at t={cta.now}: {blocked}")
        cta.now += 1 if moved else 50
        due = [e for e in cta.events if e[0] <= cta.now]
        cta.events = [e for e in cta.events if e[0] > cta.now]
        for _, act in sorted(due, key=lambda e: e[0]):
            act()


def random_items(rng):
    return [rng.randint(1, 5) for _ in range(rng.randint(1, 6))]


def test_protocol_runs_to_the_end():
    for s in range(80):
        rng = random.Random(s)
        cta = simulate(random_items(rng), s)
        assert not cta.abort and cta.status == 0


@pytest.mark.parametrize("what", ["kv", "q", "sf", "cd"])
def test_lost_arrival_ends_every_role(what):
    for s in range(30):
        rng = random.Random(100 + s)
        items = random_items(rng)
        total = sum(items)
        k = rng.randrange(len(items) if what == "kv" else total)
        cta = simulate(items, s, lose=f"{what}{k}")
        assert cta.abort and cta.status == 6


def late_runs(per_warp, seeds, what):
    hangs = 0
    for s in seeds:
        rng = random.Random(500 + s)
        items = random_items(rng)
        k = rng.randrange(sum(items))
        try:
            simulate(items, s, late=f"{what}{k}", per_warp=per_warp)
        except Hang:
            hangs += 1
    return hangs


@pytest.mark.parametrize("what", ["sf", "q"])
def test_arrival_at_the_wait_bound_leaves_no_warp_behind(what):
    assert late_runs(False, range(40), what) == 0


def test_model_finds_per_warp_decisions_unsafe():
    # negative control: with per-warp decisions, a chunk's copy landing right at the bound lets some
    # warps go on to the group barrier after the staging of lse and D that the others never reach
    assert late_runs(True, range(120), "q") >= 3
