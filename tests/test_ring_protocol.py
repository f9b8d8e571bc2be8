"""The decode kernel's shared-memory ring protocol, checked on the CPU.

The decode kernel moves K/V items through ring slots guarded by mbarriers
whose waits see only the parity of a phase.  A waiter that falls two phases
behind a barrier would pass on an old phase and read a slot whose copy has not
landed.  This model replays the protocol with randomized agent speeds and
out-of-order copy completion:
  * a producer fills K and V slots (refilling a slot only after its previous
    item was released);
  * the QK streams (two at head_dim 256: the even and the odd units; one at
    head_dim 128: every unit) each take their units through their own K slots;
  * the PV warps take every unit's V slot and its handoff buffer (unit i uses
    buffer i % 4).
The slot and phase formulas are the closed forms of the kernel's ring (struct
Ring in decode.cu); the kernel reaches them by stepping a RingPos per item,
and a test below checks that the stepping gives the closed forms.  The
model also shows that one ring whose K slots alternate between the two streams
does fail (a stream reads a slot before its copy lands), which is why each
stream has its own K slots.
"""
import random

import pytest


class Bar:
    def __init__(self):
        self.n = 0  # completed phases (one arrival completes a phase in this model)

    def arrive(self):
        self.n += 1

    def passes(self, phase):  # try_wait.parity(phase & 1)
        return (self.n & 1) != (phase & 1)


def k_slots(nslots, streams):
    """K slots per stream (Ring::k_slots): nslots // 6, at least one; a single
    stream gets at least two, so its next unit's K is in flight meanwhile."""
    k = max(1, nslots // 6)
    return max(k, 2) if streams == 1 else k


def kernel_ring(nslots, streams=2):
    kK = k_slots(nslots, streams)
    nV = nslots - streams * kK
    return dict(kslot=lambda i: (i % streams) * kK + (i // streams) % kK, kuse=lambda i: (i // streams) // kK,
                vslot=lambda i: streams * kK + i % nV, vuse=lambda i: i // nV)


def shared_ring(nslots):
    return dict(kslot=lambda i: (2 * i) % nslots, kuse=lambda i: (2 * i) // nslots,
                vslot=lambda i: (2 * i + 1) % nslots, vuse=lambda i: (2 * i + 1) // nslots)


def simulate(n_units, nslots, ring, seed, nhb=4, streams=2):
    rnd = random.Random(seed)
    kslot, kuse, vslot, vuse = ring["kslot"], ring["kuse"], ring["vslot"], ring["vuse"]
    full = [Bar() for _ in range(nslots)]
    empty = [Bar() for _ in range(nslots)]
    hfull = [Bar() for _ in range(nhb)]
    hempty = [Bar() for _ in range(nhb)]
    content, hand, pending = [None] * nslots, [None] * nhb, []

    def producer():
        for i in range(n_units):
            for kind, s, u in (("K", kslot(i), kuse(i)), ("V", vslot(i), vuse(i))):
                if u > 0:
                    while not empty[s].passes(u - 1):
                        yield
                pending.append((s, (kind, i)))
                yield

    def qk(st):
        for i in range(st, n_units, streams):
            s, u = kslot(i), kuse(i)
            while not full[s].passes(u):
                yield
            assert content[s] == ("K", i), f"QK stream {st}, unit {i} read {content[s]} from slot {s}"
            yield
            empty[s].arrive()
            hb = i % nhb
            if i >= nhb:
                while not hempty[hb].passes(i // nhb - 1):
                    yield
            hand[hb] = i
            hfull[hb].arrive()
            yield

    def pv():
        for i in range(n_units):
            hb = i % nhb
            while not hfull[hb].passes(i // nhb):
                yield
            assert hand[hb] == i, f"PV unit {i} read handoff {hand[hb]}"
            s, u = vslot(i), vuse(i)
            while not full[s].passes(u):
                yield
            assert content[s] == ("V", i), f"PV unit {i} read {content[s]} from slot {s}"
            yield
            empty[s].arrive()
            hempty[hb].arrive()
            yield

    agents = {"producer": producer(), "pv": pv()}
    for st in range(streams):
        agents[f"qk{st}"] = qk(st)
    speed = {k: rnd.uniform(0.1, 1.0) for k in agents}
    for _ in range(200000):
        if not agents and not pending:
            return
        if pending and rnd.random() < 0.3:  # some issued copy lands (any order)
            s, item = pending.pop(rnd.randrange(len(pending)))
            content[s] = item
            full[s].arrive()
            continue
        names = list(agents)
        k = rnd.choices(names, weights=[speed[n] for n in names])[0]
        try:
            next(agents[k])
        except StopIteration:
            del agents[k]
    raise AssertionError("deadlock")


@pytest.mark.parametrize("streams", [1, 2])
@pytest.mark.parametrize("nslots", [4, 6, 8, 12])
def test_kernel_ring_never_reads_an_unlanded_slot(nslots, streams):
    for seed in range(400):
        simulate(random.Random(seed).randint(1, 30), nslots, kernel_ring(nslots, streams), seed, streams=streams)


def test_alternating_k_slots_do_race():
    failures = 0
    for seed in range(1500):
        try:
            simulate(random.Random(seed).randint(1, 20), 6, shared_ring(6), seed)
        except AssertionError:
            failures += 1
    assert failures > 0


class RingPos:
    """The kernel's incremental ring position (slot, earlier passes)."""

    def __init__(self):
        self.s, self.use = 0, 0

    def next(self, n):
        self.s += 1
        if self.s == n:
            self.s, self.use = 0, self.use + 1


@pytest.mark.parametrize("streams", [1, 2])
@pytest.mark.parametrize("nslots", [4, 6, 8, 10, 12])
def test_stepped_positions_equal_the_closed_forms(nslots, streams):
    kK = k_slots(nslots, streams)
    nV = nslots - streams * kK
    ring = kernel_ring(nslots, streams)
    # producer: one K position per stream, swapped after every unit (two streams); one V position
    cur, oth, vp = RingPos(), RingPos(), RingPos()
    # consumers: each QK stream steps its own K position; the PV warps step the V position
    qk = [RingPos() for _ in range(streams)]
    pv = RingPos()
    for i in range(200):
        assert ((i % streams) * kK + cur.s, cur.use) == (ring["kslot"](i), ring["kuse"](i))
        cur.next(kK)
        if streams == 2:
            cur, oth = oth, cur
        assert (streams * kK + vp.s, vp.use) == (ring["vslot"](i), ring["vuse"](i))
        vp.next(nV)
        st = i % streams
        assert (st * kK + qk[st].s, qk[st].use) == (ring["kslot"](i), ring["kuse"](i))
        qk[st].next(kK)
        assert (streams * kK + pv.s, pv.use) == (ring["vslot"](i), ring["vuse"](i))
        pv.next(nV)


def cta_units(ngps, g0, g1, qw):
    """The units of one CTA (granules [g0, g1) of the (sequence, KV head) pairs
    laid end to end): (pair, first granule in the pair, granules)."""
    units, base = [], 0
    for pair, ngp in enumerate(ngps):
        gi = max(g0 - base, 0)
        while gi < ngp and base + gi < g1:
            n = min(qw, ngp - gi, g1 - base - gi)
            units.append((pair, gi, n))
            gi += n
        base += ngp
    return units


@pytest.mark.parametrize("streams,qw", [(1, 8), (2, 4)])
def test_decode_step_new_token_has_one_owner(streams, qw):
    """Decode step: the stream holding the unit with a pair's newest token
    quantizes that token at its first unit of the pair, decided from that unit
    alone (the pair's last granule inside the CTA's range, and the units from
    there to it, kQW granules each, a multiple of the stream count).  Exactly
    one (CTA, stream) claims each pair, and it is the one that processes the
    unit holding the token."""
    rnd = random.Random(7)
    for _ in range(300):
        ngps = [rnd.choice([0, 1, 2, 3, 5, 8, 9, 17, 33, 128]) for _ in range(rnd.randint(1, 12))]
        U, N = sum(ngps), rnd.randint(1, 40)
        claims, holders = {}, {}
        for c in range(N):
            g0, g1 = U * c // N, U * (c + 1) // N
            seen = [None] * streams
            base = {p: sum(ngps[:p]) for p in range(len(ngps))}
            for i, (pair, gi, n) in enumerate(cta_units(ngps, g0, g1, qw)):
                st = i % streams
                if gi + n == ngps[pair]:
                    holders.setdefault(pair, []).append((c, st))
                if seen[st] != pair:  # the stream's pair start
                    seen[st] = pair
                    g_last = base[pair] + ngps[pair] - 1
                    if g_last < g1 and ((ngps[pair] - 1 - gi) // qw) % streams == 0:
                        claims.setdefault(pair, []).append((c, st))
        for pair, ngp in enumerate(ngps):
            if ngp:
                assert len(holders[pair]) == 1 and claims.get(pair) == holders[pair], (ngps, N, pair)
