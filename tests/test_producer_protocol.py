"""The KV producer's shared-memory pipeline, checked on the CPU.

The producer kernel (producer.cu) runs a loader warp and 15 compute warps per
CTA.  The loader bulk-copies work units (16 tokens x a group of heads) into
ring slots guarded by mbarriers, whose waits see only the parity of a phase;
it publishes each tile's metadata into a ring of tile entries.  A unit's heads
are tasks handed to the compute warps round-robin, so a warp has a task in
only some units and waits only on those units' slots.  Such a warp can reach
use u of a slot while use u - 1 is still in flight, where the parity test
would pass on the older phase; the loader therefore stamps each slot with the
use it fills, and a waiter first waits for the stamp.

This model replays the protocol with randomized agent speeds and out-of-order
copy completion, with the kernel's arrival counts (a unit's first task arrives
for the missing ones), tile-entry reuse and the loader's deferred tile
publication.  It checks that every task of every unit runs exactly once, on
that unit's data, that no slot is refilled while in use and that no tile entry
is read stale -- and that without the stamps a waiter does read stale data.
"""
import random

import pytest

TOK, TR = 16, 3


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.tx, self.done = count, count, 0, 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, "more arrivals than the barrier's count"
        self._complete()

    def expect(self, b):
        self.tx += b

    def complete_tx(self, b):
        self.tx -= b
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def passes(self, parity):  # mbarrier.try_wait.parity
        return (self.done & 1) != parity


class Stale(Exception):
    pass


def largest_divisor_at_most(n, cap):
    return max(d for d in range(1, min(n, cap) + 1) if n % d == 0)


def simulate_cta(units, upt, nkv, kvh, qh, S, ncw, seed, stamps=True, land_p=0.3):
    rnd = random.Random(seed)
    u0, u1 = units
    full = [Bar(1) for _ in range(S)]
    free = [Bar(ncw) for _ in range(S)]
    meta_full = [Bar(1) for _ in range(TR)]
    tile_free = [Bar(ncw) for _ in range(TR)]
    slot_unit, slot_use, entry_tile = [None] * S, [-1] * S, [None] * TR
    in_flight, done = [], {}

    def heads(u):
        return qh if u % upt >= 2 * nkv else kvh

    def loader():
        cur, tl, pending = -1, -1, False

        def publish():
            nonlocal pending
            pending = False
            te = tl % TR
            if tl >= TR:
                while not tile_free[te].passes(((tl // TR) - 1) & 1):
                    yield
            entry_tile[te] = cur
            meta_full[te].arrive()

        for i, u in enumerate(range(u0, u1)):
            n = u // upt
            if n != cur:
                if pending:
                    yield from publish()
                cur, tl, pending = n, tl + 1, True
            s, use = i % S, i // S
            if use > 0:
                if pending:
                    yield from publish()
                while not free[s].passes((use - 1) & 1):
                    yield
            slot_use[s] = use
            yield
            full[s].expect(1)
            full[s].arrive()
            in_flight.append((s, u))
            yield
        if pending:
            yield from publish()

    def warp(w):
        cur, tl, tbase = -1, -1, 0
        for i, u in enumerate(range(u0, u1)):
            n = u // upt
            if n != cur:
                if tl >= 0:
                    tile_free[tl % TR].arrive()
                cur, tl = n, tl + 1
                while not meta_full[tl % TR].passes((tl // TR) & 1):
                    yield
                if entry_tile[tl % TR] != n:
                    raise Stale(f"tile entry holds tile {entry_tile[tl % TR]}, warp expects {n}")
            nh = heads(u)
            hp = (w - tbase % ncw + ncw) % ncw
            tbase += nh
            if hp >= nh:
                continue
            s, use = i % S, i // S
            if stamps:
                while slot_use[s] != use:
                    yield
            while not full[s].passes(use & 1):
                yield
            if slot_unit[s] != u:
                raise Stale(f"slot {s} holds unit {slot_unit[s]}, warp {w} expects unit {u}")
            yield
            assert slot_unit[s] == u, "slot refilled while in use"
            done.setdefault(u, []).append(hp)
            free[s].arrive(1 + ncw - nh if hp == 0 else 1)

    agents = [loader()] + [warp(w) for w in range(ncw)]
    alive = list(range(len(agents)))
    for _ in range(2_000_000):
        if not alive and not in_flight:
            break
        if in_flight and (not alive or rnd.random() < land_p):
            s, u = in_flight.pop(rnd.randrange(len(in_flight)))  # copies land in any order
            slot_unit[s] = u
            full[s].complete_tx(1)
            continue
        a = rnd.choice(alive)
        try:
            next(agents[a])
        except StopIteration:
            alive.remove(a)
    else:
        raise AssertionError("the pipeline did not finish (deadlock)")
    for u in range(u0, u1):
        assert sorted(done.get(u, [])) == list(range(heads(u))), f"unit {u}: tasks {done.get(u)}"


def geometry(Hkv, Hq, D):
    mh = 1024 // D
    kvh = largest_divisor_at_most(Hkv, mh)
    qh = largest_divisor_at_most(Hq, mh) if Hq else 1
    nkv, nq = Hkv // kvh, (Hq // qh if Hq else 0)
    return 2 * nkv + nq, nkv, kvh, qh


SHAPES = [(8, 32, 128, 6), (4, 24, 256, 4), (1, 2, 128, 8), (8, 0, 256, 3), (3, 7, 128, 8), (6, 18, 128, 4),
          (5, 10, 256, 6), (7, 14, 128, 3)]


@pytest.mark.parametrize("Hkv,Hq,D,S", SHAPES)
@pytest.mark.parametrize("ncw", [15, 8])
def test_producer_pipeline_with_stamps(Hkv, Hq, D, S, ncw):
    upt, nkv, kvh, qh = geometry(Hkv, Hq, D)
    for T in (1, 17, 100):
        U = (T + TOK - 1) // TOK * upt
        for grid in (1, 3):
            grid = min(grid, U)
            for b in range(grid):
                for seed in range(2):
                    simulate_cta((b * U // grid, (b + 1) * U // grid), upt, nkv, kvh, qh, S, ncw, seed)


def test_parity_alone_reads_stale_slots():
    # 15 warps, units of 4 heads (8 KV heads at head_dim 256): a warp has a task
    # in about every fourth unit; slow copies leave a slot's previous use in flight.
    upt, nkv, kvh, qh = geometry(8, 0, 256)
    stale = 0
    for seed in range(40):
        try:
            simulate_cta((0, 6 * upt), upt, nkv, kvh, qh, 3, 15, seed, stamps=False, land_p=0.02)
        except Stale:
            stale += 1
    assert stale > 0
