"""Model check of the link attention kernel's K/V slot protocol (CPU, no GPU).

The roles that share the five K/V slots — the TMA producer (K and V of every key
tile, in turn), the V-zeroing warps (wait for the tile's K load, then its V
load, rotate K when rotating on read, zero V's invalid rows, arrive vz_done),
the MMA issuer (waits only for vz_done of a tile before its first S product and
for the softmax's P; commits each slot free when its products complete) and the
softmax (P from S) — are coroutines over the kernel's mbarriers, run in random
interleavings with the hardware's wait semantics (a wait for phase k passes
whenever the current phase's parity differs from k's) and copies that complete
in any order.  The issuer never waits for a load itself: that it has landed
reaches it through vz_done, which the model checks by recording, at every MMA,
whether the slot it reads holds the load it means.  The shipped protocol must
never deadlock, let a wait pass on a wrong phase or read a slot too early; the
variant whose V-zeroing warps waited only for the V loads of a slot (skipping
its K phases) is caught."""

import random

import pytest

from test_compose_protocol import Agent, Aliased, Bar

SLOTS = 5


def run(n_tiles, n_units, seed, vzero_waits_k=True, rotate=False, mma_waits_tile=True):
    rng = random.Random(seed)
    bars = {}

    def mk(name, count):
        bars[name] = Bar(name, count)

    for s in range(SLOTS):
        mk(f"kv_full{s}", 1)
        mk(f"kv_empty{s}", 1)
        mk(f"vz_done{s}", 1)
    mk("s_full", 1)
    mk("p_full", 1)
    inflight, pipe = [], []
    landed = {}  # slot -> load number whose data the slot holds
    total = n_tiles * n_units  # key tiles over the CTA's units, loads ld = 0 .. 2 total - 1

    def land(s, ld):
        def f():
            landed[s] = ld
            bars[f"kv_full{s}"].arrive()
        return f

    def producer():
        for ld in range(2 * total):
            s = ld % SLOTS
            if ld >= SLOTS:
                yield ("wait", f"kv_empty{s}", ld // SLOTS - 1)
            yield ("act", lambda s=s, ld=ld: inflight.append(land(s, ld)))

    def reads(ld):  # an MMA that reads load ld's slot: the data must be there
        def f():
            if landed.get(ld % SLOTS) != ld:
                raise Aliased(f"MMA read slot {ld % SLOTS} for load {ld} holding {landed.get(ld % SLOTS)}")
        return f

    def mma():
        ld, c = 0, 0
        for _ in range(n_units):
            yield ("wait", f"vz_done{(ld // 2) % SLOTS}", (ld // 2) // SLOTS)  # S of the unit's first tile
            yield ("act", reads(ld))
            pipe.append("s_full")
            pipe.append(f"kv_empty{ld % SLOTS}")
            for j in range(n_tiles):
                vld, nld = ld + 1, ld + 2
                yield ("wait", "p_full", c)
                c += 1
                yield ("act", reads(vld))
                more = j + 1 < n_tiles
                if more:
                    if mma_waits_tile:
                        yield ("wait", f"vz_done{(nld // 2) % SLOTS}", (nld // 2) // SLOTS)
                    yield ("act", reads(nld))
                    pipe.append("s_full")
                yield ("act", lambda vs=vld % SLOTS: pipe.append(f"kv_empty{vs}"))
                if more:
                    yield ("act", lambda ns=nld % SLOTS: pipe.append(f"kv_empty{ns}"))
                ld += 2

    def softmax():
        for t in range(total):
            yield ("wait", "s_full", t)
            yield ("act", lambda: bars["p_full"].arrive())

    def vzero():
        for t in range(total):
            ld = 2 * t
            if rotate or vzero_waits_k:  # rotate-on-read rotates K in place here
                yield ("wait", f"kv_full{ld % SLOTS}", ld // SLOTS)
            yield ("wait", f"kv_full{(ld + 1) % SLOTS}", (ld + 1) // SLOTS)
            yield ("act", lambda t=t: bars[f"vz_done{t % SLOTS}"].arrive())

    agents = [Agent("producer", producer()), Agent("mma", mma()), Agent("softmax", softmax()),
              Agent("vzero", vzero())]
    while True:
        live = [a for a in agents if not a.done]
        if not live and not inflight and not pipe:
            return "ok"
        moved = False
        if inflight and rng.random() < 0.3:
            inflight.pop(rng.randrange(len(inflight)))()
            moved = True
        elif pipe and rng.random() < 0.3:
            bars[pipe.pop(0)].arrive()
            moved = True
        else:
            rng.shuffle(live)
            for a in live:
                if a.step(bars):
                    moved = True
                    break
        if not moved:
            if inflight:
                inflight.pop(rng.randrange(len(inflight)))()
            elif pipe:
                bars[pipe.pop(0)].arrive()
            else:
                return "deadlock: " + str([(a.name, a.cur[:3] if a.cur else None) for a in agents if not a.done])


@pytest.mark.parametrize("n_tiles,n_units", [(1, 6), (2, 4), (3, 3), (8, 2), (13, 1)])
@pytest.mark.parametrize("rotate", [False, True])
def test_shipped_slot_protocol_is_safe(n_tiles, n_units, rotate):
    for seed in range(80):
        assert run(n_tiles, n_units, seed, rotate=rotate) == "ok", (n_tiles, n_units, seed)


def test_v_zeroing_that_skips_k_phases_is_caught():
    caught = 0
    for seed in range(300):
        try:
            run(1, 8, seed, vzero_waits_k=False)
        except Aliased:
            caught += 1
    assert caught > 0


def test_issuer_that_skips_the_tile_wait_is_caught():
    """Without its vz_done wait the issuer would read a K slot before the load lands."""
    caught = 0
    for seed in range(300):
        try:
            r = run(4, 2, seed, mma_waits_tile=False)
        except Aliased:
            caught += 1
            continue
        caught += r != "ok"
    assert caught > 0
