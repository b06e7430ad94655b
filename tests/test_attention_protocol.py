"""Model check of the link attention kernel's K/V slot protocol (CPU, no GPU).

The roles that share the five K/V slots — the TMA producer (K and V of every key
tile, in turn), the MMA issuer (S after K lands, P.V after V lands and its
invalid rows are zeroed, committing each slot free when its product completes),
the softmax (P from S) and the V-zeroing warps — are coroutines over the
kernel's mbarriers, run in random interleavings with the hardware's wait
semantics (a wait for phase k passes whenever the current phase's parity
differs from k's) and copies that complete in any order.  The shipped protocol
must never deadlock nor let a wait pass on a wrong phase; the variant whose
V-zeroing warps waited only for the V loads of a slot (skipping its K phases) is
caught."""

import random

import pytest

from test_compose_protocol import Agent, Aliased, Bar

SLOTS = 5


def run(n_tiles, n_units, seed, vzero_waits_k=True, rotate=False):
    rng = random.Random(seed)
    bars = {}

    def mk(name, count):
        bars[name] = Bar(name, count)

    for s in range(SLOTS):
        mk(f"kv_full{s}", 1)
        mk(f"kv_empty{s}", 1)
        mk(f"vz_done{s}", 1)
        mk(f"kr_done{s}", 1)
    mk("s_full", 1)
    mk("p_full", 1)
    inflight, pipe = [], []
    total = n_tiles * n_units  # key tiles over the CTA's units, loads ld = 0 .. 2 total - 1

    def producer():
        for ld in range(2 * total):
            s = ld % SLOTS
            if ld >= SLOTS:
                yield ("wait", f"kv_empty{s}", ld // SLOTS - 1)
            yield ("act", lambda s=s: inflight.append(f"kv_full{s}"))

    def wait_k(ld):
        yield ("wait", f"kv_full{ld % SLOTS}", ld // SLOTS)
        if rotate:
            yield ("wait", f"kr_done{(ld // 2) % SLOTS}", (ld // 2) // SLOTS)

    def mma():
        ld, c = 0, 0
        for _ in range(n_units):
            yield from wait_k(ld)                       # S of the unit's first tile
            pipe.append("s_full")
            pipe.append(f"kv_empty{ld % SLOTS}")
            for j in range(n_tiles):
                vld, nld, vt = ld + 1, ld + 2, ld // 2
                yield ("wait", f"kv_full{vld % SLOTS}", vld // SLOTS)
                yield ("wait", f"vz_done{vt % SLOTS}", vt // SLOTS)
                yield ("wait", "p_full", c)
                c += 1
                more = j + 1 < n_tiles
                if more:
                    yield from wait_k(nld)
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
            if rotate:
                yield ("wait", f"kv_full{ld % SLOTS}", ld // SLOTS)
                yield ("act", lambda t=t: bars[f"kr_done{t % SLOTS}"].arrive())
            elif vzero_waits_k:
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
            bars[inflight.pop(rng.randrange(len(inflight)))].arrive()
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
                bars[inflight.pop(rng.randrange(len(inflight)))].arrive()
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
