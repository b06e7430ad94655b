"""Model check of the link attention kernel's K/V slot protocol (CPU, no GPU).

The roles that share the five K/V slots — the TMA producer (K and V of every key
tile, in turn), the V-zeroing warps (wait for the tile's K load, then its V
load, zero V's invalid rows, arrive vz_done),
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
its K phases) is caught.  A second model covers rotate-on-read's handshake on the
Q tile (written per key frame by the softmax warps, waited for by the issuer)."""

import random

import pytest

from test_compose_protocol import Agent, Aliased, Bar

SLOTS = 5


def run(n_tiles, n_units, seed, vzero_waits_k=True, mma_waits_tile=True):
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
            if vzero_waits_k:
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
def test_shipped_slot_protocol_is_safe(n_tiles, n_units):
    for seed in range(160):
        assert run(n_tiles, n_units, seed) == "ok", (n_tiles, n_units, seed)


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


def run_frames(frames, seed, early_prep=False):
    """Rotate-on-read's Q handshake for one Q tile.  frames[u][j] is the frame of key
    tile j of unit u.  The softmax writes Q (for the unit's first frame at the unit
    start, and for the next frame after P of a frame's last tile) and arrives on
    q_ready; the issuer waits for q_ready before the unit's first S product and before
    the first S product of every new frame, and issues both P.V before the wait at a
    frame change.  Checked: every S product reads Q in its key tile's frame, and Q is
    never rewritten while an S product that reads it is still in flight.
    early_prep: the softmax writes the next frame's Q one key tile early."""
    rng = random.Random(seed)
    bars = {n: Bar(n, 1) for n in ("s_full", "p_full", "q_ready")}
    state = {"qbuf": None, "s_inflight": 0}
    pipe = []

    def s_done():
        state["s_inflight"] -= 1
        bars["s_full"].arrive()

    def issue_s(u, f):
        def act():
            if state["qbuf"] != (u, f):
                raise Aliased(f"S of unit {u} frame {f} read Q {state['qbuf']}")
            state["s_inflight"] += 1
            pipe.append(s_done)
        return act

    def prep(u, f):
        def act():
            if state["s_inflight"]:
                raise Aliased(f"Q rewritten for {(u, f)} under {state['s_inflight']} S products in flight")
            state["qbuf"] = (u, f)
            bars["q_ready"].arrive()
        return act

    def mma():
        uq = c = 0
        for u, fr in enumerate(frames):
            yield ("wait", "q_ready", uq)
            uq += 1
            yield ("act", issue_s(u, fr[0]))
            for j in range(len(fr)):
                yield ("wait", "p_full", c)
                c += 1
                if j + 1 < len(fr):
                    if fr[j + 1] != fr[j]:
                        yield ("wait", "q_ready", uq)
                        uq += 1
                    yield ("act", issue_s(u, fr[j + 1]))

    def softmax():
        yield ("act", prep(0, frames[0][0]))
        t = 0
        for u, fr in enumerate(frames):
            for j in range(len(fr)):
                if early_prep and j + 2 < len(fr) and fr[j + 2] != fr[j + 1]:
                    yield ("act", prep(u, fr[j + 2]))
                yield ("wait", "s_full", t)
                t += 1
                yield ("act", lambda: bars["p_full"].arrive())
                if not early_prep and j + 1 < len(fr) and fr[j + 1] != fr[j]:
                    yield ("act", prep(u, fr[j + 1]))
            if u + 1 < len(frames):
                yield ("act", prep(u + 1, frames[u + 1][0]))

    agents = [Agent("mma", mma()), Agent("softmax", softmax())]
    while True:
        live = [a for a in agents if not a.done]
        if not live and not pipe:
            return "ok"
        if pipe and rng.random() < 0.4:
            pipe.pop(0)()
            continue
        rng.shuffle(live)
        if not any(a.step(bars) for a in live):
            if pipe:
                pipe.pop(0)()
            else:
                return "deadlock: " + str([(a.name, a.cur[:3] if a.cur else None) for a in agents if not a.done])


def _frames(rng, n_units):
    out = []
    for _ in range(n_units):
        n = rng.randint(1, 12)
        f, fr = rng.randint(-1, 5), []
        for _ in range(n):
            if rng.random() < 0.3:
                f = rng.randint(-1, 5)
            fr.append(f)
        out.append(fr)
    return out


def test_rotate_on_read_q_handshake_is_safe():
    rng = random.Random(11)
    for seed in range(400):
        assert run_frames(_frames(rng, rng.randint(1, 5)), seed) == "ok", seed


def test_rotate_on_read_q_written_early_is_caught():
    rng = random.Random(12)
    caught = 0
    for seed in range(300):
        try:
            r = run_frames(_frames(rng, 3), seed, early_prep=True)
        except Aliased:
            caught += 1
            continue
        caught += r != "ok"
    assert caught > 0
