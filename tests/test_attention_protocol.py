"""Model check of the link attention kernel's K/V slot protocol (CPU, no GPU).

The roles that share the five K/V slots — the TMA producer (K and V of every key
tile, in turn), the V-zeroing warps (wait for the tile's K load, then its V
load, zero V's invalid rows, arrive vz_done),
the MMA issuer (waits only for vz_done of a tile before its first S product and
for the softmax's P; commits once per step to a ring of step barriers: a unit's
start frees its first K, key tile j's step frees V_j and K_(j+1)) and the
softmax (P from S) — are coroutines over the kernel's mbarriers, run in random
interleavings with the hardware's wait semantics (a wait for phase k passes
whenever the current phase's parity differs from k's) and copies that complete
in any order.  The issuer never waits for a load itself: that it has landed
reaches it through vz_done, which the model checks by recording, at every MMA,
whether the slot it reads holds the load it means.  The shipped protocol must
never deadlock, let a wait pass on a wrong phase or read a slot too early; the
variant whose V-zeroing warps waited only for the V loads of a slot (skipping
its K phases) is caught, and so is a step ring of four barriers, which runs of
one-tile units let the issuer lap.  A second model covers rotate-on-read's handshake on the
Q tile (written per key frame by the softmax warps, waited for by the issuer)."""

import random

import pytest

from test_compose_protocol import Agent, Aliased, Bar

SLOTS = 5
STEP_RING = 8


def run(tiles, seed, vzero_waits_k=True, mma_waits_tile=True, ring=STEP_RING, lagging_producer=False):
    """tiles[u]: key tiles of the CTA's unit u.  lagging_producer: the producer moves
    only once every other role is blocked and no copy or commit is in flight (a
    producer as slow as the protocol allows: the issuer runs as far ahead on the step
    barriers as the loads let it)."""
    rng = random.Random(seed)
    bars = {}

    def mk(name, count):
        bars[name] = Bar(name, count)

    for s in range(SLOTS):
        mk(f"kv_full{s}", 1)
        mk(f"vz_done{s}", 1)
    for r in range(ring):
        mk(f"kv_step{r}", 1)
    mk("s_full", 1)
    mk("p_full", 1)
    inflight, pipe = [], []
    landed = {}  # slot -> load number whose data the slot holds
    total = sum(tiles)  # key tiles over the CTA's units, loads ld = 0 .. 2 total - 1

    def land(s, ld):
        def f():
            landed[s] = ld
            bars[f"kv_full{s}"].arrive()
        return f

    def producer():
        ld, s0, free_step = 0, 0, [0] * SLOTS
        for n in tiles:
            for t in range(n):
                for kv in range(2):
                    s = ld % SLOTS
                    if ld >= SLOTS:
                        fs = free_step[s]
                        yield ("wait", f"kv_step{fs % ring}", fs // ring)
                    free_step[s] = s0 + t + kv
                    yield ("act", lambda s=s, ld=ld: inflight.append(land(s, ld)))
                    ld += 1
            s0 += n + 1

    def reads(ld):  # an MMA that reads load ld's slot: the data must be there
        def f():
            if landed.get(ld % SLOTS) != ld:
                raise Aliased(f"MMA read slot {ld % SLOTS} for load {ld} holding {landed.get(ld % SLOTS)}")
        return f

    def mma():
        ld, c, st = 0, 0, 0
        for n_tiles in tiles:
            yield ("wait", f"vz_done{(ld // 2) % SLOTS}", (ld // 2) // SLOTS)  # S of the unit's first tile
            yield ("act", reads(ld))
            pipe.append("s_full")
            pipe.append(f"kv_step{st % ring}")  # frees the unit's first K
            st += 1
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
                yield ("act", lambda r=st % ring: pipe.append(f"kv_step{r}"))  # frees V_j and K_(j+1)
                st += 1
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
        if lagging_producer:
            others = [a for a in live if a.name != "producer"]
            rng.shuffle(others)
            if any(a.step(bars) for a in others):
                continue
            if inflight:
                inflight.pop(rng.randrange(len(inflight)))()
                continue
            if pipe:
                bars[pipe.pop(0)].arrive()
                continue
            if any(a.step(bars) for a in live if a.name == "producer"):
                continue
            return "deadlock: " + str([(a.name, a.cur[:3] if a.cur else None) for a in agents if not a.done])
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


@pytest.mark.parametrize("tiles", [[1] * 6, [2] * 4, [3] * 3, [8] * 2, [13], [1] * 12,
                                   [1, 3, 1, 1, 2, 1, 1, 5], [4, 1, 1, 1, 1, 6]])
@pytest.mark.parametrize("lagging_producer", [False, True])
def test_shipped_slot_protocol_is_safe(tiles, lagging_producer):
    for seed in range(160):
        assert run(tiles, seed, lagging_producer=lagging_producer) == "ok", (tiles, seed)


def test_step_ring_of_four_is_caught():
    """Runs of one-tile units let the issuer complete five steps past the one the
    producer waits for: four barriers alias a phase."""
    caught = 0
    for seed in range(20):
        try:
            r = run([1] * 12, seed, ring=4, lagging_producer=True)
        except Aliased:
            caught += 1
            continue
        caught += r != "ok"
    assert caught > 0


def test_v_zeroing_that_skips_k_phases_is_caught():
    caught = 0
    for seed in range(300):
        try:
            run([1] * 8, seed, vzero_waits_k=False)
        except Aliased:
            caught += 1
    assert caught > 0


def test_issuer_that_skips_the_tile_wait_is_caught():
    """Without its vz_done wait the issuer would read a K slot before the load lands."""
    caught = 0
    for seed in range(300):
        try:
            r = run([4, 4], seed, mma_waits_tile=False)
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
