"""Model check of the decode kernel's ring protocol (CPU, no GPU).

A producer thread fills stage i % S with page i (a copy that completes in any
order) once the stage's previous page was released; consumer warp w takes pages
w, w + 4, .. : it waits for its page's stage, reads it and releases it.  With the
hardware's parity waits (a wait for phase k passes whenever the current phase's
parity differs from k's), a consumer must see every phase of its stages in
order, so every stage has to belong to one consumer warp: S a multiple of the
four warps.  The shipped S = 8 never deadlocks nor passes a wait on a wrong
phase; S = 9, where two warps share a stage, is caught."""

import random

import pytest

from test_compose_protocol import Agent, Aliased, Bar

WARPS = 4


def run(stages, n_pages, seed):
    rng = random.Random(seed)
    bars = {}
    for s in range(stages):
        bars[f"full{s}"] = Bar(f"full{s}", 1)
        bars[f"empty{s}"] = Bar(f"empty{s}", 1)
    inflight, holds = [], {}

    def land(s, i):
        def f():
            holds[s] = i
            bars[f"full{s}"].arrive()
        return f

    def consumer(w):
        for i in range(w, n_pages, WARPS):
            s = i % stages
            yield ("wait", f"full{s}", (i // stages))

            def read(s=s, i=i):
                if holds.get(s) != i:
                    raise Aliased(f"warp {w} read stage {s} for page {i} holding {holds.get(s)}")
            yield ("act", read)
            yield ("act", lambda s=s: bars[f"empty{s}"].arrive())

    agents = [Agent("producer", producer_waits(stages, n_pages, inflight, land))]
    agents += [Agent(f"warp{w}", consumer(w)) for w in range(WARPS)]
    while True:
        live = [a for a in agents if not a.done]
        if not live and not inflight:
            return "ok"
        moved = False
        if inflight and rng.random() < 0.3:
            inflight.pop(rng.randrange(len(inflight)))()
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
            else:
                return "deadlock"


def producer_waits(stages, n_pages, inflight, land):
    """The producer: page i waits for the release of page i - stages (phase i // stages - 1)."""
    for i in range(n_pages):
        s = i % stages
        if i >= stages:
            yield ("wait", f"empty{s}", i // stages - 1)
        yield ("act", lambda s=s, i=i: inflight.append(land(s, i)))


@pytest.mark.parametrize("n_pages", [1, 5, 17, 64])
def test_stages_owned_by_one_warp_are_safe(n_pages):
    for seed in range(100):
        assert run(8, n_pages, seed) == "ok", (n_pages, seed)


def test_a_stage_shared_by_two_warps_is_caught():
    bad = 0
    for seed in range(300):
        try:
            bad += run(9, 64, seed) != "ok"
        except Aliased:
            bad += 1
    assert bad > 0
