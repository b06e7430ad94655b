"""Model check of the composition kernel's barrier protocol (CPU, no GPU).

Every role of compose_kernel — the T and S producers, the MMA issuer, the eight
epilogue warps and the asynchronous completions (TMA copies, MMA commits) — is a
coroutine over the mbarriers it waits on and arrives at; random interleavings run
them with the hardware's wait semantics: a wait for phase k passes whenever the
barrier's current phase parity differs from k's, so a wait can wrongly pass on an
older phase of the same parity.  TMA copies complete in random order.  The test
asserts that the shipped protocol never deadlocks and that no wait ever passes
on a phase other than the one it means, and that the variant with one S ring
shared by the two epilogue halves is caught (the hazard the kernel's per-half
rings exist to avoid)."""

import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.P = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, (self.name, "more arrivals than the phase expects")
        if self.pending == 0:
            self.P += 1
            self.pending = self.count


class Aliased(Exception):
    pass


class Agent:
    def __init__(self, name, gen):
        self.name, self.gen, self.cur, self.done = name, gen, None, False

    def step(self, bars):
        if self.done:
            return False
        if self.cur is None:
            try:
                self.cur = next(self.gen)
            except StopIteration:
                self.done = True
                return True
        op = self.cur
        if op[0] == "wait":
            bar, k = bars[op[1]], op[2]
            passes = (bar.P & 1) != (k & 1)
            if passes and bar.P != k + 1:
                raise Aliased(f"{self.name}: wait for phase {k} of {op[1]} passed at phase count {bar.P}")
            if not passes:
                return False
            self.cur = None
            return True
        self.cur = None
        op[1]()
        return True


def run(n, need_t, seed, shared_ring=False, ring=3):
    """One random interleaving of a CTA folding n chain elements."""
    rng = random.Random(seed)
    bars = {}

    def mk(name, count):
        bars[name] = Bar(name, count)

    for i in range(2):
        mk(f"b_full{i}", 1)
        mk(f"b_empty{i}", 8)
    rings = 1 if shared_ring else 2
    for h in range(rings):
        for s in range(ring):
            mk(f"s_full{h}_{s}", 1)
            mk(f"s_empty{h}_{s}", 4)
    for x in ("a_s", "a_t"):
        mk(x, 8)
    for x in ("d_s", "d_t"):
        mk(x, 1)
    n_steps = n - 1
    inflight, pipe = [], []

    def block(h, q, u):
        """(ring, block number) of rows 64 h + 32 q of S(u)."""
        if shared_ring:
            return 0, 4 * u + 2 * h + q
        return h, 2 * u + q

    def prod_t():
        for j in range(n_steps):
            if j >= 2:
                yield ("wait", f"b_empty{j & 1}", (j - 2) >> 1)
            yield ("act", lambda j=j: inflight.append(f"b_full{j & 1}"))

    def prod_s():
        for u in range(n):
            for q in range(2):
                for h in range(2):
                    rg, w = block(h, q, u)
                    sl = w % ring
                    if w >= ring:
                        yield ("wait", f"s_empty{rg}_{sl}", w // ring - 1)
                    yield ("act", lambda rg=rg, sl=sl: inflight.append(f"s_full{rg}_{sl}"))

    def mma():
        for k in range(n_steps):
            yield ("wait", f"b_full{k & 1}", k >> 1)
            yield ("wait", "a_s", k)
            yield ("act", lambda: pipe.append("d_s"))
            if need_t:
                yield ("wait", "a_t", k)
                yield ("act", lambda: pipe.append("d_t"))

    def epi(w):
        hf = w >> 2
        su = [0]

        def s_emit():
            for q in range(2):
                rg, b = block(hf, q, su[0])
                sl = b % ring
                yield ("wait", f"s_full{rg}_{sl}", b // ring)
                yield ("act", lambda rg=rg, sl=sl: bars[f"s_empty{rg}_{sl}"].arrive())
            su[0] += 1

        yield from s_emit()
        if n_steps > 0:
            yield ("act", lambda: bars["a_s"].arrive())
            if need_t:
                yield ("act", lambda: bars["a_t"].arrive())
        for k in range(n_steps - 1):
            yield ("wait", "d_s", k)
            if not need_t:
                yield ("act", lambda k=k: bars[f"b_empty{k & 1}"].arrive())
            yield from s_emit()
            yield ("act", lambda: bars["a_s"].arrive())
            if need_t:
                yield ("wait", "d_t", k)
                yield ("act", lambda k=k: bars[f"b_empty{k & 1}"].arrive())
                yield ("act", lambda: bars["a_t"].arrive())
        if n_steps > 0:
            yield ("wait", "d_s", n_steps - 1)
            yield from s_emit()
            if need_t:
                yield ("wait", "d_t", n_steps - 1)

    agents = [Agent("prod_t", prod_t()), Agent("prod_s", prod_s()), Agent("mma", mma())]
    agents += [Agent(f"epi{w}", epi(w)) for w in range(8)]
    while True:
        live = [a for a in agents if not a.done]
        if not live and not inflight and not pipe:
            return "ok"
        moved = False
        if inflight and rng.random() < 0.3:  # a copy completes, in any order
            bars[inflight.pop(rng.randrange(len(inflight)))].arrive()
            moved = True
        elif pipe and rng.random() < 0.3:    # MMA commits complete in order
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


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 25])
@pytest.mark.parametrize("need_t", [False, True])
def test_shipped_protocol_is_safe(n, need_t):
    for seed in range(60 if n < 10 else 15):
        assert run(n, need_t, seed) == "ok", (n, need_t, seed)


def test_one_ring_shared_by_both_halves_is_caught():
    caught = 0
    for seed in range(200):
        try:
            run(4, False, seed, shared_ring=True)
        except Aliased:
            caught += 1
    assert caught > 0
