"""Model check, on the CPU, of the P hand-off protocol between the softmax warps of one query
tile and the MMA warp (the forward, which hands P over in two halves on two barriers per
step, and the FP8 kernel, with one; the backward's hand-offs follow the same rules with its S
and dP tiles as each step's input).

The hand-off is a hardware named barrier: the four softmax warps `bar.arrive`, the MMA warp
`bar.sync`s, and a phase completes when 4 + 1 warps have arrived (a warp counts as 32 threads
of the 160).  `bar.sync` has no timeout, so the protocol must guarantee by itself that the MMA
warp is never left waiting.  The model runs the two programs under random interleavings with a
failure injected (a K or V tile that never arrives, or an abort raised by another part of the
CTA), and checks that every run ends and that every completed phase holds exactly the arrivals
of one step.  It also checks that the model catches the rule the kernels no longer use (after a
failure, arrive for every remaining step at once), which lets arrivals fill a phase without
the MMA warp."""
import random

import pytest

WARPS = 4            # softmax warps of one tile
COUNT = WARPS + 1    # warps per barrier phase (160 threads)
TIMEOUT = 50         # ticks a bounded wait lasts before it gives up


class Barrier:
    """A named barrier: arrivals accumulate; at COUNT the phase completes and resets."""

    def __init__(self):
        self.pending = []          # (who, step) of the current phase
        self.phases = []           # completed phases
        self.generation = 0

    def arrive(self, who, step):
        self.pending.append((who, step))
        if len(self.pending) == COUNT:
            self.phases.append(self.pending)
            self.pending = []
            self.generation += 1


def run(nt, withheld, abort_at, paced, seed, halves=1):
    """One interleaving.  withheld: ring tile never loaded (K_j = 2j, V_j = 2j + 1) or None;
    abort_at: tick at which another part of the CTA raises the abort flag, or None; halves:
    barriers per step (the forward hands P over in two halves, keys 0-63 then 64-127, on two
    barriers; each softmax warp arrives on them in that order, and the MMA warp syncs on them in
    that order).  Returns 'ok' or 'deadlock', and the barriers."""
    rng = random.Random(seed)
    bars = [Barrier() for _ in range(halves)]
    state = {"t": 0, "abort": False}
    s_issue = {}                 # step -> tick at which S(j) is issued
    S_LATENCY = 3

    def loaded(u):
        return u != withheld

    def s_done(j):
        return j in s_issue and state["t"] >= s_issue[j] + S_LATENCY

    # The programs are generators that yield a wait condition: ('wait', pred, honour_abort),
    # ('sync', barrier, generation_to_pass) or ('step',).  A bounded wait fails after TIMEOUT ticks.
    def mma():
        for j in range(nt + 1):
            if j >= 1:
                ok = yield ("wait", lambda j=j: loaded(2 * (j - 1) + 1), True)
                if not ok:
                    return
                for h, bar in enumerate(bars):
                    bar.arrive("mma", j - 1)
                    gen = bar.generation if bar.pending else bar.generation - 1
                    if bar.pending:
                        yield ("sync", h, gen)
            if j < nt:
                ok = yield ("wait", lambda j=j: loaded(2 * j), True)
                if not ok:
                    return
                s_issue[j] = state["t"]

    def softmax(w):
        j = 0
        while j < nt:
            ok = yield ("wait", lambda j=j: s_done(j), True)
            if not ok:
                break
            for bar in bars:
                yield ("step",)            # the softmax work for this part of P
                bar.arrive(w, j)
            j += 1
        if paced:                      # each remaining step's arrivals once S(j) is complete
            while j < nt:
                ok = yield ("wait", lambda j=j: s_done(j), False)
                if not ok:
                    return
                for bar in bars:
                    bar.arrive(w, j)
                j += 1
        else:                          # the rejected rule: arrive for every remaining step at once
            while j < nt:
                for bar in bars:
                    bar.arrive(w, j)
                j += 1

    actors = {"mma": mma()}
    actors.update({f"w{i}": softmax(f"w{i}") for i in range(WARPS)})
    waiting = {name: None for name in actors}      # current request of each actor
    started = {name: 0 for name in actors}
    live = set(actors)

    def advance(name, value):
        try:
            req = actors[name].send(value)
            waiting[name] = req
            started[name] = state["t"]
        except StopIteration:
            live.discard(name)

    for name in list(actors):
        advance(name, None)

    for _ in range(100000):
        if not live:
            return "ok", bars
        if abort_at is not None and state["t"] >= abort_at:
            state["abort"] = True
        ready = []
        for name in live:
            req = waiting[name]
            if req[0] == "step":
                ready.append((name, None))
            elif req[0] == "sync":
                if bars[req[1]].generation > req[2]:
                    ready.append((name, None))
            else:
                _, pred, honour = req
                if pred():
                    ready.append((name, True))
                elif (honour and state["abort"]) or state["t"] - started[name] >= TIMEOUT:
                    state["abort"] = True
                    ready.append((name, False))
        if ready:
            name, value = rng.choice(ready)
            advance(name, value)
        else:
            if all(waiting[n][0] == "sync" for n in live) and all(
                    bars[waiting[n][1]].generation <= waiting[n][2] for n in live):
                return "deadlock", bars    # only unbounded waits are left, and none can pass
        state["t"] += 1
    return "deadlock", bars


def phases_are_clean(bars):
    """Every completed phase of every barrier that includes the MMA warp holds one arrival of
    each softmax warp, all for the step the MMA warp waited for."""
    for bar in bars:
        for phase in bar.phases:
            steps = {step for who, step in phase if who == "mma"}
            if not steps:
                continue
            (step,) = steps
            warps = sorted(who for who, s in phase if who != "mma")
            if warps != [f"w{i}" for i in range(WARPS)] or any(s != step for who, s in phase):
                return False
    return True


CASES = [(nt, withheld, abort_at) for nt in (1, 3, 6)
         for withheld in (None, 0, 1, 2, 3, 5, 8)
         for abort_at in (None, 0, 4, 11, 27)]


@pytest.mark.parametrize("halves", [1, 2])
@pytest.mark.parametrize("nt,withheld,abort_at", CASES)
def test_paced_handoff_never_hangs(nt, withheld, abort_at, halves):
    for seed in range(25):
        outcome, bars = run(nt, withheld, abort_at, paced=True, seed=seed, halves=halves)
        assert outcome == "ok", (nt, withheld, abort_at, seed)
        assert phases_are_clean(bars), (nt, withheld, abort_at, seed, [b.phases for b in bars])


@pytest.mark.parametrize("halves", [1, 2])
def test_clean_run_hands_over_every_step(halves):
    outcome, bars = run(6, None, None, paced=True, seed=1, halves=halves)
    assert outcome == "ok"
    assert all(len(b.phases) == 6 for b in bars) and phases_are_clean(bars)


@pytest.mark.parametrize("halves", [1, 2])
def test_arriving_for_every_remaining_step_at_once_can_hang(halves):
    """The rejected rule: after an abort raised elsewhere, the softmax warps arrive for all
    their remaining steps at once; some interleaving then fills a phase without the MMA warp
    and leaves it one phase short at its bar.sync."""
    bad = 0
    for nt, withheld, abort_at in CASES:
        for seed in range(25):
            outcome, bars = run(nt, withheld, abort_at, paced=False, seed=seed, halves=halves)
            if outcome != "ok" or not phases_are_clean(bars):
                bad += 1
    assert bad > 0
