"""Model check, on the CPU, of the backward kernels' hand-off protocol (the dK/dV kernel: P^T and
dS^T per query tile on two named barriers; the dQ kernel: dS per key tile on one), with the
producer's ring and the bounded waits of every warp.

The eight compute warps `bar.arrive` and the MMA warp `bar.sync`s; a phase completes when
8 + 1 warps have arrived.  `bar.sync` has no timeout, so the protocol itself must guarantee
that the MMA warp is never left waiting.  Each kernel's warps are modelled as programs run under
random interleavings, with a failure injected (a ring tile that never arrives, as the
`fa_bwd_withheld_tile` hook does, or an abort raised elsewhere in the CTA).  Every run must end,
and every completed phase must hold the arrivals of one step only: the MMA warp's and one from
each compute warp.  The model must also catch the rule the kernels do not use (after a failure,
arrive for every remaining step at once)."""
import random

import pytest

WARPS = 8            # compute warps
COUNT = WARPS + 1    # warps per barrier phase (288 threads)
TIMEOUT = 60         # ticks a bounded wait lasts before it gives up
LAT = 3              # ticks from issue to completion of a load or a tensor-core product


class Barrier:
    """A named barrier: arrivals accumulate; at COUNT the phase completes and resets."""

    def __init__(self):
        self.pending = []
        self.phases = []
        self.generation = 0

    def arrive(self, who, step):
        self.pending.append((who, step))
        if len(self.pending) == COUNT:
            self.phases.append(self.pending)
            self.pending = []
            self.generation += 1


def _sync(bars, b, who, step):
    """The MMA warp's bar.sync: arrive, then wait for the phase its arrival belongs to."""
    bar = bars[b]
    bar.arrive(who, step)
    gen = bar.generation if bar.pending else bar.generation - 1
    return ("sync", b, gen)


def run_dkdv(n_q, stages, withheld, abort_at, paced, seed):
    """dK/dV kernel.  Ring stage u holds query tile u (Q, dO, LSE, D); withheld: a tile that is
    never loaded (the test hook withholds tile 0) or None.  Barriers: 0 = P^T handed over,
    1 = dS^T handed over."""
    t = {"now": 0, "abort": False}
    full_at, s_at, dp_at, empty_at = {}, {}, {}, {}
    bars = [Barrier(), Barrier()]

    def done(table, u):
        return u in table and t["now"] >= table[u]

    def producer():
        for u in range(n_q):
            if u >= stages:
                ok = yield ("wait", lambda u=u: done(empty_at, u - stages), True)
                if not ok:
                    return
            if u != withheld:
                full_at[u] = t["now"] + LAT

    def mma():
        if n_q == 0:
            return
        ok = yield ("wait", lambda: done(full_at, 0), True)
        if not ok:
            return
        s_at[0] = dp_at[0] = t["now"] + LAT
        for u in range(n_q):
            yield _sync(bars, 0, "mma", u)                      # P^T(u): dV(u)
            if u + 1 < n_q:
                ok = yield ("wait", lambda u=u: done(full_at, u + 1), True)
                if not ok:
                    return
                s_at[u + 1] = t["now"] + LAT                    # S^T(u+1)
            yield _sync(bars, 1, "mma", u)                      # dS^T(u): dK(u)
            empty_at[u] = t["now"] + LAT
            if u + 1 < n_q:
                dp_at[u + 1] = t["now"] + LAT                   # dP^T(u+1)

    def compute(w):
        u, np_, ok = 0, 0, True
        while u < n_q:
            ok = yield ("wait", lambda u=u: done(s_at, u), True)
            if not ok:
                break
            yield ("step",)
            bars[0].arrive(w, u)
            np_ = u + 1
            ok = yield ("wait", lambda u=u: done(dp_at, u), True)
            if not ok:
                break
            yield ("step",)
            bars[1].arrive(w, u)
            u += 1
        if ok:
            return
        if not paced:                  # the rejected rule: every remaining arrival at once
            while u < n_q:
                if np_ == u:
                    bars[0].arrive(w, u)
                    np_ += 1
                bars[1].arrive(w, u)
                u += 1
            return
        while u < n_q:                 # each arrival once the input of its step is complete
            if np_ == u:
                ok = yield ("wait", lambda u=u: done(s_at, u), False)
                if not ok:
                    return
                bars[0].arrive(w, u)
                np_ += 1
            ok = yield ("wait", lambda u=u: done(dp_at, u), False)
            if not ok:
                return
            bars[1].arrive(w, u)
            u += 1

    actors = {"producer": producer(), "mma": mma()}
    actors.update({f"w{i}": compute(f"w{i}") for i in range(WARPS)})
    return _schedule(actors, bars, t, abort_at, seed)


def run_dq(n_kv, slots, withheld, abort_at, paced, seed):
    """dQ kernel.  Ring position u holds K_{u/2} (u even) or V_{u/2} (u odd); withheld: a
    position that is never loaded (the test hook withholds V_0, position 1) or None.  Barrier
    0 = dS handed over."""
    t = {"now": 0, "abort": False}
    full_at, s_at, dp_at, empty_at = {}, {}, {}, {}
    bars = [Barrier()]

    def done(table, u):
        return u in table and t["now"] >= table[u]

    def producer():
        for u in range(2 * n_kv):
            if u >= slots:
                ok = yield ("wait", lambda u=u: done(empty_at, u - slots), True)
                if not ok:
                    return
            if u != withheld:
                full_at[u] = t["now"] + LAT

    def mma():
        def issue_s(j):
            ok = yield ("wait", lambda: done(full_at, 2 * j), True)
            if ok:
                s_at[j] = t["now"] + LAT
            return ok

        def issue_dp(j):
            ok = yield ("wait", lambda: done(full_at, 2 * j + 1), True)
            if ok:
                dp_at[j] = empty_at[2 * j + 1] = t["now"] + LAT   # V_j read by dP(j) only
            return ok

        if n_kv == 0:
            return
        ok = (yield from issue_s(0)) and (yield from issue_dp(0)) and (n_kv < 2 or (yield from issue_s(1)))
        j = 0
        while ok and j < n_kv:
            yield _sync(bars, 0, "mma", j)                      # dS(j)
            if j + 1 < n_kv and not (yield from issue_dp(j + 1)):
                return
            empty_at[2 * j] = t["now"] + LAT                    # dQ(j) reads K_j
            if j + 2 < n_kv and not (yield from issue_s(j + 2)):
                return
            j += 1

    def compute(w):
        j, ok = 0, True
        while j < n_kv:
            ok = yield ("wait", lambda j=j: done(s_at, j), True)
            if not ok:
                break
            yield ("step",)
            ok = yield ("wait", lambda j=j: done(dp_at, j), True)
            if not ok:
                break
            yield ("step",)
            bars[0].arrive(w, j)
            j += 1
        if ok:
            return
        while j < n_kv:
            if paced:
                ok = yield ("wait", lambda j=j: done(dp_at, j), False)
                if not ok:
                    return
            bars[0].arrive(w, j)
            j += 1

    actors = {"producer": producer(), "mma": mma()}
    actors.update({f"w{i}": compute(f"w{i}") for i in range(WARPS)})
    return _schedule(actors, bars, t, abort_at, seed)


def _schedule(actors, bars, t, abort_at, seed):
    """Run the programs under one random interleaving.  A program yields ('wait', pred,
    honour_abort) -- a bounded wait that fails after TIMEOUT ticks, or at once on an abort if
    it honours it, and raises the abort when it times out --, ('sync', barrier, generation) or
    ('step',).  Returns 'ok' once every program has ended, or 'deadlock' when only bar.syncs that
    can no longer pass are left."""
    rng = random.Random(seed)
    waiting, started, live = {}, {}, set(actors)

    def advance(name, value):
        try:
            waiting[name] = actors[name].send(value)
            started[name] = t["now"]
        except StopIteration:
            live.discard(name)

    for name in list(actors):
        advance(name, None)
    for _ in range(200000):
        if not live:
            return "ok", bars
        if abort_at is not None and t["now"] >= abort_at:
            t["abort"] = True
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
                elif (honour and t["abort"]) or t["now"] - started[name] >= TIMEOUT:
                    t["abort"] = True
                    ready.append((name, False))
        if ready:
            advance(*rng.choice(sorted(ready)))
        elif all(waiting[n][0] == "sync" for n in live):
            return "deadlock", bars
        t["now"] += 1
    return "deadlock", bars


def phases_are_clean(bars):
    """Every completed phase holds the MMA warp's arrival and one of each compute warp, all for
    one step."""
    for bar in bars:
        for phase in bar.phases:
            steps = {step for _, step in phase}
            warps = sorted(who for who, _ in phase)
            if len(steps) != 1 or warps != sorted(["mma"] + [f"w{i}" for i in range(WARPS)]):
                return False
    return True


DKDV_CASES = [(n_q, stages, withheld, abort_at) for n_q, stages in ((1, 2), (3, 2), (6, 2), (5, 4))
              for withheld in (None, 0, 1, 3)
              for abort_at in (None, 0, 7, 19)]
DQ_CASES = [(n_kv, withheld, abort_at) for n_kv in (1, 2, 4, 7)
            for withheld in (None, 1, 0, 4, 9)
            for abort_at in (None, 0, 9, 23)]


@pytest.mark.parametrize("n_q,stages,withheld,abort_at", DKDV_CASES)
def test_dkdv_handoff_never_hangs(n_q, stages, withheld, abort_at):
    for seed in range(12):
        outcome, bars = run_dkdv(n_q, stages, withheld, abort_at, paced=True, seed=seed)
        assert outcome == "ok", (n_q, stages, withheld, abort_at, seed)
        assert phases_are_clean(bars), (n_q, stages, withheld, abort_at, seed)


@pytest.mark.parametrize("n_kv,withheld,abort_at", DQ_CASES)
def test_dq_handoff_never_hangs(n_kv, withheld, abort_at):
    for seed in range(12):
        outcome, bars = run_dq(n_kv, 5, withheld, abort_at, paced=True, seed=seed)
        assert outcome == "ok", (n_kv, withheld, abort_at, seed)
        assert phases_are_clean(bars), (n_kv, withheld, abort_at, seed)


def test_clean_runs_hand_over_every_step():
    outcome, bars = run_dkdv(6, 2, None, None, paced=True, seed=3)
    assert outcome == "ok" and phases_are_clean(bars)
    assert [len(b.phases) for b in bars] == [6, 6]
    outcome, bars = run_dq(7, 5, None, None, paced=True, seed=3)
    assert outcome == "ok" and phases_are_clean(bars) and len(bars[0].phases) == 7


def test_arriving_for_every_remaining_step_at_once_is_caught():
    """The rejected rule: after a failure, arrive for all remaining steps at once.  Some
    interleaving then fills a phase without the MMA warp or mixes two steps in one."""
    bad = 0
    for n_q, stages, withheld, abort_at in DKDV_CASES:
        for seed in range(12):
            outcome, bars = run_dkdv(n_q, stages, withheld, abort_at, paced=False, seed=seed)
            bad += outcome != "ok" or not phases_are_clean(bars)
    assert bad > 0
    bad = 0
    for n_kv, withheld, abort_at in DQ_CASES:
        for seed in range(12):
            outcome, bars = run_dq(n_kv, 5, withheld, abort_at, paced=False, seed=seed)
            bad += outcome != "ok" or not phases_are_clean(bars)
    assert bad > 0
