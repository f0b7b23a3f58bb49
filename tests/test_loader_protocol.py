"""Deadlock check of the D = 64 attention kernel's hand-offs, at tile granularity.

Each role of a CTA (the TMA loader, the three MMA issuers and the two softmax
step parities) is modelled as an ordered program of actions; an action waits
for the actions that its barriers stand for:

* loader: per unit, the queued V tiles of units two or more back, then the
  raw q of the unit after next (single buffer: free once both parities have
  built (q+u), (q+v) of the next unit), distance tiles -2 and -1, then per
  step K(t) (stage free once the score MMA four tiles back is done), R(t+1)
  (free once the distance MMA four tiles back is done) and the queued V(t),
  issued once more than `lag` V tiles wait (stage free once the P.V four
  tiles back is done);
* score issuer: S(g) after K(g), the read of step g-2 (S buffer) and the
  unit's (q+u);
* distance issuer: tile x after R(x), every read of the tile four back (its
  ring slot) and the unit's (q+v);
* P.V issuer: PV(g) after P(g), V(g) and, for a unit's first two steps, the
  previous unit's epilogue (O accumulators);
* softmax parity p (steps with g % 2 == p): read(g) after S(g) and the
  distance tiles of step g, P(g) after the P.V of step g-2 (P buffer); after
  its first step of a unit, its half of the next unit's (q+u), (q+v) (needs
  that raw q); at the unit's end the owner of the last step runs the
  epilogue (all P.V of the unit, the other parity's (m, l)), the other hands
  over its (m, l) once the previous epilogue has read the last one.

Random schedules run every ready role until all finish or none can move.
"""
import random

import pytest

NK = NV = NR = 4


def _programs(nks, lag, flush):
    """Programs for a CTA that runs units with the given key-step counts."""
    n_units = len(nks)
    g0 = [sum(nks[:u]) for u in range(n_units)]
    x0 = [g0[u] + 2 * u for u in range(n_units)]  # global index of each unit's distance tile -2

    def tiles_of_step(u, t):  # the three ring tiles a step reads (tile e of the unit: x0 + e + 2)
        return [x0[u] + t + 2 - k for k in range(3)]

    readers = {}  # distance tile -> steps that read it
    unit_of_tile = {}
    for u in range(n_units):
        for e in range(-2, nks[u]):
            unit_of_tile[x0[u] + e + 2] = u
        for t in range(nks[u]):
            for x in tiles_of_step(u, t):
                readers.setdefault(x, []).append(g0[u] + t)
    n_tiles = sum(n + 2 for n in nks)
    unit_of_step = [u for u in range(n_units) for _ in range(nks[u])]
    G = len(unit_of_step)

    def owner(u):
        return (g0[u] + nks[u] - 1) & 1

    def build_deps(u):  # (q+u), (q+v) of unit u ready: both parities built it
        return [("B", p, u) for p in (0, 1)] if u > 0 else [("B0",)]

    progs = {}
    # ---- loader
    loader = []
    loader.append((("LQ", 0), []))
    vq, nv = [], 0  # queued V tiles (step, unit)

    def issue_v():
        nonlocal nv
        g, _ = vq.pop(0)
        loader.append((("LV", g), [("PV", g - NV)] if g >= NV else []))
        nv += 1

    nr = 0
    for u in range(n_units):
        if flush:
            while vq and vq[0][1] <= u - 2:
                issue_v()
        if u + 1 < n_units:
            # single raw q buffer: free once unit u's (q+u), (q+v) are built
            loader.append((("LQ", u + 1), build_deps(u)))
        for _ in range(2):
            loader.append((("LR", nr), [("G", nr - NR)] if nr >= NR else []))
            nr += 1
        for t in range(nks[u]):
            g = g0[u] + t
            loader.append((("LK", g), [("S", g - NK)] if g >= NK else []))
            loader.append((("LR", nr), [("G", nr - NR)] if nr >= NR else []))
            nr += 1
            vq.append((g, u))
            if len(vq) > lag:
                issue_v()
    while vq:
        issue_v()
    progs["loader"] = loader
    # ---- score issuer
    progs["S"] = [(("S", g), [("LK", g)] + ([("RD", g - 2)] if g >= 2 else []) + build_deps(unit_of_step[g]))
                  for g in range(G)]
    # ---- distance issuer
    gi = []
    for x in range(n_tiles):
        deps = [("LR", x)] + build_deps(unit_of_tile[x])
        if x >= 4:
            deps += [("RD", r) for r in readers.get(x - 4, [])]
        gi.append((("G", x), deps))
    progs["G"] = gi
    # ---- P.V issuer
    pv = []
    for u in range(n_units):
        for t in range(nks[u]):
            g = g0[u] + t
            deps = [("P", g), ("LV", g)]
            if t < 2 and u > 0:
                deps.append(("EP", u - 1))
            pv.append((("PV", g), deps))
    progs["PV"] = pv
    # ---- softmax parities
    for p in (0, 1):
        prog = [] if p else [(("B0",), [("LQ", 0)])]
        for u in range(n_units):
            own = [t for t in range(nks[u]) if (g0[u] + t) & 1 == p]
            for t in own:
                g = g0[u] + t
                prog.append((("RD", g), [("S", g)] + [("G", x) for x in tiles_of_step(u, t)]))
                prog.append((("P", g), [("PV", g - 2)] if g >= 2 else []))
                if t == own[0] and u + 1 < n_units:
                    prog.append((("B", p, u + 1), [("LQ", u + 1)]))
            if not own and u + 1 < n_units:
                last = g0[u] + nks[u] - 1
                prog.append((("B", p, u + 1), [("S", last), ("LQ", u + 1)]))
            if p == owner(u):
                prog.append((("EP", u), [("LB", u)] + [("PV", g0[u] + t) for t in range(nks[u])]))
            else:
                prog.append((("LB", u), [("EP", u - 1)] if u > 0 else []))
        progs[f"sm{p}"] = prog
    # the first unit's (q+u), (q+v): built by both parities before the loop (one action here)
    progs["sm0"].insert(1, (("B", 1, 0), []))
    return progs


def _run(progs, rng):
    done = set()
    pc = {k: 0 for k in progs}
    while True:
        ready = [k for k, prog in progs.items()
                 if pc[k] < len(prog) and all(d in done for d in prog[pc[k]][1])]
        if not ready:
            return all(pc[k] == len(progs[k]) for k in progs), pc
        k = rng.choice(ready)
        done.add(progs[k][pc[k]][0])
        pc[k] += 1


UNIT_MIXES = [
    [1] * 9,
    [1, 2, 1, 1, 3, 1, 1],
    [16, 16, 14, 12, 10],
    [3, 1, 1, 2, 1, 5, 1, 1, 1],
    [2] * 8,
]


@pytest.mark.parametrize("lag", [0, 1, 2, 3])
@pytest.mark.parametrize("nks", UNIT_MIXES)
def test_loader_queue_never_deadlocks(nks, lag):
    for seed in range(40):
        ok, pc = _run(_programs(nks, lag, flush=True), random.Random(seed))
        assert ok, f"deadlock for units {nks}, lag {lag}, seed {seed}: {pc}"


def test_model_finds_the_hazard_without_the_flush():
    """Mutation check of the model: without issuing the queued V tiles of
    units two back before the raw q load, one-step units deadlock."""
    ok, _ = _run(_programs([1] * 9, 2, flush=False), random.Random(0))
    assert not ok
