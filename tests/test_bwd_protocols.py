"""Barrier protocols of the backward's pair-term kernels, run on a model of
mbarrier phases under random schedules.

Each role of a CTA is a program of waits and arrivals on barriers that keep
a completed-phase count; a wait on parity P returns once the barrier's
current (incomplete) phase has a parity other than P, as `mbarrier.try_wait.
parity` does.  Asynchronous completions (a TMA copy landing, the MMAs behind
a `tcgen05.commit`, a bulk store reading its source) are arrivals that
happen at a random later point.  A schedule picks a random role that can
move, or a pending completion, until every role has finished; if none can
move first, the protocol deadlocks.  A wait that lets a barrier complete two
phases past the one it means would see the same parity again and block for
good, so phase skipping shows up as a deadlock too.

Modelled (the orders of `relattn_bwd_pairs.cu`):
* the pair kernel: the loader (step t's inputs into stage t % NS, refilled
  for step t + NS once the MMAs of step t have read it), the MMA thread
  (step t's MMAs after its inputs and, from step 2 on, after every pair warp
  has finished step t - 2), the eight pair warps (step t after its MMAs; the
  staging after the stores of step t - 1 have read it), the store thread;
* the products kernel: the producer (tile indices from the counter through
  an 8-slot queue, then the tile's k blocks into a ring of stages), the MMA
  thread (one of two accumulator slots per tile) and the four epilogue
  warps.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0  # completed phases

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the barrier's count"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passed(self, parity):
        return (self.phase & 1) != parity


def run(programs, bars, seed, max_moves=200000):
    """Runs generator programs yielding ("wait", bar, parity), ("arrive",
    bar) or ("async", bar) (an arrival at a random later point)."""
    rng = random.Random(seed)
    roles = {name: prog for name, prog in programs.items()}
    current = {name: next(prog, None) for name, prog in roles.items()}
    pending = []  # asynchronous arrivals
    for _ in range(max_moves):
        movable = []
        for name, op in current.items():
            if op is None:
                continue
            if op[0] == "wait" and not bars[op[1]].passed(op[2]):
                continue
            movable.append(name)
        if not movable and not pending:
            if all(op is None for op in current.values()):
                return
            stuck = {n: op for n, op in current.items() if op is not None}
            raise AssertionError(f"deadlock (seed {seed}): {stuck}")
        if pending and (not movable or rng.random() < 0.3):
            bars[pending.pop(rng.randrange(len(pending)))].arrive()
            continue
        name = rng.choice(movable)
        op = current[name]
        if op[0] == "arrive":
            bars[op[1]].arrive()
        elif op[0] == "async":
            pending.append(op[1])
        current[name] = next(roles[name], None)
    raise AssertionError("no end within the move budget")


def pair_kernel(T, NS, inject_stall=False):
    """Programs of bwd_pairs_kernel for one CTA of T key steps."""
    bars = {"q": Bar(1), "x": Bar(1), "sfree": Bar(1), "fin": Bar(1), "build": Bar(8)}
    for s in range(NS):
        bars[f"in{s}"] = Bar(1)
        bars[f"ifree{s}"] = Bar(1)
    for s in range(2):
        bars[f"m1{s}"] = Bar(1)
        bars[f"done{s}"] = Bar(8)

    def loader():
        yield ("async", "q")  # raw q and dout
        yield ("async", "in0")  # step 0 into stage 0
        if NS == 3 and T > 2 and not inject_stall:
            yield ("async", "in2")
        yield ("async", "x")  # the rest of step 0's window
        yield ("wait", "build", 0)  # the raw q in stage 1 has been read
        if T > 1:
            yield ("async", "in1")
        t = 0
        while t + NS < T and not inject_stall:
            yield ("wait", f"ifree{t % NS}", (t // NS) & 1)
            yield ("async", f"in{(t + NS) % NS}")
            t += 1

    def score_mmas(t):
        yield ("wait", f"in{t % NS}", (t // NS) & 1)
        if t == 0:
            yield ("wait", "x", 0)
        yield ("async", f"m1{t & 1}")
        yield ("async", f"ifree{t % NS}")

    def mma():
        yield ("wait", "build", 0)
        yield from score_mmas(0)
        if T > 1:
            yield from score_mmas(1)
        for t in range(T - 2):
            yield ("wait", f"done{t & 1}", (t >> 1) & 1)
            yield from score_mmas(t + 2)

    def storer():
        for t in range(T):
            yield ("wait", f"done{t & 1}", (t >> 1) & 1)
            yield ("async", "sfree")  # the bulk stores have read the staging

    def pair_warp():
        yield ("wait", "q", 0)
        yield ("arrive", "build")
        for t in range(T):
            yield ("wait", f"m1{t & 1}", (t >> 1) & 1)
            if t > 0:
                yield ("wait", "sfree", (t - 1) & 1)
            yield ("arrive", f"done{t & 1}")

    progs = {"loader": loader(), "mma": mma(), "storer": storer()}
    for w in range(8):
        progs[f"pair{w}"] = pair_warp()
    return progs, bars


@pytest.mark.parametrize("NS", [2, 3])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 7, 12])
def test_pair_kernel_protocol(T, NS):
    for seed in range(60):
        progs, bars = pair_kernel(T, NS)
        run(progs, bars, seed)


@pytest.mark.parametrize("NS", [2, 3])
def test_pair_kernel_stall_hook_deadlocks_only_past_two_steps(NS):
    """With the test hook's stall the loads stop after two steps: a CTA of two
    steps still finishes, one of three or more cannot (its bounded waits run
    out on the GPU)."""
    progs, bars = pair_kernel(2, NS, inject_stall=True)
    run(progs, bars, 0)
    progs, bars = pair_kernel(3, NS, inject_stall=True)
    with pytest.raises(AssertionError, match="deadlock"):
        run(progs, bars, 0)


def products_kernel(tiles, S=6, Q=8, ctas=1, seed=0):
    """Programs of bgemm_kernel for one CTA taking tiles from a counter; the
    other CTAs' takes are modelled by the counter skipping random indices.
    tiles: k blocks of each tile in counter order."""
    rng = random.Random(seed)
    bars = {"done": Bar(1)}
    for s in range(S):
        bars[f"full{s}"] = Bar(1)
        bars[f"empty{s}"] = Bar(1)
    for a in range(2):
        bars[f"accf{a}"] = Bar(1)
        bars[f"acce{a}"] = Bar(4)
    for q in range(Q):
        bars[f"tqf{q}"] = Bar(1)
        bars[f"tqe{q}"] = Bar(5)
    mine = [u for u in range(len(tiles)) if ctas == 1 or rng.random() < 1.0 / ctas]
    order = mine + [len(tiles)]  # the index past the end stops every role
    ring = [None] * Q  # the queue's shared-memory slots

    def take(n):  # a consumer reads slot n % Q and must find the n-th index
        u = ring[n % Q]
        assert u == order[n], f"queue slot overrun: read {u} for the {n}-th tile {order[n]}"
        return u

    def producer():
        it = 0
        for n, u in enumerate(order):
            yield ("wait", f"tqe{n % Q}", ((n // Q) & 1) ^ 1)
            ring[n % Q] = u
            yield ("arrive", f"tqf{n % Q}")
            if u >= len(tiles):
                return
            for _ in range(tiles[u]):
                yield ("wait", f"empty{it % S}", ((it // S) & 1) ^ 1)
                yield ("async", f"full{it % S}")  # the TMA loads land
                it += 1

    def mma():
        it = tl = 0
        for n in range(len(order)):
            yield ("wait", f"tqf{n % Q}", (n // Q) & 1)
            u = take(n)
            yield ("arrive", f"tqe{n % Q}")
            if u >= len(tiles):
                break
            acc = tl & 1
            if tl >= 2:
                yield ("wait", f"acce{acc}", ((tl >> 1) - 1) & 1)
            for _ in range(tiles[u]):
                yield ("wait", f"full{it % S}", (it // S) & 1)
                yield ("async", f"empty{it % S}")  # tcgen05.commit: the MMAs have read the stage
                it += 1
            yield ("async", f"accf{acc}")
            tl += 1
        yield ("async", "done")
        yield ("wait", "done", 0)

    def epilogue():
        tl = 0
        for n in range(len(order)):
            yield ("wait", f"tqf{n % Q}", (n // Q) & 1)
            u = take(n)
            yield ("arrive", f"tqe{n % Q}")
            if u >= len(tiles):
                return
            acc = tl & 1
            yield ("wait", f"accf{acc}", (tl >> 1) & 1)
            yield ("arrive", f"acce{acc}")
            tl += 1

    progs = {"producer": producer(), "mma": mma()}
    for w in range(4):
        progs[f"epi{w}"] = epilogue()
    return progs, bars, ring, order


@pytest.mark.parametrize("S", [6, 8])
@pytest.mark.parametrize("ctas", [1, 3])
def test_products_kernel_protocol(S, ctas):
    rng = random.Random(S * 10 + ctas)
    for seed in range(40):
        # DR tiles (long), DQ tiles, then DK / DV tiles of two k blocks or more
        tiles = [rng.choice([16, 32, 96]) for _ in range(3)] + [rng.randrange(2, 49) for _ in range(6)] + \
                [rng.randrange(1, 13) for _ in range(20)]
        progs, bars, _, _ = products_kernel(tiles, S=S, ctas=ctas, seed=seed)
        run(progs, bars, seed)


def test_model_catches_a_skipped_phase():
    """The model is not vacuous: a producer that does not wait for a queue
    slot to be read before writing it again overruns the slot (a consumer
    reads a later tile's index) or arrives on the slot's barrier twice in one
    phase, moving it past the phase a consumer waits for."""
    tiles = [1] * 40
    failures = 0
    for seed in range(20):
        progs, bars, ring, order = products_kernel(tiles, S=6, Q=2, seed=seed)

        def producer():  # the slot wait removed
            for n, u in enumerate(order):
                ring[n % 2] = u
                yield ("arrive", f"tqf{n % 2}")
                if u >= len(tiles):
                    return
                yield ("wait", f"empty{n % 6}", ((n // 6) & 1) ^ 1)
                yield ("async", f"full{n % 6}")

        progs["producer"] = producer()
        try:
            run(progs, bars, seed)
        except AssertionError:
            failures += 1
    assert failures == 20
