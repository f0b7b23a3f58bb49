"""The bf16 attention's unit plan and key-range split, checked on the host
(no GPU), through the library's own host code.

With more (sequence, head, 128-query tile) units than SMs, the persistent
attention kernels take their units from a table the host builds once per
shape (`txl_debug_unit_plan` returns it as the library builds it).  A unit
missing from the table leaves its outputs unwritten and a unit listed twice
writes them twice, so the table must hold every unit exactly once.  Each
CTA's row runs longest first, as its list ends with -1.  The balance is
that of list scheduling: greedy longest-first dealing followed by moves and
swaps that only lower the busiest CTA, so the busiest CTA's cost is at most
the average plus the longest unit (Graham's bound) and at most the greedy
start's; the cost of a unit is its 64-key steps (up
to the last visible key of its last query row, "Transformer-XL, explained",
method steps 3-4: query i sees keys j <= M + i) plus 1.2 steps for a unit
boundary.
"""
import ctypes
import heapq
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "transformer_xl_relative_txl_gb300", "libtxl_relattn.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        subprocess.check_call([sys.executable, os.path.join(ROOT, "transformer_xl_relative_txl_gb300", "build.py")])
    L = ctypes.CDLL(LIB)
    L.txl_debug_unit_plan.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_int,
                                                           ctypes.POINTER(ctypes.c_int)]
    L.txl_debug_unit_plan.restype = ctypes.c_int
    return L


def plan(lib, B, H, W, M, P):
    st = ctypes.c_int(0)
    assert lib.txl_debug_unit_plan(B, H, W, M, P, None, 0, st) == 0
    t = np.zeros((P, st.value), np.int32)
    assert lib.txl_debug_unit_plan(B, H, W, M, P, t.ctypes.data, t.size, st) == 0
    return t


def unit_costs(B, H, W, M):
    nqt = (W + 127) // 128
    qt = nqt - 1 - np.arange(nqt * B * H) // (B * H)  # longest query tile first
    return np.minimum(M + 128 * qt + 127, M + W - 1) // 64 + 1 + 1.2


def check(lib, B, H, W, M, P):
    t = plan(lib, B, H, W, M, P)
    cost = unit_costs(B, H, W, M)
    n = len(cost)
    rows = []
    for c in range(P):
        r = t[c]
        k = int(np.argmax(r < 0)) if (r < 0).any() else len(r)
        assert (r[k:] == -1).all(), c  # -1 ends the row and pads it
        rows.append(r[:k])
        assert (np.diff(r[:k]) > 0).all(), c  # unit index order: longest first
    assert t.shape[1] == max(len(r) for r in rows) + 1
    units = np.concatenate(rows)
    assert sorted(units.tolist()) == list(range(n))  # every unit exactly once
    load = np.array([cost[r].sum() for r in rows])
    assert load.max() <= cost.sum() / P + cost.max() + 1e-9
    greedy = greedy_max_load(cost, P)
    assert load.max() <= greedy + 1e-9
    return load.max(), greedy


def greedy_max_load(cost, P):
    """Longest-first list scheduling: each unit (already longest first) onto
    the least-loaded CTA, the lowest index on a tie."""
    heap = [(0.0, c) for c in range(P)]
    heapq.heapify(heap)
    for x in cost:
        load, c = heapq.heappop(heap)
        heapq.heappush(heap, (load + x, c))
    return max(load for load, _ in heap)


@pytest.mark.parametrize("B,H,W,M,P", [
    (22, 8, 512, 512, 152),   # base
    (8, 16, 384, 384, 152),   # large
    (8, 8, 768, 768, 152),    # wide
    (22, 8, 512, 512, 148),
    (3, 5, 300, 37, 7),
    (1, 1, 1000, 0, 3),
    (2, 3, 129, 1600, 5),
    (4, 4, 64, 7, 15),
])
def test_unit_plan(lib, B, H, W, M, P):
    busiest, greedy = check(lib, B, H, W, M, P)
    if P == 152:
        # the bench's workloads: the moves and swaps take 2 to 4 steps
        # off the busiest CTA of the greedy start (base 70.0 -> 66.8, large
        # 33.6 -> 31.6, wide 59.6 -> 55.6)
        assert busiest <= greedy - 1.9, (busiest, greedy)


def test_unit_plan_many_small_shapes(lib):
    rng = np.random.default_rng(7)
    for _ in range(60):
        B, H = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        W, M = int(rng.integers(1, 700)), int(rng.integers(0, 900))
        n = ((W + 127) // 128) * B * H
        P = int(rng.integers(1, n + 1))
        check(lib, B, H, W, M, P)


def test_unit_plan_hook_arguments(lib):
    st = ctypes.c_int(0)
    f = lib.txl_debug_unit_plan
    assert f(-1, 1, 1, 0, 1, None, 0, st) == -1
    assert f(1, 1, 1, 0, 0, None, 0, st) == -1
    buf = np.zeros(1, np.int32)
    assert f(4, 4, 256, 0, 3, buf.ctypes.data, 1, st) == -2 and st.value > 1


# ---------------------------------------------------------------------------
# The key-range split of the D = 64 attention (fewer units than SMs): work
# item it is chunk it % nsplit of unit it / nsplit; the chunks of a unit
# must cover its key steps exactly once, each at least one step, or the
# merge would weigh a missing or doubled part of the softmax.
# ---------------------------------------------------------------------------
def items_of(lib, B, H, W, M, nsplit):
    n = ctypes.c_int(0)
    assert lib.txl_debug_attention_items(B, H, W, M, nsplit, None, 0, n) == 0
    items = np.zeros((n.value, 5), np.int32)
    assert lib.txl_debug_attention_items(B, H, W, M, nsplit, items.ctypes.data, n.value, n) == 0
    return items


@pytest.fixture(scope="module")
def lib_split(lib):
    ip = ctypes.POINTER(ctypes.c_int)
    lib.txl_debug_attention_items.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_int, ip]
    lib.txl_debug_attention_items.restype = ctypes.c_int
    lib.txl_debug_attention_split.argtypes = [ctypes.c_int] * 5
    lib.txl_debug_attention_split.restype = ctypes.c_int
    return lib


def steps(qt, W, M):
    return min(M + 128 * qt + 127, M + W - 1) // 64 + 1


@pytest.mark.parametrize("W", [1, 64, 65, 128, 200, 384])
@pytest.mark.parametrize("M", [0, 7, 100, 384, 1600])
def test_split_items_cover_every_key_step_once(lib_split, W, M):
    B, H = 2, 3
    nqt = (W + 127) // 128
    for nsplit in range(1, min(steps(0, W, M), 64) + 1):
        items = items_of(lib_split, B, H, W, M, nsplit)
        assert len(items) == nqt * B * H * nsplit
        units = {}
        for it, (b, h, i0, t0, nks) in enumerate(items):
            assert nks >= 1
            u = it // nsplit
            units.setdefault(u, []).append((b, h, i0, t0, nks))
        seen = set()
        last_i0 = W
        for u in range(nqt * B * H):
            ch = units[u]
            assert len({c[:3] for c in ch}) == 1  # every chunk of a unit is the same unit
            b, h, i0 = ch[0][:3]
            assert i0 <= last_i0  # longest query tile first
            last_i0 = i0
            seen.add((b, h, i0))
            covered = [t for _, _, _, t0, nks in ch for t in range(t0, t0 + nks)]
            assert covered == list(range(steps(i0 // 128, W, M)))  # in chunk order, once each
        assert len(seen) == nqt * B * H
    # one chunk more than the shortest unit's key steps is refused
    n = ctypes.c_int(0)
    too_many = steps(0, W, M) + 1
    if too_many <= 64:
        assert lib_split.txl_debug_attention_items(B, H, W, M, too_many, None, 0, n) == -1


def split_model(B, H, W, M, sms):
    """The split choice's cost model: waves of work items times the key
    steps of the longest item plus 1.5 for a unit boundary, plus 4 for the
    merge when split; up to 16 chunks and no more than the shortest unit's
    steps; the smallest count on a tie."""
    nqt = (W + 127) // 128
    units = nqt * B * H
    if units >= sms:
        return 1
    longest, shortest = steps(nqt - 1, W, M), steps(0, W, M)
    best, best_cost = 1, -(-units // sms) * (longest + 1.5)
    for s in range(2, min(shortest, 16) + 1):
        cost = -(-units * s // sms) * (-(-longest // s) + 1.5) + 4.0
        if cost < best_cost:
            best, best_cost = s, cost
    return best


def test_split_choice(lib_split):
    f = lib_split.txl_debug_attention_split
    # the bench's workloads: only the long memory (one sequence, W = 128) splits
    assert f(1, 64, 128, 1600, 152) == 2
    for B, H, W, M in [(22, 8, 512, 512), (8, 16, 384, 384), (8, 8, 768, 768)]:
        assert f(B, H, W, M, 152) == 1
    rng = np.random.default_rng(3)
    for _ in range(300):
        B, H = int(rng.integers(1, 4)), int(rng.integers(1, 65))
        W, M = int(rng.integers(1, 400)), int(rng.integers(0, 4000))
        sms = int(rng.choice([8, 148, 152]))
        assert f(B, H, W, M, sms) == split_model(B, H, W, M, sms), (B, H, W, M, sms)
    assert f(0, 1, 1, 0, 152) == -1 and f(1, 1, 1, 0, 0) == -1
