"""The bf16 attention's unit plan, checked on the host (no GPU).

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
