"""The backward's work split, checked on the host (no GPU): the pair kernel's
CTAs and the gradient products' tiles, as the library's own mapping code
hands them out (`txl_debug_bwd_pairs_work`), against

* the causal mask of the relative attention ("Transformer-XL, explained",
  method steps 3-4: query i of the segment sees key j of [memory ; segment]
  iff j <= M + i, i.e. distance d = M + i - j >= 0): every visible pair is
  computed by exactly one pair CTA, and every gradient row sums over every
  visible pair exactly once;
* the hand-off between the two launches: every element of the pair terms G,
  P (key order) and GS (distance order) that a product tile reads inside the
  tensors' extents (reads past them are zero-filled) was written by some CTA
  of the pair kernel.  An unwritten element is uninitialised scratch.

The write rules restate the pair kernel's stores: G for every 64-key step of
the CTA's 128 rows; P only for steps holding a segment key (j >= M); GS at
the distances d = M + i - j >= 0 of the step's keys, and, by the CTA that
starts the unit, zeros past the row's last distance, up to 191 columns.  The
read rules restate the products' operand tiles: dq rows read G and GS over
the tile's k blocks of 64 columns; dk / dv rows (keys m) read G / P at
column M + m over the queries of their k blocks, plus the pairs of queries
i in [m, 128 n) that the epilogue adds for a tile whose rows start ks = M % 8
before its first query 128 n; dr rows (distances) read GS over every
sequence's queries of their k blocks.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "transformer_xl_relative_txl_gb300", "libtxl_relattn.so")
DQ, DK, DV, DR = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        subprocess.check_call([sys.executable, os.path.join(ROOT, "transformer_xl_relative_txl_gb300", "build.py")])
    L = ctypes.CDLL(LIB)
    ip = ctypes.POINTER(ctypes.c_int)
    L.txl_debug_bwd_pairs_work.argtypes = [ctypes.c_int] * 5 + [ip, ip, ctypes.c_void_p, ctypes.c_int,
                                                                ctypes.c_void_p, ctypes.c_int]
    L.txl_debug_bwd_pairs_work.restype = ctypes.c_int
    L.txl_debug_pair_split_tiles.argtypes = [ctypes.c_int] * 5
    L.txl_debug_pair_split_tiles.restype = ctypes.c_int
    return L


def work(lib, B, W, M, H, split):
    n_c, n_t = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.txl_debug_bwd_pairs_work(B, W, M, H, split, n_c, n_t, None, 0, None, 0) == 0
    ctas = np.zeros((n_c.value, 5), np.int32)
    tiles = np.zeros((n_t.value, 6), np.int32)
    assert lib.txl_debug_bwd_pairs_work(B, W, M, H, split, n_c, n_t, ctas.ctypes.data, len(ctas),
                                        tiles.ctypes.data, len(tiles)) == 0
    return ctas, tiles


def steps_of_tile(qt, W, M):
    """64-key steps a query tile needs: up to the last visible key of its
    last row."""
    return min(M + 128 * qt + 127, M + W - 1) // 64 + 1


def written(ctas, B, H, W, M):
    """Write counts of G, P and GS, [B*H, W, L] each, from the pair CTAs."""
    L = M + W
    G = np.zeros((B * H, W, L), np.int32)
    P = np.zeros_like(G)
    GS = np.zeros_like(G)
    for b, h, i0, t0, nks in ctas:
        z = b * H + h
        rows = range(i0, min(i0 + 128, W))
        for s in range(t0, t0 + nks):
            c0, c1 = 64 * s, min(64 * s + 64, L)
            G[z, i0:i0 + 128, c0:c1] += 1
            if 64 * s + 64 > M:
                P[z, i0:i0 + 128, c0:c1] += 1
            for i in rows:
                hi = M + i - 64 * s  # the step's first key
                if hi >= 0:
                    GS[z, i, max(0, hi - 63):hi + 1] += 1
        if t0 == 0:
            for i in rows:
                GS[z, i, M + i + 1:min(L, M + i + 192)] += 1
    return G, P, GS


def unwritten_reads(tiles, B, H, W, M, G, P, GS):
    """The product tiles' reads inside the extents that no pair CTA wrote,
    as (tile index, tensor) pairs."""
    L = M + W
    bad = []
    for u, (mode, z, m0, kb0, nkb, nkb_c) in enumerate(tiles):
        if mode == DQ:
            c1 = min(64 * nkb_c, L)
            if not (G[z, m0:m0 + 128, :c1] > 0).all():
                bad.append((u, "G"))
            if not (GS[z, m0:m0 + 128, :c1] > 0).all():
                bad.append((u, "GS"))
        elif mode in (DK, DV):
            A = G if mode == DK else P
            name = "G" if mode == DK else "P"
            c0, c1 = M + m0, min(M + m0 + 128, L)
            if not (A[z, 64 * kb0:64 * (kb0 + nkb), c0:c1] > 0).all():
                bad.append((u, name))
            q0 = 64 * kb0  # the k loop's first query; the epilogue adds [m, q0) below it
            for m in range(max(m0, 0), min(q0, m0 + 128, W)):
                if not (A[z, m:min(q0, W), M + m] > 0).all():
                    bad.append((u, name + " (epilogue)"))
        else:
            assert mode == DR
            for b in range(B):
                if not (GS[b * H + z, 64 * kb0:W, m0:min(m0 + 128, L)] > 0).all():
                    bad.append((u, "GS"))
    return bad


def check_coverage(ctas, tiles, B, H, W, M, split):
    L, BH, nqt = M + W, B * H, (W + 127) // 128
    ks = M % 8
    # pair CTAs: every (sequence, head, query tile) has its steps 0 .. n - 1
    # exactly once; whole units first, longest first, then the halves
    assert len(ctas) == (nqt + split) * BH
    seen = {}
    for b, h, i0, t0, nks in ctas:
        assert i0 % 128 == 0 and 0 <= i0 < W and nks >= 1
        seen.setdefault((b * H + h, i0 // 128), []).extend(range(t0, t0 + nks))
    assert len(seen) == BH * nqt
    for (z, qt), st in seen.items():
        assert sorted(st) == list(range(steps_of_tile(qt, W, M))), (z, qt)
    qts = [i0 // 128 for _, _, i0, t0, nks in ctas[:(nqt - split) * BH]]
    assert qts == sorted(qts, reverse=True)
    # product tiles: kinds in counter order, each output row once
    modes = list(tiles[:, 0])
    n_dr, n_dq = H * ((L + 127) // 128), BH * nqt
    n_k = BH * ((W + ks + 127) // 128)
    assert modes == [DR] * n_dr + [DQ] * n_dq + [DK, DV] * n_k
    rows = {DQ: np.zeros((BH, W), int), DK: np.zeros((BH, W), int), DV: np.zeros((BH, W), int),
            DR: np.zeros((H, L), int)}
    for mode, z, m0, kb0, nkb, nkb_c in tiles:
        r = rows[mode]
        r[z, max(m0, 0):m0 + 128] += 1
        if mode == DQ:
            # row i sums over keys j <= M + i and distances d = M + i - j <= M + i
            assert nkb == 2 * nkb_c and 64 * nkb_c >= min(L, M + m0 + 128)
        elif mode == DR:
            # distance d is non-zero for queries i >= d - M of every sequence
            assert nkb == B * ((W + 63) // 64 - kb0) and 64 * kb0 <= max(0, m0 - M)
        else:
            # key row m (key M + m) gets the pairs of queries i >= m: the k loop
            # covers [q0, W) from a whole query tile q0 = 64 kb0 (rows of the
            # tile before have G and P only up to their own last step), the
            # epilogue the disjoint [m, q0) of the first ks rows
            q0 = 64 * kb0
            assert 64 * (kb0 + nkb) >= W and q0 % 128 == 0 and m0 == q0 - ks
    for mode, r in rows.items():
        assert (r == 1).all(), mode


def _cases():
    for W in (1, 63, 64, 65, 128, 129, 200, 300, 512):
        for M in (0, 1, 7, 8, 37, 64, 77, 100, 128, 200):
            nqt = (W + 127) // 128
            for split in range(0, min(nqt, 2) + 1):
                if split and steps_of_tile(nqt - split, W, M) < 4:
                    break  # the host never splits units of fewer than four steps
                yield W, M, split


CASES = list(_cases())


@pytest.mark.parametrize("W,M,split", CASES, ids=[f"W{w}-M{m}-s{s}" for w, m, s in CASES])
def test_work_split(lib, W, M, split):
    B, H = 2, 2
    ctas, tiles = work(lib, B, W, M, H, split)
    check_coverage(ctas, tiles, B, H, W, M, split)
    G, P, GS = written(ctas, B, H, W, M)
    assert G.max() <= 1 and P.max() <= 1 and GS.max() <= 1  # no element written twice
    assert unwritten_reads(tiles, B, H, W, M, G, P, GS) == []


@pytest.mark.parametrize("B,H,W,M,sms", [(6, 8, 768, 768, 152), (4, 4, 640, 200, 16), (3, 1, 384, 45, 2)])
def test_work_split_at_the_chosen_split(lib, B, H, W, M, sms):
    """The split the host's cost model picks, on the wide workload's shape
    (one sequence of it: every sequence maps alike) and on small launches."""
    nqt = (W + 127) // 128
    split = lib.txl_debug_pair_split_tiles(nqt, B * H, W, M, sms)
    b = 1 if B * H * W > 20000 else B
    ctas, tiles = work(lib, b, W, M, H, split)
    check_coverage(ctas, tiles, b, H, W, M, split)
    G, P, GS = written(ctas, b, H, W, M)
    assert unwritten_reads(tiles, b, H, W, M, G, P, GS) == []


def test_read_check_catches_planted_mistakes(lib):
    """The hand-off check is not vacuous: each planted mistake leaves reads of
    unwritten scratch.  (1) dk / dv tiles whose k loop starts at the 64-block
    of their first row instead of their first whole query tile read rows of
    the tile before, past that tile's last key step; (2) no zeros past each
    row's last distance in GS; (3) P stored only for steps that start at a
    segment key, so a step holding both memory and segment keys has none."""
    B, H, W, M = 2, 2, 512, 37
    ctas, tiles = work(lib, B, W, M, H, 0)
    G, P, GS = written(ctas, B, H, W, M)
    assert unwritten_reads(tiles, B, H, W, M, G, P, GS) == []

    t1 = tiles.copy()
    k = (t1[:, 0] == DK) | (t1[:, 0] == DV)
    t1[k, 3] = np.maximum(t1[k, 2], 0) // 64
    t1[k, 4] = (W + 63) // 64 - t1[k, 3]
    assert any(name.startswith(("G", "P")) for _, name in unwritten_reads(t1, B, H, W, M, G, P, GS))

    GS2 = GS.copy()
    L = M + W
    for z in range(B * H):
        for i in range(W):
            GS2[z, i, M + i + 1:] = 0
    assert any(name == "GS" for _, name in unwritten_reads(tiles, B, H, W, M, G, P, GS2))

    P3 = np.zeros_like(P)
    for b, h, i0, t0, nks in ctas:
        for s in range(t0, t0 + nks):
            if 64 * s >= M:
                P3[b * H + h, i0:i0 + 128, 64 * s:min(64 * s + 64, L)] += 1
    assert any(name.startswith("P") for _, name in unwritten_reads(tiles, B, H, W, M, G, P3, GS))


def test_work_hook_rejects_bad_arguments(lib):
    n_c, n_t = ctypes.c_int(0), ctypes.c_int(0)
    f = lib.txl_debug_bwd_pairs_work
    assert f(-1, 8, 0, 1, 0, n_c, n_t, None, 0, None, 0) == -1
    assert f(1, 128, 0, 1, 2, n_c, n_t, None, 0, None, 0) == -1  # one query tile: at most one split
    assert f(1, 128, 0, 1, -1, n_c, n_t, None, 0, None, 0) == -1
    buf = np.zeros(5, np.int32)
    assert f(1, 256, 0, 1, 0, n_c, n_t, buf.ctypes.data, 1, None, 0) == -2
