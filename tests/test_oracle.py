"""Pins for the float64 oracle: each check ties it to something other than
itself -- a closed form, a library routine, brute force on tiny inputs, or a
fact the pages print -- so that a plausible mistake (a dropped term, a wrong
sign or index, a transposed operand) fails at least one of them.  The mutation
test at the end plants such mistakes in a copy of the oracle and checks that.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import txl_oracle as O
from synthetic import WORKLOADS, make_segments, project_r

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_printed.json")


def _rand_inputs(rng, B, W, M, H, D, extra_r=0, scale_in=1.0):
    q = rng.standard_normal((B, W, H, D)) * scale_in
    k = rng.standard_normal((B, M + W, H, D)) * scale_in
    v = rng.standard_normal((B, M + W, H, D))
    r = rng.standard_normal((M + W + extra_r, H, D)) * scale_in
    u = rng.standard_normal((H, D)) * 0.3
    vb = rng.standard_normal((H, D)) * 0.3
    return q, k, v, r, u, vb


# ----------------------------------------------------------------------------
# Pin functions.  Each takes a forward function with the oracle's signature
# fwd(q, k, v, r, u, vb, M, scale) -> (o, lse) and raises AssertionError on a
# mismatch.  The tests below run them on the oracle; the mutation test runs
# them on planted mistakes.
# ----------------------------------------------------------------------------

def pin_content_attention_matches_sdpa(fwd):
    """r = u = v = 0: the score loses both distance terms and the bias
    ("remove the two R terms and attention loses explicit distance
    information"), leaving masked softmax(q k^T * scale) v, which the library
    routine computes."""
    rng = np.random.default_rng(1)
    for (B, W, M, H, D) in [(2, 5, 3, 2, 4), (1, 7, 0, 1, 8), (1, 3, 6, 2, 2)]:
        q, k, v, r, u, vb = _rand_inputs(rng, B, W, M, H, D)
        r[:] = 0
        u[:] = 0
        vb[:] = 0
        scale = 0.7
        o, _ = fwd(q, k, v, r, u, vb, M, scale)
        i = np.arange(W)[:, None]
        j = np.arange(M + W)[None, :]
        mask = torch.from_numpy(j <= M + i)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q).permute(0, 2, 1, 3), torch.from_numpy(k).permute(0, 2, 1, 3),
            torch.from_numpy(v).permute(0, 2, 1, 3), attn_mask=mask, scale=scale)
        np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def pin_content_bias_pairs_with_keys(fwd):
    """q = r = 0: only the global content bias survives, u . k_j, which is
    ordinary attention with the query replaced by u for every row."""
    rng = np.random.default_rng(2)
    B, W, M, H, D = 1, 4, 3, 2, 4
    q, k, v, r, u, vb = _rand_inputs(rng, B, W, M, H, D)
    q[:] = 0
    r[:] = 0
    scale = 0.9
    o, _ = fwd(q, k, v, r, u, vb, M, scale)
    i = np.arange(W)[:, None]
    j = np.arange(M + W)[None, :]
    mask = torch.from_numpy(j <= M + i)
    qu = np.broadcast_to(u[None, None], (B, W, H, D)).copy()
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qu).permute(0, 2, 1, 3), torch.from_numpy(k).permute(0, 2, 1, 3),
        torch.from_numpy(v).permute(0, 2, 1, 3), attn_mask=mask, scale=scale)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def _geometric_probs(W, M, a):
    """Closed form of softmax over visible j <= M+i of scores a * (M+i-j)."""
    P = np.zeros((W, M + W))
    for i in range(W):
        n = M + i + 1
        d = M + i - np.arange(n)  # distances of the visible keys
        w = np.exp(a * d - a * (n - 1))
        P[i, :n] = w / w.sum()
    return P


def pin_distance_term_closed_form(fwd):
    """k = 0 and u = 0 remove the content terms.  With r_d = gamma * d * e_0
    and the distance-side query q_i + v = e_0 the score is scale*gamma*(M+i-j):
    a geometric distribution over the visible keys.  Checked twice: once with
    the global distance bias v carrying e_0 and once with the query itself,
    so both halves of (q_i + v) are exercised."""
    B, W, M, H, D = 1, 5, 3, 1, 4
    gamma, scale = 0.37, 0.8
    L = M + W
    k = np.zeros((B, L, H, D))
    v = np.zeros((B, L, H, D))
    v[0, :, 0, :] = np.random.default_rng(3).standard_normal((L, D))
    r = np.zeros((L, H, D))
    r[:, 0, 0] = gamma * np.arange(L)
    u = np.zeros((H, D))
    P = _geometric_probs(W, M, scale * gamma)
    expect = P @ v[0, :, 0]
    for mode in ("bias", "query"):
        q = np.zeros((B, W, H, D))
        vb = np.zeros((H, D))
        if mode == "bias":
            vb[0, 0] = 1.0
        else:
            q[0, :, 0, 0] = 1.0
        o, _ = fwd(q, k, v, r, u, vb, M, scale)
        np.testing.assert_allclose(o[0, :, 0], expect, rtol=0, atol=1e-12, err_msg=mode)


def pin_scale_zero_uniform(fwd):
    """scale = 0: every visible key gets the same weight, so o_i is the mean
    of v_0 .. v_{M+i} and lse_i = log(M+i+1)."""
    rng = np.random.default_rng(4)
    B, W, M, H, D = 2, 6, 4, 2, 3
    q, k, v, r, u, vb = _rand_inputs(rng, B, W, M, H, D)
    o, lse = fwd(q, k, v, r, u, vb, M, 0.0)
    for i in range(W):
        np.testing.assert_allclose(o[:, i], v[:, :M + i + 1].mean(axis=1), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, i], math.log(M + i + 1), rtol=0, atol=1e-12)


def pin_single_key(fwd):
    """W = 1, M = 0: the only visible key is the query's own position, so
    o = v_0 and lse is the one score, scale*((q+u).k_0 + (q+v).r_0)."""
    rng = np.random.default_rng(5)
    q, k, v, r, u, vb = _rand_inputs(rng, 2, 1, 0, 3, 4)
    o, lse = fwd(q, k, v, r, u, vb, 0, 0.6)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)
    s = 0.6 * (np.einsum("bhd,bhd->bh", q[:, 0] + u, k[:, 0]) +
               np.einsum("bhd,hd->bh", q[:, 0] + vb, r[0]))
    np.testing.assert_allclose(lse[:, :, 0], s, rtol=0, atol=1e-12)


def pin_bruteforce(fwd):
    """Explicit (i, j) loops with the distance formed per pair."""
    rng = np.random.default_rng(6)
    for trial in range(25):
        W = int(rng.integers(1, 8))
        M = int(rng.integers(0, 8))
        D = int(rng.choice([2, 4, 8]))
        H = int(rng.integers(1, 3))
        B = int(rng.integers(1, 3))
        q, k, v, r, u, vb = _rand_inputs(rng, B, W, M, H, D, extra_r=int(rng.integers(0, 3)))
        scale = float(rng.uniform(0.1, 1.0))
        o1, l1 = fwd(q, k, v, r, u, vb, M, scale)
        o2, l2 = O.relattn_forward_bruteforce(q, k, v, r, u, vb, M, scale)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def _global_banded(qs, ks, vs, r, u, vb, W, M, scale, with_lse=False):
    """Attention over the whole concatenated stream at global positions t:
    query t of segment tau sees keys t' in [tau*W - M_tau, t] with
    M_tau = min(M, tau*W), distance t - t'.  Explicit loops, one head."""
    T = qs.shape[0]
    o = np.zeros_like(qs)
    lse = np.zeros(T)
    for t in range(T):
        tau = t // W
        lo = tau * W - min(M, tau * W)
        idx = np.arange(lo, t + 1)
        s = np.array([scale * ((qs[t] + u) @ ks[tp] + (qs[t] + vb) @ r[t - tp]) for tp in idx])
        e = np.exp(s - s.max())
        o[t] = (e / e.sum()) @ vs[idx]
        lse[t] = s.max() + np.log(e.sum())
    return (o, lse) if with_lse else o


def pin_recurrence(fwd):
    """Segment by segment with the memory roll equals one attention over the
    concatenated stream at global positions (distance = global i - j)."""
    rng = np.random.default_rng(7)
    for (W, M, S) in [(4, 4, 3), (3, 5, 4), (5, 2, 3), (4, 0, 2), (2, 7, 5)]:
        H, D = 2, 4
        T = W * S
        qs = rng.standard_normal((1, T, H, D))
        ks = rng.standard_normal((1, T, H, D))
        vs = rng.standard_normal((1, T, H, D))
        r = rng.standard_normal((M + W, H, D))
        u = rng.standard_normal((H, D)) * 0.3
        vb = rng.standard_normal((H, D)) * 0.3
        mem_k = np.zeros((1, 0, H * D))
        mem_v = np.zeros((1, 0, H * D))
        got = []
        for tau in range(S):
            sl = slice(tau * W, (tau + 1) * W)
            m_tau = mem_k.shape[1]
            kb = np.concatenate([mem_k.reshape(1, m_tau, H, D), ks[:, sl]], axis=1)
            vb_ = np.concatenate([mem_v.reshape(1, m_tau, H, D), vs[:, sl]], axis=1)
            o, _ = fwd(qs[:, sl], kb, vb_, r, u, vb, m_tau, 0.5)
            got.append(o)
            mem_k = O.mem_update(mem_k, ks[:, sl].reshape(1, W, H * D), M)
            mem_v = O.mem_update(mem_v, vs[:, sl].reshape(1, W, H * D), M)
        got = np.concatenate(got, axis=1)
        for h in range(H):
            ref = _global_banded(qs[0, :, h], ks[0, :, h], vs[0, :, h], r[:, h],
                                 u[h], vb[h], W, M, 0.5)
            np.testing.assert_allclose(got[0, :, h], ref, rtol=0, atol=1e-12)


PINS = [pin_content_attention_matches_sdpa, pin_content_bias_pairs_with_keys,
        pin_distance_term_closed_form, pin_scale_zero_uniform, pin_single_key,
        pin_bruteforce, pin_recurrence]


def _oracle_fwd(q, k, v, r, u, vb, M, scale):
    return O.relattn_forward(q, k, v, r, u, vb, M, scale)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pins(pin):
    pin(_oracle_fwd)


def test_rows_route_matches_forward():
    rng = np.random.default_rng(8)
    B, W, M, H, D = 2, 9, 5, 2, 4
    q, k, v, r, u, vb = _rand_inputs(rng, B, W, M, H, D, extra_r=3)
    o, lse = O.relattn_forward(q, k, v, r, u, vb, M, 0.4)
    rows = [0, 3, 8]
    o2, l2 = O.relattn_rows(q, k, v, r, u, vb, M, 0.4, 1, 1, rows)
    np.testing.assert_allclose(o2, o[1, rows, 1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lse[1, 1, rows], rtol=0, atol=1e-12)


def test_probabilities_rows_and_mask():
    rng = np.random.default_rng(9)
    W, M = 6, 3
    q, k, v, r, u, vb = _rand_inputs(rng, 1, W, M, 2, 4)
    _, _, p = O.relattn_forward(q, k, v, r, u, vb, M, 0.5, return_probs=True)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
    for i in range(W):
        assert np.all(p[..., i, M + i + 1:] == 0)
        assert np.all(p[..., i, :M + i + 1] > 0)


# ----------------------------------------------------------------------------
# Facts the pages print
# ----------------------------------------------------------------------------

def test_printed_segment_shapes():
    g = json.load(open(GOLDEN))["segment_shapes"]
    wl = WORKLOADS["tiny"]
    assert (wl.W, wl.d_model, wl.H, wl.segments) == (g["seg_len"], g["dim"], g["heads"], g["segments"])
    seg = make_segments(wl, n_segments=wl.segments)
    R = O.sinusoid_rel(wl.M + wl.W, wl.d_model)
    r = project_r(R, seg.W_r, wl.H, wl.D, wl.dtype)
    mem_k = np.zeros((wl.B, 0, wl.H * wl.D))
    mem_v = np.zeros((wl.B, 0, wl.H * wl.D))
    for tau in range(wl.segments):
        m_tau = mem_k.shape[1]
        ks, vs, qs = seg.seg("k", tau), seg.seg("v", tau), seg.seg("q", tau)
        kb = np.concatenate([mem_k.reshape(wl.B, m_tau, wl.H, wl.D), ks], axis=1)
        vb = np.concatenate([mem_v.reshape(wl.B, m_tau, wl.H, wl.D), vs], axis=1)
        _, _, p = O.relattn_forward(qs, kb, vb, r, seg.bias_u, seg.bias_v, m_tau,
                                    return_probs=True)
        assert p.shape[2:] == (g["queries"][tau], g["positions"][tau])
        mem_k = O.mem_update(mem_k, ks.reshape(wl.B, wl.W, -1), wl.M)
        mem_v = O.mem_update(mem_v, vs.reshape(wl.B, wl.W, -1), wl.M)


def test_printed_shift_invariance():
    """rel(5,3) = rel(105,103): with the content terms removed (k = u = 0) the
    score of global pair (5,3) equals that of (105,103) when the query rows
    match, although the pairs sit in different segments at different local
    positions."""
    g = json.load(open(GOLDEN))["shift_invariance"]
    (t1, s1), (t2, s2) = g["pairs"]
    assert t1 - s1 == t2 - s2 == g["distance"]
    W, M, H, D = 8, 8, 2, 4
    S = (t2 // W) + 1
    rng = np.random.default_rng(10)
    qs = rng.standard_normal((1, S * W, H, D))
    qs[0, t2] = qs[0, t1]
    ks = np.zeros((1, S * W, H, D))
    vs = rng.standard_normal((1, S * W, H, D))
    r = rng.standard_normal((M + W, H, D))
    u = np.zeros((H, D))
    vb = rng.standard_normal((H, D))

    def raw_score(t, tp):
        tau = t // W
        m_tau = min(M, tau * W)
        lo = tau * W - m_tau
        sl = slice(tau * W, (tau + 1) * W)
        _, lse, p = O.relattn_forward(qs[:, sl], ks[:, lo:(tau + 1) * W], vs[:, lo:(tau + 1) * W],
                                      r, u, vb, m_tau, 0.5, return_probs=True)
        i, j = t - tau * W, tp - lo
        return np.log(p[0, :, i, j]) + lse[0, :, i]

    np.testing.assert_allclose(raw_score(t1, s1), raw_score(t2, s2), rtol=0, atol=1e-12)


def test_segment_cost_model():
    """The simulation's per-segment cost W(W+M) counts every pair; the causal
    mask removes the strictly-upper half of the current block, which is what
    the counted flops use."""
    g = json.load(open(GOLDEN))["segment_cost"]
    W, M = g["W"], g["M"]
    assert W * (W + M) == g["cost"]
    i = np.arange(W)[:, None]
    j = np.arange(M + W)[None, :]
    visible = int((j <= M + i).sum())
    assert visible == g["cost"] - W * (W - 1) // 2
    assert O.counted_flops(1, 1, 1, W, M) == 6 * visible
    assert O.counted_flops(22, 8, 64, 512, 512) == 26_592_411_648


# ----------------------------------------------------------------------------
# Sinusoid
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n,dim", [(8, 16), (1024, 512), (40, 6)])
def test_sinusoid_closed_form(n, dim):
    R = O.sinusoid_rel(n, dim)
    assert R.shape == (n, dim)
    # distance 0: sin 0 = 0, cos 0 = 1
    np.testing.assert_array_equal(R[0, 0::2], 0.0)
    np.testing.assert_array_equal(R[0, 1::2], 1.0)
    # each (sin, cos) pair lies on the unit circle
    np.testing.assert_allclose(R[:, 0::2] ** 2 + R[:, 1::2] ** 2, 1.0, atol=1e-14)
    # pair 0 has frequency 10000^0 = 1: the library's sin / cos of d itself
    d = np.arange(n)
    np.testing.assert_allclose(R[:, 0], np.sin(d), atol=1e-15)
    np.testing.assert_allclose(R[:, 1], np.cos(d), atol=1e-15)
    if n > 1:
        # frequencies read back from distance 1 fall geometrically by
        # 10000^(-2/dim) per pair, down to 10000^(-(dim-2)/dim)
        w = np.arctan2(R[1, 0::2], R[1, 1::2])
        np.testing.assert_allclose(w[1:] / w[:-1], 10000.0 ** (-2.0 / dim), rtol=1e-12)
        np.testing.assert_allclose(w[-1], 10000.0 ** (-(dim - 2) / dim), rtol=1e-12)


def test_sinusoid_angle_addition():
    """R[d1+d2] follows from R[d1] and R[d2] by the angle-addition identities,
    so the angle is linear in the distance."""
    R = O.sinusoid_rel(64, 10)
    for d1, d2 in [(3, 5), (17, 40), (0, 63), (31, 31)]:
        s1, c1 = R[d1, 0::2], R[d1, 1::2]
        s2, c2 = R[d2, 0::2], R[d2, 1::2]
        np.testing.assert_allclose(R[d1 + d2, 0::2], s1 * c2 + c1 * s2, atol=1e-13)
        np.testing.assert_allclose(R[d1 + d2, 1::2], c1 * c2 - s1 * s2, atol=1e-13)


def test_sinusoid_rejects_odd_dim():
    with pytest.raises(ValueError):
        O.sinusoid_rel(4, 7)


# ----------------------------------------------------------------------------
# Memory roll
# ----------------------------------------------------------------------------

def test_mem_update_keeps_last_rows():
    rng = np.random.default_rng(11)
    mem = rng.standard_normal((2, 5, 3))
    h = rng.standard_normal((2, 4, 3))
    out = O.mem_update(mem, h, 6)
    np.testing.assert_array_equal(out[:, :2], mem[:, 3:])
    np.testing.assert_array_equal(out[:, 2:], h)
    # memory still growing: keep everything
    np.testing.assert_array_equal(O.mem_update(mem[:, :1], h, 6), np.concatenate([mem[:, :1], h], 1))
    # window longer than the memory: only the newest rows
    np.testing.assert_array_equal(O.mem_update(mem, h, 3), h[:, 1:])
    assert O.mem_update(mem, h, 0).shape == (2, 0, 3)


def test_mem_update_composes():
    """Two rolls of W rows equal one roll of the 2W rows."""
    rng = np.random.default_rng(12)
    mem = rng.standard_normal((1, 7, 2))
    h1 = rng.standard_normal((1, 3, 2))
    h2 = rng.standard_normal((1, 3, 2))
    for m in [0, 2, 5, 7, 13]:
        a = O.mem_update(O.mem_update(mem, h1, m), h2, m)
        b = O.mem_update(mem, np.concatenate([h1, h2], 1), m)
        np.testing.assert_array_equal(a, b)


# ----------------------------------------------------------------------------
# Mutation test: plausible mistakes planted in a copy of the oracle must each
# fail at least one pin.
# ----------------------------------------------------------------------------

def _mutant(kind):
    def fwd(q, k, v, r, u, vb, M, scale):
        q, k, v, r = map(np.asarray, (q, k, v, r))
        B, W, H, D = q.shape
        o = np.zeros((B, W, H, D))
        lse = np.zeros((B, H, W))
        for b in range(B):
            for h in range(H):
                qh, kh, vh, rh = q[b, :, h], k[b, :, h], v[b, :, h], r[:, h]
                uu, vv = u[h], vb[h]
                if kind == "swap_u_v":
                    uu, vv = vv, uu
                if kind == "drop_u":
                    uu = 0 * uu
                ac = (qh + uu) @ kh.T
                g = (np.broadcast_to(vv, qh.shape) if kind == "drop_q_in_bd" else qh + vv) @ rh.T
                i = np.arange(W)[:, None]
                j = np.arange(M + W)[None, :]
                dist = {"sign": M - i + j - 2 * M + (W - 1), "no_mem_offset": i - j,
                        "off_by_one": M + i - j + 1}.get(kind, M + i - j)
                visible = (M + i - j) >= (1 if kind == "strict_mask" else 0)
                bd = np.take_along_axis(g, np.clip(dist, 0, rh.shape[0] - 1), axis=1)
                if kind == "drop_bd":
                    bd = 0 * bd
                sc = 1.0 if kind == "no_scale" else scale
                s = np.where(visible, sc * (ac + bd), -np.inf)
                if kind == "strict_mask":
                    s[:, 0] = np.where(np.isinf(s[:, 0]), 0.0, s[:, 0])
                m = s.max(1, keepdims=True)
                e = np.exp(s - m)
                l = e.sum(1, keepdims=True) + (1e-3 if kind == "epsilon" else 0.0)
                o[b, :, h] = (e / l) @ (vh if kind != "transpose_v" else vh[::-1])
                lse[b, h] = (m + np.log(l))[:, 0]
        return o, lse
    return fwd


MUTANTS = ["swap_u_v", "drop_u", "drop_q_in_bd", "sign", "no_mem_offset", "off_by_one",
           "strict_mask", "drop_bd", "no_scale", "epsilon", "transpose_v"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(kind):
    fwd = _mutant(kind)
    caught = []
    for pin in PINS:
        try:
            pin(fwd)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {kind!r}"


def test_unmutated_copy_passes_all_pins():
    fwd = _mutant("none")
    for pin in PINS:
        pin(fwd)


# ----------------------------------------------------------------------------
# The oracle's segment recurrence (run_segments), pinned by itself: it gives
# the expected values of every multi-segment GPU test, so the function that
# runs the segments -- not a copy of its loop -- is checked against one
# attention over the concatenated stream at global positions.
# ----------------------------------------------------------------------------

RECURRENCE_CASES = [(4, 4, 3), (3, 5, 4), (5, 2, 3), (4, 0, 2), (2, 7, 5), (3, 9, 6)]


def pin_segment_recurrence(run):
    """``run`` has run_segments' signature.  Per segment tau: M_tau is
    min(M, tau*W) ("Long-context transformers": the memory is the last M
    rows of [memory ; segment], empty before the first segment), and o, lse
    equal the banded attention over the whole stream (each query sees the
    M_tau rows before its segment and its segment up to itself)."""
    rng = np.random.default_rng(11)
    for (W, M, S) in RECURRENCE_CASES:
        H, D = 2, 3
        T = W * S
        qs = rng.standard_normal((2, T, H, D))
        ks = rng.standard_normal((2, T, H, D))
        vs = rng.standard_normal((2, T, H, D))
        r = rng.standard_normal((M + W + T, H, D))  # spare rows: a memory too long stays a wrong value
        u = rng.standard_normal((H, D)) * 0.3
        vb = rng.standard_normal((H, D)) * 0.3
        segs = lambda a: [a[:, t * W:(t + 1) * W] for t in range(S)]
        out = run(segs(qs), segs(ks), segs(vs), r, u, vb, M, 0.7)
        assert len(out) == S
        for tau, (o, lse, m_tau) in enumerate(out):
            assert m_tau == min(M, tau * W), (W, M, tau, m_tau)
            assert o.shape == (2, W, H, D) and lse.shape == (2, H, W)
        for b in range(2):
            for h in range(H):
                ref_o, ref_l = _global_banded(qs[b, :, h], ks[b, :, h], vs[b, :, h], r[:, h], u[h], vb[h],
                                              W, M, 0.7, with_lse=True)
                got_o = np.concatenate([o[b, :, h] for o, _, _ in out])
                got_l = np.concatenate([lse[b, h] for _, lse, _ in out])
                np.testing.assert_allclose(got_o, ref_o, rtol=0, atol=1e-12)
                np.testing.assert_allclose(got_l, ref_l, rtol=0, atol=1e-12)


def test_run_segments_pinned():
    pin_segment_recurrence(O.run_segments)


def _run_segments_mutant(kind):
    """A copy of the recurrence with one plausible mistake planted."""
    def run(q_segs, k_segs, v_segs, r, bias_u, bias_v, M, scale=None):
        B, W, H, D = q_segs[0].shape
        mem_k = np.zeros((B, 0, H, D))
        mem_v = np.zeros((B, 0, H, D))
        out = []

        def roll(mem, new, keep_src=None):
            cat = np.concatenate([mem, new], axis=1)
            if kind == "keep_first_rows":
                return cat[:, :min(M, cat.shape[1])]
            if kind == "no_truncation":
                return cat
            if kind == "segment_only":
                return new[:, new.shape[1] - min(M, W):]
            return cat[:, cat.shape[1] - min(M, cat.shape[1]):]

        for qs, ks, vs in zip(q_segs, k_segs, v_segs):
            if kind == "roll_before_attention":
                mem_k, mem_v = roll(mem_k, ks), roll(mem_v, vs)
            m_tau = mem_k.shape[1]
            kb = np.concatenate([mem_k, ks], axis=1)
            vb_ = np.concatenate([mem_v, vs], axis=1)
            o, lse = O.relattn_forward(qs, kb, vb_, r, bias_u, bias_v, m_tau, scale)
            out.append((o, lse, m_tau))
            if kind != "roll_before_attention":
                mem_k = roll(mem_k, qs if kind == "memory_from_queries" else ks)
                mem_v = roll(mem_v, ks if kind == "values_memory_from_keys" else vs)
        return out
    return run


RECURRENCE_MUTANTS = ["roll_before_attention", "keep_first_rows", "no_truncation", "segment_only",
                      "memory_from_queries", "values_memory_from_keys"]


@pytest.mark.parametrize("kind", RECURRENCE_MUTANTS)
def test_recurrence_pin_catches_planted_mistake(kind):
    with pytest.raises(AssertionError):
        pin_segment_recurrence(_run_segments_mutant(kind))


def test_recurrence_unmutated_copy_passes():
    pin_segment_recurrence(_run_segments_mutant("none"))
