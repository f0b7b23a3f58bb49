"""Pins for the oracle's backward (gradients of the relative attention).

The backward is tied to things other than itself: central finite differences
of the pinned forward, automatic differentiation of an independent forward
written with torch ops, and identities the score's structure forces.  A
mutation test plants plausible mistakes in a copy of the backward and checks
that each fails at least one pin.
"""

import numpy as np
import pytest
import torch

from oracle import txl_oracle as O


def _inputs(seed, B, W, M, H, D, extra_r=1):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, W, H, D)) * 0.8
    k = rng.standard_normal((B, M + W, H, D)) * 0.8
    v = rng.standard_normal((B, M + W, H, D))
    r = rng.standard_normal((M + W + extra_r, H, D)) * 0.8
    u = rng.standard_normal((H, D)) * 0.3
    vb = rng.standard_normal((H, D)) * 0.3
    dout = rng.standard_normal((B, W, H, D))
    return q, k, v, r, u, vb, dout


def _oracle_bwd(q, k, v, r, u, vb, M, dout, scale):
    return O.relattn_backward(q, k, v, r, u, vb, M, dout, scale, memory_grads=True)


def _loss(args, M, dout, scale):
    o, _ = O.relattn_forward(*args, M, scale)
    return float((dout * o).sum())


# ----------------------------------------------------------------------------
# Pin functions: each takes a backward with the signature
# bwd(q, k, v, r, u, vb, M, dout, scale) -> dict (the oracle's keys, with
# dk_all / dv_all) and raises AssertionError on a mismatch.
# ----------------------------------------------------------------------------

def pin_finite_differences(bwd):
    """Central differences of L = sum(dout * o), o from the pinned forward,
    for every input element, on tiny shapes with and without memory.  The
    segment rows of k and v are compared with dk / dv, every row with
    dk_all / dv_all."""
    for (B, W, M, H, D) in [(2, 3, 2, 2, 3), (1, 4, 0, 1, 2)]:
        q, k, v, r, u, vb, dout = _inputs(7 + M, B, W, M, H, D)
        scale = 0.6
        got = bwd(q, k, v, r, u, vb, M, dout, scale)
        args = [q, k, v, r, u, vb]
        names = ["dq", "dk_all", "dv_all", "dr", "dbias_u", "dbias_v"]
        eps = 1e-6
        for n, (x, name) in enumerate(zip(args, names)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                keep = x[idx]
                x[idx] = keep + eps
                lp = _loss(args, M, dout, scale)
                x[idx] = keep - eps
                lm = _loss(args, M, dout, scale)
                x[idx] = keep
                fd[idx] = (lp - lm) / (2 * eps)
            np.testing.assert_allclose(got[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)
        np.testing.assert_allclose(got["dk"], got["dk_all"][:, M:], rtol=0, atol=0)
        np.testing.assert_allclose(got["dv"], got["dv_all"][:, M:], rtol=0, atol=0)


def _torch_forward(q, k, v, r, u, vb, M, scale):
    """The forward written again with torch ops, the distance of every pair
    gathered from r directly (no shift of a computed row)."""
    B, W, H, D = q.shape
    L = k.shape[1]
    i = torch.arange(W)[:, None]
    j = torch.arange(L)[None, :]
    dist = M + i - j
    vis = dist >= 0
    rg = r[dist.clamp(min=0)]  # [W, L, H, D]
    ac = torch.einsum("bihd,bjhd->bhij", q + u, k)
    bd = torch.einsum("bihd,ijhd->bhij", q + vb, rg)
    s = (scale * (ac + bd)).masked_fill(~vis, float("-inf"))
    p = torch.softmax(s, dim=-1)
    return torch.einsum("bhij,bjhd->bihd", p, v)


def pin_autograd(bwd):
    """Reverse-mode automatic differentiation of the torch forward (checked
    against the oracle forward first) on shapes too large for finite
    differences: several memory lengths and an unused extra distance row."""
    for (B, W, M, H, D, extra) in [(2, 6, 5, 2, 8, 3), (1, 9, 0, 3, 4, 0), (2, 4, 11, 1, 16, 2)]:
        q, k, v, r, u, vb, dout = _inputs(31 + W, B, W, M, H, D, extra)
        scale = 1.0 / np.sqrt(D)
        ts = [torch.tensor(x, requires_grad=True) for x in (q, k, v, r, u, vb)]
        o = _torch_forward(*ts, M, scale)
        o_ref, _ = O.relattn_forward(q, k, v, r, u, vb, M, scale)
        np.testing.assert_allclose(o.detach().numpy(), o_ref, rtol=0, atol=1e-12)
        (o * torch.from_numpy(dout)).sum().backward()
        got = bwd(q, k, v, r, u, vb, M, dout, scale)
        for t, name in zip(ts, ["dq", "dk_all", "dv_all", "dr", "dbias_u", "dbias_v"]):
            np.testing.assert_allclose(got[name], t.grad.numpy(), rtol=1e-9, atol=1e-11, err_msg=name)


def pin_structural_identities(bwd):
    """Identities the score forces, at any size:
    * q enters through (q + u) and (q + v), so summed over batch and rows,
      dq = dbias_u + dbias_v per head;
    * adding one vector to every key (or every distance row) adds a per-row
      constant to the scores, which the softmax ignores: sum_j dk_all = 0
      and sum_d dr = 0;
    * o is linear in v, so sum(dv_all * v) = L;
    * a distance row no pair uses gets no gradient."""
    B, W, M, H, D = 3, 7, 6, 2, 5
    q, k, v, r, u, vb, dout = _inputs(99, B, W, M, H, D, extra_r=4)
    scale = 0.4
    g = bwd(q, k, v, r, u, vb, M, dout, scale)
    np.testing.assert_allclose(g["dq"].sum(axis=(0, 1)), g["dbias_u"] + g["dbias_v"], rtol=0, atol=1e-11)
    np.testing.assert_allclose(g["dk_all"].sum(axis=1), 0, atol=1e-11)
    np.testing.assert_allclose(g["dr"].sum(axis=0), 0, atol=1e-11)
    L = _loss([q, k, v, r, u, vb], M, dout, scale)
    np.testing.assert_allclose((g["dv_all"] * v).sum(), L, rtol=1e-12, atol=1e-11)
    np.testing.assert_array_equal(g["dr"][M + W:], 0)


PINS = [pin_finite_differences, pin_autograd, pin_structural_identities]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_backward_pins(pin):
    pin(_oracle_bwd)


def test_backward_first_segment_and_output_shapes():
    """M = 0 (empty memory, the first segment): dk / dv cover all key rows;
    with memory they cover the segment rows only."""
    for M in (0, 3):
        q, k, v, r, u, vb, dout = _inputs(5, 2, 4, M, 2, 3)
        g = O.relattn_backward(q, k, v, r, u, vb, M, dout)
        assert g["dq"].shape == q.shape
        assert g["dk"].shape == q.shape and g["dv"].shape == q.shape
        assert g["dr"].shape == r.shape
        assert g["dbias_u"].shape == u.shape and g["dbias_v"].shape == vb.shape


# ----------------------------------------------------------------------------
# Mutation test
# ----------------------------------------------------------------------------

def _mutant(kind):
    def bwd(q, k, v, r, u, vb, M, dout, scale):
        B, W, H, D = q.shape
        L = k.shape[1]
        n_r = r.shape[0]
        out = {"dq": np.zeros(q.shape), "dk_all": np.zeros(k.shape), "dv_all": np.zeros(v.shape),
               "dr": np.zeros(r.shape), "dbias_u": np.zeros(u.shape), "dbias_v": np.zeros(vb.shape)}
        i = np.arange(W)[:, None]
        j = np.arange(L)[None, :]
        dist = M + i - j
        vis = dist >= 0
        for b in range(B):
            for h in range(H):
                qu = q[b, :, h] + u[h]
                qv = q[b, :, h] + (u[h] if kind == "qv_uses_u" else vb[h])
                kh, vh, rh, do = k[b, :, h], v[b, :, h], r[:, h], dout[b, :, h]
                g = qv @ rh.T
                s = np.where(vis, scale * (qu @ kh.T + np.take_along_axis(g, np.clip(dist, 0, n_r - 1), 1)),
                             -np.inf)
                e = np.exp(s - s.max(1, keepdims=True))
                P = e / e.sum(1, keepdims=True)
                dP = do @ vh.T
                delta = 0.0 if kind == "no_delta" else (P * dP).sum(1, keepdims=True)
                G = (1.0 if kind == "no_scale" else scale) * P * (dP - delta)
                dg = np.zeros((W, n_r))
                ii, jj = np.nonzero(vis)
                dd = dist[ii, jj] + (1 if kind == "dist_off_by_one" else 0)
                dd = np.clip(dd, 0, n_r - 1)
                np.add.at(dg, (ii, dd) if kind != "dist_transposed" else (ii, np.clip(jj, 0, n_r - 1)),
                          G[ii, jj])
                d_qu = G @ kh
                d_qv = dg @ rh
                out["dq"][b, :, h] = d_qu + (0 if kind == "dq_drops_qv" else d_qv)
                out["dk_all"][b, :, h] = G.T @ (qv if kind == "dk_uses_qv" else qu)
                out["dv_all"][b, :, h] = (P if kind != "dv_uses_g" else G).T @ do
                out["dr"][:, h] += dg.T @ (qu if kind == "dr_uses_qu" else qv)
                out["dbias_u"][h] += (d_qv if kind == "bias_swapped" else d_qu).sum(0)
                out["dbias_v"][h] += (d_qu if kind == "bias_swapped" else d_qv).sum(0)
        out["dk"] = out["dk_all"][:, M:]
        out["dv"] = out["dv_all"][:, M:]
        return out
    return bwd


MUTANTS = ["no_delta", "no_scale", "dist_off_by_one", "dist_transposed", "dq_drops_qv", "dk_uses_qv",
           "dv_uses_g", "dr_uses_qu", "bias_swapped", "qv_uses_u"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_backward_pins_catch_planted_mistake(kind):
    bwd = _mutant(kind)
    caught = []
    for pin in PINS:
        try:
            pin(bwd)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {kind!r}"


def test_backward_unmutated_copy_passes_all_pins():
    bwd = _mutant("none")
    for pin in PINS:
        pin(bwd)
