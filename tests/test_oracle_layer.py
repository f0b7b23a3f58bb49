"""Pins for the oracle's layer and stack: closed forms of the normalisation,
special cases that remove one block, the equivalence of caching the memory
as rows or as projected keys and values, the growth of the reach with depth,
and a mutation test."""

import numpy as np
import pytest

from oracle import txl_oracle as O


def _params(rng, d, H, D, dff, scale=0.3):
    shapes = dict(Wq=(d, H * D), WkE=(d, H * D), WkR=(d, H * D), Wv=(d, H * D), u=(H, D), v=(H, D),
                  Wo=(H * D, d), W1=(d, dff), b1=(dff,), W2=(dff, d), b2=(d,))
    P = {k: rng.standard_normal(s) * scale for k, s in shapes.items()}
    P.update(g1=1.0 + 0.2 * rng.standard_normal(d), b1n=0.1 * rng.standard_normal(d),
             g2=1.0 + 0.2 * rng.standard_normal(d), b2n=0.1 * rng.standard_normal(d))
    return P


def _case(seed=0, B=2, W=5, M=3, H=2, D=4, dff=16, extra=2):
    rng = np.random.default_rng(seed)
    d = H * D
    P = _params(rng, d, H, D, dff)
    h = rng.standard_normal((B, W, d))
    mem = rng.standard_normal((B, M, d))
    R = O.sinusoid_rel(M + W + extra, d)
    return P, h, mem, R, H


# ----------------------------------------------------------------------------
# Pin functions: each takes (layer, norm) with the oracle's signatures.
# ----------------------------------------------------------------------------

def pin_norm_closed_forms(layer, norm):
    """A row with mean m and population std s maps to (x - m) / (s + 1e-6);
    a constant row maps to beta; gamma and beta act per column."""
    x = np.array([[1.0, 2.0, 3.0, 6.0]])
    m, s = 3.0, np.sqrt(((x - 3.0) ** 2).mean())
    np.testing.assert_allclose(norm(x, np.ones(4), np.zeros(4)), (x - m) / (s + 1e-6), rtol=1e-14)
    np.testing.assert_allclose(norm(np.full((2, 3), 7.0), np.ones(3), np.array([0.5, -1.0, 2.0])),
                               [[0.5, -1.0, 2.0]] * 2, atol=1e-12)
    g, b = np.array([2.0, -1.0, 0.5, 3.0]), np.array([0.1, 0.2, 0.3, 0.4])
    np.testing.assert_allclose(norm(x, g, b), g * norm(x, np.ones(4), np.zeros(4)) + b, rtol=1e-13)


def pin_no_attention_output(layer, norm):
    """W_o = 0 removes the attention: out = LN2(x + FFN(x)), x = LN1(h)."""
    P, h, mem, R, H = _case(1)
    P["Wo"] = np.zeros_like(P["Wo"])
    x = norm(h, P["g1"], P["b1n"])
    f = np.maximum(0, x @ P["W1"] + P["b1"]) @ P["W2"] + P["b2"]
    np.testing.assert_allclose(layer(h, mem, P, R, H), norm(x + f, P["g2"], P["b2n"]), rtol=1e-12, atol=1e-12)


def pin_constant_ffn(layer, norm):
    """W1 = 0 and b1 = c (> 0 and < 0): the FFN adds the constant row
    ReLU(c) W2 + b2, whatever its input."""
    P, h, mem, R, H = _case(2)
    P["W1"] = np.zeros_like(P["W1"])
    rng = np.random.default_rng(9)
    P["b1"] = rng.standard_normal(P["b1"].shape)
    P2 = dict(P, Wo=np.zeros_like(P["Wo"]))
    x = norm(h, P2["g1"], P2["b1n"])
    const = np.maximum(0, P["b1"]) @ P["W2"] + P["b2"]
    np.testing.assert_allclose(layer(h, mem, P2, R, H), norm(x + const, P["g2"], P["b2n"]), rtol=1e-12,
                               atol=1e-12)


def pin_memory_as_projected_rows(layer, norm):
    """Caching the memory's projected keys and values gives the layer of the
    cached rows: the projections act row by row."""
    P, h, mem, R, H = _case(3, M=6)
    B, M, d = mem.shape
    kv = ((mem @ P["WkE"]).reshape(B, M, H, -1), (mem @ P["Wv"]).reshape(B, M, H, -1))
    np.testing.assert_allclose(layer(h, None, P, R, H, mem_kv=kv), layer(h, mem, P, R, H), rtol=1e-11, atol=1e-12)


def pin_reach_grows_with_depth(layer, norm):
    """Three segments through two layers with M = W: changing segment 0
    leaves layer 1's output on segment 2 unchanged (its memory holds segment
    1's input rows only) but changes layer 2's (its memory holds layer 1's
    outputs on segment 1, which read segment 0)."""
    rng = np.random.default_rng(4)
    B, W, H, D, dff = 1, 4, 2, 4, 8
    d = H * D
    layers = [_params(rng, d, H, D, dff), _params(rng, d, H, D, dff)]
    segs = [rng.standard_normal((B, W, d)) for _ in range(3)]
    R = O.sinusoid_rel(2 * W, d)

    def run(segments):
        mems = [np.zeros((B, 0, d)), np.zeros((B, 0, d))]
        outs = []
        for x in segments:
            per = []
            for n, P in enumerate(layers):
                y = layer(x, mems[n], P, R, H)
                mems[n] = O.mem_update(mems[n], x, W)
                per.append(y)
                x = y
            outs.append(per)
        return outs

    a = run(segs)
    segs2 = [segs[0] + rng.standard_normal(segs[0].shape)] + segs[1:]
    b = run(segs2)
    np.testing.assert_array_equal(a[2][0], b[2][0])
    assert np.abs(a[2][1] - b[2][1]).max() > 1e-6


PINS = [pin_norm_closed_forms, pin_no_attention_output, pin_constant_ffn, pin_memory_as_projected_rows,
        pin_reach_grows_with_depth]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_layer_pins(pin):
    pin(O.layer_forward, O.layer_norm)


def test_stack_matches_layer_loop():
    """stack_forward is the per-layer loop with each layer's memory its own
    input rows (the oracle's two entry points agree)."""
    rng = np.random.default_rng(5)
    B, W, M, H, D, dff = 2, 3, 4, 2, 4, 8
    d = H * D
    layers = [_params(rng, d, H, D, dff) for _ in range(3)]
    segs = [rng.standard_normal((B, W, d)) for _ in range(3)]
    R = O.sinusoid_rel(M + W, d)
    got = O.stack_forward(segs, layers, R, H, M)
    mems = [np.zeros((B, 0, d))] * 3
    for t, x in enumerate(segs):
        for n, P in enumerate(layers):
            y = O.layer_forward(x, mems[n], P, R, H)
            mems[n] = O.mem_update(mems[n], x, M)
            np.testing.assert_allclose(got[t][n], y, rtol=1e-13)
            x = y


# ----------------------------------------------------------------------------
# Mutation test
# ----------------------------------------------------------------------------

def _mutant(kind):
    def norm(x, g, b, eps=1e-6):
        x = np.asarray(x, dtype=np.float64)
        mean = x.mean(-1, keepdims=True)
        if kind == "eps_in_root":
            return g * (x - mean) / np.sqrt(x.var(-1, keepdims=True) + 1e-2) + b
        return g * (x - mean) / (x.std(-1, keepdims=True) + eps) + b

    def layer(h, mem, P, R, H, scale=None, mem_kv=None):
        h = np.asarray(h, dtype=np.float64)
        B, W, d = h.shape
        if mem_kv is not None:
            k = np.concatenate([mem_kv[0], (h @ P["WkE"]).reshape(B, W, H, -1)], 1)
            v = np.concatenate([mem_kv[1], (h @ P["Wv"]).reshape(B, W, H, -1)], 1)
            M = k.shape[1] - W
        else:
            mem = np.zeros((B, 0, d)) if mem is None else mem
            M = mem.shape[1]
            ext = np.concatenate([mem, h], 1)
            k = (ext @ (P["Wq"] if kind == "key_from_query" else P["WkE"])).reshape(B, M + W, H, -1)
            v = (ext @ P["Wv"]).reshape(B, M + W, H, -1)
        q = (h @ P["Wq"]).reshape(B, W, H, -1)
        r = (R @ P["WkR"]).reshape(R.shape[0], H, -1)
        a, _ = O.relattn_forward(q, k, v, r, P["u"], P["v"], M, scale)
        y = a.reshape(B, W, -1) @ (np.eye(d) if kind == "no_wo" else P["Wo"])
        x = norm((0 if kind == "no_residual" else h) + y, P["g1"], P["b1n"])
        pre = x @ P["W1"] + P["b1"]
        f = (pre if kind == "no_relu" else np.maximum(0, pre)) @ P["W2"] + P["b2"]
        return norm(x + f, P["g2"], P["b2n"])
    return layer, norm


MUTANTS = ["eps_in_root", "key_from_query", "no_wo", "no_residual", "no_relu"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_layer_pins_catch_planted_mistake(kind):
    layer, norm = _mutant(kind)
    caught = []
    for pin in PINS:
        try:
            pin(layer, norm)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {kind!r}"


def test_layer_unmutated_copy_passes_all_pins():
    layer, norm = _mutant("none")
    for pin in PINS:
        pin(layer, norm)


def test_reach_pin_catches_memory_of_outputs():
    """Caching each layer's output rather than its input breaks the reach
    pin: layer 1 on segment 2 then depends on segment 0 through its memory."""
    rng = np.random.default_rng(4)
    B, W, H, D, dff = 1, 4, 2, 4, 8
    d = H * D
    layers = [_params(rng, d, H, D, dff), _params(rng, d, H, D, dff)]
    segs = [rng.standard_normal((B, W, d)) for _ in range(3)]
    R = O.sinusoid_rel(2 * W, d)

    def run(segments):
        mems = [np.zeros((B, 0, d)), np.zeros((B, 0, d))]
        outs = []
        for x in segments:
            per = []
            for n, P in enumerate(layers):
                y = O.layer_forward(x, mems[n], P, R, H)
                mems[n] = O.mem_update(mems[n], y, W)  # the mistake: outputs cached
                per.append(y)
                x = y
            outs.append(per)
        return outs

    a = run(segs)
    b = run([segs[0] + rng.standard_normal(segs[0].shape)] + segs[1:])
    assert not np.array_equal(a[2][0], b[2][0])
