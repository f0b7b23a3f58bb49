"""Plain float64 CPU oracle for Transformer-XL relative-position attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this module: only the test suite, the entry point's ``smoke()`` check and
the benchmark's CPU-baseline leg use it.  It shares no code with the CUDA
library (no kernels, helpers, tables or constants); both sides receive the
same seeded inputs from the ``synthetic`` package and nothing else.

Every function is written for a reader checking it by eye against the pages:
no blocking, fusion or reordering beyond the definition.  NumPy matmuls serve
as plain library steps; all arithmetic is float64 on the exact values the GPU
sees (bf16 / fp32 inputs widen to float64 without rounding).

Sources (page title, then section / step / equation):

* "Transformer-XL, explained" -- method steps 2-5 (memory with stop-gradient,
  keys and values over [memory ; segment], queries from the segment only, the
  four-term relative score, the distance term computed once per distance and
  shifted into place), the symbol legend (SG, concatenation memory-first,
  R_{i-j} a parameter-free sinusoid of the distance, separate key projections
  W_{k,E} / W_{k,R}, global biases u and v) and the shift-invariance remark
  rel(5,3) = rel(105,103) = 2.
* "Long-context transformers" interactive simulation -- the segment
  recurrence equations h~ = [stop_grad(mem) ; h], K,V = h~ W, Q = h W_q,
  mem = last M rows of h~, and softmax(Q K^T / sqrt(d)) V.
* "Implementing Transformer-XL" (recurrent-memory chapter) --
  ``relative_attention``: score scaled by 1/sqrt(d_head) after all terms, the
  causal mask letting query i see every memory row plus current rows <= i,
  max-subtracted softmax, then P V.

Readings taken where the pages are silent or disagree (all listed in the
design notes):

* score:  s[i,j] = scale * ((q_i + u) . k_j + (q_i + v) . r_{M+i-j}), the four
  terms of step 4 grouped by their query-side factor;
* distance origin:  d = M + i - j in concatenated indexing (global i - j);
* no distance clipping, no softmax epsilon;
* sinusoid layout interleaved: R[d, 2k] = sin(d w_k), R[d, 2k+1] = cos(d w_k),
  w_k = 10000^(-2k/dim);
* memory = the layer's input rows, rolled as projected K/V rows;
* backward: the stop-gradient drops the memory rows' dk / dv only; r, u and
  v are shared by every pair and take their whole gradient;
* layer: post-residual normalisation with the population standard deviation
  plus 1e-6 (outside the root), ReLU feed-forward with biases, output
  projection after the attention ("Implementing Transformer-XL").

Parity status: every function here is pinned by tests in
``tests/test_oracle.py`` (closed forms, library routines, brute force); the
backward by ``tests/test_oracle_backward.py`` (finite differences of the
forward, automatic differentiation of an independent torch forward, and
identities of the score's structure); the layer and the stack by
``tests/test_oracle_layer.py`` (closed forms of the normalisation, blocks
switched off, the memory cached as rows or as projected keys and values, the
reach growing with depth).
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "sinusoid_rel",
    "relattn_forward",
    "relattn_forward_bruteforce",
    "relattn_rows",
    "relattn_backward",
    "mem_update",
    "run_segments",
    "counted_flops",
    "layer_norm",
    "layer_forward",
    "stack_forward",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def sinusoid_rel(n_dist: int, dim: int) -> np.ndarray:
    """Raw distance table R[n_dist, dim] (float64).

    "Transformer-XL, explained", symbol legend: R_{i-j} is a sinusoidal
    encoding of the distance with no trained parameters; "What it adds to
    earlier relative positions": fixed sinusoids, so any distance (also one
    longer than seen in training) has an encoding -- hence no clipping.

    Layout reading: interleaved pairs, R[d, 2k] = sin(d * w_k) and
    R[d, 2k+1] = cos(d * w_k) with w_k = 10000 ** (-2k / dim).
    """
    if dim <= 0 or dim % 2:
        raise ValueError("dim must be a positive even number")
    if n_dist < 0:
        raise ValueError("n_dist must be >= 0")
    d = np.arange(n_dist, dtype=np.float64)[:, None]
    k = np.arange(dim // 2, dtype=np.float64)[None, :]
    w = np.power(10000.0, -2.0 * k / dim)
    angle = d * w
    R = np.empty((n_dist, dim), dtype=np.float64)
    R[:, 0::2] = np.sin(angle)
    R[:, 1::2] = np.cos(angle)
    return R


def _one_head(qh, kh, vh, rh, u, vb, M, scale):
    """Relative attention for one (batch, head) pair, all in float64.

    qh [W, D] queries of the current segment; kh, vh [M+W, D] keys / values
    over [memory ; segment] (memory first); rh [n_r, D] projected distance
    keys, row d = distance d; u, vb [D] global content / distance biases.
    """
    W = qh.shape[0]
    L = kh.shape[0]
    n_r = rh.shape[0]
    # Step 4: content addressing + global content bias  ->  (q_i + u) . k_j
    ac = (qh + u) @ kh.T  # [W, L]
    # Step 5: the distance term against every available distance once ...
    g = (qh + vb) @ rh.T  # [W, n_r], g[i, d] = (q_i + v) . r_d
    # ... then each row shifted into place: key j of query i sits at
    # distance d = M + i - j (concatenated indexing, memory first).
    i = np.arange(W)[:, None]
    j = np.arange(L)[None, :]
    dist = M + i - j
    visible = dist >= 0  # mask: query i sees memory + current rows <= i
    bd = np.take_along_axis(g, np.clip(dist, 0, n_r - 1), axis=1)
    s = scale * (ac + bd)
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)  # every row has >= 1 visible key (j = M+i)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e / l) @ vh  # values carry no distance term
    lse = (m + np.log(l))[:, 0]
    return o, lse, e / l


def _check_shapes(q, k, v, r, bias_u, bias_v, M):
    B, W, H, D = q.shape
    if k.shape != (B, M + W, H, D) or v.shape != (B, M + W, H, D):
        raise ValueError(f"k/v must be [B, M+W, H, D] = {(B, M + W, H, D)}")
    if r.ndim != 3 or r.shape[1:] != (H, D) or r.shape[0] < M + W:
        raise ValueError("r must be [n_r >= M+W, H, D]")
    if bias_u.shape != (H, D) or bias_v.shape != (H, D):
        raise ValueError("bias_u / bias_v must be [H, D]")
    return B, W, H, D


def relattn_forward(q, k, v, r, bias_u, bias_v, M, scale=None, return_probs=False):
    """Relative multi-head attention of one segment over [memory ; segment].

    q [B, W, H, D]; k, v [B, M+W, H, D] (memory rows first); r [n_r, H, D]
    with n_r >= M+W, row d = distance d; bias_u, bias_v [H, D].
    Returns o [B, W, H, D] and lse [B, H, W] (natural log of the softmax
    normaliser including the row max), optionally the probabilities
    [B, H, W, M+W].

    scale defaults to 1/sqrt(D) (the simulation's softmax(QK^T/sqrt(d)) and
    the layer's division by sqrt(d_head) after all score terms).
    """
    q, k, v, r = _f64(q), _f64(k), _f64(v), _f64(r)
    bias_u, bias_v = _f64(bias_u), _f64(bias_v)
    B, W, H, D = _check_shapes(q, k, v, r, bias_u, bias_v, M)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros((B, W, H, D))
    lse = np.zeros((B, H, W))
    probs = np.zeros((B, H, W, M + W)) if return_probs else None
    for b in range(B):
        for h in range(H):
            oh, lh, ph = _one_head(q[b, :, h], k[b, :, h], v[b, :, h], r[:, h],
                                   bias_u[h], bias_v[h], M, float(scale))
            o[b, :, h] = oh
            lse[b, h] = lh
            if return_probs:
                probs[b, h] = ph
    if return_probs:
        return o, lse, probs
    return o, lse


def _one_head_backward(qh, kh, vh, rh, u, vb, M, scale, doh):
    """Gradients of L = sum(doh * o) for one (batch, head) pair, float64.

    Follows the forward of ``_one_head`` backwards, step by step:
      o = P V                     ->  dV = P^T dO,  dP = dO V^T
      P = softmax over visible j  ->  dS = P * (dP - rowsum(P * dP))
      s = scale * (ac + bd)       ->  G = scale * dS (zero where masked)
      ac = (q + u) K^T            ->  d(q+u) = G K,  dK = G^T (q+u)
      bd[i, j] = g[i, M+i-j]      ->  dg[i, d] = sum of G[i, j] over j = M+i-d
      g = (q + v) r^T             ->  d(q+v) = dg r,  dr = dg^T (q+v)
    Returns d(q+u) [W, D], d(q+v) [W, D], dK, dV [M+W, D] (every row) and
    dr [n_r, D].
    """
    W = qh.shape[0]
    L = kh.shape[0]
    n_r = rh.shape[0]
    qu = qh + u
    qv = qh + vb
    ac = qu @ kh.T
    g = qv @ rh.T
    i = np.arange(W)[:, None]
    j = np.arange(L)[None, :]
    dist = M + i - j
    visible = dist >= 0
    bd = np.take_along_axis(g, np.clip(dist, 0, n_r - 1), axis=1)
    s = np.where(visible, scale * (ac + bd), -np.inf)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    P = e / e.sum(axis=1, keepdims=True)
    dV = P.T @ doh
    dP = doh @ vh.T
    dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
    G = scale * dS  # P is 0 on masked pairs, so G is too
    d_qu = G @ kh
    dK = G.T @ qu
    dg = np.zeros((W, n_r))
    ii, jj = np.nonzero(visible)
    np.add.at(dg, (ii, dist[ii, jj]), G[ii, jj])
    d_qv = dg @ rh
    dr = dg.T @ qv
    return d_qu, d_qv, dK, dV, dr


def relattn_backward(q, k, v, r, bias_u, bias_v, M, dout, scale=None, memory_grads=False):
    """Gradients of the relative attention of one segment (float64).

    Differentiates L = sum(dout * o) with o = relattn_forward(...).  Returns a
    dict with dq [B, W, H, D], dk and dv [B, W, H, D] for the segment's own
    key / value rows, dr [n_r, H, D], dbias_u and dbias_v [H, D].

    "Transformer-XL, explained", method step 2 and the symbol SG(.): the
    memory is read as a fixed input and backpropagation stays inside the
    current segment, so the memory rows of k and v (rows 0 .. M-1) get no
    gradient.  ``memory_grads=True`` also returns ``dk_all`` / ``dv_all``
    [B, M+W, H, D] -- the plain derivatives over every key row, for tests
    only (they are what the stop-gradient discards).  r, u and v are shared
    parameters of every pair, so they take the whole gradient.
    """
    q, k, v, r = _f64(q), _f64(k), _f64(v), _f64(r)
    bias_u, bias_v, dout = _f64(bias_u), _f64(bias_v), _f64(dout)
    B, W, H, D = _check_shapes(q, k, v, r, bias_u, bias_v, M)
    if dout.shape != q.shape:
        raise ValueError("dout must be [B, W, H, D]")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.zeros((B, W, H, D))
    dk_all = np.zeros((B, M + W, H, D))
    dv_all = np.zeros((B, M + W, H, D))
    dr = np.zeros(r.shape)
    dbu = np.zeros((H, D))
    dbv = np.zeros((H, D))
    for b in range(B):
        for h in range(H):
            d_qu, d_qv, dK, dV, drh = _one_head_backward(q[b, :, h], k[b, :, h], v[b, :, h], r[:, h],
                                                         bias_u[h], bias_v[h], M, float(scale), dout[b, :, h])
            dq[b, :, h] = d_qu + d_qv  # q enters through both (q + u) and (q + v)
            dk_all[b, :, h] = dK
            dv_all[b, :, h] = dV
            dr[:, h] += drh
            dbu[h] += d_qu.sum(axis=0)
            dbv[h] += d_qv.sum(axis=0)
    out = {"dq": dq, "dk": dk_all[:, M:].copy(), "dv": dv_all[:, M:].copy(), "dr": dr,
           "dbias_u": dbu, "dbias_v": dbv}
    if memory_grads:
        out["dk_all"] = dk_all
        out["dv_all"] = dv_all
    return out


def relattn_rows(q, k, v, r, bias_u, bias_v, M, scale, b, h, rows):
    """Output rows o[b, rows, h, :] and lse[b, h, rows] computed one at a time.

    Used to check sampled outputs of full-size launches: each requested query
    row is evaluated on its own with the same definition as relattn_forward.
    """
    qh = _f64(q[b, :, h])
    kh = _f64(k[b, :, h])
    vh = _f64(v[b, :, h])
    rh = _f64(r[:, h])
    u = _f64(bias_u[h])
    vb = _f64(bias_v[h])
    rows = np.asarray(rows, dtype=np.int64)
    o = np.zeros((rows.size, qh.shape[1]))
    lse = np.zeros(rows.size)
    for n, i in enumerate(rows):
        L = M + int(i) + 1  # visible keys j = 0 .. M+i
        ac = kh[:L] @ (qh[i] + u)
        dist = M + int(i) - np.arange(L)
        bd = rh[dist] @ (qh[i] + vb)
        s = scale * (ac + bd)
        m = s.max()
        e = np.exp(s - m)
        o[n] = (e @ vh[:L]) / e.sum()
        lse[n] = m + np.log(e.sum())
    return o, lse


def relattn_forward_bruteforce(q, k, v, r, bias_u, bias_v, M, scale=None):
    """The same operation with explicit (i, j) loops and the distance formed
    directly per pair -- an independent route used only on tiny shapes."""
    q, k, v, r = _f64(q), _f64(k), _f64(v), _f64(r)
    bias_u, bias_v = _f64(bias_u), _f64(bias_v)
    B, W, H, D = _check_shapes(q, k, v, r, bias_u, bias_v, M)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros((B, W, H, D))
    lse = np.zeros((B, H, W))
    for b in range(B):
        for h in range(H):
            for i in range(W):
                scores = []
                for j in range(M + W):
                    d = M + i - j
                    if d < 0:
                        continue  # key lies after the query
                    content = 0.0
                    position = 0.0
                    for x in range(D):
                        content += (q[b, i, h, x] + bias_u[h, x]) * k[b, j, h, x]
                        position += (q[b, i, h, x] + bias_v[h, x]) * r[d, h, x]
                    scores.append((j, scale * (content + position)))
                mx = max(sc for _, sc in scores)
                z = sum(np.exp(sc - mx) for _, sc in scores)
                for j, sc in scores:
                    o[b, i, h] += np.exp(sc - mx) / z * v[b, j, h]
                lse[b, h, i] = mx + np.log(z)
    return o, lse


def mem_update(mem, h, m):
    """Memory roll: the last min(m, m_prev + w) rows of [mem ; h].

    Simulation: mem_tau = last M rows of h~_tau = [stop_grad(mem_{tau-1}) ; h_tau].
    mem [B, m_prev, C] and h [B, w, C]; rows are copied, never changed.
    """
    mem = np.asarray(mem)
    h = np.asarray(h)
    cat = np.concatenate([mem, h], axis=1)
    keep = min(m, cat.shape[1])
    return cat[:, cat.shape[1] - keep:].copy()


def run_segments(q_segs, k_segs, v_segs, r, bias_u, bias_v, M, scale=None):
    """Segment-level recurrence over consecutive segments.

    q_segs, k_segs, v_segs: lists of [B, W, H, D] per segment (projected rows
    of each segment).  The first segment sees an empty memory; afterwards the
    memory is the last M rows of [memory ; segment] (rolled as projected K/V
    rows).  Returns a list of (o, lse, M_tau) per segment.
    """
    B, W, H, D = np.asarray(q_segs[0]).shape
    mem_k = np.zeros((B, 0, H, D))
    mem_v = np.zeros((B, 0, H, D))
    out = []
    for qs, ks, vs in zip(q_segs, k_segs, v_segs):
        m_tau = mem_k.shape[1]
        kb = np.concatenate([_f64(mem_k), _f64(ks)], axis=1)
        vb_ = np.concatenate([_f64(mem_v), _f64(vs)], axis=1)
        o, lse = relattn_forward(qs, kb, vb_, r, bias_u, bias_v, m_tau, scale)
        out.append((o, lse, m_tau))
        C = H * D
        mem_k = mem_update(_f64(mem_k).reshape(B, m_tau, C), _f64(ks).reshape(B, W, C), M)
        mem_v = mem_update(_f64(mem_v).reshape(B, m_tau, C), _f64(vs).reshape(B, W, C), M)
        mem_k = mem_k.reshape(B, -1, H, D)
        mem_v = mem_v.reshape(B, -1, H, D)
    return out


def counted_flops(B, H, D, W, M):
    """Counted work of one segment: three contractions (q.k, q.r, p.v), two
    flops per multiply-add, over the visible (query, key) pairs only:
    W*M memory pairs plus W(W+1)/2 causal pairs in the current segment."""
    return 6 * B * H * D * (W * M + W * (W + 1) // 2)


# ----------------------------------------------------------------------------
# The layer and the stack around the attention
# ----------------------------------------------------------------------------

def layer_norm(x, gamma, beta, eps=1e-6):
    """Normalisation over the last axis as "Implementing Transformer-XL"
    writes it (recurrent-memory chapter, layer_norm): subtract the mean,
    divide by the population standard deviation plus eps (eps outside the
    root), then scale by gamma and shift by beta."""
    x = _f64(x)
    mean = x.mean(axis=-1, keepdims=True)
    std = x.std(axis=-1, keepdims=True)
    return _f64(gamma) * (x - mean) / (std + eps) + _f64(beta)


def _heads(x, H):
    B, T, C = x.shape
    return x.reshape(B, T, H, C // H)


def layer_forward(h, mem, P, R, H, scale=None, mem_kv=None):
    """One Transformer-XL layer on a segment, float64.

    h [B, W, d]: the layer's input rows of the segment; mem [B, M, d]: its
    input rows of the previous segment (the memory, read as a fixed input);
    P: weights -- Wq, WkE, WkR, Wv [d, H*D], u, v [H, D], Wo [H*D, d],
    g1, b1n, g2, b2n [d] (the two normalisations), W1 [d, d_ff], b1 [d_ff],
    W2 [d_ff, d], b2 [d]; R [n_r, d]: the raw distance table.

    "Implementing Transformer-XL", recurrent-memory chapter, forward and
    feed_forward: the attention over [memory ; segment] with the output
    projection, then x = LN1(h + attention), out = LN2(x + FFN(x)) with
    FFN(x) = ReLU(x W1 + b1) W2 + b2.  Keys and values come from
    [memory ; segment] through the content key and value projections, the
    distance keys from R through W_{k,R} ("Transformer-XL, explained", symbol
    legend), queries from the segment.

    mem_kv = (k_mem, v_mem) [B, M, H, D]: the memory given as its projected
    keys and values instead of its rows (the same numbers, since the
    projections act row by row); mem is then unused.
    """
    h = _f64(h)
    B, W, d = h.shape
    hk = h @ _f64(P["WkE"])
    hv = h @ _f64(P["Wv"])
    if mem_kv is not None:
        k = np.concatenate([_f64(mem_kv[0]), _heads(hk, H)], axis=1)
        v = np.concatenate([_f64(mem_kv[1]), _heads(hv, H)], axis=1)
        M = k.shape[1] - W
    else:
        mem = np.zeros((B, 0, d)) if mem is None else _f64(mem)
        M = mem.shape[1]
        ext = np.concatenate([mem, h], axis=1)
        k = _heads(ext @ _f64(P["WkE"]), H)
        v = _heads(ext @ _f64(P["Wv"]), H)
    q = _heads(h @ _f64(P["Wq"]), H)
    r = _heads((_f64(R) @ _f64(P["WkR"]))[None], H)[0]
    a, _ = relattn_forward(q, k, v, r, P["u"], P["v"], M, scale)
    y = a.reshape(B, W, -1) @ _f64(P["Wo"])
    x = layer_norm(h + y, P["g1"], P["b1n"])
    f = np.maximum(0.0, x @ _f64(P["W1"]) + _f64(P["b1"])) @ _f64(P["W2"]) + _f64(P["b2"])
    return layer_norm(x + f, P["g2"], P["b2n"])


def stack_forward(segments, layers, R, H, M, scale=None):
    """A stack of layers over consecutive segments, float64.

    segments: list of [B, W, d] inputs; layers: list of weight dicts.  Layer
    n's memory is its own input rows of the previous segment, the last M
    rows of [memory ; input] ("Transformer-XL, explained", method steps 2 and
    6: every layer caches its states, and layer n of segment t+1 reads layer
    n-1 of segment t, so the reach grows with depth).  Returns, per segment,
    the list of every layer's output.
    """
    mems = [None] * len(layers)
    out = []
    for h in segments:
        x = _f64(h)
        outs = []
        for n, P in enumerate(layers):
            y = layer_forward(x, mems[n], P, R, H, scale)
            prev = np.zeros((x.shape[0], 0, x.shape[2])) if mems[n] is None else mems[n]
            mems[n] = mem_update(prev, x, M)
            outs.append(y)
            x = y
        out.append(outs)
    return out

