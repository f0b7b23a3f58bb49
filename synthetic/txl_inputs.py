"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the
benchmark.

This module holds no arithmetic of the attention method itself: it draws the
random hidden states and weights, applies the input projections (the step
upstream of the attention path, Q = h W_q, K = h W_{k,E}, V = h W_v,
r = R W_{k,R}) and rounds to the storage type.  The raw distance table R is
always passed in by the caller.

Recipe (one generator per workload): ``np.random.default_rng([seed, cfg_id])``;
draw order hidden, W_q, W_k, W_v, W_r, u, v; hidden ~ N(0, 1); weights, u and v
~ N(0, 0.02^2).  fp32 workloads project in float64 and round to float32;
bf16 workloads draw and project in float32 and round to bf16 (round to
nearest even).  These shapes stand in for the language-modelling benchmarks
the pages quote (enwik8, WikiText-103, ...), which are not used.
"""

from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "round_bf16",
    "bf16_bits",
    "Segments",
    "make_segments",
    "make_prefilled",
    "project_r",
    "make_dout",
    "make_layer_weights",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int
    B: int
    H: int
    D: int
    d_model: int
    W: int
    M: int
    segments: int
    dtype: str  # "f32" or "bf16"

    @property
    def steady_segment(self) -> int:
        """First segment index (0-based) whose memory is full."""
        return -(-self.M // self.W)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 0, 1, 2, 8, 16, 4, 4, 3, "f32"),
        Workload("base", 1, 22, 8, 64, 512, 512, 512, 8, "bf16"),
        Workload("large", 2, 16, 16, 64, 1024, 384, 384, 8, "bf16"),
        Workload("wide", 3, 8, 8, 128, 1024, 768, 768, 6, "bf16"),
        Workload("long", 4, 4, 16, 64, 1024, 128, 1600, 16, "bf16"),
    ]
}


def round_bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even); returned as float32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def bf16_bits(x) -> np.ndarray:
    """uint16 storage of values that are already exactly bfloat16."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _round(x, dtype):
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return round_bf16(x)
    raise ValueError(dtype)


@dataclasses.dataclass
class Segments:
    """Projected rows of consecutive segments, already rounded.

    q, k, v: [B, n_seg * W, H, D] float32 holding exactly representable values
    of the storage type.  W_r: [dim, H*D] float64.  bias_u, bias_v: [H, D]
    float32 (kept in fp32 by the library's interface).
    """

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    W_r: np.ndarray
    bias_u: np.ndarray
    bias_v: np.ndarray
    W: int
    dtype: str

    def seg(self, name, tau):
        a = getattr(self, name)
        return a[:, tau * self.W:(tau + 1) * self.W]


def _draw(rng, shape, std, f32):
    if f32:
        return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
    return rng.standard_normal(shape) * std


def make_segments(wl: Workload, seed: int = 0, n_segments: int | None = None,
                  batch: int | None = None, rows: int | None = None) -> Segments:
    """Draw hidden states for n_segments segments and project them.

    ``rows`` overrides the total number of rows (n_segments * W by default),
    which the prefilled-memory workloads use.
    """
    n_seg = wl.segments if n_segments is None else n_segments
    B = wl.B if batch is None else batch
    HD = wl.H * wl.D
    n_rows = n_seg * wl.W if rows is None else rows
    f32 = wl.dtype == "bf16"
    rng = np.random.default_rng([seed, wl.cfg_id])
    hidden = _draw(rng, (B, n_rows, wl.d_model), 1.0, f32)
    W_q = _draw(rng, (wl.d_model, HD), 0.02, f32)
    W_k = _draw(rng, (wl.d_model, HD), 0.02, f32)
    W_v = _draw(rng, (wl.d_model, HD), 0.02, f32)
    W_r = rng.standard_normal((wl.d_model, HD)) * 0.02
    u = rng.standard_normal((wl.H, wl.D)) * 0.02
    vb = rng.standard_normal((wl.H, wl.D)) * 0.02

    def proj(Wm):
        y = hidden.reshape(-1, wl.d_model) @ Wm
        return _round(y, wl.dtype).reshape(B, n_rows, wl.H, wl.D)

    return Segments(q=proj(W_q), k=proj(W_k), v=proj(W_v), W_r=W_r,
                    bias_u=u.astype(np.float32), bias_v=vb.astype(np.float32),
                    W=wl.W, dtype=wl.dtype)


def make_prefilled(wl: Workload, M: int, seed: int = 0, batch: int | None = None):
    """One segment whose memory is pre-filled with M seeded rows.

    Returns (q [B, W, H, D], k [B, M+W, H, D], v [B, M+W, H, D], Segments).
    """
    s = make_segments(wl, seed=seed, batch=batch, rows=M + wl.W)
    return s.q[:, M:], s.k, s.v, s


def project_r(R, W_r, H, D, dtype):
    """r = R W_{k,R}, reshaped to [n_dist, H, D] and rounded to dtype."""
    R = np.asarray(R, dtype=np.float64)
    y = R @ np.asarray(W_r, dtype=np.float64)
    return _round(y, dtype).reshape(R.shape[0], H, D)


def make_dout(wl: Workload, seed: int = 0, batch: int | None = None) -> np.ndarray:
    """Output gradient dL/do [B, W, H, D] for the backward: its own generator
    ``np.random.default_rng([seed, cfg_id, 1])`` (the forward's draws are
    unchanged), entries ~ N(0, 1) rounded to the workload's storage type."""
    B = wl.B if batch is None else batch
    rng = np.random.default_rng([seed, wl.cfg_id, 1])
    g = _draw(rng, (B, wl.W, wl.H, wl.D), 1.0, wl.dtype == "bf16")
    return _round(g, wl.dtype)


def make_layer_weights(d_model: int, H: int, D: int, d_ff: int, seed: int = 0, layer: int = 0) -> dict:
    """Weights of one layer: ``np.random.default_rng([seed, 7, layer])``,
    draw order W_q, W_k, W_v, W_r, W_o, W_1, W_2 (matrices ~ N(0, 0.02^2),
    rounded to bf16, row-major [in, out]), then u, v ~ N(0, 0.02^2), b_1,
    b_2 ~ N(0, 0.02^2), the normalisations' gains ~ 1 + N(0, 0.1^2) and
    shifts ~ N(0, 0.02^2) (float32)."""
    rng = np.random.default_rng([seed, 7, layer])
    HD = H * D
    mats = {}
    for name, shape in (("W_q", (d_model, HD)), ("W_k", (d_model, HD)), ("W_v", (d_model, HD)),
                        ("W_r", (d_model, HD)), ("W_o", (HD, d_model)), ("W_1", (d_model, d_ff)),
                        ("W_2", (d_ff, d_model))):
        mats[name] = round_bf16(rng.standard_normal(shape, dtype=np.float32) * np.float32(0.02))
    f32 = lambda shape, std, mean=0.0: (mean + rng.standard_normal(shape) * std).astype(np.float32)
    mats.update(bias_u=f32((H, D), 0.02), bias_v=f32((H, D), 0.02), b_1=f32((d_ff,), 0.02),
                b_2=f32((d_model,), 0.02), ln1_gamma=f32((d_model,), 0.1, 1.0), ln1_beta=f32((d_model,), 0.02),
                ln2_gamma=f32((d_model,), 0.1, 1.0), ln2_beta=f32((d_model,), 0.02))
    return mats

