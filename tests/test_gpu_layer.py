"""GPU parity of txl_layer_forward (one Transformer-XL layer, the attention
memory as rings of projected keys and values) against the oracle's layer and
stack.  Tolerance: every intermediate (q, k, v, r, the attention output, the
projections, the FFN hidden layer, the normalised rows) is stored in bf16, a
relative rounding of 2^-9 each; after the normalisations the outputs are
O(1), and the measured error stays well inside rel-L2 <= 1e-2 and
max |err| <= 0.1."""

import numpy as np
import pytest
import torch

from oracle import txl_oracle as O
from synthetic import make_layer_weights, round_bf16

from gpu_util import dev

pytestmark = pytest.mark.gpu

REL_L2, ATOL = 1e-2, 1e-1

# oracle weight names for the library's
ORACLE_NAMES = {"W_q": "Wq", "W_k": "WkE", "W_v": "Wv", "W_r": "WkR", "bias_u": "u", "bias_v": "v", "W_o": "Wo",
                "ln1_gamma": "g1", "ln1_beta": "b1n", "W_1": "W1", "b_1": "b1", "W_2": "W2", "b_2": "b2",
                "ln2_gamma": "g2", "ln2_beta": "b2n"}


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import transformer_xl_relative_txl_gb300 as lib  # fails loudly if not built

    torch.cuda.set_device(0)
    lib.txl_get_device_status()
    return lib


def _weights(d, H, D, dff, layer=0, packed=False):
    """Oracle and device weights; packed puts W_q, W_k, W_v back to back in
    one [3, d, H*D] allocation (the layer's batched-projection path)."""
    w = make_layer_weights(d, H, D, dff, seed=3, layer=layer)
    P = {ORACLE_NAMES[k]: v.astype(np.float64) for k, v in w.items()}
    dw = {k: torch.from_numpy(v).to(dev()).to(torch.bfloat16 if k.startswith("W_") else torch.float32).contiguous()
          for k, v in w.items()}
    if packed:
        qkv = torch.stack([dw["W_q"], dw["W_k"], dw["W_v"]])
        dw["W_q"], dw["W_k"], dw["W_v"] = qkv[0], qkv[1], qkv[2]
    return P, dw


def _close(got, want, what):
    err = got.astype(np.float64) - want
    rel = np.linalg.norm(err) / np.linalg.norm(want)
    mx = np.abs(err).max()
    assert np.all(np.isfinite(got)), what
    assert rel <= REL_L2 and mx <= ATOL, f"{what}: rel-L2 {rel:.3e}, max abs {mx:.3e}"
    return rel


@pytest.mark.parametrize("B,W,M,H,D,dff,packed", [
    (2, 128, 128, 4, 64, 1024, False),  # ring of M+W rows: the append runs inside the attention kernel
    (2, 128, 128, 4, 64, 1024, True),   # the same, q/k/v projections as one batched GEMM launch
    (1, 72, 40, 2, 64, 256, True),      # memory, segment and rows (72) off the tile grids
    (2, 64, 0, 2, 128, 512, False),     # first segment, D = 128
    (3, 64, 64, 16, 64, 128, True),     # d_model = 1024, the widest normalisation
    (1, 100, 64, 2, 64, 136, False),    # d_ff = 136: a GEMM k and n off the 64-column grid
])
def test_layer_matches_oracle(txl, B, W, M, H, D, dff, packed):
    d = H * D
    P, dw = _weights(d, H, D, dff, packed=packed)
    rng = np.random.default_rng(B * 1000 + W + M)
    h = round_bf16(rng.standard_normal((B, W, d)).astype(np.float32)).astype(np.float64)
    mem = round_bf16(rng.standard_normal((B, M, d)).astype(np.float32)).astype(np.float64)
    # the memory's projected keys and values, as a previous call would have cached them (bf16)
    k_mem = round_bf16((mem @ P["WkE"]).astype(np.float32)).reshape(B, M, H, D)
    v_mem = round_bf16((mem @ P["Wv"]).astype(np.float32)).reshape(B, M, H, D)
    n_r = M + W
    R = round_bf16(O.sinusoid_rel(n_r, d).astype(np.float32))
    cap = M + W
    start = 0
    k_ring = torch.zeros(B, cap, H, D, device=dev(), dtype=torch.bfloat16)
    v_ring = torch.zeros_like(k_ring)
    k_ring[:, :M] = torch.from_numpy(k_mem).to(dev()).to(torch.bfloat16)
    v_ring[:, :M] = torch.from_numpy(v_mem).to(dev()).to(torch.bfloat16)
    hd = torch.from_numpy(h.astype(np.float32)).to(dev()).to(torch.bfloat16)
    Rd = torch.from_numpy(R).to(dev()).to(torch.bfloat16)
    out = torch.empty_like(hd)
    ws = torch.empty(txl.txl_layer_workspace_bytes(B, W, d, H, D, dff, n_r), device=dev(), dtype=torch.uint8)
    s2, m2 = txl.txl_layer_forward(hd, out, k_ring, v_ring, start, M, dw, Rd, ws)
    assert txl.txl_get_device_status() == 0
    assert (s2, m2) == (0, M + W)
    want = O.layer_forward(h, None, P, R.astype(np.float64), H, mem_kv=(k_mem, v_mem))
    _close(out.float().cpu().numpy(), want, "layer output")
    # the segment's projected rows were appended after the memory
    new_k = k_ring[:, M:M + W].float().cpu().numpy().reshape(B, W, d)
    new_v = v_ring[:, M:M + W].float().cpu().numpy().reshape(B, W, d)
    _close(new_k, h @ P["WkE"], "appended keys")
    _close(new_v, h @ P["Wv"], "appended values")
    assert torch.equal(k_ring[:, :M].cpu(), torch.from_numpy(k_mem).to(torch.bfloat16))  # memory untouched


def test_layer_base_size(txl):
    """The layer at the bench's shapes (B=22 W=512 M=512, 8 heads of 64,
    d_ff=2048, packed projections, a ring of M+W rows) in one call, against
    the oracle's layer on every output row."""
    B, W, M, H, D, dff = 22, 512, 512, 8, 64, 2048
    d = H * D
    P, dw = _weights(d, H, D, dff, packed=True)
    rng = np.random.default_rng(11)
    h = round_bf16(rng.standard_normal((B, W, d)).astype(np.float32)).astype(np.float64)
    mem = round_bf16(rng.standard_normal((B, M, d)).astype(np.float32)).astype(np.float64)
    k_mem = round_bf16((mem @ P["WkE"]).astype(np.float32)).reshape(B, M, H, D)
    v_mem = round_bf16((mem @ P["Wv"]).astype(np.float32)).reshape(B, M, H, D)
    n_r = M + W
    R = round_bf16(O.sinusoid_rel(n_r, d).astype(np.float32))
    cap = M + W
    k_ring = torch.zeros(B, cap, H, D, device=dev(), dtype=torch.bfloat16)
    v_ring = torch.zeros_like(k_ring)
    k_ring[:, :M] = torch.from_numpy(k_mem).to(dev()).to(torch.bfloat16)
    v_ring[:, :M] = torch.from_numpy(v_mem).to(dev()).to(torch.bfloat16)
    hd = torch.from_numpy(h.astype(np.float32)).to(dev()).to(torch.bfloat16)
    Rd = torch.from_numpy(R).to(dev()).to(torch.bfloat16)
    out = torch.empty_like(hd)
    ws = torch.empty(txl.txl_layer_workspace_bytes(B, W, d, H, D, dff, n_r), device=dev(), dtype=torch.uint8)
    assert txl.txl_layer_forward(hd, out, k_ring, v_ring, 0, M, dw, Rd, ws) == (0, M + W)
    assert txl.txl_get_device_status() == 0
    want = O.layer_forward(h, None, P, R.astype(np.float64), H, mem_kv=(k_mem, v_mem))
    _close(out.float().cpu().numpy(), want, "layer output at base size")


def test_stack_matches_oracle(txl):
    """Two layers over four segments (B=2, W=64, M=64, d=128): each layer
    keeps its own rings (M+W rows) and reads the last M of them; every
    layer's output against the oracle's stack, which caches hidden rows."""
    B, W, M, H, D, dff, S, N = 2, 64, 64, 2, 64, 256, 4, 2
    d = H * D
    layers = [_weights(d, H, D, dff, layer=n) for n in range(N)]
    rng = np.random.default_rng(77)
    segs = [round_bf16(rng.standard_normal((B, W, d)).astype(np.float32)).astype(np.float64) for _ in range(S)]
    n_r = M + W
    R = round_bf16(O.sinusoid_rel(n_r, d).astype(np.float32))
    Rd = torch.from_numpy(R).to(dev()).to(torch.bfloat16)
    want = O.stack_forward(segs, [P for P, _ in layers], R.astype(np.float64), H, M)
    cap = M + W
    rings = [(torch.zeros(B, cap, H, D, device=dev(), dtype=torch.bfloat16),
              torch.zeros(B, cap, H, D, device=dev(), dtype=torch.bfloat16)) for _ in range(N)]
    state = [(0, 0)] * N  # per layer: ring row of the memory's first row, memory rows
    ws = torch.empty(txl.txl_layer_workspace_bytes(B, W, d, H, D, dff, n_r), device=dev(), dtype=torch.uint8)
    for t in range(S):
        x = torch.from_numpy(segs[t].astype(np.float32)).to(dev()).to(torch.bfloat16)
        for n in range(N):
            start, m = state[n]
            y = torch.empty_like(x)
            s2, m2 = txl.txl_layer_forward(x, y, rings[n][0], rings[n][1], start, m, layers[n][1], Rd, ws)
            keep = min(m2, M)
            state[n] = ((s2 + m2 - keep) % cap, keep)  # the next memory: the last M rows
            _close(y.float().cpu().numpy(), want[t][n], f"segment {t} layer {n}")
            x = y
    assert txl.txl_get_device_status() == 0


def test_stack_entry_matches_oracle(txl):
    """txl_stack_forward: three layers in one call per segment over four
    segments (B=2, W=64, M=64, d=128), the layers' rings advancing together;
    the last layer's output against the oracle's stack."""
    B, W, M, H, D, dff, S, N = 2, 64, 64, 2, 64, 256, 4, 3
    d = H * D
    layers = [_weights(d, H, D, dff, layer=n, packed=(n == 1)) for n in range(N)]
    rng = np.random.default_rng(78)
    segs = [round_bf16(rng.standard_normal((B, W, d)).astype(np.float32)).astype(np.float64) for _ in range(S)]
    n_r = M + W
    R = round_bf16(O.sinusoid_rel(n_r, d).astype(np.float32))
    Rd = torch.from_numpy(R).to(dev()).to(torch.bfloat16)
    want = O.stack_forward(segs, [P for P, _ in layers], R.astype(np.float64), H, M)
    cap = M + W
    k_rings = [torch.zeros(B, cap, H, D, device=dev(), dtype=torch.bfloat16) for _ in range(N)]
    v_rings = [torch.zeros(B, cap, H, D, device=dev(), dtype=torch.bfloat16) for _ in range(N)]
    ws = torch.empty(txl.txl_stack_workspace_bytes(B, W, d, H, D, dff, n_r), device=dev(), dtype=torch.uint8)
    start, m = 0, 0
    for t in range(S):
        x = torch.from_numpy(segs[t].astype(np.float32)).to(dev()).to(torch.bfloat16)
        y = torch.empty_like(x)
        s2, m2 = txl.txl_stack_forward(x, y, k_rings, v_rings, start, m, [dw for _, dw in layers], Rd, ws)
        keep = min(m2, M)
        start, m = (s2 + m2 - keep) % cap, keep
        _close(y.float().cpu().numpy(), want[t][N - 1], f"segment {t}, last layer")
    assert txl.txl_get_device_status() == 0
    with pytest.raises(txl.TxlError) as e:  # two layers sharing a ring
        txl.txl_stack_forward(x, y, [k_rings[0], k_rings[0], k_rings[2]], v_rings, start, m,
                              [dw for _, dw in layers], Rd, ws)
    assert e.value.status == 3


def test_layer_rejects_bad_arguments(txl):
    B, W, M, H, D, dff = 1, 64, 0, 2, 64, 128
    d = H * D
    _, dw = _weights(d, H, D, dff)
    h = torch.zeros(B, W, d, device=dev(), dtype=torch.bfloat16)
    ring = torch.zeros(B, 128, H, D, device=dev(), dtype=torch.bfloat16)
    R = torch.zeros(M + W, d, device=dev(), dtype=torch.bfloat16)
    need = txl.txl_layer_workspace_bytes(B, W, d, H, D, dff, M + W)
    small = torch.empty(need - 256, device=dev(), dtype=torch.uint8)
    with pytest.raises(txl.TxlError) as e:  # workspace too small
        txl.txl_layer_forward(h, torch.empty_like(h), ring, ring.clone(), 0, 0, dw, R, small)
    assert e.value.status == 1
    ws = torch.empty(need, device=dev(), dtype=torch.uint8)
    with pytest.raises(txl.TxlError) as e:  # output over the input
        txl.txl_layer_forward(h, h, ring, ring.clone(), 0, 0, dw, R, ws)
    assert e.value.status == 3
    assert txl.txl_get_device_status() == 0
