"""GPU parity of txl_relattn_backward against the float64 oracle's backward.

The forward runs first on the device (its o and lse feed the backward, as in
training); the oracle differentiates the same seeded inputs from scratch.
Tolerances: fp32 inputs max |err| <= 1e-5 * max(1, max |want|); bf16 inputs
rel-L2 <= 5e-3 and max |err| <= 2e-2 * max(1, max |want|) per gradient
tensor.  On the bf16 path G = scale P (dP - Delta) enters the gradient
products rounded to bf16 (2^-9 relative), beside the forward's bf16 o in
Delta.  The two bias gradients are [H, D] sums over every (sequence, query)
row of d(q+u) and d(q+v), whose terms largely cancel: their norm is a small
residue of the summed magnitudes, so the same per-term rounding is a larger
fraction of it (up to 6e-3 measured at the large workload, against about
2e-3 for every other gradient).  Their rel-L2 bound is 1e-2; the max |err|
bound is the same as for the others.
"""

import numpy as np
import pytest
import torch

from oracle import txl_oracle as O
from synthetic import make_dout

from gpu_util import dev, prefilled_case, to_dev, torch_dtype, workload

pytestmark = pytest.mark.gpu

KEYS = ["dq", "dk", "dv", "dr", "dbias_u", "dbias_v"]


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import transformer_xl_relative_txl_gb300 as lib  # fails loudly if not built

    torch.cuda.set_device(0)
    lib.txl_get_device_status()
    return lib


def _case(B, H, D, W, M, dtype, n_r_extra=0, seed=0):
    wl = workload(B, H, D, W, M, dtype)
    q, k, v, r, bu, bv = prefilled_case(wl, seed=seed, n_r_extra=n_r_extra)
    dout = make_dout(wl, seed=seed)
    return q, k, v, r, bu, bv, dout


def _run(txl, q, k, v, r, bu, bv, dout, M, dtype, o_dtype=None, scale=None):
    td = torch_dtype(dtype)
    od = td if o_dtype is None else torch_dtype(o_dtype)
    qd, kd, vd, rd = (to_dev(x, td) for x in (q, k, v, r))
    bud, bvd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    B, W, H, D = q.shape
    o = torch.empty(qd.shape, device=dev(), dtype=od)
    lse = torch.empty(B, H, W, device=dev(), dtype=torch.float32)
    txl.txl_relattn_forward(qd, kd, vd, rd, bud, bvd, o, lse, M=M, scale=scale)
    g = txl.txl_relattn_backward(qd, kd, vd, rd, bud, bvd, o, lse, to_dev(dout, od), M=M, scale=scale)
    assert txl.txl_get_device_status() == 0
    return {key: t.cpu().numpy() for key, t in g.items()}


def _compare(got, want, dtype):
    for key in KEYS:
        a = got[key].astype(np.float64)
        b = want[key]
        assert a.shape == b.shape, key
        assert np.all(np.isfinite(a)), key
        scale = max(1.0, float(np.abs(b).max()) if b.size else 1.0)
        err = np.abs(a - b).max() if a.size else 0.0
        if dtype == "f32":
            assert err <= 1e-5 * scale, f"{key}: max abs {err:.3e} (scale {scale:.3e})"
        else:
            rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
            rel_bound = 1e-2 if key.startswith("dbias") else 5e-3
            assert rel <= rel_bound and err <= 2e-2 * scale, f"{key}: rel-L2 {rel:.3e}, max abs {err:.3e}"


CASES = [
    # B, H, D, W, M, dtype, n_r_extra
    (1, 2, 8, 4, 4, "f32", 0),       # the tiny configuration
    (1, 2, 8, 4, 0, "f32", 0),       # first segment: empty memory
    (2, 2, 16, 37, 29, "f32", 3),    # ragged, unused distance rows
    (1, 1, 5, 6, 2, "f32", 1),       # odd head dim (scalar row loads)
    (2, 2, 64, 130, 70, "bf16", 0),  # several tiles, ragged
    (1, 2, 128, 64, 0, "bf16", 2),
    (1, 1, 64, 5, 3, "bf16", 0),     # fewer rows than a warp
    (1, 2, 256, 40, 24, "f32", 0),   # largest head dim
    # bf16, D = 64: the tensor-core kernels
    (2, 3, 64, 300, 37, "bf16", 5),  # memory not a multiple of the key step
    (1, 2, 64, 256, 0, "bf16", 0),   # first segment, whole tiles
    (1, 2, 64, 128, 512, "bf16", 0), # memory longer than the segment
    (3, 1, 64, 64, 64, "bf16", 64),  # half a query tile
    # bf16, D = 128: the tensor-core kernels (memory a multiple of 8 rows)
    (2, 2, 128, 200, 136, "bf16", 3),  # several tiles, ragged
    (1, 3, 128, 300, 512, "bf16", 0),  # memory longer than the segment
    (2, 1, 128, 7, 8, "bf16", 1),      # fewer rows than a warp
    (3, 5, 128, 64, 0, "bf16", 7),     # odd head count, half a tile, empty memory
    # bf16, memory not a multiple of 8: the dk / dv tiles start before column M
    (1, 2, 128, 130, 37, "bf16", 0),
    (2, 2, 128, 300, 77, "bf16", 2),   # several dk / dv tiles, each shifted by 5 keys
    (2, 1, 64, 9, 15, "bf16", 0),      # fewer rows than a warp, shifted by 7
    (1, 1, 64, 520, 1, "bf16", 0),     # five dk / dv tiles, shifted by 1
]


@pytest.mark.parametrize("B,H,D,W,M,dtype,extra", CASES)
def test_backward_matches_oracle(txl, B, H, D, W, M, dtype, extra):
    q, k, v, r, bu, bv, dout = _case(B, H, D, W, M, dtype, extra)
    scale = D ** -0.5
    got = _run(txl, q, k, v, r, bu, bv, dout, M, dtype)
    want = O.relattn_backward(q, k, v, r, bu, bv, M, dout, scale)
    _compare(got, want, dtype)
    assert np.all(got["dr"][M + W:] == 0)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("B,H,W,M,extra", [
    (2, 3, 300, 40, 5),    # several tiles, ragged, unused distance rows
    (1, 2, 256, 0, 0),     # first segment, whole tiles
    (1, 2, 128, 512, 0),   # memory longer than the segment
    (2, 1, 7, 8, 1),       # fewer rows than a warp
    (2, 2, 260, 45, 3),    # memory not a multiple of 8
])
def test_backward_d64_each_path(txl, path, B, H, W, M, extra):
    """D = 64 through each tensor-core path, forced by the test hook: 1 the
    fused kernels, 2 the materialised pair terms (the library's choice),
    against the oracle; the
    pair-term path also bit for bit between two calls (every sum has a fixed
    order there)."""
    q, k, v, r, bu, bv, dout = _case(B, H, 64, W, M, "bf16", extra)
    txl.txl_debug_force_bwd_path(path)
    try:
        got = _run(txl, q, k, v, r, bu, bv, dout, M, "bf16")
        again = _run(txl, q, k, v, r, bu, bv, dout, M, "bf16")
    finally:
        txl.txl_debug_force_bwd_path(0)
    want = O.relattn_backward(q, k, v, r, bu, bv, M, dout, 64 ** -0.5)
    _compare(got, want, "bf16")
    assert np.all(got["dr"][M + W:] == 0)
    if path == 2:
        for key in KEYS:
            assert np.array_equal(got[key], again[key]), key


@pytest.mark.parametrize("D,M", [(128, 8), (64, 0), (64, 8)])
def test_backward_one_query_row(txl, D, M):
    """W = 1: one softmax row over M + 1 keys.  dv = p dout has no
    cancellation and meets the rel-L2 bound.  Every other gradient is built
    from g = scale p (dout.v_j - Delta), whose difference nearly cancels when
    the row has few keys (with M = 0 the exact gradient is zero); there the
    bf16 o that Delta = dout.o takes from the forward decides the relative
    error, so those gradients are held to the max |err| bound only."""
    q, k, v, r, bu, bv, dout = _case(1, 1, D, 1, M, "bf16")
    got = _run(txl, q, k, v, r, bu, bv, dout, M, "bf16")
    want = O.relattn_backward(q, k, v, r, bu, bv, M, dout, D ** -0.5)
    a, b = got["dv"].astype(np.float64), want["dv"]
    assert np.linalg.norm(a - b) / np.linalg.norm(b) <= 5e-3
    for key in KEYS:
        a, b = got[key].astype(np.float64), want[key]
        assert np.all(np.isfinite(a)), key
        assert np.abs(a - b).max() <= 2e-2 * max(1.0, np.abs(b).max()), key


def test_backward_fp32_output_gradient_with_bf16_inputs(txl):
    """bf16 q, k, v, r with an fp32 o and dout."""
    q, k, v, r, bu, bv, dout = _case(2, 2, 64, 70, 60, "bf16")
    got = _run(txl, q, k, v, r, bu, bv, dout, 60, "bf16", o_dtype="f32")
    want = O.relattn_backward(q, k, v, r, bu, bv, 60, dout, 64 ** -0.5)
    _compare(got, want, "bf16")


def test_backward_custom_scale(txl):
    q, k, v, r, bu, bv, dout = _case(1, 2, 16, 9, 7, "f32")
    got = _run(txl, q, k, v, r, bu, bv, dout, 7, "f32", scale=0.31)
    want = O.relattn_backward(q, k, v, r, bu, bv, 7, dout, 0.31)
    _compare(got, want, "f32")


@pytest.mark.parametrize("D,dtype,o_dtype", [(64, "bf16", "f32"), (64, "f32", "f32"), (64, "bf16", "bf16"),
                                             (128, "bf16", "bf16")])
def test_backward_deterministic(txl, D, dtype, o_dtype):
    """Bit-identical on repeated calls.  (The fused D = 64 kernels, which the
    library takes for bf16 o and dout when M is not a multiple of 8, add dr
    by atomic fp32 adds in any order; there dr agrees to fp32 rounding.  At
    M = 72 every bf16 case here takes the pair-term path, which sums in a
    fixed order.)"""
    q, k, v, r, bu, bv, dout = _case(2, 2, D, 130, 72, dtype)
    a = _run(txl, q, k, v, r, bu, bv, dout, 72, dtype, o_dtype=o_dtype)
    b = _run(txl, q, k, v, r, bu, bv, dout, 72, dtype, o_dtype=o_dtype)
    for key in KEYS:
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("D", [64, 128])
def test_backward_captured_in_a_graph(txl, D):
    """The pair-term backward (three kernels, each launched behind the one
    before it with programmatic serialisation, and a tile counter the first
    zeroes for the second) captured into a CUDA graph after one eager call
    (which allocates the scratch) and replayed twice: bit for bit the eager
    result each time."""
    q, k, v, r, bu, bv, dout = _case(2, 2, D, 200, 136, "bf16")
    td = torch.bfloat16
    qd, kd, vd, rd = (to_dev(x, td) for x in (q, k, v, r))
    bud, bvd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    o = torch.empty(qd.shape, device=dev(), dtype=td)
    lse = torch.empty(2, 2, 200, device=dev(), dtype=torch.float32)
    txl.txl_relattn_forward(qd, kd, vd, rd, bud, bvd, o, lse, M=136)
    gd = to_dev(dout, td)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()  # the library keeps scratch per stream: warm up the capture stream
    with torch.cuda.stream(side):
        eager = txl.txl_relattn_backward(qd, kd, vd, rd, bud, bvd, o, lse, gd, M=136)
    torch.cuda.synchronize()
    want = {key: t.clone() for key, t in eager.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        txl.txl_relattn_backward(qd, kd, vd, rd, bud, bvd, o, lse, gd, M=136, grads=eager)
    for _ in range(2):
        for t in eager.values():
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert txl.txl_get_device_status() == 0
        for key in KEYS:
            assert torch.equal(eager[key], want[key]), key


def test_backward_d128_scratch_reuse(txl):
    """The D = 128 tensor-core path keeps its pair terms in a scratch buffer
    reused across calls: a call after one of another shape (which leaves
    nonzero pair terms where this call's layout has zeros to read) must still
    match the oracle."""
    big = _case(2, 2, 128, 250, 264, "bf16", seed=1)
    _run(txl, *big, 264, "bf16")
    q, k, v, r, bu, bv, dout = _case(1, 2, 128, 190, 40, "bf16", seed=2)
    got = _run(txl, q, k, v, r, bu, bv, dout, 40, "bf16")
    want = O.relattn_backward(q, k, v, r, bu, bv, 40, dout, 128 ** -0.5)
    _compare(got, want, "bf16")


def test_backward_d128_chunked(txl):
    """The D = 128 tensor-core path over a batch split into chunks of
    sequences (here one per chunk, forced by a small scratch cap): dq, dk and
    dv are per-sequence work and come out bit-identical to one chunk; dr and
    the bias gradients, which sum over the sequences, match the oracle."""
    q, k, v, r, bu, bv, dout = _case(3, 2, 128, 200, 136, "bf16", 2)
    whole = _run(txl, q, k, v, r, bu, bv, dout, 136, "bf16")
    try:
        txl.txl_debug_set_bwd_chunk_bytes(2 << 20)  # one sequence's scratch is about 1.6 MB
        parts = _run(txl, q, k, v, r, bu, bv, dout, 136, "bf16")
    finally:
        txl.txl_debug_set_bwd_chunk_bytes(0)
    for key in ("dq", "dk", "dv"):
        assert np.array_equal(parts[key], whole[key]), key
    want = O.relattn_backward(q, k, v, r, bu, bv, 136, dout, 128 ** -0.5)
    _compare(parts, want, "bf16")
    assert np.all(parts["dr"][136 + 200:] == 0)


@pytest.mark.parametrize("D,path", [(64, 1), (64, 2), (128, 0)])
def test_backward_bounded_wait_reports_timeout(txl, D, path):
    """The backward's loads stop after its first two key steps (test hook),
    so the bounded waits of the roles that need later steps run out (50 ms):
    the kernels unwind, the status word reports the timeout, and the next
    call computes correctly.  D = 64 on each tensor-core path."""
    q, k, v, r, bu, bv, dout = _case(1, 2, D, 128, 256, "bf16")  # six key steps
    td = torch.bfloat16
    qd, kd, vd, rd = (to_dev(x, td) for x in (q, k, v, r))
    bud, bvd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    o = torch.empty(qd.shape, device=dev(), dtype=td)
    lse = torch.empty(1, 2, 128, device=dev(), dtype=torch.float32)
    txl.txl_relattn_forward(qd, kd, vd, rd, bud, bvd, o, lse, M=256)
    assert txl.txl_get_device_status() == 0
    assert txl.txl_debug_set_wait_limit_ns(50_000_000) == 0
    try:
        txl.txl_debug_force_bwd_path(path)
        assert txl.txl_debug_inject_stall(True) == 0
        txl.txl_relattn_backward(qd, kd, vd, rd, bud, bvd, o, lse, to_dev(dout, td), M=256)
        assert txl.txl_get_device_status() == 5  # TXL_ERR_DEVICE_TIMEOUT
        assert txl.txl_get_device_status() == 0  # the word was cleared
        got = _run(txl, q, k, v, r, bu, bv, dout, 256, "bf16")
    finally:
        txl.txl_debug_inject_stall(False)
        txl.txl_debug_set_wait_limit_ns(2_000_000_000)
        txl.txl_debug_force_bwd_path(0)
    want = O.relattn_backward(q, k, v, r, bu, bv, 256, dout, D ** -0.5)
    _compare(got, want, "bf16")


def test_backward_base_size_sampled_head(txl):
    """The base workload at full size (B=22, H=8, D=64, W=512, M=512) in one
    call; the oracle checks every gradient of one head (dq, dk, dv of all 22
    sequences, and dr, dbias_u, dbias_v, which sum over them)."""
    B, H, D, W, M = 22, 8, 64, 512, 512
    q, k, v, r, bu, bv, dout = _case(B, H, D, W, M, "bf16")
    got = _run(txl, q, k, v, r, bu, bv, dout, M, "bf16")
    h = 3
    sl = slice(h, h + 1)
    want = O.relattn_backward(q[:, :, sl], k[:, :, sl], v[:, :, sl], r[:, sl], bu[sl], bv[sl], M, dout[:, :, sl],
                              D ** -0.5)
    head = {"dq": got["dq"][:, :, sl], "dk": got["dk"][:, :, sl], "dv": got["dv"][:, :, sl],
            "dr": got["dr"][:, sl], "dbias_u": got["dbias_u"][sl], "dbias_v": got["dbias_v"][sl]}
    _compare(head, want, "bf16")


@pytest.mark.parametrize("name,heads", [("large", [11]), ("wide", [5]), ("long", None)])
def test_backward_full_size(txl, name, heads):
    """The other workloads at full size in one call each: large (D = 64),
    wide (D = 128) and long (W = 128 over M = 1600 rows), all three on the
    tensor cores; every gradient of the listed heads (every
    head of long) against the oracle's backward of the same inputs."""
    from synthetic import WORKLOADS

    wl = WORKLOADS[name]
    B, H, D, W, M = wl.B, wl.H, wl.D, wl.W, wl.M
    q, k, v, r, bu, bv, dout = _case(B, H, D, W, M, "bf16")
    got = _run(txl, q, k, v, r, bu, bv, dout, M, "bf16")
    for h in (range(H) if heads is None else heads):
        sl = slice(h, h + 1)
        want = O.relattn_backward(q[:, :, sl], k[:, :, sl], v[:, :, sl], r[:, sl], bu[sl], bv[sl], M,
                                  dout[:, :, sl], D ** -0.5)
        head = {"dq": got["dq"][:, :, sl], "dk": got["dk"][:, :, sl], "dv": got["dv"][:, :, sl],
                "dr": got["dr"][:, sl], "dbias_u": got["dbias_u"][sl], "dbias_v": got["dbias_v"][sl]}
        _compare(head, want, "bf16")


def test_backward_rejects_bad_arguments(txl):
    q, k, v, r, bu, bv, dout = _case(1, 2, 8, 4, 4, "f32")
    qd, kd, vd, rd = (to_dev(x, torch.float32) for x in (q, k, v, r))
    bud, bvd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    o = torch.empty(qd.shape, device=dev())
    lse = torch.empty(1, 2, 4, device=dev())
    txl.txl_relattn_forward(qd, kd, vd, rd, bud, bvd, o, lse, M=4)
    dd = to_dev(dout, torch.float32)
    # an output aliasing an input
    with pytest.raises(txl.TxlError) as e:
        txl.txl_relattn_backward(qd, kd, vd, rd, bud, bvd, o, lse, dd, M=4, grads={"dq": dd})
    assert e.value.status == 3
    # two outputs overlapping each other
    buf = torch.empty(qd.shape, device=dev())
    with pytest.raises(txl.TxlError) as e:
        txl.txl_relattn_backward(qd, kd, vd, rd, bud, bvd, o, lse, dd, M=4, grads={"dk": buf, "dv": buf})
    assert e.value.status == 3
    assert txl.txl_get_device_status() == 0
