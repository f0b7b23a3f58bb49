"""GPU parity of the ring-buffer memory: txl_relattn_forward_ring against
txl_relattn_forward on the same rows laid out linearly (bit for bit: the same
kernels run) and against the oracle, and txl_mem_ring_append against the
oracle's memory roll (bit-exact)."""

import numpy as np
import pytest
import torch

from oracle import txl_oracle as O
from synthetic import make_segments, project_r

from gpu_util import assert_bf16_close, dev, prefilled_case, to_dev, torch_dtype, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import transformer_xl_relative_txl_gb300 as lib  # fails loudly if not built

    torch.cuda.set_device(0)
    lib.txl_get_device_status()
    return lib


def _ring_of(x, M, cap, start, fill=99.0):
    """[B, cap, H, D] ring holding memory rows x[:, :M] from ring row start;
    the other rows hold `fill`, which must never be read."""
    ring = torch.full((x.shape[0], cap) + tuple(x.shape[2:]), fill, device=x.device, dtype=x.dtype)
    idx = (start + torch.arange(M, device=x.device)) % cap
    ring[:, idx] = x[:, :M]
    return ring


CASES = [
    # B, H, D, W, M, cap, start, dtype
    (2, 2, 64, 256, 512, 512, 128, "bf16"),    # read in place
    (2, 2, 64, 130, 512, 640, 576, "bf16"),    # read in place, the memory wraps
    (1, 2, 64, 128, 1600, 1664, 1216, "bf16"), # few units: split key ranges, wraps
    (2, 2, 64, 96, 320, 448, 37, "bf16"),      # start off the tile grid: linearised
    (2, 2, 64, 70, 100, 128, 64, "bf16"),      # M off the tile grid: linearised
    (1, 2, 128, 64, 192, 256, 200, "bf16"),    # D = 128: linearised
    (1, 2, 8, 4, 4, 6, 5, "f32"),              # fp32: linearised
    (2, 2, 64, 64, 0, 128, 0, "bf16"),         # no memory
]


@pytest.mark.parametrize("B,H,D,W,M,cap,start,dtype", CASES)
def test_ring_forward_equals_linear(txl, B, H, D, W, M, cap, start, dtype):
    q, k, v, r, bu, bv = prefilled_case(workload(B, H, D, W, M, dtype))
    td = torch_dtype(dtype)
    qd, kd, vd, rd = (to_dev(x, td) for x in (q, k, v, r))
    bud, bvd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    o_lin = torch.empty(qd.shape, device=dev(), dtype=td)
    lse_lin = torch.empty(B, H, W, device=dev())
    txl.txl_relattn_forward(qd, kd, vd, rd, bud, bvd, o_lin, lse_lin, M=M)
    k_ring, v_ring = _ring_of(kd, M, cap, start), _ring_of(vd, M, cap, start)
    o = torch.empty(qd.shape, device=dev(), dtype=td)
    lse = torch.empty(B, H, W, device=dev())
    txl.txl_relattn_forward_ring(qd, k_ring, v_ring, start, M, kd[:, M:].contiguous(), vd[:, M:].contiguous(), rd,
                                 bud, bvd, o, lse)
    assert txl.txl_get_device_status() == 0
    assert torch.equal(o, o_lin)
    assert torch.equal(lse, lse_lin)
    want, _ = O.relattn_forward(q, k, v, r, bu, bv, M)
    got = o.float().cpu().numpy()
    if dtype == "f32":
        assert np.abs(got - want).max() <= 1e-5
    else:
        assert_bf16_close(got, want, "ring forward")


@pytest.mark.parametrize("cap,start,m,w,dtype", [
    (512, 128, 512, 256, "bf16"),   # full ring: the oldest 256 rows are pushed out
    (640, 576, 300, 200, "bf16"),   # not full, writes wrap
    (64, 10, 30, 100, "f32"),       # more new rows than the ring holds
    (100, 0, 0, 37, "f32"),         # empty ring
    (128, 127, 128, 1, "bf16"),     # one row, full ring
    (96, 5, 20, 0, "bf16"),         # nothing to append
])
def test_ring_append_bit_exact(txl, cap, start, m, w, dtype):
    B, C = 3, 48
    rng = np.random.default_rng(cap * 7 + start + m + w)
    td = torch_dtype(dtype)
    ring = torch.from_numpy(rng.standard_normal((B, cap, C)).astype(np.float32)).to(dev()).to(td)
    big = torch.from_numpy(rng.standard_normal((B, w + 9, C)).astype(np.float32)).to(dev()).to(td)
    h = big[:, 4:4 + w]  # rows inside a larger buffer: batch stride (w + 9) * C
    idx = (start + np.arange(m)) % cap
    mem_lin = ring.cpu().float().numpy()[:, idx]
    s2, m2 = txl.txl_mem_ring_append(ring, start, m, h)
    assert txl.txl_get_device_status() == 0
    want = O.mem_update(mem_lin, h.cpu().float().numpy(), cap)
    assert m2 == want.shape[1]
    got = ring.cpu().float().numpy()[:, (s2 + np.arange(m2)) % cap]
    assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("B,H,D,W,M,cap,start,dtype", [
    (2, 2, 64, 128, 512, 640, 128, "bf16"),    # one launch: slots for the new rows, wraps
    (1, 2, 64, 128, 1600, 1728, 1664, "bf16"), # one launch with split key ranges
    (2, 2, 64, 64, 0, 128, 0, "bf16"),         # one launch, empty memory
    (2, 2, 64, 128, 512, 512, 128, "bf16"),    # full ring: read in place, then the appends
    (2, 2, 64, 100, 256, 512, 64, "bf16"),     # W off the tile grid
    (1, 2, 8, 4, 4, 6, 5, "f32"),              # fp32
])
def test_ring_append_call_equals_sequence(txl, B, H, D, W, M, cap, start, dtype):
    q, k, v, r, bu, bv = prefilled_case(workload(B, H, D, W, M, dtype))
    td = torch_dtype(dtype)
    qd, kd, vd, rd = (to_dev(x, td) for x in (q, k, v, r))
    bud, bvd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    ks, vs = kd[:, M:].contiguous(), vd[:, M:].contiguous()
    rings = [_ring_of(kd, M, cap, start), _ring_of(vd, M, cap, start)]
    ref = [x.clone() for x in rings]
    o1 = torch.empty(qd.shape, device=dev(), dtype=td)
    l1 = torch.empty(B, H, W, device=dev())
    txl.txl_relattn_forward_ring(qd, ref[0], ref[1], start, M, ks, vs, rd, bud, bvd, o1, l1)
    s1, m1 = txl.txl_mem_ring_append(ref[0], start, M, ks)
    txl.txl_mem_ring_append(ref[1], start, M, vs)
    o2 = torch.empty(qd.shape, device=dev(), dtype=td)
    l2 = torch.empty(B, H, W, device=dev())
    s2, m2 = txl.txl_relattn_forward_ring_append(qd, rings[0], rings[1], start, M, ks, vs, rd, bud, bvd, o2, l2)
    assert txl.txl_get_device_status() == 0
    assert (s1, m1) == (s2, m2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for got, want in zip(rings, ref):
        idx = (s2 + torch.arange(m2, device=dev())) % cap
        assert torch.equal(got[:, idx], want[:, idx])


def test_ring_recurrence_matches_oracle(txl):
    """Five segments through a ring of M = 128 rows (W = 64, bf16, D = 64):
    attention reads the ring in place, then the segment's k, v rows are
    appended; every segment's output against the oracle's recurrence."""
    B, H, D, W, M, S = 2, 2, 64, 64, 128, 5
    wl = workload(B, H, D, W, M)
    seg = make_segments(wl, n_segments=S)
    r = project_r(O.sinusoid_rel(M + W, wl.d_model), seg.W_r, H, D, "bf16")
    rd = to_dev(r, torch.bfloat16)
    bud, bvd = to_dev(seg.bias_u, torch.float32), to_dev(seg.bias_v, torch.float32)
    k_ring = torch.zeros(B, M, H, D, device=dev(), dtype=torch.bfloat16)
    v_ring = torch.zeros_like(k_ring)
    expect = O.run_segments([seg.seg("q", t) for t in range(S)], [seg.seg("k", t) for t in range(S)],
                            [seg.seg("v", t) for t in range(S)], r, seg.bias_u, seg.bias_v, M)
    start, m = 0, 0
    for t in range(S):
        qd = to_dev(seg.seg("q", t), torch.bfloat16)
        ks, vs = to_dev(seg.seg("k", t), torch.bfloat16), to_dev(seg.seg("v", t), torch.bfloat16)
        o = torch.empty(qd.shape, device=dev(), dtype=torch.float32)
        txl.txl_relattn_forward_ring(qd, k_ring, v_ring, start, m, ks, vs, rd, bud, bvd, o)
        eo, _, em = expect[t]
        assert em == m
        assert_bf16_close(o.cpu().numpy(), eo, f"segment {t}")
        s_k, m_k = txl.txl_mem_ring_append(k_ring, start, m, ks)
        s_v, m_v = txl.txl_mem_ring_append(v_ring, start, m, vs)
        assert (s_k, m_k) == (s_v, m_v)
        start, m = s_k, m_k
    assert txl.txl_get_device_status() == 0


def test_ring_rejects_bad_arguments(txl):
    q = torch.zeros(1, 4, 2, 64, device=dev(), dtype=torch.bfloat16)
    ring = torch.zeros(1, 8, 2, 64, device=dev(), dtype=torch.bfloat16)
    r = torch.zeros(12, 2, 64, device=dev(), dtype=torch.bfloat16)
    u = torch.zeros(2, 64, device=dev())
    o = torch.empty_like(q)
    with pytest.raises(txl.TxlError) as e:  # M > cap
        txl.txl_relattn_forward_ring(q, ring, ring, 0, 9, q, q, r, u, u, o)
    assert e.value.status == 1
    with pytest.raises(txl.TxlError) as e:  # start outside the ring
        txl.txl_relattn_forward_ring(q, ring, ring, 8, 4, q, q, r, u, u, o)
    assert e.value.status == 1
    with pytest.raises(txl.TxlError) as e:  # output over the ring
        txl.txl_relattn_forward_ring(q, ring, ring, 0, 4, q, q, r, u, u, ring[:, :4])
    assert e.value.status == 3
    with pytest.raises(txl.TxlError) as e:  # appending a ring to itself
        txl.txl_mem_ring_append(ring, 0, 4, ring[:, 2:4])
    assert e.value.status == 3
    assert txl.txl_get_device_status() == 0
