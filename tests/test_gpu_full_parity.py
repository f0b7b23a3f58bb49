"""Element-wise parity at the workloads' full sizes, every segment.

Each bf16 workload runs all of its segments from an empty memory through the
call the benchmark times -- ``txl_relattn_forward_roll`` (attention and the
memory roll in one launch, bf16 output, no lse), so the roll of segment tau
feeds segment tau+1 -- and every element of every segment's output is
compared with the oracle's segment recurrence (``run_segments``) on the same
inputs.  The same inputs then go through ``txl_relattn_forward`` with lse: its
output must equal the rolled call's bit for bit, and every lse element is
compared with the oracle's.  The memory each roll writes must equal the
oracle's roll bit for bit.

The long workload (W=128, M=1600, 16 segments) runs on the split path (64
units, fewer than the SMs) and also as a ring of M+W rows through
``txl_relattn_forward_ring_append``.  The memory-length sweep at W=128 (M =
0, 384, 1600, 3200 pre-filled rows) runs ``txl_relattn_forward`` alone, as
the benchmark times it.

"Transformer-XL, explained", method steps 2-5 (memory, keys and values over
[memory ; segment], the relative score); "Long-context transformers",
segment recurrence (the memory is the last M rows of [memory ; segment]).
Tolerances: bf16 inputs with fp32 accumulation, rel-L2 <= 5e-3 and
max |err| <= 2e-2 against the float64 oracle.
"""

import numpy as np
import pytest
import torch

from oracle import txl_oracle as O
from synthetic import WORKLOADS, make_prefilled, make_segments, project_r

from gpu_util import assert_bf16_close, dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import transformer_xl_relative_txl_gb300 as lib  # fails loudly if not built

    torch.cuda.set_device(0)
    lib.txl_get_device_status()
    return lib


def _workload_inputs(wl):
    seg = make_segments(wl)
    S = wl.segments
    r = project_r(O.sinusoid_rel(wl.M + wl.W, wl.d_model), seg.W_r, wl.H, wl.D, "bf16")
    qs = [seg.seg("q", t) for t in range(S)]
    ks = [seg.seg("k", t) for t in range(S)]
    vs = [seg.seg("v", t) for t in range(S)]
    return seg, r, qs, ks, vs


def _check_segment(what, o_gpu, lse_gpu, eo, el):
    assert_bf16_close(o_gpu, eo, f"{what}: o")
    assert_bf16_close(lse_gpu, el, f"{what}: lse")


@pytest.mark.parametrize("name", ["base", "large", "wide", "long"])
def test_every_segment_rolled(txl, name):
    wl = WORKLOADS[name]
    seg, r, qs, ks, vs = _workload_inputs(wl)
    expect = O.run_segments(qs, ks, vs, r, seg.bias_u, seg.bias_v, wl.M)
    B, W, H, D, C = wl.B, wl.W, wl.H, wl.D, wl.H * wl.D
    rd = to_dev(r, torch.bfloat16)
    ud, vd = to_dev(seg.bias_u, torch.float32), to_dev(seg.bias_v, torch.float32)
    bf = torch.bfloat16
    # segment 0: an empty memory; each roll writes the head of the next buffer
    m_tau = 0
    kcur = torch.empty(B, W, H, D, device=dev(), dtype=bf)
    vcur = torch.empty(B, W, H, D, device=dev(), dtype=bf)
    mem_k = np.zeros((B, 0, C), np.float32)
    mem_v = np.zeros((B, 0, C), np.float32)
    for tau in range(wl.segments):
        kcur[:, m_tau:] = to_dev(ks[tau], bf)
        vcur[:, m_tau:] = to_dev(vs[tau], bf)
        q = to_dev(qs[tau], bf)
        keep = min(wl.M, m_tau + W)
        knext = torch.empty(B, keep + W, H, D, device=dev(), dtype=bf)
        vnext = torch.empty(B, keep + W, H, D, device=dev(), dtype=bf)
        o = torch.empty(q.shape, device=dev(), dtype=bf)
        got_keep = txl.txl_relattn_forward_roll(q, kcur, vcur, rd, ud, vd, o, knext[:, :keep], vnext[:, :keep],
                                                wl.M, M=m_tau)
        o2 = torch.empty(q.shape, device=dev(), dtype=bf)
        lse = torch.empty(B, H, W, device=dev(), dtype=torch.float32)
        txl.txl_relattn_forward(q, kcur, vcur, rd, ud, vd, o2, lse, M=m_tau)
        assert txl.txl_get_device_status() == 0
        eo, el, em = expect[tau]
        assert em == m_tau and got_keep == keep
        assert torch.equal(o, o2), f"{name} segment {tau}: the rolled call's output differs"
        _check_segment(f"{name} segment {tau} (M_tau={m_tau})", o.float().cpu().numpy(), lse.cpu().numpy(), eo, el)
        # the roll: exactly the oracle's memory for the next segment
        mem_k = O.mem_update(mem_k, ks[tau].reshape(B, W, C), wl.M)
        mem_v = O.mem_update(mem_v, vs[tau].reshape(B, W, C), wl.M)
        assert np.array_equal(knext[:, :keep].float().cpu().numpy().reshape(B, keep, C), mem_k), f"k memory {tau}"
        assert np.array_equal(vnext[:, :keep].float().cpu().numpy().reshape(B, keep, C), mem_v), f"v memory {tau}"
        kcur, vcur, m_tau = knext, vnext, keep
    assert m_tau == wl.M


def test_every_segment_ring_long(txl):
    """The long workload's 16 segments with the memory as a ring of M+W rows
    (txl_relattn_forward_ring_append, as the benchmark's ring step runs it)."""
    wl = WORKLOADS["long"]
    seg, r, qs, ks, vs = _workload_inputs(wl)
    expect = O.run_segments(qs, ks, vs, r, seg.bias_u, seg.bias_v, wl.M)
    B, W, H, D = wl.B, wl.W, wl.H, wl.D
    cap = wl.M + W
    bf = torch.bfloat16
    rd = to_dev(r, bf)
    ud, vd = to_dev(seg.bias_u, torch.float32), to_dev(seg.bias_v, torch.float32)
    k_ring = torch.zeros(B, cap, H, D, device=dev(), dtype=bf)
    v_ring = torch.zeros(B, cap, H, D, device=dev(), dtype=bf)
    start, m_tau = 0, 0
    for tau in range(wl.segments):
        q, k_seg, v_seg = to_dev(qs[tau], bf), to_dev(ks[tau], bf), to_dev(vs[tau], bf)
        o = torch.empty(q.shape, device=dev(), dtype=bf)
        lse = torch.empty(B, H, W, device=dev(), dtype=torch.float32)
        s2, m2 = txl.txl_relattn_forward_ring_append(q, k_ring, v_ring, start, m_tau, k_seg, v_seg, rd, ud, vd, o,
                                                     lse)
        assert txl.txl_get_device_status() == 0
        eo, el, em = expect[tau]
        assert em == m_tau
        _check_segment(f"ring segment {tau} (M_tau={m_tau})", o.float().cpu().numpy(), lse.cpu().numpy(), eo, el)
        keep = min(wl.M, m2)  # the next memory: the last M rows the ring holds
        start, m_tau = (s2 + m2 - keep) % cap, keep
    assert m_tau == wl.M


@pytest.mark.parametrize("M", [0, 384, 1600, 3200])
def test_memory_length_sweep(txl, M):
    base = WORKLOADS["long"]
    wl = base.__class__(base.name, base.cfg_id, base.B, base.H, base.D, base.d_model, base.W, M, 1, "bf16")
    q, k, v, s = make_prefilled(wl, M)
    r = project_r(O.sinusoid_rel(M + wl.W, wl.d_model), s.W_r, wl.H, wl.D, "bf16")
    bf = torch.bfloat16
    qd, kd, vd, rd = (to_dev(x, bf) for x in (q, k, v, r))
    ud, vbd = to_dev(s.bias_u, torch.float32), to_dev(s.bias_v, torch.float32)
    o = torch.empty(qd.shape, device=dev(), dtype=bf)
    txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o, M=M)
    o2 = torch.empty(qd.shape, device=dev(), dtype=bf)
    lse = torch.empty(wl.B, wl.H, wl.W, device=dev(), dtype=torch.float32)
    txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o2, lse, M=M)
    assert txl.txl_get_device_status() == 0
    assert torch.equal(o, o2)
    eo, el = O.relattn_forward(q, k, v, r, s.bias_u, s.bias_v, M)
    _check_segment(f"M={M}", o.float().cpu().numpy(), lse.cpu().numpy(), eo, el)
