"""txl_relattn_forward captured into a CUDA graph, and the library's own
memory: the unit plan made without blocking the host, and its release.

A shape with more (batch, head, query-tile) units than SMs runs from a
host-made unit plan, made and uploaded on its first call.  Captured on a
first call, the forward must not allocate: it keeps the snake order, and the
graph's result equals the eager call's bit for bit (which CTA runs a unit
does not change the unit's arithmetic)."""

import time

import numpy as np
import pytest
import torch

from gpu_util import dev, prefilled_case, to_dev, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import transformer_xl_relative_txl_gb300 as lib  # fails loudly if not built

    torch.cuda.set_device(0)
    lib.txl_get_device_status()
    return lib


def test_forward_captured_on_first_call(txl):
    # The kernel's one-time set-up (its shared-memory attribute, the status
    # word) comes from an ordinary call on a small shape first.
    q0, k0, v0, r0, bu0, bv0 = prefilled_case(workload(1, 2, 64, 128, 64, "bf16"))
    o0 = torch.empty(q0.shape, device=dev(), dtype=torch.bfloat16)
    txl.txl_relattn_forward(*(to_dev(x, torch.bfloat16) for x in (q0, k0, v0, r0)), to_dev(bu0, torch.float32),
                            to_dev(bv0, torch.float32), o0, None, M=64)
    torch.cuda.synchronize()
    # 2 x 83 heads x 1 query tile = 166 units (> the SMs); a shape no other test uses
    B, H, D, W, M = 2, 83, 64, 128, 64
    assert B * H * ((W + 127) // 128) > torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v, r, bu, bv = prefilled_case(workload(B, H, D, W, M, "bf16"))
    qd, kd, vd, rd = (to_dev(x, torch.bfloat16) for x in (q, k, v, r))
    ud, vbd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    o_graph = torch.empty(qd.shape, device=dev(), dtype=torch.bfloat16)
    o_eager = torch.empty_like(o_graph)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o_graph, None, M=M)
    g.replay()
    torch.cuda.synchronize()
    txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o_eager, None, M=M)  # makes the plan
    torch.cuda.synchronize()
    assert txl.txl_get_device_status() == 0
    assert torch.equal(o_graph, o_eager)
    assert np.all(np.isfinite(o_eager.float().cpu().numpy()))
    # a second eager call sees the plan's upload complete; captured after
    # that, the forward runs from the plan and replays to the same result
    txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o_eager, None, M=M)
    torch.cuda.synchronize()
    o_graph2 = torch.empty_like(o_graph)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o_graph2, None, M=M)
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_graph2, o_eager)


def test_first_call_of_a_shape_does_not_block(txl):
    """The first call of a shape with more units than SMs makes its unit plan
    and uploads it on the caller's stream: the host returns while the stream
    is still busy with earlier work.  A call of the same shape on a second
    stream, made before that upload has run, waits for it on the device and
    gives the same result."""
    B, H, D, W, M = 3, 61, 64, 128, 64  # 183 units; a shape no other test uses
    assert B * H > torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v, r, bu, bv = prefilled_case(workload(B, H, D, W, M, "bf16"))
    qd, kd, vd, rd = (to_dev(x, torch.bfloat16) for x in (q, k, v, r))
    ud, vbd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    o1 = torch.empty(qd.shape, device=dev(), dtype=torch.bfloat16)
    o2 = torch.empty_like(o1)
    o3 = torch.empty_like(o1)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        torch.cuda._sleep(1_000_000_000)  # about half a second of spinning on s1
        t0 = time.perf_counter()
        txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o1, None, M=M)
        dt = time.perf_counter() - t0
        still_busy = not s1.query()
    with torch.cuda.stream(s2):
        txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o2, None, M=M)
    torch.cuda.synchronize()
    txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o3, None, M=M)
    torch.cuda.synchronize()
    assert txl.txl_get_device_status() == 0
    assert still_busy, "the call waited for the stream"
    assert dt < 0.2, f"the first call took {dt:.3f} s on the host"
    assert torch.equal(o1, o3) and torch.equal(o2, o3)


def test_release_cached(txl):
    """txl_release_cached frees the scratch and plans; later calls make them
    again and give the same results."""
    B, H, D, W, M = 4, 16, 64, 128, 1600  # split: per-stream scratch
    q, k, v, r, bu, bv = prefilled_case(workload(B, H, D, W, M, "bf16"))
    qd, kd, vd, rd = (to_dev(x, torch.bfloat16) for x in (q, k, v, r))
    ud, vbd = to_dev(bu, torch.float32), to_dev(bv, torch.float32)
    o1 = torch.empty(qd.shape, device=dev(), dtype=torch.bfloat16)
    o2 = torch.empty_like(o1)
    txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o1, None, M=M)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    txl.txl_release_cached()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 > free0
    txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o2, None, M=M)
    torch.cuda.synchronize()
    assert txl.txl_get_device_status() == 0
    assert torch.equal(o1, o2)
