"""txl_relattn_forward captured into a CUDA graph.

A shape with more (batch, head, query-tile) units than SMs runs from a
host-made unit plan, made and uploaded on its first call.  Captured on a
first call, the forward must not allocate: it keeps the snake order, and the
graph's result equals the eager call's bit for bit (which CTA runs a unit
does not change the unit's arithmetic)."""

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
    # captured again, now with the plan: replays to the same result
    o_graph2 = torch.empty_like(o_graph)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        txl.txl_relattn_forward(qd, kd, vd, rd, ud, vbd, o_graph2, None, M=M)
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_graph2, o_eager)
