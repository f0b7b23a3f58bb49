"""txl_relattn_forward_static: the forward for callers that cannot allocate.

Some callers must not call cudaMalloc: a host that hands all device memory to
its own pool at start-up, code running inside another library's allocator
callbacks, or a loop that must never stall on the allocator (cudaMalloc and
cudaFree can synchronise the device).  This entry point keeps the scratch of
split launches in a fixed device array inside the library instead.

It is compared with txl_relattn_forward on two calls in a row: the same
kernels run, so the outputs must agree bit for bit.  A launch with few units
splits its key ranges (the path that needs scratch), one with many units does
not.  The file is collected last, so a run that stops at its first failure
has run every other test before it.
"""

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


def _inputs(B, H, D, W, M):
    wl = workload(B, H, D, W, M)
    q, k, v, r, bu, bv = prefilled_case(wl)
    return [to_dev(x, torch.bfloat16) for x in (q, k, v, r)] + [to_dev(bu, torch.float32), to_dev(bv, torch.float32)]


@pytest.mark.parametrize("B,H,D,W,M", [
    (4, 16, 64, 128, 1600),  # 64 units: key ranges split across CTAs
    (2, 2, 64, 300, 200),    # 12 units, split
    (22, 8, 64, 512, 512),   # 704 units: no split
])
def test_static_matches_forward_twice(txl, B, H, D, W, M):
    q, k, v, r, bu, bv = _inputs(B, H, D, W, M)
    outs = []
    for fn in (txl.txl_relattn_forward, txl.txl_relattn_forward_static,
               txl.txl_relattn_forward, txl.txl_relattn_forward_static):
        o = torch.empty(q.shape, device=dev(), dtype=torch.bfloat16)
        lse = torch.empty(B, H, W, device=dev(), dtype=torch.float32)
        fn(q, k, v, r, bu, bv, o, lse, M=M)
        outs.append((o, lse))
    assert txl.txl_get_device_status() == 0
    ref_o, ref_l = outs[0]
    for o, lse in outs[1:]:
        assert torch.equal(o, ref_o)
        assert torch.equal(lse, ref_l)


def test_static_allocates_nothing(txl):
    """On a stream the library has not seen, the static entry point leaves the
    device's free memory unchanged; the allocating one, on another new
    stream, takes its split scratch (so the measurement can see it)."""
    B, H, D, W, M = 4, 16, 64, 128, 1600
    q, k, v, r, bu, bv = _inputs(B, H, D, W, M)
    o = torch.empty(q.shape, device=dev(), dtype=torch.bfloat16)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    free0, _ = torch.cuda.mem_get_info()
    with torch.cuda.stream(s1):
        txl.txl_relattn_forward_static(q, k, v, r, bu, bv, o, M=M)
        txl.txl_relattn_forward_static(q, k, v, r, bu, bv, o, M=M)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    with torch.cuda.stream(s2):
        txl.txl_relattn_forward(q, k, v, r, bu, bv, o, M=M)
    torch.cuda.synchronize()
    free2, _ = torch.cuda.mem_get_info()
    assert txl.txl_get_device_status() == 0
    assert free1 == free0
    assert free2 < free1


def test_static_split_captured_and_replayed(txl):
    """The static entry point captured into a CUDA graph on a split launch
    (64 units, key ranges split across CTAs) and replayed twice: each replay
    equals the eager forward bit for bit, so the merge counters the launch
    uses are back at zero after every replay.  One ordinary call comes first
    (it resolves the library's device symbols, which may load device code)."""
    B, H, D, W, M = 4, 16, 64, 128, 1600
    q, k, v, r, bu, bv = _inputs(B, H, D, W, M)
    o_ref = torch.empty(q.shape, device=dev(), dtype=torch.bfloat16)
    l_ref = torch.empty(B, H, W, device=dev(), dtype=torch.float32)
    txl.txl_relattn_forward(q, k, v, r, bu, bv, o_ref, l_ref, M=M)
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(l_ref)
    txl.txl_relattn_forward_static(q, k, v, r, bu, bv, o, lse, M=M)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        txl.txl_relattn_forward_static(q, k, v, r, bu, bv, o, lse, M=M)
    for _ in range(2):
        o.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert txl.txl_get_device_status() == 0
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, l_ref)
