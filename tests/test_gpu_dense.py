"""txl_dense, the layer's dense products on this library's tensor-core GEMM,
against float64 products of the same bf16 operands.

The kernel accumulates in fp32 and rounds once to bf16, so each element may
differ from the exact value by half a bf16 ulp (2^-9 relative) plus the fp32
accumulation error; the bound below allows 2^-8 relative plus 1e-3 of the
tensor's largest value.  Shapes cover ragged m, n and k (the tiles' zero
fill and clipped stores), the column-tile widths the launcher picks (128
and 256) and each of 64, 128 and 256 forced by the test hook, a batch of three packed weight matrices, the bias and the ReLU,
and the base layer's two feed-forward shapes.
"""

import numpy as np
import pytest
import torch

from synthetic import round_bf16

from gpu_util import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import transformer_xl_relative_txl_gb300 as lib  # fails loudly if not built

    torch.cuda.set_device(0)
    lib.txl_get_device_status()
    return lib


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev()).to(torch.bfloat16)


@pytest.mark.parametrize("m,n,k,batch,bias,relu", [
    (300, 200, 136, 1, True, True),       # every dimension ragged; 128-column tiles
    (5120, 512, 512, 1, True, False),     # 256-column tiles (one wave of 80 tiles)
    (1000, 72, 64, 3, False, False),      # a batch of three weight matrices, n below one tile
    (1, 8, 8, 1, True, True),             # a single row
    (11264, 2048, 512, 1, True, True),    # base layer, W_1 with b_1 and the ReLU
    (11264, 512, 2048, 1, True, False),   # base layer, W_2 with b_2
    (11264, 512, 512, 3, False, False),   # base layer, packed W_q / W_k / W_v
])
def test_dense_matches_float64(txl, m, n, k, batch, bias, relu):
    rng = np.random.default_rng(m * 7 + n * 3 + k + batch)
    x = round_bf16(rng.standard_normal((m, k)).astype(np.float32))
    W = round_bf16((rng.standard_normal((batch, k, n)) * 0.05).astype(np.float32))
    b = (rng.standard_normal(n) * 0.1).astype(np.float32) if bias else None
    y = torch.empty(batch, m, n, device=dev(), dtype=torch.bfloat16)
    txl.txl_dense(_bf(x), _bf(W), y, bias=torch.from_numpy(b).to(dev()) if bias else None, relu=relu)
    assert txl.txl_get_device_status() == 0
    want = np.einsum("mk,zkn->zmn", x.astype(np.float64), W.astype(np.float64))
    if bias:
        want = want + b.astype(np.float64)
    if relu:
        want = np.maximum(want, 0.0)
    got = y.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    bound = 2.0 ** -8 * np.abs(want) + 1e-3 * np.abs(want).max()
    assert np.all(err <= bound), f"max err {err.max():.3e}, worst excess {(err - bound).max():.3e}"


@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("m,n,k,bias,relu", [
    (300, 200, 264, True, True),        # ragged in every dimension, k over two 128-deep stages
    (11264, 512, 2048, True, False),    # base layer, W_2 with b_2
])
def test_dense_each_tile_width(txl, bn, m, n, k, bias, relu):
    """Every column-tile width of the GEMM, forced through the test hook."""
    rng = np.random.default_rng(m + n + k + bn)
    x = round_bf16(rng.standard_normal((m, k)).astype(np.float32))
    W = round_bf16((rng.standard_normal((1, k, n)) * 0.05).astype(np.float32))
    b = (rng.standard_normal(n) * 0.1).astype(np.float32) if bias else None
    y = torch.empty(1, m, n, device=dev(), dtype=torch.bfloat16)
    txl.txl_debug_force_dense_tile_n(bn)
    try:
        txl.txl_dense(_bf(x), _bf(W), y, bias=torch.from_numpy(b).to(dev()) if bias else None, relu=relu)
    finally:
        txl.txl_debug_force_dense_tile_n(0)
    assert txl.txl_get_device_status() == 0
    want = np.einsum("mk,zkn->zmn", x.astype(np.float64), W.astype(np.float64))
    if bias:
        want = want + b.astype(np.float64)
    if relu:
        want = np.maximum(want, 0.0)
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - want)
    bound = 2.0 ** -8 * np.abs(want) + 1e-3 * np.abs(want).max()
    assert np.all(err <= bound), f"max err {err.max():.3e}, worst excess {(err - bound).max():.3e}"


def test_dense_deterministic_and_errors(txl):
    rng = np.random.default_rng(5)
    x = _bf(round_bf16(rng.standard_normal((257, 64)).astype(np.float32)))
    W = _bf(round_bf16(rng.standard_normal((64, 96)).astype(np.float32)))
    y1 = torch.empty(257, 96, device=dev(), dtype=torch.bfloat16)
    y2 = torch.empty_like(y1)
    txl.txl_dense(x, W, y1)
    txl.txl_dense(x, W, y2)
    assert torch.equal(y1, y2)
    txl.txl_dense(x[:0], W, y1[:0])  # m = 0: an empty call
    with pytest.raises(txl.TxlError) as e:  # n not a multiple of 8
        txl.txl_dense(x, W[:, :90].contiguous(), torch.empty(257, 90, device=dev(), dtype=torch.bfloat16))
    assert e.value.status == 2
    with pytest.raises(txl.TxlError) as e:  # the output over the input
        big = torch.zeros(257 * 96 + 257 * 64, device=dev(), dtype=torch.bfloat16)
        txl.txl_dense(big[:257 * 64].view(257, 64), W, big[:257 * 96].view(257, 96))
    assert e.value.status == 3
    assert txl.txl_get_device_status() == 0
