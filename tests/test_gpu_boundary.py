"""The C ABI's error contract on a GPU: invalid arguments are rejected on the
host with the documented codes and nothing is launched; empty calls succeed;
a bounded wait that runs out inside the tensor-core kernel is reported
through the device status word and leaves the context usable."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import txl_oracle as O

from gpu_util import assert_bf16_close, dev, prefilled_case, run_forward, workload

pytestmark = pytest.mark.gpu

OK, INVALID, UNSUPPORTED, ALIAS, CUDA, TIMEOUT = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import transformer_xl_relative_txl_gb300 as m

    torch.cuda.set_device(0)
    return m


def _bufs(B=1, W=8, M=8, H=2, D=64, dtype=torch.bfloat16, n_r=None):
    n_r = M + W if n_r is None else n_r
    q = torch.randn(B, W, H, D, device=dev()).to(dtype)
    k = torch.randn(B, M + W, H, D, device=dev()).to(dtype)
    v = torch.randn(B, M + W, H, D, device=dev()).to(dtype)
    r = torch.randn(n_r, H, D, device=dev()).to(dtype)
    u = torch.zeros(H, D, device=dev())
    vb = torch.zeros(H, D, device=dev())
    o = torch.empty(B, W, H, D, device=dev(), dtype=dtype)
    return q, k, v, r, u, vb, o


def _fwd(txl, q, k, v, r, u, vb, o, lse=None, B=1, W=8, M=8, H=2, D=64, n_r=None, dt=1, odt=1, scale=0.125):
    n_r = M + W if n_r is None else n_r
    p = lambda t: None if t is None else t.data_ptr()
    return txl.lib.txl_relattn_forward(p(q), p(k), p(v), p(r), p(u), p(vb), p(o), p(lse), B, W, M, H, D, n_r,
                                       scale, dt, odt, None)


def test_forward_argument_errors(txl):
    q, k, v, r, u, vb, o = _bufs()
    o.fill_(3.0)
    sentinel = o.clone()
    assert _fwd(txl, q, k, v, r, u, vb, o) == OK
    torch.cuda.synchronize()
    assert not torch.equal(o, sentinel)
    o.copy_(sentinel)
    assert _fwd(txl, None, k, v, r, u, vb, o) == INVALID
    assert _fwd(txl, q, k, v, r, None, vb, o) == INVALID
    assert _fwd(txl, q, k, v, r, u, vb, o, n_r=15) == INVALID           # n_r < M + W
    assert _fwd(txl, q, k, v, r, u, vb, o, M=-1) == INVALID
    assert _fwd(txl, q, k, v, r, u, vb, o, H=0) == INVALID
    assert _fwd(txl, q, k, v, r, u, vb, o, dt=7) == INVALID
    assert _fwd(txl, q, k, v, r, u, vb, o, scale=float("nan")) == INVALID
    assert _fwd(txl, q, k, v, r, u, vb, o, D=32) == UNSUPPORTED         # bf16 path: D in {64, 128}
    qq = torch.empty(q.numel() * 2 + 8, device=dev(), dtype=torch.bfloat16)
    assert txl.lib.txl_relattn_forward(qq.data_ptr() + 2, k.data_ptr(), v.data_ptr(), r.data_ptr(),
                                       u.data_ptr(), vb.data_ptr(), o.data_ptr(), None, 1, 8, 8, 2, 64, 16,
                                       0.125, 1, 1, None) == INVALID     # misaligned q
    assert _fwd(txl, q, k, v, r, u, vb, q) == ALIAS                      # o overlaps q
    assert txl.lib.txl_relattn_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(), u.data_ptr(),
                                       vb.data_ptr(), k.data_ptr() + 1024, None, 1, 8, 8, 2, 64, 16, 0.125,
                                       1, 1, None) == ALIAS              # o inside k
    lse = torch.empty(1, 2, 8, device=dev())
    assert _fwd(txl, q, k, v, r, u, vb, o, lse=lse) == OK
    torch.cuda.synchronize()
    o.copy_(sentinel)
    assert txl.lib.txl_relattn_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(), u.data_ptr(),
                                       vb.data_ptr(), o.data_ptr(), o.data_ptr() + 64, 1, 8, 8, 2, 64, 16,
                                       0.125, 1, 1, None) == ALIAS  # lse inside o
    # fp32 path limits
    qf, kf, vf, rf, uf, vbf, of = _bufs(dtype=torch.float32, D=300)
    assert _fwd(txl, qf, kf, vf, rf, uf, vbf, of, D=300, dt=0, odt=0) == UNSUPPORTED
    qf, kf, vf, rf, uf, vbf, of = _bufs(dtype=torch.float32)
    assert _fwd(txl, qf, kf, vf, rf, uf, vbf, of, dt=0, odt=1) == UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.equal(o, sentinel)  # rejected calls launched nothing
    assert txl.txl_get_device_status() == OK


def test_forward_empty_calls(txl):
    assert txl.lib.txl_relattn_forward(None, None, None, None, None, None, None, None, 0, 8, 8, 2, 64, 16,
                                       0.125, 1, 1, None) == OK
    assert txl.lib.txl_relattn_forward(None, None, None, None, None, None, None, None, 3, 0, 8, 2, 64, 8,
                                       0.125, 1, 1, None) == OK


def test_mem_update_errors(txl):
    buf = torch.zeros(2, 12, 16, device=dev())
    out = torch.zeros(2, 12, 16, device=dev())
    m_out = ctypes.c_int(-1)
    P = lambda t, off=0: t.data_ptr() + off * 4
    lib = txl.lib
    # valid: keep last 8 of [mem(4) ; h(8)]
    assert lib.txl_mem_update(P(buf), 4, P(buf, 4 * 16), 8, P(out), 8, 2, 16, 12 * 16, 12 * 16, 12 * 16,
                              ctypes.byref(m_out), 0, None) == OK
    assert m_out.value == 8
    # in-place roll: output overlaps the rows it reads
    assert lib.txl_mem_update(P(buf), 4, P(buf, 4 * 16), 8, P(buf), 8, 2, 16, 12 * 16, 12 * 16, 12 * 16,
                              None, 0, None) == ALIAS
    assert lib.txl_mem_update(None, 4, P(buf), 2, P(out), 6, 2, 16, 192, 192, 192, None, 0, None) == INVALID
    assert lib.txl_mem_update(P(buf), 4, P(buf), 2, None, 6, 2, 16, 192, 192, 192, None, 0, None) == INVALID
    assert lib.txl_mem_update(P(buf), -1, P(buf), 2, P(out), 6, 2, 16, 192, 192, 192, None, 0, None) == INVALID
    assert lib.txl_mem_update(P(buf), 4, P(buf, 64), 8, P(out), 8, 2, 16, 10, 192, 192, None, 0, None) == INVALID
    # memory limit 0 and empty batches are valid no-ops
    assert lib.txl_mem_update(P(buf), 4, P(buf, 64), 8, P(out), 0, 2, 16, 192, 192, 192,
                              ctypes.byref(m_out), 0, None) == OK and m_out.value == 0
    assert lib.txl_mem_update(None, 4, None, 8, None, 8, 0, 16, 0, 0, 0, None, 0, None) == OK


def test_sinusoid_errors(txl):
    R = torch.empty(8, 16, device=dev())
    assert txl.lib.txl_sinusoid_rel(R.data_ptr(), 8, 15, 0, None) == INVALID
    assert txl.lib.txl_sinusoid_rel(None, 8, 16, 0, None) == INVALID
    assert txl.lib.txl_sinusoid_rel(R.data_ptr(), -1, 16, 0, None) == INVALID
    assert txl.lib.txl_sinusoid_rel(None, 0, 16, 0, None) == OK


def test_status_strings(txl):
    assert txl.txl_status_string(TIMEOUT) == "TXL_ERR_DEVICE_TIMEOUT"
    assert txl.txl_version() == 160


def test_bounded_wait_reports_timeout_and_context_survives(txl):
    """The loader stops after the first key tile (test hook), so the MMA and
    softmax roles' bounded waits run out (50 ms); the kernel unwinds, the
    status word reports the timeout, and the next call computes correctly."""
    wl = workload(1, 2, 64, 256, 256)  # 4 key tiles per query tile
    q, k, v, r, bu, bv = prefilled_case(wl)
    assert txl.txl_debug_set_wait_limit_ns(50_000_000) == OK
    try:
        assert txl.txl_debug_inject_stall(True) == OK
        td = lambda a, t=torch.bfloat16: torch.from_numpy(np.ascontiguousarray(a)).to(dev()).to(t)
        o = torch.empty(q.shape, device=dev(), dtype=torch.float32)
        txl.txl_relattn_forward(td(q), td(k), td(v), td(r), td(bu, torch.float32), td(bv, torch.float32), o,
                                None, M=wl.M)
        assert txl.txl_get_device_status() == TIMEOUT
        assert txl.txl_get_device_status() == OK  # the word was cleared
    finally:
        txl.txl_debug_inject_stall(False)
        txl.txl_debug_set_wait_limit_ns(2_000_000_000)
    o2, _ = run_forward(q, k, v, r, bu, bv, wl.M, "bf16", o_dtype="f32")
    eo, _ = O.relattn_forward(q, k, v, r, bu, bv, wl.M)
    assert_bf16_close(o2, eo)
