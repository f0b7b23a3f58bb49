"""GPU parity: every kernel of the path against the float64 oracle on the same
seeded inputs, through the C ABI (via the thin binding)."""


import numpy as np
import pytest
import torch

from oracle import txl_oracle as O
from synthetic import WORKLOADS, make_prefilled, make_segments, project_r

from gpu_util import (BF16_ATOL, F32_ATOL, assert_bf16_close, dev, prefilled_case, run_forward, to_dev,
                      torch_dtype, workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import transformer_xl_relative_txl_gb300 as txl  # fails loudly if not built

    torch.cuda.set_device(0)
    txl.txl_get_device_status()
    yield txl


# ----------------------------------------------------------------------------
# K4: sinusoid table
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n,dim", [(8, 16), (1, 2), (1024, 512), (1536, 1024), (1728, 1024), (3328, 1024),
                                   (777, 6)])
def test_sinusoid_f32(_lib, n, dim):
    R = torch.empty(n, dim, device=dev())
    _lib.txl_sinusoid_rel(R)
    err = np.abs(R.cpu().numpy().astype(np.float64) - O.sinusoid_rel(n, dim)).max()
    assert err <= 1e-6, err


def test_sinusoid_bf16(_lib):
    n, dim = 1728, 1024
    R = torch.empty(n, dim, device=dev(), dtype=torch.bfloat16)
    _lib.txl_sinusoid_rel(R)
    want = O.sinusoid_rel(n, dim)
    got = R.float().cpu().numpy().astype(np.float64)
    # within half a bf16 ulp of the exact value (plus the fp32 error)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 1e-30))) - 7)
    assert np.all(np.abs(got - want) <= 0.5 * ulp + 1e-6)


# ----------------------------------------------------------------------------
# K3: memory roll (bit-exact)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("m_prev,w,m,C", [(0, 4, 4, 16), (4, 4, 4, 16), (512, 512, 512, 512),
                                          (1600, 128, 1600, 1024), (128, 128, 1600, 1024),
                                          (7, 3, 5, 33), (3, 7, 5, 9), (5, 2, 0, 8), (0, 0, 4, 8),
                                          (10, 6, 12, 1), (37, 5, 40, 1000)])
def test_mem_roll_bit_exact(_lib, dtype, m_prev, w, m, C):
    B = 3
    rng = np.random.default_rng(m_prev * 131 + w * 7 + m + C)
    td = torch_dtype(dtype)
    pad_m, pad_h, pad_o = 2, 1, 3  # extra rows: batch strides differ from the row counts
    mem = torch.from_numpy(rng.standard_normal((B, m_prev + pad_m, C)).astype(np.float32)).to(dev()).to(td)
    h = torch.from_numpy(rng.standard_normal((B, w + pad_h, C)).astype(np.float32)).to(dev()).to(td)
    keep = min(m, m_prev + w)
    out = torch.full((B, keep + pad_o, C), -7.0, device=dev(), dtype=td)
    got_m = _lib.txl_mem_update(mem[:, :m_prev], h[:, :w], out, m)
    assert got_m == keep
    want = O.mem_update(mem[:, :m_prev].cpu().float().numpy(), h[:, :w].cpu().float().numpy(), m)
    got = out[:, :keep].cpu().float().numpy()
    assert got.shape == want.shape
    assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32))
    assert torch.all(out[:, keep:] == -7.0)  # nothing written past m'


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("m_prev,w,m,C", [(512, 512, 512, 512), (37, 5, 40, 1000), (7, 3, 5, 33), (0, 6, 4, 8)])
def test_mem_update_kv_bit_exact(_lib, dtype, m_prev, w, m, C):
    """Keys and values rolled in one call: each equals its own txl_mem_update
    and the oracle's roll, bit for bit."""
    B = 3
    rng = np.random.default_rng(m_prev * 17 + w * 5 + m + C)
    td = torch_dtype(dtype)
    t = lambda rows: torch.from_numpy(rng.standard_normal((B, rows, C)).astype(np.float32)).to(dev()).to(td)
    km, vm, kh, vh = t(m_prev + 2), t(m_prev + 2), t(w + 1), t(w + 1)
    keep = min(m, m_prev + w)
    ko = torch.full((B, keep + 3, C), -7.0, device=dev(), dtype=td)
    vo = torch.full((B, keep + 3, C), -7.0, device=dev(), dtype=td)
    ks = torch.empty_like(ko)
    vs = torch.empty_like(vo)
    got_m = _lib.txl_mem_update_kv(km[:, :m_prev], vm[:, :m_prev], kh[:, :w], vh[:, :w], ko, vo, m)
    _lib.txl_mem_update(km[:, :m_prev], kh[:, :w], ks, m)
    _lib.txl_mem_update(vm[:, :m_prev], vh[:, :w], vs, m)
    assert got_m == keep
    assert _lib.txl_get_device_status() == 0
    for o, sep, mem, h in ((ko, ks, km, kh), (vo, vs, vm, vh)):
        assert torch.equal(o[:, :keep], sep[:, :keep])
        want = O.mem_update(mem[:, :m_prev].cpu().float().numpy(), h[:, :w].cpu().float().numpy(), m)
        assert np.array_equal(o[:, :keep].cpu().float().numpy(), want.astype(np.float32))
        assert torch.all(o[:, keep:] == -7.0)


def test_mem_update_kv_rejects_overlap(_lib):
    B, C = 2, 64
    buf = torch.zeros(B, 40, C, device=dev(), dtype=torch.bfloat16)
    h = torch.zeros(B, 8, C, device=dev(), dtype=torch.bfloat16)
    mem = torch.zeros(B, 8, C, device=dev(), dtype=torch.bfloat16)
    with pytest.raises(_lib.TxlError, match="ALIAS"):  # the two outputs overlap
        _lib.txl_mem_update_kv(mem, mem, h, h, buf[:, :10], buf[:, 5:15], 8)
    other = torch.zeros(B, 40, C, device=dev(), dtype=torch.bfloat16)
    with pytest.raises(_lib.TxlError, match="ALIAS"):  # k's output is v's input
        _lib.txl_mem_update_kv(other[:, :8], other[:, 10:18], h, h, other[:, 10:22], buf[:, :12], 12)


# ----------------------------------------------------------------------------
# K2: exact fp32 path
# ----------------------------------------------------------------------------

def test_tiny_fp32_three_segments(_lib):
    """The pages' toy: seg_len 4, dim 16, 2 heads, three segments carrying
    memory (first one empty), roll and attention on the GPU."""
    wl = WORKLOADS["tiny"]
    seg = make_segments(wl)
    R = O.sinusoid_rel(wl.M + wl.W, wl.d_model)
    r = project_r(R, seg.W_r, wl.H, wl.D, wl.dtype)
    expect = O.run_segments([seg.seg("q", t) for t in range(3)], [seg.seg("k", t) for t in range(3)],
                            [seg.seg("v", t) for t in range(3)], r, seg.bias_u, seg.bias_v, wl.M)
    L, C = wl.M + wl.W, wl.H * wl.D
    kb = [torch.zeros(wl.B, L, C, device=dev()) for _ in range(2)]
    vb = [torch.zeros(wl.B, L, C, device=dev()) for _ in range(2)]
    m_tau = 0
    rd, ud, vd = to_dev(r, torch.float32), to_dev(seg.bias_u, torch.float32), to_dev(seg.bias_v, torch.float32)
    for tau in range(3):
        cur = tau % 2
        kb[cur][:, m_tau:m_tau + wl.W] = to_dev(seg.seg("k", tau), torch.float32).view(wl.B, wl.W, C)
        vb[cur][:, m_tau:m_tau + wl.W] = to_dev(seg.seg("v", tau), torch.float32).view(wl.B, wl.W, C)
        q = to_dev(seg.seg("q", tau), torch.float32)
        o = torch.empty_like(q)
        lse = torch.empty(wl.B, wl.H, wl.W, device=dev())
        k = kb[cur][:, :m_tau + wl.W].reshape(wl.B, m_tau + wl.W, wl.H, wl.D).contiguous()
        v = vb[cur][:, :m_tau + wl.W].reshape(wl.B, m_tau + wl.W, wl.H, wl.D).contiguous()
        _lib.txl_relattn_forward(q, k, v, rd, ud, vd, o, lse, M=m_tau)
        eo, el, em = expect[tau]
        assert em == m_tau == [0, 4, 4][tau]
        assert np.abs(o.cpu().numpy() - eo).max() <= F32_ATOL
        assert np.abs(lse.cpu().numpy() - el).max() <= F32_ATOL
        nxt = 1 - cur
        m_new = _lib.txl_mem_update(kb[cur][:, :m_tau], kb[cur][:, m_tau:m_tau + wl.W], kb[nxt], wl.M)
        _lib.txl_mem_update(vb[cur][:, :m_tau], vb[cur][:, m_tau:m_tau + wl.W], vb[nxt], wl.M)
        m_tau = m_new
    assert _lib.txl_get_device_status() == 0


@pytest.mark.parametrize("B,H,D,W,M", [(1, 2, 8, 4, 4), (2, 3, 16, 37, 50), (1, 1, 1, 5, 0), (2, 2, 64, 130, 7),
                                       (1, 2, 256, 9, 300), (1, 1, 33, 1, 0)])
def test_fp32_shapes(B, H, D, W, M):
    wl = workload(B, H, D, W, M, "f32")
    q, k, v, r, bu, bv = prefilled_case(wl, n_r_extra=3)
    o, lse = run_forward(q, k, v, r, bu, bv, M, "f32")
    eo, el = O.relattn_forward(q, k, v, r, bu, bv, M)
    assert np.abs(o - eo).max() <= F32_ATOL
    assert np.abs(lse - el).max() <= F32_ATOL


# ----------------------------------------------------------------------------
# K1: bf16 tensor-core path, several tiles and ragged tails
# ----------------------------------------------------------------------------

SHAPES = [
    (1, 1, 64, 1, 0),      # a single key
    (1, 2, 64, 128, 0),    # one full tile, empty memory
    (2, 2, 64, 200, 150),  # ragged query tile, memory not a tile multiple
    (1, 2, 64, 300, 384),  # three query tiles
    (2, 1, 64, 64, 1000),  # short segment, long memory
    (1, 2, 128, 200, 150),
    (2, 1, 128, 256, 128),
    (1, 1, 128, 129, 1),
    # more units than SMs, so every CTA runs several: one-step units (the
    # loader's queued V tiles of a unit two back go out before the next raw q
    # load) and two-step units.  The units come from the batch: H stays at 8
    # (d_model 512), so the value entries keep the workloads' size.
    (64, 8, 64, 64, 0),
    (40, 8, 64, 100, 20),
]


@pytest.mark.parametrize("B,H,D,W,M", SHAPES)
@pytest.mark.parametrize("o_dtype", ["bf16", "f32"])
def test_bf16_shapes(B, H, D, W, M, o_dtype):
    wl = workload(B, H, D, W, M)
    q, k, v, r, bu, bv = prefilled_case(wl, n_r_extra=5)
    o, lse = run_forward(q, k, v, r, bu, bv, M, "bf16", o_dtype=o_dtype)
    eo, el = O.relattn_forward(q, k, v, r, bu, bv, M)
    assert_bf16_close(o, eo, f"o {B,H,D,W,M}")
    assert np.abs(lse - el).max() <= BF16_ATOL


def test_bf16_scale_and_biases_matter():
    """A scale other than 1/sqrt(D) and large biases: catches a dropped term."""
    wl = workload(1, 2, 64, 160, 96)
    q, k, v, r, bu, bv = prefilled_case(wl)
    bu = bu * 40
    bv = bv * 40
    o, _ = run_forward(q, k, v, r, bu, bv, wl.M, "bf16", o_dtype="f32", scale=0.2)
    eo, _ = O.relattn_forward(q, k, v, r, bu, bv, wl.M, scale=0.2)
    assert_bf16_close(o, eo)


def test_bf16_segments_with_roll(_lib):
    """Four consecutive segments from empty memory (M_tau = 0, 256, 384, 384),
    roll and attention on the GPU, against the oracle's recurrence."""
    wl = workload(2, 2, 64, 256, 384)
    wl = wl.__class__(wl.name, wl.cfg_id, wl.B, wl.H, wl.D, wl.d_model, wl.W, wl.M, 4, "bf16")
    seg = make_segments(wl)
    r = project_r(O.sinusoid_rel(wl.M + wl.W, wl.d_model), seg.W_r, wl.H, wl.D, "bf16")
    expect = O.run_segments([seg.seg("q", t) for t in range(4)], [seg.seg("k", t) for t in range(4)],
                            [seg.seg("v", t) for t in range(4)], r, seg.bias_u, seg.bias_v, wl.M)
    L, C = wl.M + wl.W, wl.H * wl.D
    bufs = [[torch.zeros(wl.B, L, C, device=dev(), dtype=torch.bfloat16) for _ in range(2)] for _ in range(2)]
    rd = to_dev(r, torch.bfloat16)
    ud, vd = to_dev(seg.bias_u, torch.float32), to_dev(seg.bias_v, torch.float32)
    m_tau = 0
    for tau in range(4):
        cur = tau % 2
        kb, vb = bufs[cur]
        kb[:, m_tau:m_tau + wl.W] = to_dev(seg.seg("k", tau), torch.bfloat16).view(wl.B, wl.W, C)
        vb[:, m_tau:m_tau + wl.W] = to_dev(seg.seg("v", tau), torch.bfloat16).view(wl.B, wl.W, C)
        q = to_dev(seg.seg("q", tau), torch.bfloat16)
        o = torch.empty(q.shape, device=dev(), dtype=torch.float32)
        k = kb[:, :m_tau + wl.W].reshape(wl.B, m_tau + wl.W, wl.H, wl.D).contiguous()
        v = vb[:, :m_tau + wl.W].reshape(wl.B, m_tau + wl.W, wl.H, wl.D).contiguous()
        _lib.txl_relattn_forward(q, k, v, rd, ud, vd, o, None, M=m_tau)
        eo, _, em = expect[tau]
        assert em == m_tau
        assert_bf16_close(o.cpu().numpy(), eo, f"segment {tau}")
        nk, nv = bufs[1 - cur]
        m_new = _lib.txl_mem_update(kb[:, :m_tau], kb[:, m_tau:m_tau + wl.W], nk, wl.M)
        _lib.txl_mem_update(vb[:, :m_tau], vb[:, m_tau:m_tau + wl.W], nv, wl.M)
        m_tau = m_new
    assert _lib.txl_get_device_status() == 0


def test_bf16_deterministic():
    wl = workload(2, 2, 64, 300, 200)
    q, k, v, r, bu, bv = prefilled_case(wl)
    o1, l1 = run_forward(q, k, v, r, bu, bv, wl.M, "bf16")
    o2, l2 = run_forward(q, k, v, r, bu, bv, wl.M, "bf16")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ----------------------------------------------------------------------------
# Attention with the memory roll in one call (txl_relattn_forward_roll)
# ----------------------------------------------------------------------------

ROLL_CASES = [
    # B, H, D, W, M, m        (M+W-m' a multiple of 64 -> written by the attention kernel)
    (2, 2, 64, 128, 64, 64),     # fused: kept rows are segment rows
    (2, 1, 64, 256, 256, 256),   # fused
    (1, 2, 64, 64, 1000, 1000),  # fused: kept rows start inside the memory
    (1, 1, 64, 128, 0, 512),     # fused: m > M+W keeps every row
    (1, 2, 64, 300, 384, 100),   # fused: 684-100 = 584 is not a multiple of 64 -> separate roll
    (2, 2, 64, 200, 150, 150),   # separate roll (350-150 = 200)
    (1, 2, 128, 200, 150, 64),   # D = 128: 350-64 = 286 is not a multiple of 64 -> separate roll
    (2, 2, 128, 256, 128, 128),  # D = 128 fused: kept rows are segment rows
    (1, 2, 128, 64, 1000, 1000), # D = 128 fused: kept rows start inside the memory
    (1, 1, 128, 128, 0, 512),    # D = 128 fused: every row kept
    (2, 2, 64, 128, 64, 0),      # m = 0: no roll
    (64, 8, 64, 64, 0, 64),      # fused, 512 one-step units (several per CTA), every row kept
    (24, 8, 64, 128, 64, 64),    # fused, 192 two-step units
]


@pytest.mark.parametrize("B,H,D,W,M,m", ROLL_CASES)
def test_forward_roll(_lib, B, H, D, W, M, m):
    wl = workload(B, H, D, W, M)
    q, k, v, r, bu, bv = prefilled_case(wl, n_r_extra=3)
    L, keep = M + W, min(m, M + W)
    qd, kd, vd, rd = (to_dev(x, torch.bfloat16) for x in (q, k, v, r))
    o = torch.empty(qd.shape, device=dev(), dtype=torch.bfloat16)
    # memory outputs: the head of larger buffers (batch stride != keep rows), prefilled with a sentinel
    rows = max(keep, 1) + 37
    km = torch.full((B, rows, H, D), 7.0, device=dev(), dtype=torch.bfloat16)
    vm = torch.full((B, rows, H, D), -7.0, device=dev(), dtype=torch.bfloat16)
    got_keep = _lib.txl_relattn_forward_roll(qd, kd, vd, rd, to_dev(bu, torch.float32), to_dev(bv, torch.float32),
                                             o, km[:, :max(keep, 1)], vm[:, :max(keep, 1)], m, M=M)
    assert _lib.txl_get_device_status() == 0
    assert got_keep == keep
    eo, _ = O.relattn_forward(q, k, v, r, bu, bv, M)
    assert_bf16_close(o.float().cpu().numpy(), eo, f"o {B,H,D,W,M,m}")
    C = H * D
    for dev_out, src, fill in ((km, k, 7.0), (vm, v, -7.0)):
        out = dev_out.float().cpu().numpy()
        want = O.mem_update(src[:, :M].reshape(B, M, C), src[:, M:].reshape(B, W, C), m).reshape(B, keep, H, D)
        assert np.array_equal(out[:, :keep], want), "kept rows differ"
        assert np.all(out[:, keep:] == fill), "rows past m' were written"


@pytest.mark.parametrize("name", ["base", "wide"])
def test_forward_roll_full_size_segments(_lib, name):
    """Base (D = 64) and wide (D = 128) workloads, three segments from a full
    memory: each call's fused roll feeds the next call, against the separate
    attention + roll calls."""
    wl = WORKLOADS[name]
    seg = make_segments(wl, n_segments=3)
    r = project_r(O.sinusoid_rel(wl.M + wl.W, wl.d_model), seg.W_r, wl.H, wl.D, "bf16")
    L = wl.M + wl.W
    rd = to_dev(r, torch.bfloat16)
    ud, vd = to_dev(seg.bias_u, torch.float32), to_dev(seg.bias_v, torch.float32)
    q0, k0, v0, _ = make_prefilled(wl, wl.M, seed=1)
    bufs = {n: [torch.empty(wl.B, L, wl.H, wl.D, device=dev(), dtype=torch.bfloat16) for _ in range(2)]
            for n in ("fk", "fv", "sk", "sv")}
    for n, src in (("fk", k0), ("fv", v0), ("sk", k0), ("sv", v0)):
        bufs[n][0].copy_(to_dev(src, torch.bfloat16))
    for tau in range(3):
        cur, nxt = tau % 2, 1 - tau % 2
        qt = to_dev(seg.seg("q", tau), torch.bfloat16)
        for n in ("fk", "sk"):
            bufs[n][cur][:, wl.M:] = to_dev(seg.seg("k", tau), torch.bfloat16)
        for n in ("fv", "sv"):
            bufs[n][cur][:, wl.M:] = to_dev(seg.seg("v", tau), torch.bfloat16)
        of = torch.empty(qt.shape, device=dev(), dtype=torch.bfloat16)
        os_ = torch.empty(qt.shape, device=dev(), dtype=torch.bfloat16)
        _lib.txl_relattn_forward_roll(qt, bufs["fk"][cur], bufs["fv"][cur], rd, ud, vd, of,
                                      bufs["fk"][nxt][:, :wl.M], bufs["fv"][nxt][:, :wl.M], wl.M, M=wl.M)
        _lib.txl_relattn_forward(qt, bufs["sk"][cur], bufs["sv"][cur], rd, ud, vd, os_, None, M=wl.M)
        C = wl.H * wl.D
        for n in ("sk", "sv"):
            b = bufs[n][cur].view(wl.B, L, C)
            _lib.txl_mem_update(b[:, :wl.M], b[:, wl.M:], bufs[n][nxt].view(wl.B, L, C), wl.M)
        assert torch.equal(of, os_), f"segment {tau}: outputs differ"
        assert torch.equal(bufs["fk"][nxt][:, :wl.M], bufs["sk"][nxt][:, :wl.M]), f"segment {tau}: k memory"
        assert torch.equal(bufs["fv"][nxt][:, :wl.M], bufs["sv"][nxt][:, :wl.M]), f"segment {tau}: v memory"
    assert _lib.txl_get_device_status() == 0
