"""Helpers shared by the GPU parity tests: seeded inputs on the device, the
oracle's expected values on the same (rounded) inputs, and the tolerances."""

import numpy as np
import torch

from oracle import txl_oracle as O
from synthetic import Workload, make_prefilled, make_segments, project_r

# Tolerances: fp32 path max |err| <= 1e-5; bf16-in / fp32-accumulate path
# rel-L2 <= 5e-3 and max |err| <= 2e-2 (both against the float64 oracle on the
# identical rounded inputs).
F32_ATOL = 1e-5
BF16_REL_L2 = 5e-3
BF16_ATOL = 2e-2


def dev():
    return torch.device("cuda:0")


def to_dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(dev()).to(dtype).contiguous()


def torch_dtype(name):
    return torch.bfloat16 if name == "bf16" else torch.float32


def workload(B, H, D, W, M, dtype="bf16", cfg_id=100):
    d_model = H * D + (H * D) % 2  # the sinusoid width must be even
    return Workload(f"t{B}x{H}x{D}x{W}x{M}", cfg_id, B, H, D, d_model, W, M, 1, dtype)


def prefilled_case(wl, seed=0, n_r_extra=0):
    """q, k, v (float32 arrays of exactly-representable values), r, biases."""
    q, k, v, s = make_prefilled(wl, wl.M, seed=seed)
    R = O.sinusoid_rel(wl.M + wl.W + n_r_extra, wl.d_model)
    r = project_r(R, s.W_r, wl.H, wl.D, wl.dtype)
    return q, k, v, r, s.bias_u, s.bias_v


def run_forward(q, k, v, r, bu, bv, M, dtype, o_dtype=None, with_lse=True, scale=None):
    import transformer_xl_relative_txl_gb300 as txl

    td = torch_dtype(dtype)
    od = td if o_dtype is None else torch_dtype(o_dtype)
    qd, kd, vd, rd = (to_dev(x, td) for x in (q, k, v, r))
    o = torch.empty(qd.shape, device=dev(), dtype=od)
    B, W, H, D = q.shape
    lse = torch.empty(B, H, W, device=dev(), dtype=torch.float32) if with_lse else None
    txl.txl_relattn_forward(qd, kd, vd, rd, to_dev(bu, torch.float32), to_dev(bv, torch.float32), o, lse,
                            M=M, scale=scale)
    assert txl.txl_get_device_status() == 0
    return o.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None)


def assert_bf16_close(got, want, what=""):
    err = got.astype(np.float64) - want
    rel = np.linalg.norm(err) / max(np.linalg.norm(want), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert rel <= BF16_REL_L2 and mx <= BF16_ATOL, f"{what}: rel-L2 {rel:.3e}, max abs {mx:.3e}"
    return rel, mx
