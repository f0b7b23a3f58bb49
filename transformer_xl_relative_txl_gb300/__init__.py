"""Transformer-XL relative-position attention for GB300 (sm_103a).

Thin ctypes binding of the C ABI in ``include/txl_relattn.h``: each function
has the C entry point's name and only marshals torch tensors (device memory,
CUDA streams) into pointers, sizes and dtype codes.  All computation runs in
the library's CUDA kernels; there is no fallback.  Importing fails loudly if
the library has not been built (``python transformer_xl_relative_txl_gb300/build.py``).
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "TXL_F32", "TXL_BF16", "TxlError", "lib", "library_path",
    "txl_relattn_forward", "txl_relattn_forward_static", "txl_relattn_forward_roll", "txl_relattn_forward_ring",
    "txl_relattn_forward_ring_append", "txl_relattn_backward", "txl_mem_update", "txl_mem_update_kv",
    "txl_mem_ring_append",
    "txl_layer_forward", "txl_layer_workspace_bytes", "LAYER_WEIGHT_NAMES", "txl_dense", "txl_stack_forward",
    "txl_stack_workspace_bytes",
    "txl_sinusoid_rel",
    "txl_get_device_status", "txl_release_cached", "txl_status_string", "txl_version",
    "txl_debug_set_wait_limit_ns", "txl_debug_inject_stall", "txl_debug_force_split",
    "txl_debug_set_bwd_chunk_bytes",
    "txl_debug_force_dense_tile_n",
    "txl_debug_force_bwd_path",
    "txl_debug_pair_split_tiles",
    "txl_debug_bwd_pairs_work",
    "txl_debug_unit_plan",
    "txl_debug_attention_split",
    "txl_debug_attention_items",
]

TXL_F32 = 0
TXL_BF16 = 1
_STATUS = {0: "TXL_OK", 1: "TXL_ERR_INVALID_ARG", 2: "TXL_ERR_UNSUPPORTED", 3: "TXL_ERR_ALIAS",
           4: "TXL_ERR_CUDA", 5: "TXL_ERR_DEVICE_TIMEOUT"}

library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtxl_relattn.so")
if not os.path.exists(library_path):
    raise ImportError(
        f"{library_path} is missing: build it with `python transformer_xl_relative_txl_gb300/build.py`")
lib = ctypes.CDLL(library_path)

_p, _i, _ll, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
lib.txl_relattn_forward.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _i, _i, _p]
lib.txl_relattn_forward.restype = _i
lib.txl_relattn_forward_static.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _i, _i, _p]
lib.txl_relattn_forward_static.restype = _i
lib.txl_relattn_forward_roll.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                                         _p, _p, _i, _ll, ctypes.POINTER(_i), _p]
lib.txl_relattn_forward_roll.restype = _i
lib.txl_relattn_backward.argtypes = [_p] * 15 + [_i, _i, _i, _i, _i, _i, _f, _i, _i, _p]
lib.txl_relattn_backward.restype = _i
lib.txl_relattn_forward_ring.argtypes = [_p, _p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _f,
                                         _i, _i, _p]
lib.txl_relattn_forward_ring.restype = _i
lib.txl_relattn_forward_ring_append.argtypes = [_p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i,
                                                _f, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i), _p]
lib.txl_relattn_forward_ring_append.restype = _i
lib.txl_mem_ring_append.argtypes = [_p, _i, _i, _i, _p, _i, _i, _i, _ll, ctypes.POINTER(_i), ctypes.POINTER(_i),
                                    _i, _p]
lib.txl_mem_ring_append.restype = _i
LAYER_WEIGHT_NAMES = ("W_q", "W_k", "W_v", "W_r", "bias_u", "bias_v", "W_o", "ln1_gamma", "ln1_beta", "W_1", "b_1",
                      "W_2", "b_2", "ln2_gamma", "ln2_beta")


class _LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_WEIGHT_NAMES]


lib.txl_layer_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
lib.txl_layer_workspace_bytes.restype = ctypes.c_size_t
lib.txl_layer_forward.argtypes = [_p, _p, _p, _p, _i, _i, _i, ctypes.POINTER(_LayerWeights), _p, _i, _i, _i, _i, _i,
                                  _i, _i, _f, _p, ctypes.c_size_t, ctypes.POINTER(_i), ctypes.POINTER(_i), _p]
lib.txl_layer_forward.restype = _i
lib.txl_stack_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
lib.txl_stack_workspace_bytes.restype = ctypes.c_size_t
lib.txl_stack_forward.argtypes = [_p, _p, _i, ctypes.POINTER(_p), ctypes.POINTER(_p), _i, _i, _i,
                                  ctypes.POINTER(_LayerWeights), _p, _i, _i, _i, _i, _i, _i, _i, _f, _p,
                                  ctypes.c_size_t, ctypes.POINTER(_i), ctypes.POINTER(_i), _p]
lib.txl_stack_forward.restype = _i
lib.txl_dense.argtypes = [_p, _p, _p, _i, _i, _i, _i, _ll, _ll, _p, _i, _p]
lib.txl_dense.restype = _i
lib.txl_mem_update.argtypes = [_p, _i, _p, _i, _p, _i, _i, _i, _ll, _ll, _ll, ctypes.POINTER(_i), _i, _p]
lib.txl_mem_update.restype = _i
lib.txl_mem_update_kv.argtypes = [_p, _p, _i, _p, _p, _i, _p, _p, _i, _i, _i, _ll, _ll, _ll, ctypes.POINTER(_i), _i,
                                  _p]
lib.txl_mem_update_kv.restype = _i
lib.txl_sinusoid_rel.argtypes = [_p, _i, _i, _i, _p]
lib.txl_sinusoid_rel.restype = _i
lib.txl_get_device_status.argtypes = [_p]
lib.txl_get_device_status.restype = _i
lib.txl_release_cached.argtypes = []
lib.txl_release_cached.restype = _i
lib.txl_status_string.argtypes = [_i]
lib.txl_status_string.restype = ctypes.c_char_p
lib.txl_version.argtypes = []
lib.txl_version.restype = _i
lib.txl_debug_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
lib.txl_debug_set_wait_limit_ns.restype = _i
lib.txl_debug_inject_stall.argtypes = [_i]
lib.txl_debug_inject_stall.restype = _i
lib.txl_debug_force_split.argtypes = [_i]
lib.txl_debug_force_split.restype = _i
lib.txl_debug_set_bwd_chunk_bytes.argtypes = [ctypes.c_ulonglong]
lib.txl_debug_set_bwd_chunk_bytes.restype = _i
lib.txl_debug_force_dense_tile_n.argtypes = [_i]
lib.txl_debug_force_dense_tile_n.restype = _i
lib.txl_debug_force_bwd_path.argtypes = [_i]
lib.txl_debug_force_bwd_path.restype = _i
lib.txl_debug_pair_split_tiles.argtypes = [_i, _i, _i, _i, _i]
lib.txl_debug_pair_split_tiles.restype = _i
lib.txl_debug_bwd_pairs_work.argtypes = [_i, _i, _i, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i), _p, _i, _p,
                                         _i]
lib.txl_debug_bwd_pairs_work.restype = _i
lib.txl_debug_unit_plan.argtypes = [_i, _i, _i, _i, _i, _p, _i, ctypes.POINTER(_i)]
lib.txl_debug_unit_plan.restype = _i
lib.txl_debug_attention_split.argtypes = [_i, _i, _i, _i, _i]
lib.txl_debug_attention_split.restype = _i
lib.txl_debug_attention_items.argtypes = [_i, _i, _i, _i, _i, _p, _i, ctypes.POINTER(_i)]
lib.txl_debug_attention_items.restype = _i


class TxlError(RuntimeError):
    """A nonzero txl_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)}")


def _check(status: int, where: str):
    if status != 0:
        raise TxlError(status, where)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return TXL_BF16
    if t == torch.float32:
        return TXL_F32
    raise ValueError(f"unsupported dtype {t}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live in device memory")
    return t.data_ptr() or None


def txl_relattn_forward(q, k, v, r, bias_u, bias_v, o, lse=None, M=None, scale=None, stream=None):
    """o <- relative attention of q [B,W,H,D] over k, v [B,M+W,H,D] with
    distance keys r [n_r,H,D] and biases bias_u, bias_v [H,D] (fp32).
    lse [B,H,W] fp32 is optional.  scale defaults to 1/sqrt(D)."""
    return _forward(lib.txl_relattn_forward, "txl_relattn_forward", q, k, v, r, bias_u, bias_v, o, lse, M, scale,
                    stream)


def txl_relattn_forward_static(q, k, v, r, bias_u, bias_v, o, lse=None, M=None, scale=None, stream=None):
    """txl_relattn_forward without any allocation: split key ranges keep
    their partial results in the library's fixed device array."""
    return _forward(lib.txl_relattn_forward_static, "txl_relattn_forward_static", q, k, v, r, bias_u, bias_v, o,
                    lse, M, scale, stream)


def txl_relattn_backward(q, k, v, r, bias_u, bias_v, o, lse, dout, M=None, scale=None, grads=None, stream=None):
    """Gradients of txl_relattn_forward for dout = dL/do: returns a dict of
    fp32 tensors dq [B,W,H,D], dk and dv [B,W,H,D] (the segment's key and
    value rows; memory rows get none), dr [n_r,H,D], dbias_u and dbias_v
    [H,D].  o and lse are the forward's outputs; o and dout share a dtype.
    ``grads`` may pass preallocated output tensors under the same keys."""
    B, W, H, D = q.shape
    if M is None:
        M = k.shape[1] - W
    for t in (q, k, v, r, bias_u, bias_v, o, lse, dout):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if k.shape != (B, M + W, H, D) or v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shape mismatch between q, k, v, o, dout")
    if r.dim() != 3 or r.shape[1:] != (H, D) or bias_u.shape != (H, D) or bias_v.shape != (H, D):
        raise ValueError("r must be [n_r, H, D]; biases [H, D]")
    if bias_u.dtype != torch.float32 or bias_v.dtype != torch.float32:
        raise ValueError("biases are fp32")
    if lse.shape != (B, H, W) or lse.dtype != torch.float32:
        raise ValueError("lse must be fp32 [B, H, W]")
    if not (q.dtype == k.dtype == v.dtype == r.dtype) or o.dtype != dout.dtype:
        raise ValueError("q, k, v, r share a dtype; so do o and dout")
    shapes = {"dq": q.shape, "dk": q.shape, "dv": q.shape, "dr": r.shape, "dbias_u": bias_u.shape,
              "dbias_v": bias_v.shape}
    g = dict(grads or {})
    for key, shp in shapes.items():
        if key not in g:
            g[key] = torch.empty(shp, device=q.device, dtype=torch.float32)
        t = g[key]
        if t.shape != shp or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{key} must be a contiguous fp32 tensor of shape {tuple(shp)}")
    if scale is None:
        scale = D ** -0.5
    st = lib.txl_relattn_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(bias_u), _ptr(bias_v), _ptr(o),
                                  _ptr(lse), _ptr(dout), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                                  _ptr(g["dr"]), _ptr(g["dbias_u"]), _ptr(g["dbias_v"]), B, W, M, H, D,
                                  r.shape[0], float(scale), _dtype_code(q.dtype), _dtype_code(o.dtype),
                                  _stream(stream))
    _check(st, "txl_relattn_backward")
    return g


def txl_relattn_forward_ring(q, k_mem, v_mem, start, M, k_seg, v_seg, r, bias_u, bias_v, o, lse=None, scale=None,
                             stream=None):
    """Relative attention of q [B,W,H,D] over [memory ; segment]: memory row
    m (m < M) is row (start + m) % cap of the rings k_mem, v_mem [B,cap,H,D];
    the segment's keys and values are k_seg, v_seg [B,W,H,D]."""
    B, W, H, D = q.shape
    for t in (q, k_seg, v_seg, r, bias_u, bias_v, o) + ((lse,) if lse is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if k_mem.dim() != 4 or k_mem.shape[0] != B or k_mem.shape[2:] != (H, D) or v_mem.shape != k_mem.shape:
        raise ValueError("k_mem, v_mem must be [B, cap, H, D]")
    if not (k_mem.is_contiguous() and v_mem.is_contiguous()):
        raise ValueError("rings must be contiguous")
    if k_seg.shape != q.shape or v_seg.shape != q.shape or o.shape != q.shape:
        raise ValueError("k_seg, v_seg, o must be [B, W, H, D]")
    if r.dim() != 3 or r.shape[1:] != (H, D) or bias_u.shape != (H, D) or bias_v.shape != (H, D):
        raise ValueError("r must be [n_r, H, D]; biases [H, D]")
    if not (q.dtype == k_mem.dtype == v_mem.dtype == k_seg.dtype == v_seg.dtype == r.dtype):
        raise ValueError("q, rings, segment rows and r must share a dtype")
    if scale is None:
        scale = D ** -0.5
    st = lib.txl_relattn_forward_ring(_ptr(q), _ptr(k_mem), _ptr(v_mem), k_mem.shape[1], int(start), int(M),
                                      _ptr(k_seg), _ptr(v_seg), _ptr(r), _ptr(bias_u), _ptr(bias_v), _ptr(o),
                                      _ptr(lse), B, W, H, D, r.shape[0], float(scale), _dtype_code(q.dtype),
                                      _dtype_code(o.dtype), _stream(stream))
    _check(st, "txl_relattn_forward_ring")
    return o


def txl_relattn_forward_ring_append(q, k_mem, v_mem, start, M, k_seg, v_seg, r, bias_u, bias_v, o, lse=None,
                                    scale=None, stream=None):
    """txl_relattn_forward_ring, then the segment's k, v rows appended to
    the rings; returns the rings' new (start, m)."""
    B, W, H, D = q.shape
    for t in (q, k_mem, v_mem, k_seg, v_seg, r, bias_u, bias_v, o) + ((lse,) if lse is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if k_mem.dim() != 4 or k_mem.shape[0] != B or k_mem.shape[2:] != (H, D) or v_mem.shape != k_mem.shape:
        raise ValueError("k_mem, v_mem must be [B, cap, H, D]")
    if k_seg.shape != q.shape or v_seg.shape != q.shape or o.shape != q.shape:
        raise ValueError("k_seg, v_seg, o must be [B, W, H, D]")
    if r.dim() != 3 or r.shape[1:] != (H, D) or bias_u.shape != (H, D) or bias_v.shape != (H, D):
        raise ValueError("r must be [n_r, H, D]; biases [H, D]")
    if not (q.dtype == k_mem.dtype == v_mem.dtype == k_seg.dtype == v_seg.dtype == r.dtype):
        raise ValueError("q, rings, segment rows and r must share a dtype")
    if scale is None:
        scale = D ** -0.5
    s_out, m_out = ctypes.c_int(0), ctypes.c_int(0)
    st = lib.txl_relattn_forward_ring_append(_ptr(k_mem), _ptr(v_mem), k_mem.shape[1], int(start), int(M), _ptr(q),
                                             _ptr(k_seg), _ptr(v_seg), _ptr(r), _ptr(bias_u), _ptr(bias_v),
                                             _ptr(o), _ptr(lse), B, W, H, D, r.shape[0], float(scale),
                                             _dtype_code(q.dtype), _dtype_code(o.dtype), ctypes.byref(s_out),
                                             ctypes.byref(m_out), _stream(stream))
    _check(st, "txl_relattn_forward_ring_append")
    return s_out.value, m_out.value


def txl_layer_workspace_bytes(B, W, d_model, H, D, d_ff, n_r):
    return int(lib.txl_layer_workspace_bytes(B, W, d_model, H, D, d_ff, n_r))


def txl_layer_forward(h, out, k_mem, v_mem, start, M, weights, R, workspace, scale=None, stream=None):
    """One layer on the segment h [B, W, d_model] (bf16) into out; the
    attention memory is the rings k_mem, v_mem [B, cap, H, D] holding M
    projected rows from ring row `start`; weights: dict with
    LAYER_WEIGHT_NAMES (bf16 matrices [in, out], fp32 vectors); R: the raw
    distance table [n_r, d_model] bf16; workspace: uint8 device tensor of at
    least txl_layer_workspace_bytes(...) bytes.  Returns the rings' new
    (start, m)."""
    B, W, d_model = h.shape
    _, cap, H, D = k_mem.shape
    d_ff = weights["W_1"].shape[1]
    for t in (h, out, k_mem, v_mem, R, workspace) + tuple(weights[n] for n in LAYER_WEIGHT_NAMES):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if out.shape != h.shape or h.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("h and out must be bf16 [B, W, d_model]")
    if v_mem.shape != k_mem.shape or k_mem.shape[0] != B or k_mem.dtype != torch.bfloat16:
        raise ValueError("rings must be bf16 [B, cap, H, D]")
    if scale is None:
        scale = D ** -0.5
    wts = _layer_struct(weights, d_model, H, D)
    s_out, m_out = ctypes.c_int(0), ctypes.c_int(0)
    st = lib.txl_layer_forward(_ptr(h), _ptr(out), _ptr(k_mem), _ptr(v_mem), cap, int(start), int(M),
                               ctypes.byref(wts), _ptr(R), R.shape[0], B, W, d_model, H, D, d_ff, float(scale),
                               _ptr(workspace), workspace.numel() * workspace.element_size(), ctypes.byref(s_out),
                               ctypes.byref(m_out), _stream(stream))
    _check(st, "txl_layer_forward")
    return s_out.value, m_out.value


def _layer_struct(weights, d_model, H, D):
    for t in (weights[n] for n in LAYER_WEIGHT_NAMES):
        if not t.is_contiguous():
            raise ValueError("weights must be contiguous")
    for n in ("W_q", "W_k", "W_v", "W_r", "W_o", "W_1", "W_2"):
        if weights[n].dtype != torch.bfloat16:
            raise ValueError(f"{n} must be bf16")
    for n in ("bias_u", "bias_v", "ln1_gamma", "ln1_beta", "b_1", "b_2", "ln2_gamma", "ln2_beta"):
        if weights[n].dtype != torch.float32:
            raise ValueError(f"{n} must be fp32")
    return _LayerWeights(*[_ptr(weights[n]) for n in LAYER_WEIGHT_NAMES])


def txl_stack_workspace_bytes(B, W, d_model, H, D, d_ff, n_r):
    return int(lib.txl_stack_workspace_bytes(B, W, d_model, H, D, d_ff, n_r))


def txl_stack_forward(h, out, k_mems, v_mems, start, M, weights, R, workspace, scale=None, stream=None):
    """len(weights) layers of txl_layer_forward on the segment h [B, W,
    d_model] (bf16), the last layer's output into out; k_mems, v_mems: one
    ring pair [B, cap, H, D] per layer, all holding M rows from ring row
    `start`; weights: one dict per layer; workspace: uint8 device tensor of
    at least txl_stack_workspace_bytes(...) bytes.  Returns the rings' common
    new (start, m)."""
    B, W, d_model = h.shape
    L = len(weights)
    if L < 1 or len(k_mems) != L or len(v_mems) != L:
        raise ValueError("one ring pair and one weight dict per layer")
    _, cap, H, D = k_mems[0].shape
    d_ff = weights[0]["W_1"].shape[1]
    for t in (h, out, R, workspace) + tuple(k_mems) + tuple(v_mems):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if out.shape != h.shape or h.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("h and out must be bf16 [B, W, d_model]")
    for km, vm in zip(k_mems, v_mems):
        if km.shape != (B, cap, H, D) or vm.shape != km.shape or km.dtype != torch.bfloat16 or vm.dtype != km.dtype:
            raise ValueError("rings must be bf16 [B, cap, H, D], the same for every layer")
    if scale is None:
        scale = D ** -0.5
    ws = (_LayerWeights * L)(*[_layer_struct(w, d_model, H, D) for w in weights])
    kp = (_p * L)(*[_ptr(x) for x in k_mems])
    vp = (_p * L)(*[_ptr(x) for x in v_mems])
    s_out, m_out = ctypes.c_int(0), ctypes.c_int(0)
    st = lib.txl_stack_forward(_ptr(h), _ptr(out), L, kp, vp, cap, int(start), int(M), ws, _ptr(R), R.shape[0], B, W,
                               d_model, H, D, d_ff, float(scale), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), ctypes.byref(s_out), ctypes.byref(m_out),
                               _stream(stream))
    _check(st, "txl_stack_forward")
    return s_out.value, m_out.value


def txl_dense(x, W, y, bias=None, relu=False, stream=None):
    """y = x W (+ bias) (then ReLU): x [m, k], W [k, n] or [batch, k, n],
    y [m, n] or [batch, m, n] (bf16, contiguous); bias fp32 [n] or None."""
    if x.dim() != 2:
        raise ValueError("x must be [m, k]")
    m, k = x.shape
    Wb = W if W.dim() == 3 else W.unsqueeze(0)
    yb = y if y.dim() == 3 else y.unsqueeze(0)
    batch, k2, n = Wb.shape
    if k2 != k or yb.shape != (batch, m, n):
        raise ValueError("shape mismatch between x, W, y")
    for t in (x, W, y) + ((bias,) if bias is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if not (x.dtype == W.dtype == y.dtype == torch.bfloat16):
        raise ValueError("x, W, y must be bf16")
    if bias is not None and (bias.dtype != torch.float32 or bias.shape != (n,)):
        raise ValueError("bias must be fp32 [n]")
    st = lib.txl_dense(_ptr(x), _ptr(W), _ptr(y), m, n, k, batch, k * n, m * n, _ptr(bias), 1 if relu else 0,
                       _stream(stream))
    _check(st, "txl_dense")
    return y


def txl_mem_ring_append(mem, start, m, h, stream=None):
    """Append the rows of h [B, w, ...] (row-contiguous, any batch stride) to
    the ring mem [B, cap, ...] that holds m rows from ring row `start`;
    returns the new (start, m)."""
    B, cap = mem.shape[0], mem.shape[1]
    C = math.prod(mem.shape[2:])
    w = h.shape[1]
    if not mem.is_contiguous():
        raise ValueError("the ring must be contiguous")
    if h.shape[0] != B or math.prod(h.shape[2:]) != C or (w > 0 and not h[0].is_contiguous()):
        raise ValueError("h must be [B, w, ...] with rows of the ring's width")
    if mem.dtype != h.dtype:
        raise ValueError("mem and h must share a dtype")
    s_out, m_out = ctypes.c_int(0), ctypes.c_int(0)
    st = lib.txl_mem_ring_append(_ptr(mem), cap, int(start), int(m), _ptr(h) if w > 0 else None, w, B, C,
                                 h.stride(0) if B > 1 else w * C, ctypes.byref(s_out), ctypes.byref(m_out),
                                 _dtype_code(mem.dtype), _stream(stream))
    _check(st, "txl_mem_ring_append")
    return s_out.value, m_out.value


def _forward(fn, name, q, k, v, r, bias_u, bias_v, o, lse, M, scale, stream):
    B, W, H, D = q.shape
    if M is None:
        M = k.shape[1] - W
    for t in (q, k, v, r, bias_u, bias_v, o) + ((lse,) if lse is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if k.shape != (B, M + W, H, D) or v.shape != k.shape or o.shape != q.shape:
        raise ValueError("shape mismatch between q, k, v, o")
    if r.dim() != 3 or r.shape[1:] != (H, D) or bias_u.shape != (H, D) or bias_v.shape != (H, D):
        raise ValueError("r must be [n_r, H, D]; biases [H, D]")
    if bias_u.dtype != torch.float32 or bias_v.dtype != torch.float32:
        raise ValueError("biases are fp32")
    if lse is not None and (lse.shape != (B, H, W) or lse.dtype != torch.float32):
        raise ValueError("lse must be fp32 [B, H, W]")
    if not (q.dtype == k.dtype == v.dtype == r.dtype):
        raise ValueError("q, k, v, r must share a dtype")
    if scale is None:
        scale = D ** -0.5
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(bias_u), _ptr(bias_v), _ptr(o), _ptr(lse), B, W, M, H, D,
            r.shape[0], float(scale), _dtype_code(q.dtype), _dtype_code(o.dtype), _stream(stream))
    _check(st, name)
    return o


def txl_relattn_forward_roll(q, k, v, r, bias_u, bias_v, o, k_mem_out, v_mem_out, m, lse=None, M=None, scale=None,
                             stream=None) -> int:
    """txl_relattn_forward, then the memory roll of k and v: k_mem_out and
    v_mem_out [B, >= m', H, D] (row-contiguous views; batch strides may be
    any, equal for both) receive the last m' = min(m, M+W) rows of k and v.
    Returns m'."""
    B, W, H, D = q.shape
    if M is None:
        M = k.shape[1] - W
    for t in (q, k, v, r, bias_u, bias_v, o) + ((lse,) if lse is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if k.shape != (B, M + W, H, D) or v.shape != k.shape or o.shape != q.shape:
        raise ValueError("shape mismatch between q, k, v, o")
    if r.dim() != 3 or r.shape[1:] != (H, D) or bias_u.shape != (H, D) or bias_v.shape != (H, D):
        raise ValueError("r must be [n_r, H, D]; biases [H, D]")
    if bias_u.dtype != torch.float32 or bias_v.dtype != torch.float32:
        raise ValueError("biases are fp32")
    if lse is not None and (lse.shape != (B, H, W) or lse.dtype != torch.float32):
        raise ValueError("lse must be fp32 [B, H, W]")
    if not (q.dtype == k.dtype == v.dtype == r.dtype == k_mem_out.dtype == v_mem_out.dtype):
        raise ValueError("q, k, v, r and the memory outputs must share a dtype")
    keep = min(m, M + W)
    for t, name in ((k_mem_out, "k_mem_out"), (v_mem_out, "v_mem_out")):
        if t.dim() != 4 or t.shape[0] != B or t.shape[2:] != (H, D) or t.shape[1] < keep:
            raise ValueError(f"{name} must be [B, >= m', H, D]")
        if t.stride(3) != 1 or t.stride(2) != D or (t.shape[1] > 1 and t.stride(1) != H * D):
            raise ValueError(f"{name} rows must be contiguous")
    if k_mem_out.stride(0) != v_mem_out.stride(0):
        raise ValueError("k_mem_out and v_mem_out must share a batch stride")
    if scale is None:
        scale = D ** -0.5
    m_out = ctypes.c_int(0)
    st = lib.txl_relattn_forward_roll(_ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(bias_u), _ptr(bias_v), _ptr(o),
                                      _ptr(lse), B, W, M, H, D, r.shape[0], float(scale), _dtype_code(q.dtype),
                                      _dtype_code(o.dtype), _ptr(k_mem_out), _ptr(v_mem_out), m,
                                      k_mem_out.stride(0), ctypes.byref(m_out), _stream(stream))
    _check(st, "txl_relattn_forward_roll")
    return m_out.value


def _rows_view(t, name):
    if t.dim() != 3 or t.stride(2) != 1 or (t.shape[1] > 1 and t.stride(1) != t.shape[2]):
        raise ValueError(f"{name} must be a [B, rows, C] view with contiguous rows")
    return t.stride(0)


def txl_mem_update(mem, h, mem_out, m, stream=None) -> int:
    """mem_out[:, :m'] <- last m' = min(m, m_prev + w) rows of [mem ; h].

    mem [B, m_prev, C], h [B, w, C], mem_out [B, >= m', C]: row-contiguous
    views (batch strides may differ).  Returns m'."""
    B, m_prev, C = mem.shape
    w = h.shape[1]
    if h.shape[0] != B or h.shape[2] != C or mem_out.shape[0] != B or mem_out.shape[2] != C:
        raise ValueError("mem, h, mem_out disagree on B or C")
    if not (mem.dtype == h.dtype == mem_out.dtype):
        raise ValueError("dtype mismatch")
    mem_bs = _rows_view(mem, "mem")
    h_bs = _rows_view(h, "h")
    out_bs = _rows_view(mem_out, "mem_out")
    keep = min(m, m_prev + w)
    if mem_out.shape[1] < keep:
        raise ValueError("mem_out has too few rows")
    m_out = ctypes.c_int(0)
    st = lib.txl_mem_update(_ptr(mem) if m_prev > 0 else None, m_prev, _ptr(h) if w > 0 else None, w,
                            _ptr(mem_out), m, B, C, mem_bs, h_bs, out_bs, ctypes.byref(m_out),
                            _dtype_code(mem.dtype), _stream(stream))
    _check(st, "txl_mem_update")
    return m_out.value


def txl_mem_update_kv(k_mem, v_mem, k_h, v_h, k_out, v_out, m, stream=None) -> int:
    """txl_mem_update of keys and of values in one launch: [B, rows, C]
    row-contiguous views; each pair (k_mem, v_mem), (k_h, v_h), (k_out,
    v_out) shares its shape and batch stride.  Returns m'."""
    B, m_prev, C = k_mem.shape
    w = k_h.shape[1]
    for a, b, name in ((k_mem, v_mem, "mem"), (k_h, v_h, "h"), (k_out, v_out, "out")):
        if a.shape != b.shape or _rows_view(a, "k_" + name) != _rows_view(b, "v_" + name):
            raise ValueError(f"k_{name} and v_{name} must share shape and batch stride")
    if k_h.shape[0] != B or k_h.shape[2] != C or k_out.shape[0] != B or k_out.shape[2] != C:
        raise ValueError("mem, h, out disagree on B or C")
    if not (k_mem.dtype == v_mem.dtype == k_h.dtype == v_h.dtype == k_out.dtype == v_out.dtype):
        raise ValueError("dtype mismatch")
    keep = min(m, m_prev + w)
    if k_out.shape[1] < keep:
        raise ValueError("out has too few rows")
    m_out = ctypes.c_int(0)
    st = lib.txl_mem_update_kv(_ptr(k_mem) if m_prev > 0 else None, _ptr(v_mem) if m_prev > 0 else None, m_prev,
                               _ptr(k_h) if w > 0 else None, _ptr(v_h) if w > 0 else None, w, _ptr(k_out),
                               _ptr(v_out), m, B, C, _rows_view(k_mem, "k_mem"), _rows_view(k_h, "k_h"),
                               _rows_view(k_out, "k_out"), ctypes.byref(m_out), _dtype_code(k_mem.dtype),
                               _stream(stream))
    _check(st, "txl_mem_update_kv")
    return m_out.value


def txl_sinusoid_rel(R, stream=None):
    """R [n_dist, dim] <- sin / cos of distance times 10000^(-2k/dim), interleaved."""
    if R.dim() != 2 or not R.is_contiguous():
        raise ValueError("R must be a contiguous [n_dist, dim] tensor")
    st = lib.txl_sinusoid_rel(_ptr(R), R.shape[0], R.shape[1], _dtype_code(R.dtype), _stream(stream))
    _check(st, "txl_sinusoid_rel")
    return R


def txl_get_device_status(stream=None) -> int:
    return lib.txl_get_device_status(_stream(stream))


def txl_release_cached() -> None:
    """Frees the library's cached scratch and unit plans of the current device
    (synchronises it first)."""
    _check(lib.txl_release_cached(), "txl_release_cached")


def txl_status_string(status: int) -> str:
    return lib.txl_status_string(status).decode()


def txl_version() -> int:
    return lib.txl_version()


def txl_debug_set_wait_limit_ns(ns: int) -> int:
    return lib.txl_debug_set_wait_limit_ns(ns)


def txl_debug_inject_stall(on: bool) -> int:
    return lib.txl_debug_inject_stall(1 if on else 0)


def txl_debug_force_split(nsplit):
    """Test hook: force the D = 64 forward's split count (0: its cost model)."""
    _check(lib.txl_debug_force_split(int(nsplit)), "txl_debug_force_split")


def txl_debug_set_bwd_chunk_bytes(nbytes):
    """Test hook: cap on one chunk's scratch in the D = 128 tensor-core
    backward (0: the default, 1 GiB)."""
    _check(lib.txl_debug_set_bwd_chunk_bytes(int(nbytes)), "txl_debug_set_bwd_chunk_bytes")


def txl_debug_force_dense_tile_n(bn):
    """Test hook: fix txl_dense's column tile (64, 128 or 256; 0: its cost
    model)."""
    _check(lib.txl_debug_force_dense_tile_n(int(bn)), "txl_debug_force_dense_tile_n")


def txl_debug_force_bwd_path(path):
    """Test hook: the bf16 D = 64 backward's path (1: fused kernels, 2: pair
    terms materialised; 0: the library's choice)."""
    _check(lib.txl_debug_force_bwd_path(int(path)), "txl_debug_force_bwd_path")


def txl_debug_pair_split_tiles(n_query_tiles, seq_heads, W, M, sms):
    """Test hook (host only): the number of longest query tiles the
    backward's pair kernel splits into two CTAs per unit."""
    return lib.txl_debug_pair_split_tiles(int(n_query_tiles), int(seq_heads), int(W), int(M), int(sms))


def txl_debug_bwd_pairs_work(B, W, M, H, split_qt):
    """Test hook (host only): the backward pair kernel's CTAs as rows
    (b, h, i0, t0, nks) and the products' tiles as rows (mode, z, m0, kb0,
    nkb, nkb_c), two int32 arrays, for B sequences with the split_qt longest
    query tiles split."""
    import numpy as np

    n_ctas, n_tiles = _i(0), _i(0)
    args = [int(B), int(W), int(M), int(H), int(split_qt), ctypes.byref(n_ctas), ctypes.byref(n_tiles)]
    rc = lib.txl_debug_bwd_pairs_work(*args, None, 0, None, 0)
    if rc != 0:
        raise TxlError(1, "txl_debug_bwd_pairs_work")
    ctas = np.zeros((n_ctas.value, 5), np.int32)
    tiles = np.zeros((n_tiles.value, 6), np.int32)
    rc = lib.txl_debug_bwd_pairs_work(*args, ctas.ctypes.data, ctas.shape[0], tiles.ctypes.data, tiles.shape[0])
    if rc != 0:
        raise TxlError(1, "txl_debug_bwd_pairs_work")
    return ctas, tiles


def txl_debug_unit_plan(B, H, W, M, ctas):
    """Test hook (host only): the bf16 attention's unit plan for `ctas`
    persistent CTAs, an int32 array [ctas, stride] of unit indices, -1
    ending each CTA's row."""
    import numpy as np

    stride = _i(0)
    if lib.txl_debug_unit_plan(int(B), int(H), int(W), int(M), int(ctas), None, 0, ctypes.byref(stride)) != 0:
        raise TxlError(1, "txl_debug_unit_plan")
    table = np.zeros((int(ctas), stride.value), np.int32)
    if lib.txl_debug_unit_plan(int(B), int(H), int(W), int(M), int(ctas), table.ctypes.data, table.size,
                               ctypes.byref(stride)) != 0:
        raise TxlError(1, "txl_debug_unit_plan")
    return table


def txl_debug_attention_split(B, H, W, M, sms):
    """Test hook (host only): the chunks per unit the D = 64 attention
    splits its key steps into on a device of `sms` SMs (1: no split)."""
    return lib.txl_debug_attention_split(int(B), int(H), int(W), int(M), int(sms))


def txl_debug_attention_items(B, H, W, M, nsplit):
    """Test hook (host only): the attention's work items for nsplit chunks
    per unit, an int32 array of rows (b, h, i0, t0, nks) in launch order."""
    import numpy as np

    n = _i(0)
    args = [int(B), int(H), int(W), int(M), int(nsplit)]
    if lib.txl_debug_attention_items(*args, None, 0, ctypes.byref(n)) != 0:
        raise TxlError(1, "txl_debug_attention_items")
    items = np.zeros((n.value, 5), np.int32)
    if lib.txl_debug_attention_items(*args, items.ctypes.data, n.value, ctypes.byref(n)) != 0:
        raise TxlError(1, "txl_debug_attention_items")
    return items
