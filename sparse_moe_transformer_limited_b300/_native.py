"""ctypes binding of libbeam_moe.so (the C ABI in include/beam_moe.h).

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream; every step of the layer runs in the library's kernels.
There is no fallback: if the library is missing or cannot load, importing
the functions raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbeam_moe.so")

BEAM_OK = 0
BEAM_ERR_INVALID_ARG = 1
BEAM_ERR_UNSUPPORTED = 2
BEAM_ERR_WORKSPACE = 3
BEAM_ERR_CUDA = 4
BEAM_ERR_TIMEOUT = 5
BEAM_ERR_DEVICE_FLAG = 6

FLAG_PRE_NORM = 1
FLAG_FP32_OUT = 2
FLAG_RETURN_SCORES = 4
FLAG_FP8_EXPERTS = 8
FLAG_NVFP4_EXPERTS = 16
FLAG_PREFILL_WEIGHT_MAJOR = 32

# names of the workspace buffers, in beam_moe_workspace_layout() order
LAYOUT_NAMES = ("xn", "part", "topk_idx", "topk_w", "counts", "offsets", "row_token",
                "row_weight", "xperm", "act", "oacc", "n_units", "blk_hist", "blk_off",
                "units_gu", "units_dn", "pair_row", "router_w3", "router_units",
                "x_scale", "act_q", "act_scale", "x_sf", "act_sf", "arrive")

# every symbol include/beam_moe.h declares
EXPORTED = ("beam_moe_workspace_size", "beam_moe_route", "beam_moe_route_static",
            "beam_moe_forward", "beam_dense_workspace_size", "beam_dense_mlp_forward",
            "beam_residual_step", "beam_status", "beam_last_error_string",
            "beam_moe_workspace_layout", "beam_debug_wait_timeout", "beam_profile_enable",
            "beam_profile_read", "beam_quantize_e4m3_rows", "beam_moe_forward_fp8",
            "beam_dense_mlp_forward_fp8", "beam_dense_workspace_layout",
            "beam_quantize_nvfp4", "beam_moe_forward_nvfp4", "beam_dense_mlp_forward_nvfp4",
            "beam_attention_workspace_size", "beam_attention_forward",
            "beam_attention_workspace_layout", "beam_moe_forward_routed", "beam_ep_dispatch",
            "beam_ep_combine")


class BeamError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"beam status {code}: {msg}")
        self.code = code


class Params(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int),
                ("I", ctypes.c_int), ("n_group", ctypes.c_int), ("topk_group", ctypes.c_int),
                ("top_k", ctypes.c_int), ("routed_scale", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("residual_k", ctypes.c_int),
                ("flags", ctypes.c_int)]


class DenseParams(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("residual_k", ctypes.c_int),
                ("flags", ctypes.c_int)]


class AttnParams(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("n_q", ctypes.c_int),
                ("n_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("window", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("residual_k", ctypes.c_int), ("flags", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the library once; raise if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run "
                              "`python -m sparse_moe_transformer_limited_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
        P = ctypes.POINTER(Params)
        L.beam_moe_workspace_size.argtypes = [P]
        L.beam_moe_workspace_size.restype = sz
        L.beam_moe_workspace_layout.argtypes = [P, ctypes.POINTER(sz), i32]
        L.beam_moe_workspace_layout.restype = i32
        L.beam_moe_route.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.beam_moe_route.restype = i32
        L.beam_moe_route_static.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
        L.beam_moe_route_static.restype = i32
        L.beam_moe_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.beam_moe_forward.restype = i32
        D = ctypes.POINTER(DenseParams)
        L.beam_dense_workspace_size.argtypes = [D]
        L.beam_dense_workspace_size.restype = sz
        L.beam_dense_workspace_layout.argtypes = [D, ctypes.POINTER(sz), i32]
        L.beam_dense_workspace_layout.restype = i32
        L.beam_dense_mlp_forward.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.beam_dense_mlp_forward.restype = i32
        L.beam_quantize_e4m3_rows.argtypes = [vp, ctypes.c_longlong, i32, vp, vp, vp]
        L.beam_quantize_e4m3_rows.restype = i32
        L.beam_moe_forward_fp8.argtypes = [P] + [vp] * 15 + [sz, vp]
        L.beam_moe_forward_fp8.restype = i32
        L.beam_dense_mlp_forward_fp8.argtypes = [D] + [vp] * 11 + [sz, vp]
        L.beam_dense_mlp_forward_fp8.restype = i32
        L.beam_quantize_nvfp4.argtypes = [vp, ctypes.c_longlong, i32, i32, vp, vp, vp, vp]
        L.beam_quantize_nvfp4.restype = i32
        L.beam_moe_forward_nvfp4.argtypes = [P] + [vp] * 18 + [sz, vp]
        L.beam_moe_forward_nvfp4.restype = i32
        L.beam_dense_mlp_forward_nvfp4.argtypes = [D] + [vp] * 14 + [sz, vp]
        L.beam_dense_mlp_forward_nvfp4.restype = i32
        A = ctypes.POINTER(AttnParams)
        L.beam_attention_workspace_size.argtypes = [A]
        L.beam_attention_workspace_size.restype = sz
        L.beam_attention_workspace_layout.argtypes = [A, ctypes.POINTER(sz), i32]
        L.beam_attention_workspace_layout.restype = i32
        L.beam_attention_forward.argtypes = [A] + [vp] * 9 + [sz, vp]
        L.beam_attention_forward.restype = i32
        L.beam_moe_forward_routed.argtypes = [P] + [vp] * 10 + [sz, vp]
        L.beam_moe_forward_routed.restype = i32
        L.beam_ep_dispatch.argtypes = [P, i32] + [vp] * 7 + [sz, vp]
        L.beam_ep_dispatch.restype = i32
        L.beam_ep_combine.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, f32, i32, i32, vp, vp]
        L.beam_ep_combine.restype = i32
        L.beam_residual_step.argtypes = [vp, vp, i32, i32, i32, vp, f32, i32, i32, vp, vp]
        L.beam_residual_step.restype = i32
        L.beam_status.argtypes = [vp]
        L.beam_status.restype = i32
        L.beam_last_error_string.argtypes = []
        L.beam_last_error_string.restype = ctypes.c_char_p
        L.beam_debug_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        L.beam_debug_wait_timeout.restype = i32
        L.beam_profile_enable.argtypes = [i32]
        L.beam_profile_enable.restype = None
        L.beam_profile_read.argtypes = [ctypes.c_char_p, sz, ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(i32), i32]
        L.beam_profile_read.restype = i32
        _lib = L
    return _lib


def _check(code: int):
    if code != BEAM_OK:
        raise BeamError(code, lib().beam_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_params(T, H, E, I, n_group=8, topk_group=4, top_k=8, routed_scale=2.5,
                rms_eps=1e-6, residual_k=0, flags=0) -> Params:
    return Params(T, H, E, I, n_group, topk_group, top_k, routed_scale, rms_eps, residual_k,
                  flags)


def workspace_size(p: Params) -> int:
    n = lib().beam_moe_workspace_size(ctypes.byref(p))
    if n == 0:
        raise BeamError(BEAM_ERR_INVALID_ARG, lib().beam_last_error_string().decode())
    return int(n)


def workspace_layout(p: Params) -> dict:
    arr = (ctypes.c_size_t * len(LAYOUT_NAMES))()
    n = lib().beam_moe_workspace_layout(ctypes.byref(p), arr, len(LAYOUT_NAMES))
    if n == 0:
        raise BeamError(BEAM_ERR_INVALID_ARG, lib().beam_last_error_string().decode())
    return {LAYOUT_NAMES[i]: int(arr[i]) for i in range(n)}


def dense_workspace_size(p: DenseParams) -> int:
    n = lib().beam_dense_workspace_size(ctypes.byref(p))
    if n == 0:
        raise BeamError(BEAM_ERR_INVALID_ARG, lib().beam_last_error_string().decode())
    return int(n)


def dense_workspace_layout(p: DenseParams) -> dict:
    arr = (ctypes.c_size_t * len(LAYOUT_NAMES))()
    n = lib().beam_dense_workspace_layout(ctypes.byref(p), arr, len(LAYOUT_NAMES))
    if n == 0:
        raise BeamError(BEAM_ERR_INVALID_ARG, lib().beam_last_error_string().decode())
    return {LAYOUT_NAMES[i]: int(arr[i]) for i in range(n)}


def alloc_workspace(p: Params, device="cuda") -> torch.Tensor:
    return torch.empty(workspace_size(p), dtype=torch.uint8, device=device)


def route(p: Params, x, w_router, bias=None, pre_gain=None, topk_idx=None, topk_w=None,
          scores=None, workspace=None, stream=None):
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((p.T, p.top_k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((p.T, p.top_k), dtype=torch.float32, device=dev)
    if scores is None and (p.flags & FLAG_RETURN_SCORES):
        scores = torch.empty((p.T, p.E), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(p, dev)
    _check(lib().beam_moe_route(ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(bias),
                                _ptr(pre_gain), _ptr(topk_idx), _ptr(topk_w), _ptr(scores),
                                _ptr(workspace), workspace.numel(), _stream(stream)))
    return topk_idx, topk_w, scores


def route_static(p: Params, x, w_router, bias=None, pre_gain=None, topk_idx=None,
                 topk_w=None, scores=None, stream=None):
    """beam_moe_route_static: the router with its scratch in a fixed array
    inside the library (no workspace, no allocation by the library)."""
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((p.T, p.top_k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((p.T, p.top_k), dtype=torch.float32, device=dev)
    if scores is None and (p.flags & FLAG_RETURN_SCORES):
        scores = torch.empty((p.T, p.E), dtype=torch.float32, device=dev)
    _check(lib().beam_moe_route_static(ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(bias),
                                       _ptr(pre_gain), _ptr(topk_idx), _ptr(topk_w),
                                       _ptr(scores), _stream(stream)))
    return topk_idx, topk_w, scores


def forward(p: Params, x, w_router, w_gate, w_up, w_down, bias=None, pre_gain=None,
            post_gain=None, out=None, topk_idx=None, topk_w=None, workspace=None, stream=None):
    dev = x.device
    if out is None:
        dt = torch.float32 if (p.flags & FLAG_FP32_OUT) else torch.bfloat16
        out = torch.empty((p.T, p.H), dtype=dt, device=dev)
    if workspace is None:
        workspace = alloc_workspace(p, dev)
    _check(lib().beam_moe_forward(ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(bias),
                                  _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(pre_gain),
                                  _ptr(post_gain), _ptr(out), _ptr(topk_idx), _ptr(topk_w),
                                  _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def forward_routed(p: Params, x, topk_idx, topk_w, w_gate, w_up, w_down, pre_gain=None,
                   post_gain=None, out=None, workspace=None, stream=None):
    """beam_moe_forward_routed: the sublayer with the routing given."""
    dev = x.device
    if out is None:
        dt = torch.float32 if (p.flags & FLAG_FP32_OUT) else torch.bfloat16
        out = torch.empty((p.T, p.H), dtype=dt, device=dev)
    if workspace is None:
        workspace = alloc_workspace(p, dev)
    _check(lib().beam_moe_forward_routed(ctypes.byref(p), _ptr(x), _ptr(topk_idx), _ptr(topk_w),
                                         _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(pre_gain),
                                         _ptr(post_gain), _ptr(out), _ptr(workspace),
                                         workspace.numel(), _stream(stream)))
    return out


def ep_dispatch(p: Params, n_ranks: int, x, topk_idx, workspace=None, stream=None):
    """beam_ep_dispatch: (send_x [T*k,H] bf16, send_expert [T*k], pair_row
    [T*k], send_counts [n_ranks]) for the pairs of this rank's tokens."""
    dev = x.device
    R = p.T * p.top_k
    send_x = torch.empty((R, p.H), dtype=torch.bfloat16, device=dev)
    send_expert = torch.empty(R, dtype=torch.int32, device=dev)
    pair_row = torch.empty(R, dtype=torch.int32, device=dev)
    send_counts = torch.zeros(n_ranks, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(p, dev)
    _check(lib().beam_ep_dispatch(ctypes.byref(p), n_ranks, _ptr(x), _ptr(topk_idx),
                                  _ptr(send_x), _ptr(send_expert), _ptr(pair_row),
                                  _ptr(send_counts), _ptr(workspace), workspace.numel(),
                                  _stream(stream)))
    return send_x, send_expert, pair_row, send_counts


def ep_combine(recv_y, pair_row, topk_w, h_prev=None, post_gain=None, eps=1e-6, residual_k=0,
               out_f32=False, out=None, stream=None):
    """beam_ep_combine: the source rank's weighted combine of the returned
    expert outputs, then the output or the post-norm + residual."""
    T, K = topk_w.shape
    H = recv_y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32 if out_f32 else torch.bfloat16,
                          device=recv_y.device)
    _check(lib().beam_ep_combine(T, K, H, _ptr(recv_y), _ptr(pair_row), _ptr(topk_w),
                                 _ptr(h_prev), _ptr(post_gain), eps, residual_k, int(out_f32),
                                 _ptr(out), _stream(stream)))
    return out


def dense_forward(T, H, I, x, w_gate, w_up, w_down, pre_gain=None, post_gain=None,
                  rms_eps=1e-6, residual_k=0, flags=0, out=None, workspace=None, stream=None):
    """beam_dense_mlp_forward: the dense SwiGLU MLP sublayer."""
    p = DenseParams(T, H, I, rms_eps, residual_k, flags)
    if out is None:
        dt = torch.float32 if (flags & FLAG_FP32_OUT) else torch.bfloat16
        out = torch.empty((T, H), dtype=dt, device=x.device)
    if workspace is None:
        workspace = torch.empty(dense_workspace_size(p), dtype=torch.uint8, device=x.device)
    _check(lib().beam_dense_mlp_forward(ctypes.byref(p), _ptr(x), _ptr(w_gate), _ptr(w_up),
                                        _ptr(w_down), _ptr(pre_gain), _ptr(post_gain), _ptr(out),
                                        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def quantize_e4m3_rows(w, stream=None):
    """beam_quantize_e4m3_rows over the last dimension of a bf16 tensor:
    returns (codes uint8 of w's shape, row scales fp32 of w.shape[:-1])."""
    K = w.shape[-1]
    rows = w.numel() // K if K else 0
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    sc = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _check(lib().beam_quantize_e4m3_rows(_ptr(w), rows, K, _ptr(q), _ptr(sc), _stream(stream)))
    return q, sc


def forward_fp8(p: Params, x, w_router, gate_q, up_q, down_q, bias=None, pre_gain=None,
                post_gain=None, out=None, topk_idx=None, topk_w=None, workspace=None,
                stream=None):
    """beam_moe_forward_fp8; gate_q, up_q, down_q are (codes, row scales)
    pairs as quantize_e4m3_rows returns them. p.flags must hold
    FLAG_FP8_EXPERTS."""
    dev = x.device
    if out is None:
        dt = torch.float32 if (p.flags & FLAG_FP32_OUT) else torch.bfloat16
        out = torch.empty((p.T, p.H), dtype=dt, device=dev)
    if workspace is None:
        workspace = alloc_workspace(p, dev)
    _check(lib().beam_moe_forward_fp8(
        ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(gate_q[0]), _ptr(gate_q[1]),
        _ptr(up_q[0]), _ptr(up_q[1]), _ptr(down_q[0]), _ptr(down_q[1]), _ptr(pre_gain),
        _ptr(post_gain), _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return out


def dense_forward_fp8(T, H, I, x, gate_q, up_q, down_q, pre_gain=None, post_gain=None,
                      rms_eps=1e-6, residual_k=0, flags=FLAG_FP8_EXPERTS, out=None,
                      workspace=None, stream=None):
    """beam_dense_mlp_forward_fp8; weights as (codes, row scales) pairs."""
    p = DenseParams(T, H, I, rms_eps, residual_k, flags)
    if out is None:
        dt = torch.float32 if (flags & FLAG_FP32_OUT) else torch.bfloat16
        out = torch.empty((T, H), dtype=dt, device=x.device)
    if workspace is None:
        workspace = torch.empty(dense_workspace_size(p), dtype=torch.uint8, device=x.device)
    _check(lib().beam_dense_mlp_forward_fp8(
        ctypes.byref(p), _ptr(x), _ptr(gate_q[0]), _ptr(gate_q[1]), _ptr(up_q[0]),
        _ptr(up_q[1]), _ptr(down_q[0]), _ptr(down_q[1]), _ptr(pre_gain), _ptr(post_gain),
        _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def quantize_nvfp4(w, rows_per_group=None, stream=None):
    """beam_quantize_nvfp4 over the last dimension of a bf16 tensor whose
    leading dimensions flatten to a multiple of 128 rows. rows_per_group
    defaults to the second-to-last dimension (one scale per matrix of a
    [E, N, K] expert tensor). Returns (codes uint8 [..., K/2], block scales
    uint8 [rows * K / 16] in the SF-group layout, group scales fp32)."""
    K = w.shape[-1]
    rows = w.numel() // K
    if rows_per_group is None:
        rows_per_group = w.shape[-2] if w.dim() >= 2 else rows
    codes = torch.empty(w.shape[:-1] + (K // 2,), dtype=torch.uint8, device=w.device)
    sf = torch.empty(rows * K // 16, dtype=torch.uint8, device=w.device)
    g = torch.empty(rows // rows_per_group, dtype=torch.float32, device=w.device)
    _check(lib().beam_quantize_nvfp4(_ptr(w), rows, K, rows_per_group, _ptr(codes), _ptr(sf),
                                     _ptr(g), _stream(stream)))
    return codes, sf, g


def forward_nvfp4(p: Params, x, w_router, gate_q, up_q, down_q, bias=None, pre_gain=None,
                  post_gain=None, out=None, topk_idx=None, topk_w=None, workspace=None,
                  stream=None):
    """beam_moe_forward_nvfp4; gate_q, up_q, down_q are (codes, block scales,
    group scales) as quantize_nvfp4 returns them. p.flags must hold
    FLAG_NVFP4_EXPERTS."""
    dev = x.device
    if out is None:
        dt = torch.float32 if (p.flags & FLAG_FP32_OUT) else torch.bfloat16
        out = torch.empty((p.T, p.H), dtype=dt, device=dev)
    if workspace is None:
        workspace = alloc_workspace(p, dev)
    _check(lib().beam_moe_forward_nvfp4(
        ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(bias),
        *[_ptr(t) for q in (gate_q, up_q, down_q) for t in q],
        _ptr(pre_gain), _ptr(post_gain), _ptr(out), _ptr(topk_idx), _ptr(topk_w),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def dense_forward_nvfp4(T, H, I, x, gate_q, up_q, down_q, pre_gain=None, post_gain=None,
                        rms_eps=1e-6, residual_k=0, flags=FLAG_NVFP4_EXPERTS, out=None,
                        workspace=None, stream=None):
    """beam_dense_mlp_forward_nvfp4; weights as (codes, block scales, group
    scales) triples."""
    p = DenseParams(T, H, I, rms_eps, residual_k, flags)
    if out is None:
        dt = torch.float32 if (flags & FLAG_FP32_OUT) else torch.bfloat16
        out = torch.empty((T, H), dtype=dt, device=x.device)
    if workspace is None:
        workspace = torch.empty(dense_workspace_size(p), dtype=torch.uint8, device=x.device)
    _check(lib().beam_dense_mlp_forward_nvfp4(
        ctypes.byref(p), _ptr(x), *[_ptr(t) for q in (gate_q, up_q, down_q) for t in q],
        _ptr(pre_gain), _ptr(post_gain), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out


def make_attn_params(T, H=5120, n_q=48, n_kv=8, head_dim=128, window=512, rope_theta=10000.0,
                     rms_eps=1e-6, residual_k=0, flags=0) -> AttnParams:
    return AttnParams(T, H, n_q, n_kv, head_dim, window, rope_theta, rms_eps, residual_k, flags)


def attention_workspace_size(p: AttnParams) -> int:
    n = lib().beam_attention_workspace_size(ctypes.byref(p))
    if n == 0:
        raise BeamError(BEAM_ERR_INVALID_ARG, lib().beam_last_error_string().decode())
    return int(n)


ATTN_LAYOUT_NAMES = ("x", "proj", "q", "k", "vt", "rope", "attn", "y", "units_qkvg", "units_o",
                     "n_units")


def attention_workspace_layout(p: AttnParams) -> dict:
    arr = (ctypes.c_size_t * len(ATTN_LAYOUT_NAMES))()
    n = lib().beam_attention_workspace_layout(ctypes.byref(p), arr, len(ATTN_LAYOUT_NAMES))
    if n == 0:
        raise BeamError(BEAM_ERR_INVALID_ARG, lib().beam_last_error_string().decode())
    return {ATTN_LAYOUT_NAMES[i]: int(arr[i]) for i in range(n)}


def attention_forward(p: AttnParams, h, w_qkvg, w_o, q_gain=None, k_gain=None, pre_gain=None,
                      post_gain=None, out=None, workspace=None, stream=None):
    """beam_attention_forward: the attention sublayer over one sequence."""
    if out is None:
        dt = torch.float32 if (p.flags & FLAG_FP32_OUT) else torch.bfloat16
        out = torch.empty((p.T, p.H), dtype=dt, device=h.device)
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(p), dtype=torch.uint8, device=h.device)
    _check(lib().beam_attention_forward(ctypes.byref(p), _ptr(h), _ptr(w_qkvg), _ptr(w_o),
                                        _ptr(q_gain), _ptr(k_gain), _ptr(pre_gain),
                                        _ptr(post_gain), _ptr(out), _ptr(workspace),
                                        workspace.numel(), _stream(stream)))
    return out


def residual_step(h_prev, sub_out, k, post_gain=None, eps=1e-6, apply_norm=True, out=None,
                  stream=None):
    T, H = h_prev.shape
    if out is None:
        out = torch.empty_like(h_prev)
    _check(lib().beam_residual_step(_ptr(h_prev), _ptr(sub_out), T, H, k, _ptr(post_gain),
                                    eps, int(bool(apply_norm)),
                                    int(sub_out.dtype == torch.float32), _ptr(out),
                                    _stream(stream)))
    return out


def status(stream=None) -> int:
    """Synchronise the stream and read (and clear) the device error flag."""
    code = lib().beam_status(_stream(stream))
    return int(code)


def last_error() -> str:
    return lib().beam_last_error_string().decode()


def debug_wait_timeout(timeout_ns: int, stream=None):
    _check(lib().beam_debug_wait_timeout(ctypes.c_uint64(timeout_ns), _stream(stream)))


def profile_enable(on: bool = True):
    """Bracket every library kernel launch with CUDA events (on its stream)."""
    lib().beam_profile_enable(1 if on else 0)


def profile_read() -> dict:
    """{kernel name: (total ms, launches)} since the last read; clears it."""
    n_max = 64
    names = ctypes.create_string_buffer(4096)
    ms = (ctypes.c_double * n_max)()
    cnt = (ctypes.c_int * n_max)()
    n = lib().beam_profile_read(names, 4096, ms, cnt, n_max)
    keys = names.value.decode().split("\n")[:n]
    return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(keys)}
