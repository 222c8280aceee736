"""Beam MoE sublayer on one B300 (sm_103a): Python binding of libbeam_moe.so.

The layer (router, group-limited top-8, normalised x2.5 weights, token
permutation, SwiGLU experts, weighted combine, post-RMSNorm and the scaled
residual update; BF16, E4M3 or NVFP4 expert weights), the dense MLP and the
attention sublayer runs in the library's CUDA kernels; this package only
marshals torch tensors into the C ABI declared in include/beam_moe.h.
"""
from ._native import (BeamError, Params, make_params, workspace_size, workspace_layout,
                      alloc_workspace, route, route_static, forward, dense_forward, DenseParams, residual_step, status, last_error,
                      debug_wait_timeout, lib, LIB_PATH, EXPORTED, FLAG_PRE_NORM,
                      FLAG_FP32_OUT, FLAG_RETURN_SCORES, FLAG_FP8_EXPERTS, profile_enable,
                      profile_read, quantize_e4m3_rows, forward_fp8, dense_forward_fp8,
                      dense_workspace_size, dense_workspace_layout, FLAG_NVFP4_EXPERTS,
                      quantize_nvfp4, forward_nvfp4, dense_forward_nvfp4, AttnParams,
                      make_attn_params, attention_workspace_size, attention_forward,
                      attention_workspace_layout, FLAG_PREFILL_WEIGHT_MAJOR, forward_routed,
                      ep_dispatch, ep_combine)

__all__ = ["BeamError", "Params", "make_params", "workspace_size", "workspace_layout",
           "alloc_workspace", "route", "route_static", "forward", "dense_forward", "DenseParams", "residual_step", "status", "last_error",
           "debug_wait_timeout", "lib", "LIB_PATH", "EXPORTED", "FLAG_PRE_NORM",
           "FLAG_FP32_OUT", "FLAG_RETURN_SCORES", "FLAG_FP8_EXPERTS", "profile_enable",
           "profile_read", "quantize_e4m3_rows", "forward_fp8", "dense_forward_fp8",
           "dense_workspace_size", "dense_workspace_layout", "FLAG_NVFP4_EXPERTS",
           "quantize_nvfp4", "forward_nvfp4", "dense_forward_nvfp4", "AttnParams",
           "make_attn_params", "attention_workspace_size", "attention_forward",
           "attention_workspace_layout", "FLAG_PREFILL_WEIGHT_MAJOR", "forward_routed",
           "ep_dispatch", "ep_combine"]
