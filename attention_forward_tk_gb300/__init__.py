"""GB300-native fused attention forward.

O = softmax(scale * Q K^T [+ causal mask]) V with the per-row log-sum-exp, on
bf16 [B, H, N, D] tensors, computed by hand-written sm_103a CUDA kernels behind
a C ABI (``include/tk_attn.h``).  This package is the thin Python binding over
that library: argument marshalling only.  The shared library is loaded on first
use; if it is missing or cannot be loaded, every call raises.  The library
also holds the backward pass (dQ, dK, dV), Based linear attention and a bf16
GEMM (C = A B^T) on the same TMA / tensor-core pipeline.
"""
from .api import (  # noqa: F401
    TkAttnError,
    attention,
    attention_backward,
    attention_forward,
    attention_forward_host,
    attention_forward_splitkv,
    based_forward,
    gemm_bf16,
    last_device_error,
    library,
    status_string,
    tk_attn_bwd,
    tk_attn_bwd_check_args,
    tk_attn_bwd_workspace_bytes,
    tk_attn_check_args,
    tk_attn_fwd,
    tk_attn_fwd_host,
    tk_attn_fwd_host_check_args,
    tk_attn_fwd_host_workspace_bytes,
    tk_attn_fwd_qk,
    tk_attn_fwd_splitkv,
    tk_attn_last_device_error,
    tk_attn_splitkv_workspace_bytes,
    tk_attn_status_string,
    tk_attn_version,
    tk_based_check_args,
    tk_based_fwd,
    tk_based_fwd_linear,
    tk_gemm_bf16,
    tk_gemm_bf16_check_args,
    version,
)
