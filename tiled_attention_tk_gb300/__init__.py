"""GB300-native (sm_103a) fused attention forward.

``fwd(q, k, v, causal, scale) -> (O, LSE)`` computes, per (batch, head),
O = softmax(scale QK^T [+ causal mask]) V and the natural-log row
log-sum-exp (queries and keys of equal length, or Nq queries at the end of
Nkv keys) in one CUDA kernel (TMA producer, tcgen05 MMAs into tensor
memory, online softmax), through the C ABI declared in include/tk_attn.h.
PyTorch only provides device memory and streams.
"""
from ._lib import STATUS, STATUS_NAMES, TkError, library_path, load, strerror
from .attention import (based, bwd, bwd_workspace_bytes, device_status, fwd, fwd_kv_raw, fwd_raw, fwd_workspace_bytes,
                        fwd_ws_raw, gemm, gemm_uses_pairs, gemm_workspace_bytes, hedgehog, selftest_timeout, based_workspace_bytes,
                        hedgehog_workspace_bytes)

__all__ = ["fwd", "fwd_raw", "fwd_kv_raw", "fwd_ws_raw", "fwd_workspace_bytes", "bwd", "gemm", "gemm_uses_pairs", "gemm_workspace_bytes", "based", "based_workspace_bytes", "hedgehog", "hedgehog_workspace_bytes", "bwd_workspace_bytes", "device_status", "selftest_timeout", "TkError", "STATUS",
           "STATUS_NAMES", "library_path", "load", "strerror"]
