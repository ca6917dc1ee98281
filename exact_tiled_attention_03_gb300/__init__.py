"""GB300-native exact attention forward (sm_103a CUDA behind a C ABI).

The kernels live in ``lib/libfa_gb300.so`` (built from ``csrc/`` by
``build.py``); ``_capi`` binds the C entry points by name. ``attention``
is the convenience call: it allocates O and LSE with torch (device memory
is the only thing torch provides here) and runs ``fa_forward`` on the
current stream.
"""
from __future__ import annotations

from ._capi import (FA_ERR_CUDA, FA_ERR_INVALID_ARG, FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED,
                    FA_ERR_WORKSPACE, FA_OK, FA_VERIFY_MAX_SQ, FAError, check, fa_backward,
                    fa_backward_workspace_size, fa_device_status,
                    fa_forward, fa_forward_fp8, fa_forward_ws, fa_prefill_forward,
                    fa_status_string,
                    fa_verify_auto_splits, fa_verify_forward, fa_verify_workspace_size,
                    fa_workspace_size, load)

__all__ = [
    "attention", "attention_fp8", "attention_backward", "fa_backward",
    "fa_backward_workspace_size", "fa_forward", "fa_forward_fp8", "fa_forward_ws", "fa_prefill_forward", "fa_verify_forward",
    "fa_workspace_size", "fa_verify_workspace_size", "fa_verify_auto_splits", "fa_status_string",
    "fa_device_status", "FAError", "check", "load", "FA_OK", "FA_ERR_INVALID_ARG",
    "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT", "FA_ERR_WORKSPACE", "FA_VERIFY_MAX_SQ",
]


def attention(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """O, LSE = attention(Q, K, V) for contiguous bf16 CUDA tensors [B, H, S, d].

    Returns O (bf16, like q) and LSE (fp32 [B, H, Sq]). Raises FAError on a
    non-OK status.
    """
    import math

    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor [B, H, S, d]")
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    check(fa_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream), "fa_forward")
    return o, lse


def attention_fp8(q8, k8, v8, causal: bool = False, scale: float | None = None,
                  descale=(1.0, 1.0, 1.0), stream=None):
    """O, LSE for contiguous E4M3 CUDA tensors [B, H, S, 128] (torch.float8_e4m3fn
    or uint8 bytes) with per-tensor descales (q, k, v); runs ``fa_forward_fp8``.

    Returns O (bf16 [B, H, Sq, 128]) and LSE (fp32 [B, H, Sq]). Raises FAError on a
    non-OK status.
    """
    import math

    import torch

    for name, t in (("q", q8), ("k", k8), ("v", v8)):
        if (t.dtype not in (torch.float8_e4m3fn, torch.uint8) or not t.is_cuda
                or not t.is_contiguous() or t.dim() != 4):
            raise ValueError(f"{name} must be a contiguous 4-D E4M3 CUDA tensor [B, H, S, d]")
    if scale is None:
        scale = 1.0 / math.sqrt(q8.shape[-1])
    B, H, Sq, d = q8.shape
    Sk = k8.shape[2]
    o = torch.empty((B, H, Sq, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q8.device)
    check(fa_forward_fp8(q8, k8, v8, o, lse, B, H, Sq, Sk, d, causal, scale, descale[0],
                         descale[1], descale[2], stream), "fa_forward_fp8")
    return o, lse


def attention_backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None,
                       stream=None):
    """dQ, dK, dV of O = attention(Q, K, V) given the forward's O and LSE and the
    upstream gradient dO (contiguous bf16 CUDA tensors [B, H, S, d]; LSE fp32
    [B, H, Sq] as ``attention`` returns it); runs ``fa_backward`` with a
    workspace from the stream-ordered allocator. Raises FAError on a non-OK
    status.
    """
    import math

    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor [B, H, S, d]")
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    check(fa_backward(q, k, v, o, lse, do, dq, dk, dv, B, H, Sq, Sk, d, causal, scale, None, 0,
                      stream), "fa_backward")
    return dq, dk, dv
