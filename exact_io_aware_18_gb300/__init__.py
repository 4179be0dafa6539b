"""Exact IO-aware attention for GB300 (sm_103a): forward and backward.

The compute lives in libfa.so (hand-written CUDA: tcgen05 tensor cores, TMEM
accumulators, TMA copies) behind the C ABI of ``include/fa.h``; this package
is its thin Python binding.  PyTorch only supplies device memory and streams.

    from exact_io_aware_18_gb300 import attention_fwd, attention_bwd
    o, lse = attention_fwd(q, k, v, causal=True)           # bf16 [B,H,N,d]
    dq, dk, dv = attention_bwd(q, k, v, o, do, lse, causal=True)
"""

from __future__ import annotations

import math

import torch

from . import _lib
from ._lib import (FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT, FA_ERR_INVALID_ARG, FA_ERR_MISALIGNED,
                   FA_ERR_NO_MEMORY, FA_ERR_UNSUPPORTED, FA_OK, FaError, error_string, fa_bwd,
                   fa_bwd_dkdv, fa_bwd_dq, fa_bwd_dq_preprocess, fa_bwd_f32, fa_bwd_gqa,
                   fa_bwd_noalloc, fa_bwd_preprocess, fa_bwd_workspace_bytes, fa_device_status,
                   fa_fp8_quantize, fa_fwd, fa_fwd_f32, fa_fwd_fp8, fa_fwd_gqa, fa_fwd_splitkv,
                   fa_fwd_splitkv_workspace_bytes, fa_selftest_wait_timeout,
                   fa_set_wait_timeout_ns, lib_path, load)

__all__ = [
    "attention_fwd", "attention_bwd", "fa_fwd", "fa_bwd", "fa_bwd_preprocess", "fa_bwd_dkdv",
    "fa_bwd_dq", "fa_bwd_dq_preprocess", "fa_bwd_noalloc", "fa_fwd_gqa", "fa_bwd_gqa",
    "fa_fwd_splitkv",
    "fa_fwd_splitkv_workspace_bytes", "attention_decode", "fa_fp8_quantize", "fa_fwd_fp8",
    "fp8_quantize", "attention_fwd_fp8",
    "fa_bwd_workspace_bytes", "fa_fwd_f32", "fa_bwd_f32", "fa_device_status",
    "fa_set_wait_timeout_ns", "fa_selftest_wait_timeout", "FaError", "error_string", "load",
    "lib_path", "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED",
    "FA_ERR_CUDA", "FA_ERR_DEVICE_TIMEOUT", "FA_ERR_NO_MEMORY",
]


def default_scale(d: int) -> float:
    """1/sqrt(d) rounded to the float the C ABI receives."""
    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))


def attention_fwd(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocates O and LSE and runs fa_fwd (bf16) or fa_fwd_f32 (fp32).

    With fewer K/V heads than query heads (bf16 only), grouped-query
    attention: fa_fwd_gqa.
    """
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if q.dtype == torch.float32:
        fa_fwd_f32(q, k, v, o, lse, causal, scale, stream)
    elif k.shape[1] != H:
        fa_fwd_gqa(q, k, v, o, lse, causal, scale, stream)
    else:
        fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def attention_decode(q, k, v, scale: float | None = None, n_splits: int = 0, workspace=None,
                     stream=None):
    """Allocates O and LSE and runs fa_fwd_splitkv: few queries [B,Hq,Nq,d] against
    many keys [B,Hkv,Nk,d], every query reading every key."""
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd_splitkv(q, k, v, o, lse, scale, n_splits, workspace, stream)
    return o, lse


def fp8_quantize(x, signs, stream=None):
    """Allocates and returns (codes uint8 [B,H,N,d], scales float32 [B,H,ceil(N/128)]):
    x (bf16) rotated by diag(signs) H / sqrt(d), E4M3 per 128-row tile."""
    B, H, N, d = x.shape
    codes = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    scales = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=x.device)
    fa_fp8_quantize(x, signs, codes, scales, stream)
    return codes, scales


def attention_fwd_fp8(q, k, v, signs, causal: bool = False, scale: float | None = None,
                      stream=None):
    """FP8 forward with incoherent processing: Q and K (bf16) rotated and
    quantised with fa_fp8_quantize, then fa_fwd_fp8 (V stays bf16).  Returns
    O (bf16) and LSE (float32)."""
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    signs = _lib._host_signs(signs, d)
    q8, qs = fp8_quantize(q, signs, stream)
    k8, ks = fp8_quantize(k, signs, stream)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd_fp8(q8, qs, k8, ks, v, o, lse, causal, scale, stream)
    return o, lse


def attention_bwd(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
                  workspace=None, stream=None):
    """Allocates FP32 dQ, dK, dV and runs fa_bwd (bf16) or fa_bwd_f32 (fp32).

    With fewer K/V heads than query heads (bf16 only): fa_bwd_gqa, and dK, dV
    have the K/V heads' shape.
    """
    d = q.shape[-1]
    scale = default_scale(d) if scale is None else scale
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty_like(dk)
    if q.dtype == torch.float32:
        fa_bwd_f32(q, k, v, o, do, lse, dq, dk, dv, causal, scale, workspace, stream)
    elif k.shape[1] != q.shape[1]:
        fa_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, causal, scale, workspace, stream)
    else:
        fa_bwd(q, k, v, o, do, lse, dq, dk, dv, causal, scale, workspace, stream)
    return dq, dk, dv
