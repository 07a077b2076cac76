"""Exact scaled-dot-product attention for GB300 (sm_103a), behind a small C ABI.

``fa_fwd`` / ``fa_bwd`` and friends mirror include/fa.h one to one (see
``_lib``). ``forward`` and ``backward`` are conveniences that allocate outputs
and workspace with torch and call them; torch is used for device memory and
streams only.
"""
from __future__ import annotations

import math

from ._lib import (FAError, fa_accumulate, fa_bwd, fa_bwd_noalloc,  # noqa: F401
                   fa_bwd_varlen, fa_bwd_workspace_bytes, fa_debug_set, fa_debug_set_events,
                   fa_debug_set_trace, fa_fwd, fa_fwd_fp8, fa_fwd_varlen, fa_get_device_error,
                   fa_merge, fa_quantize_fp8, fa_to_bf16, load)


def _dims(q, k, cu_seqlens):
    if cu_seqlens is not None:
        T, Hq, d = q.shape
        return cu_seqlens.numel() - 1, Hq, k.shape[1], T, k.shape[0], d
    B, Sq, Hq, d = q.shape
    return B, Hq, k.shape[2], Sq, k.shape[1], d


def forward(q, k, v, causal=False, scale=None, cu_seqlens=None, out=None, lse=None, stream=None,
            cu_seqlens_k=None):
    """O, LSE for bf16 q/k/v ([B,S,H,d] dense or [T,H,d] packed with int32 cu_seqlens;
    cu_seqlens_k gives the keys their own boundaries, k/v then [Tk,Hkv,d])."""
    import torch
    B, Hq, Hkv, Sq, Sk, d = _dims(q, k, cu_seqlens)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        shape = (Hq, Sq) if cu_seqlens is not None else (B, Hq, Sq)
        lse = torch.empty(shape, dtype=torch.float32, device=q.device)
    if cu_seqlens_k is not None:
        fa_fwd_varlen(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, cu_seqlens,
                      cu_seqlens_k, stream)
    else:
        fa_fwd(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, cu_seqlens, stream)
    return out, lse


def backward(q, k, v, o, lse, dout, causal=False, scale=None, cu_seqlens=None, workspace=None,
             stream=None, cu_seqlens_k=None):
    """dQ, dK, dV (bf16) for the forward above."""
    import torch
    B, Hq, Hkv, Sq, Sk, d = _dims(q, k, cu_seqlens)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nbytes = fa_bwd_workspace_bytes(B, Hq, Sq, d, Sq if cu_seqlens is not None else 0)
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if cu_seqlens_k is not None:
        fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale,
                      cu_seqlens, cu_seqlens_k, workspace, nbytes, stream)
    else:
        fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale,
               cu_seqlens, workspace, nbytes, stream)
    return dq, dk, dv


def quantize_fp8(x, layout):
    """e4m3 codes and scales of a bf16 [B,S,H,d] tensor: layout 0 (Q, K) gives
    codes [B,S,H,d] and scales [B,H,ceil(S/128)]; layout 1 (V) gives codes
    [B,H,d,S_pad] (keys contiguous, S_pad = S rounded up to 16) and scales [B,H]."""
    import torch
    B, S, H, d = x.shape
    if layout == 0:
        codes = torch.empty((B, S, H, d), dtype=torch.uint8, device=x.device)
        scales = torch.empty((B, H, (S + 127) // 128), dtype=torch.float32, device=x.device)
    else:
        codes = torch.empty((B, H, d, (S + 15) // 16 * 16), dtype=torch.uint8, device=x.device)
        scales = torch.empty((B, H), dtype=torch.float32, device=x.device)
    fa_quantize_fp8(x, B, S, H, d, layout, codes, scales)
    return codes, scales


def forward_fp8(q8, q_scale, k8, k_scale, vt8, v_scale, causal=False, scale=None, out=None,
                lse=None, stream=None):
    """O (bf16), LSE for e4m3 inputs from quantize_fp8 (dense layouts, d = 128)."""
    import torch
    B, Sq, Hq, d = q8.shape
    Sk, Hkv = k8.shape[1], k8.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = torch.empty((B, Sq, Hq, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q8.device)
    fa_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, out, lse, B, Hq, Hkv, Sq, Sk, d, causal,
               scale, stream)
    return out, lse
