"""torch.autograd.Function over the C ABI.

Mirrors the wrapper on "Triton 05: Flash Attention", section torch.autograd.Function
래핑: the forward saves q, k, v, o and the logsumexp (never S or P), the backward
returns dq, dk, dv and None for the causal flag; sm_scale defaults to d ** -0.5.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import binding


class FlashAttentionFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal: bool = False, scale: Optional[float] = None):
        scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
        o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal = causal
        ctx.scale = scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, do.contiguous(), causal=ctx.causal,
                                      scale=ctx.scale)
        return dq, dk, dv, None, None


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
              scale: Optional[float] = None) -> torch.Tensor:
    """Differentiable exact attention over [B, H, N, d] fp16/bf16 CUDA tensors."""
    return FlashAttentionFunction.apply(q, k, v, causal, scale)


class VarlenAttentionFunction(torch.autograd.Function):
    """The same pair over sequences packed along the token axis (cu_seqlens boundaries)."""

    @staticmethod
    def forward(ctx, q, k, v, cu_q, cu_k, max_q: int, max_k: int, causal: bool = False,
                scale: Optional[float] = None, cu_q_host=None, cu_k_host=None):
        scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
        o, lse = binding.attn_fwd_varlen(q, k, v, cu_q, cu_k, max_q, max_k, causal=causal,
                                         scale=scale, cu_seqlens_q_host=cu_q_host,
                                         cu_seqlens_k_host=cu_k_host)
        ctx.save_for_backward(q, k, v, o, lse, cu_q, cu_k)
        ctx.max_q, ctx.max_k, ctx.causal, ctx.scale = max_q, max_k, causal, scale
        ctx.host = (cu_q_host, cu_k_host)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, cu_q, cu_k = ctx.saved_tensors
        dq, dk, dv = binding.attn_bwd_varlen(q, k, v, o, lse, do.contiguous(), cu_q, cu_k,
                                             ctx.max_q, ctx.max_k, causal=ctx.causal,
                                             scale=ctx.scale, cu_seqlens_q_host=ctx.host[0],
                                             cu_seqlens_k_host=ctx.host[1])
        return dq, dk, dv, None, None, None, None, None, None, None, None


def attention_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                     cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, max_seqlen_q: int,
                     max_seqlen_k: int, causal: bool = False, scale: Optional[float] = None,
                     cu_seqlens_q_host: Optional[torch.Tensor] = None,
                     cu_seqlens_k_host: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Differentiable exact attention over packed [total, H, d] sequences (int32 device
    cu_seqlens of B + 1 entries, and optionally their CPU copies, which only order the work;
    see binding.attn_fwd_varlen)."""
    return VarlenAttentionFunction.apply(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                                         max_seqlen_k, causal, scale, cu_seqlens_q_host,
                                         cu_seqlens_k_host)
