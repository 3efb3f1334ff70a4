"""PyTorch custom operators over the C ABI.

``torch.ops.ffpa.attn_fwd`` and ``torch.ops.ffpa.attn_varlen_fwd`` wrap
``ffpa_fwd`` / ``ffpa_fwd_varlen`` as opaque operators: torch.compile and
other tracers see one node with a shape-only fake implementation and never
look inside, and eager calls go straight to the CUDA kernels through the
binding.  ``ffpa_attn_func`` takes the argument list of
``torch.nn.functional.scaled_dot_product_attention`` (the FFPA API
reference, ``ffpa_attn.ffpa_attn_func``, uses the same list), so it can
replace that call for the supported cases: bf16/fp16 CUDA tensors,
64 <= D <= 1024 with D % 8 == 0 (D % 64 == 0 for varlen and for the
backward), no dropout.  The dense operator is
differentiable through ``ffpa_bwd`` (the backward kernels; a mask enters
the recomputed scores, but no gradient is formed for the mask itself), and
the varlen operator through ``ffpa_bwd_varlen``.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _binding


@torch.library.custom_op("ffpa::attn_fwd", mutates_args=())
def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, attn_mask: Optional[torch.Tensor],
             is_causal: bool, scale: Optional[float],
             enable_gqa: bool) -> tuple[torch.Tensor, torch.Tensor]:
    """O [B,Hq,Nq,D] and LSE [B,Hq,Nq] (fp32) of exact attention."""
    return _binding.ffpa_fwd(q, k, v, attn_mask=attn_mask, is_causal=is_causal, scale=scale,
                             enable_gqa=enable_gqa, return_lse=True)


@attn_fwd.register_fake
def _attn_fwd_fake(q, k, v, attn_mask, is_causal, scale, enable_gqa):
    B, Hq, Nq, _ = q.shape
    return (torch.empty_like(q, memory_format=torch.contiguous_format),
            q.new_empty((B, Hq, Nq), dtype=torch.float32))


def _attn_fwd_setup_context(ctx, inputs, output):
    q, k, v, attn_mask, is_causal, scale, enable_gqa = inputs
    o, lse = output
    ctx.save_for_backward(q, k, v, o, lse, attn_mask)
    ctx.is_causal, ctx.scale, ctx.enable_gqa = is_causal, scale, enable_gqa
    # An output the loss does not use arrives in backward as None (not as a
    # tensor of zeros), so the LSE check below needs no device read.
    ctx.set_materialize_grads(False)


def _check_grads(grad_o, grad_lse):
    if grad_lse is not None:
        raise NotImplementedError("gradients through the returned LSE are not supported")
    if grad_o is None:
        raise NotImplementedError("backward without a gradient for O")


def _attn_fwd_backward(ctx, grad_o, grad_lse):
    if ctx.needs_input_grad[3]:
        raise NotImplementedError("no gradient is formed for attn_mask")
    _check_grads(grad_o, grad_lse)
    q, k, v, o, lse, attn_mask = ctx.saved_tensors
    dq, dk, dv = _binding.ffpa_bwd(grad_o.contiguous(), q, k, v, o, lse, is_causal=ctx.is_causal,
                                   scale=ctx.scale, enable_gqa=ctx.enable_gqa, attn_mask=attn_mask)
    return dq, dk, dv, None, None, None, None


attn_fwd.register_autograd(_attn_fwd_backward, setup_context=_attn_fwd_setup_context)


@torch.library.custom_op("ffpa::attn_varlen_fwd", mutates_args=())
def attn_varlen_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                    cu_seqlens_k: Optional[torch.Tensor], max_seqlen_q: int, max_seqlen_k: int,
                    causal: bool, softmax_scale: Optional[float],
                    enable_gqa: bool) -> tuple[torch.Tensor, torch.Tensor]:
    """O [Tq,Hq,D] and LSE [Hq,Tq] (fp32) of packed variable-length attention."""
    return _binding.ffpa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                                    max_seqlen_k, causal=causal, softmax_scale=softmax_scale,
                                    enable_gqa=enable_gqa, return_lse=True)


@attn_varlen_fwd.register_fake
def _attn_varlen_fwd_fake(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal,
                          softmax_scale, enable_gqa):
    Tq, Hq, _ = q.shape
    return (torch.empty_like(q, memory_format=torch.contiguous_format),
            q.new_empty((Hq, Tq), dtype=torch.float32))


def _attn_varlen_setup_context(ctx, inputs, output):
    (q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, softmax_scale,
     enable_gqa) = inputs
    o, lse = output
    ctx.save_for_backward(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k)
    ctx.max_q, ctx.max_k = max_seqlen_q, max_seqlen_k
    ctx.causal, ctx.scale, ctx.enable_gqa = causal, softmax_scale, enable_gqa
    ctx.set_materialize_grads(False)


def _attn_varlen_backward(ctx, grad_o, grad_lse):
    _check_grads(grad_o, grad_lse)
    q, k, v, o, lse, cu_q, cu_k = ctx.saved_tensors
    dq, dk, dv = _binding.ffpa_bwd_varlen(grad_o.contiguous(), q, k, v, o, lse, cu_q, cu_k,
                                          ctx.max_q, ctx.max_k, softmax_scale=ctx.scale,
                                          causal=ctx.causal, enable_gqa=ctx.enable_gqa)
    return dq, dk, dv, None, None, None, None, None, None, None


attn_varlen_fwd.register_autograd(_attn_varlen_backward, setup_context=_attn_varlen_setup_context)


def ffpa_attn_func(query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                   attn_mask: Optional[torch.Tensor] = None, dropout_p: float = 0.0,
                   is_causal: bool = False, scale: Optional[float] = None,
                   enable_gqa: bool = False, *, return_lse: bool = False):
    """Drop-in for ``F.scaled_dot_product_attention`` on [B,H,N,D] tensors.

    Causal masking is tail-aligned (query row r sees keys k <= r + Nkv - Nq),
    which equals SDPA's top-left alignment when Nq == Nkv.  Returns O, or
    (O, LSE) with return_lse."""
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not supported by this forward kernel")
    o, lse = torch.ops.ffpa.attn_fwd(query, key, value, attn_mask, bool(is_causal), scale,
                                     bool(enable_gqa))
    return (o, lse) if return_lse else o


def ffpa_attn_varlen_func(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                          cu_seqlens_q: torch.Tensor, cu_seqlens_k: Optional[torch.Tensor],
                          max_seqlen_q: int, max_seqlen_k: int, dropout_p: float = 0.0,
                          softmax_scale: Optional[float] = None, causal: bool = False,
                          enable_gqa: bool = False, *, return_lse: bool = False):
    """Packed THD variable-length forward (q [Tq,Hq,D], k/v [Tk,Hkv,D])."""
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not supported by this forward kernel")
    o, lse = torch.ops.ffpa.attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, int(max_seqlen_q),
                                            int(max_seqlen_k), bool(causal), softmax_scale,
                                            bool(enable_gqa))
    return (o, lse) if return_lse else o
