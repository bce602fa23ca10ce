"""Differentiable entry points over the C ABI: ``varlen_attention`` and flash_attn-style wrappers.

mtlattn 0.3.0 ("Use") names ``varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_kv,
max_seqlen_q, scale=None, causal=False)`` with a sliding ``window`` and an additive
``attn_bias`` (a bool mask becomes a 0 / -inf bias; a bias that requires grad is refused), and
differentiable flash_attn-compatible wrappers ``flash_attn_varlen_qkvpacked_func(qkv,
cu_seqlens, max_seqlen)`` and ``flash_attn_varlen_kvpacked_func(q, kv, cu_q, cu_k, max_q,
max_k)``; and ``latent_attention`` on split nope / rope operands.  Everything here is argument marshalling and autograd plumbing: the forward and the
backward are the library's kernels (``vlf_attn_varlen_fwd`` / ``vlf_attn_varlen_bwd``).

flash_attn's ``window_size=(left, right)`` counts keys on each side of the diagonal; the window
of this library is the pages' "last W keys" (W keys ending at the diagonal), so ``(left, 0)``
under causal masking, or ``(left, -1)`` without it (only a lower bound), is W = left + 1.  Other
window shapes, dropout, ALiBi slopes and returning the probabilities are refused rather than
approximated.
"""
from __future__ import annotations

import torch

from . import (VLF_ERR_INVALID, VLF_ERR_UNSUPPORTED, VlfError, vlf_attn_varlen_bwd,
               vlf_attn_varlen_bwd_latent, vlf_attn_varlen_fwd, vlf_attn_varlen_fwd_latent,
               vlf_bias_bands)


def mask_to_bias(mask: torch.Tensor) -> torch.Tensor:
    """A bool mask (True: the pair takes part) as the additive fp32 bias the kernels take:
    0 where True, -inf where False.  Other dtypes are returned as fp32 unchanged."""
    if mask.dtype == torch.bool:
        bias = torch.zeros(mask.shape, dtype=torch.float32, device=mask.device)
        return bias.masked_fill_(~mask, float("-inf"))
    return mask.float() if mask.dtype != torch.float32 else mask


def window_from_flash(window_size, causal: bool) -> int:
    """flash_attn ``window_size=(left, right)`` -> this library's window W (0: none)."""
    if window_size is None:
        return 0
    left, right = int(window_size[0]), int(window_size[1])
    if left < 0 and right < 0:
        return 0
    if left >= 0 and ((causal and right in (0, -1)) or (not causal and right < 0)):
        return left + 1
    raise VlfError(VLF_ERR_UNSUPPORTED, f"window_size={tuple(window_size)} with causal={causal}: "
                   "only a window ending at the diagonal is supported")


class _VarlenAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q, max_seqlen_kv, scale,
                causal, window, bias):
        # the bias bands (which keys the bias leaves each row) serve the forward and backward
        bands = None if bias is None else vlf_bias_bands(bias, cu_seqlens_q, cu_seqlens_kv)
        out, lse = vlf_attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q,
                                       max_seqlen_kv, scale=scale, causal=causal, window=window,
                                       bias=bias, bias_bands=bands)
        ctx.save_for_backward(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_kv)
        ctx.bias, ctx.bands = bias, bands
        ctx.args = (max_seqlen_q, max_seqlen_kv, scale, causal, window)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse, cu_q, cu_kv = ctx.saved_tensors
        max_q, max_kv, scale, causal, window = ctx.args
        dq, dk, dv = vlf_attn_varlen_bwd(dout.contiguous(), q, k, v, out, lse, cu_q, cu_kv,
                                         max_q, max_kv, scale=scale, causal=causal,
                                         window=window, bias=ctx.bias, bias_bands=ctx.bands)
        return dq, dk, dv, None, None, None, None, None, None, None, None


def varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q, max_seqlen_kv=None,
                     scale=None, causal=False, window=0, attn_bias=None):
    """Attention over packed variable-length sequences (mtlattn 0.3.0, "Use"), differentiable in
    q, k and v.  q [total_q, H_q, D_qk], k [total_kv, H_kv, D_qk], v [total_kv, H_kv, D_v];
    ``attn_bias`` fp32 (or bool mask) [total_q, H_q or 1, max_seqlen_kv], constant."""
    bias = None
    if attn_bias is not None:
        if attn_bias.requires_grad:
            raise VlfError(VLF_ERR_UNSUPPORTED, "the bias is treated as a constant; a bias that "
                           "requires grad is refused")
        bias = mask_to_bias(attn_bias).contiguous()
        if max_seqlen_kv is None:
            max_seqlen_kv = int(bias.shape[2])
    if max_seqlen_kv is None:
        max_seqlen_kv = int((cu_seqlens_kv[1:] - cu_seqlens_kv[:-1]).max().item()) \
            if cu_seqlens_kv.numel() > 1 else 0
    return _VarlenAttention.apply(q.contiguous(), k.contiguous(), v.contiguous(), cu_seqlens_q,
                                  cu_seqlens_kv, int(max_seqlen_q), int(max_seqlen_kv), scale,
                                  bool(causal), int(window or 0), bias)


class _LatentAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q_nope, q_rope, k_nope, k_rope, v, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q,
                max_seqlen_kv, scale, causal, window, bias):
        out, lse = vlf_attn_varlen_fwd_latent(q_nope, q_rope, k_nope, k_rope, v, cu_seqlens_q,
                                              cu_seqlens_kv, max_seqlen_q, max_seqlen_kv,
                                              scale=scale, causal=causal, window=window, bias=bias)
        ctx.save_for_backward(q_nope, q_rope, k_nope, k_rope, v, out, lse, cu_seqlens_q,
                              cu_seqlens_kv)
        ctx.bias = bias
        ctx.args = (max_seqlen_q, max_seqlen_kv, scale, causal, window)
        return out

    @staticmethod
    def backward(ctx, dout):
        q_nope, q_rope, k_nope, k_rope, v, out, lse, cu_q, cu_kv = ctx.saved_tensors
        max_q, max_kv, scale, causal, window = ctx.args
        grads = vlf_attn_varlen_bwd_latent(dout.contiguous(), q_nope, q_rope, k_nope, k_rope, v,
                                           out, lse, cu_q, cu_kv, max_q, max_kv, scale=scale,
                                           causal=causal, window=window, bias=ctx.bias)
        return (*grads, None, None, None, None, None, None, None, None)


def latent_attention(q_nope, q_rope, k_nope, k_rope, v, cu_seqlens_q, cu_seqlens_kv,
                     max_seqlen_q, max_seqlen_kv=None, scale=None, causal=False, window=0,
                     attn_bias=None):
    """Latent attention with split operands (triton-msl part 2, "Latent attention"),
    differentiable in all five: score = q_nope . k_nope + q_rope . k_rope (contraction 192 =
    128 + 64), output width 128.  k_rope [total_kv, 1 or H_kv, 64]: one rope key may serve every
    head (its gradient is then summed over heads).  ``attn_bias`` as in varlen_attention."""
    bias = None
    if attn_bias is not None:
        if attn_bias.requires_grad:
            raise VlfError(VLF_ERR_UNSUPPORTED, "the bias is treated as a constant; a bias that "
                           "requires grad is refused")
        bias = mask_to_bias(attn_bias).contiguous()
        if max_seqlen_kv is None:
            max_seqlen_kv = int(bias.shape[2])
    if max_seqlen_kv is None:
        max_seqlen_kv = int((cu_seqlens_kv[1:] - cu_seqlens_kv[:-1]).max().item()) \
            if cu_seqlens_kv.numel() > 1 else 0
    return _LatentAttention.apply(q_nope.contiguous(), q_rope.contiguous(), k_nope.contiguous(),
                                  k_rope.contiguous(), v.contiguous(), cu_seqlens_q,
                                  cu_seqlens_kv, int(max_seqlen_q), int(max_seqlen_kv), scale,
                                  bool(causal), int(window or 0), bias)


def _refuse_flash_extras(dropout_p, alibi_slopes, return_attn_probs):
    if dropout_p:
        raise VlfError(VLF_ERR_UNSUPPORTED, "dropout is not supported")
    if alibi_slopes is not None:
        raise VlfError(VLF_ERR_UNSUPPORTED, "alibi_slopes: pass the ALiBi terms as attn_bias")
    if return_attn_probs:
        raise VlfError(VLF_ERR_UNSUPPORTED, "return_attn_probs is not supported")


def flash_attn_varlen_func(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                           dropout_p=0.0, softmax_scale=None, causal=False, window_size=(-1, -1),
                           alibi_slopes=None, deterministic=False, return_attn_probs=False,
                           attn_bias=None):
    """flash_attn-style call on separate q, k, v (results are deterministic either way)."""
    _refuse_flash_extras(dropout_p, alibi_slopes, return_attn_probs)
    return varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                            scale=softmax_scale, causal=causal,
                            window=window_from_flash(window_size, causal), attn_bias=attn_bias)


def flash_attn_varlen_qkvpacked_func(qkv, cu_seqlens, max_seqlen, dropout_p=0.0,
                                     softmax_scale=None, causal=False, window_size=(-1, -1),
                                     alibi_slopes=None, deterministic=False,
                                     return_attn_probs=False, attn_bias=None):
    """qkv [total, 3, H, D] (self-attention: one cu_seqlens).  q, k, v are taken as contiguous
    copies of the packed slices; the gradient flows back into qkv through them."""
    _refuse_flash_extras(dropout_p, alibi_slopes, return_attn_probs)
    if qkv.dim() != 4 or qkv.shape[1] != 3:
        raise VlfError(VLF_ERR_INVALID, "qkv must be [total_tokens, 3, heads, head_dim]")
    q, k, v = qkv.unbind(1)
    return varlen_attention(q, k, v, cu_seqlens, cu_seqlens, max_seqlen, max_seqlen,
                            scale=softmax_scale, causal=causal,
                            window=window_from_flash(window_size, causal), attn_bias=attn_bias)


def flash_attn_varlen_kvpacked_func(q, kv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                                    max_seqlen_k, dropout_p=0.0, softmax_scale=None, causal=False,
                                    window_size=(-1, -1), alibi_slopes=None, deterministic=False,
                                    return_attn_probs=False, attn_bias=None):
    """q [total_q, H_q, D], kv [total_k, 2, H_kv, D]."""
    _refuse_flash_extras(dropout_p, alibi_slopes, return_attn_probs)
    if kv.dim() != 4 or kv.shape[1] != 2:
        raise VlfError(VLF_ERR_INVALID, "kv must be [total_tokens, 2, kv_heads, head_dim]")
    k, v = kv.unbind(1)
    return varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                            scale=softmax_scale, causal=causal,
                            window=window_from_flash(window_size, causal), attn_bias=attn_bias)
