"""Autograd wrapper: a ``DotProductAttention``-like module over the C ABI.

TransformerEngine users call attention as a module ([2448] minimal repro:
``te.DotProductAttention(num_attention_heads, kv_channels, num_gqa_groups,
qkv_format="thd", attn_mask_type="padding_causal", softmax_scale)`` called as
``dpa(q, k, v, cu_seqlens_q=..., cu_seqlens_kv=..., max_seqlen_q=..., max_seqlen_kv=...)``,
then ``.sum().backward()``; [2892] adds ``cu_seqlens_q_padded`` /
``cu_seqlens_kv_padded``). This module keeps that call shape. The forward stashes
``out`` and ``lse`` for the backward, as TransformerEngine's fused attention does
([2448]: ``fused_attn_bwd`` takes ``out`` and the softmax aux tensor), and every
step of both passes runs in ``libteattn.so``; this file only reshapes and routes
tensors.

Readings where the pages are silent:

* The output is ``[T_q, hq * d]`` (heads flattened, padded rows kept), the shape
  TransformerEngine's module returns for packed input; pad rows are exactly 0.
* ``attn_mask_type`` ``"causal"`` / ``"no_mask"`` / ``"causal_bottom_right"`` mean
  their ``padding_*`` forms: with packed input the real lengths always mask.
* ``qkv_format="bshd"`` (``[B, S, h, d]``, contiguous) is the packed layout with
  padded offsets ``b * S``; no data moves. ``"sbhd"`` (``[S, B, h, d]``, the
  layout of [3216]) runs on the library's sequence-major entry points. In both,
  ``cu_seqlens_q/kv`` are optional real lengths (default: all S tokens).

Pages cited, by title (keys are the pages' issue numbers):
  [2448] "Inconsistent fused_attn_bwd results of dk, dv under THD layout + GQA on multiple calls"
  [3216] "flash-attn-4 4.0.0b11: DotProductAttention batched backward returns wrong dQ/dK/dV at head_dim=256 on Blackwell (sm_100)"
  [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
"""

from __future__ import annotations

import math

import torch

from . import _binding as _b

_MASK_ALIASES = {
    "padding": "padding", "no_mask": "padding",
    "padding_causal": "padding_causal", "causal": "padding_causal",
    "padding_causal_bottom_right": "padding_causal_bottom_right",
    "causal_bottom_right": "padding_causal_bottom_right",
}


def _mask_name(mask):
    if isinstance(mask, str):
        if mask not in _MASK_ALIASES:
            raise ValueError(f"unknown attn_mask_type {mask!r}")
        return _MASK_ALIASES[mask]
    return mask


class THDAttentionFunction(torch.autograd.Function):
    """``out = attention(q, k, v)`` over packed sequences with a fused backward.

    ``q [T_q, hq, d]``, ``k, v [T_kv, hkv, d]`` contiguous CUDA tensors; returns
    ``(out [T_q, hq, d], lse [T_q, hq])``. The backward returns ``dq, dk, dv`` (GQA
    dk/dv summed over each head group) and no gradient for the index tensors."""

    @staticmethod
    def forward(ctx, q, k, v, cu_q, cu_kv, cu_q_pad, cu_kv_pad, scale, mask, max_q, max_kv):
        out, lse = _b.fwd(q, k, v, cu_q, cu_kv, cu_q_pad, cu_kv_pad, scale, mask, max_q, max_kv)
        ctx.save_for_backward(q, k, v, out, lse, cu_q, cu_kv, cu_q_pad, cu_kv_pad)
        ctx.args = (scale, mask, max_q, max_kv)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse, cu_q, cu_kv, cu_q_pad, cu_kv_pad = ctx.saved_tensors
        scale, mask, max_q, max_kv = ctx.args
        # e.g. the expanded ones of .sum().backward(): the kernels want dense rows
        dout = dout.contiguous()
        dq, dk, dv = _b.bwd(q, k, v, out, dout, lse, cu_q, cu_kv, cu_q_pad, cu_kv_pad, scale,
                            mask, max_q, max_kv)
        return dq, dk, dv, None, None, None, None, None, None, None, None


class SBHDAttentionFunction(torch.autograd.Function):
    """The same over the sequence-major layout: ``q [S_q, B, hq, d]``, ``k, v
    [S_kv, B, hkv, d]``, real lengths ``cu_q, cu_kv``; returns ``(out, lse [S_q, B,
    hq])``."""

    @staticmethod
    def forward(ctx, q, k, v, cu_q, cu_kv, scale, mask):
        out, lse = _b.fwd_sbhd(q, k, v, cu_q, cu_kv, scale, mask)
        ctx.save_for_backward(q, k, v, out, lse, cu_q, cu_kv)
        ctx.args = (scale, mask)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse, cu_q, cu_kv = ctx.saved_tensors
        scale, mask = ctx.args
        dq, dk, dv = _b.bwd_sbhd(q, k, v, out, dout.contiguous(), lse, cu_q, cu_kv, scale, mask)
        return dq, dk, dv, None, None, None, None


def _full_lengths(B, S, device):
    return torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device=device)


def _bshd_to_thd(x, cu_real, S):
    # a view, never a copy: a non-contiguous input fails here instead of moving data
    B = x.shape[0]
    cu_pad = _full_lengths(B, S, x.device)
    if cu_real is None:
        cu_real = cu_pad
    return x.view(B * S, x.shape[2], x.shape[3]), cu_real, cu_pad


def dot_product_attention(q, k, v, cu_seqlens_q=None, cu_seqlens_kv=None,
                          cu_seqlens_q_padded=None, cu_seqlens_kv_padded=None,
                          max_seqlen_q=0, max_seqlen_kv=0, attn_mask_type="padding_causal",
                          softmax_scale=None, qkv_format="thd", return_lse=False):
    """Differentiable attention over packed sequences; see the module docstring.

    ``thd``: ``q [T_q, hq, d]``, ``k, v [T_kv, hkv, d]``; ``cu_seqlens_q/kv`` (int32
    ``[B+1]``) are required and the padded ones default to them. ``bshd``: ``q [B,
    S_q, hq, d]``, ``k, v [B, S_kv, hkv, d]``; ``sbhd``: ``q [S_q, B, hq, d]``, ``k, v
    [S_kv, B, hkv, d]``; for both, ``cu_seqlens_*`` are optional real lengths
    (default: full). ``softmax_scale`` defaults to ``1 / sqrt(d)``. Returns ``[T_q,
    hq * d]`` (``[B, S_q, hq * d]`` for bshd, ``[S_q, B, hq * d]`` for sbhd), plus
    the fp32 lse (``[T_q, hq]``, ``[B * S_q, hq]``, ``[S_q, B, hq]``) when
    ``return_lse``."""
    mask = _mask_name(attn_mask_type)
    if qkv_format == "bshd":
        if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
            raise ValueError("bshd tensors must be [B, S, h, d]")
        Bq, Sq = q.shape[:2]
        Sk = k.shape[1]
        if k.shape[0] != Bq or v.shape[:2] != k.shape[:2]:
            raise ValueError("bshd q, k, v must share the batch size; k and v the length")
        if cu_seqlens_q_padded is not None or cu_seqlens_kv_padded is not None:
            raise ValueError("bshd takes no padded cu_seqlens: its padded offsets are b * S")
        q3, cu_q, cu_q_pad = _bshd_to_thd(q, cu_seqlens_q, Sq)
        k3, cu_kv, cu_kv_pad = _bshd_to_thd(k, cu_seqlens_kv, Sk)
        v3 = v.view(Bq * Sk, v.shape[2], v.shape[3])
        shape = (Bq, Sq, q.shape[2] * q.shape[3])
    elif qkv_format == "sbhd":
        if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
            raise ValueError("sbhd tensors must be [S, B, h, d]")
        if cu_seqlens_q_padded is not None or cu_seqlens_kv_padded is not None:
            raise ValueError("sbhd takes no padded cu_seqlens: every entry spans S tokens")
        Sq, B = q.shape[:2]
        cu_q = _full_lengths(B, Sq, q.device) if cu_seqlens_q is None else cu_seqlens_q
        cu_kv = _full_lengths(B, k.shape[0], q.device) if cu_seqlens_kv is None else cu_seqlens_kv
        scale = 1.0 / math.sqrt(q.shape[-1]) if softmax_scale is None else float(softmax_scale)
        out, lse = SBHDAttentionFunction.apply(q, k, v, cu_q, cu_kv, scale, mask)
        out = out.view(Sq, B, q.shape[2] * q.shape[3])
        return (out, lse) if return_lse else out
    elif qkv_format == "thd":
        if cu_seqlens_q is None or cu_seqlens_kv is None:
            raise ValueError("thd needs cu_seqlens_q and cu_seqlens_kv")
        q3, k3, v3 = q, k, v
        cu_q, cu_kv = cu_seqlens_q, cu_seqlens_kv
        cu_q_pad = cu_seqlens_q if cu_seqlens_q_padded is None else cu_seqlens_q_padded
        cu_kv_pad = cu_seqlens_kv if cu_seqlens_kv_padded is None else cu_seqlens_kv_padded
        shape = (q.shape[0], q.shape[1] * q.shape[2])
    else:
        raise NotImplementedError(f"qkv_format {qkv_format!r}: 'thd', 'bshd' or 'sbhd'")
    scale = 1.0 / math.sqrt(q.shape[-1]) if softmax_scale is None else float(softmax_scale)
    out, lse = THDAttentionFunction.apply(q3, k3, v3, cu_q, cu_kv, cu_q_pad, cu_kv_pad, scale,
                                          mask, int(max_seqlen_q or 0), int(max_seqlen_kv or 0))
    out = out.view(shape)
    return (out, lse) if return_lse else out


class DotProductAttention(torch.nn.Module):
    """Module form of :func:`dot_product_attention` with TransformerEngine's
    constructor arguments ([2448] minimal repro); no parameters, no state."""

    def __init__(self, num_attention_heads, kv_channels, num_gqa_groups=None,
                 attn_mask_type="padding_causal", softmax_scale=None, qkv_format="thd",
                 attention_dropout=0.0):
        super().__init__()
        if attention_dropout != 0.0:
            raise NotImplementedError("attention dropout is not supported")
        self.num_attention_heads = int(num_attention_heads)
        self.kv_channels = int(kv_channels)
        self.num_gqa_groups = int(num_gqa_groups or num_attention_heads)
        if self.num_attention_heads % self.num_gqa_groups != 0:
            raise ValueError("num_attention_heads must be a multiple of num_gqa_groups")
        self.attn_mask_type = _mask_name(attn_mask_type)
        self.softmax_scale = softmax_scale
        self.qkv_format = qkv_format

    def forward(self, q, k, v, cu_seqlens_q=None, cu_seqlens_kv=None, cu_seqlens_q_padded=None,
                cu_seqlens_kv_padded=None, max_seqlen_q=None, max_seqlen_kv=None,
                attn_mask_type=None, qkv_format=None):
        fmt = qkv_format or self.qkv_format
        if q.shape[-2] != self.num_attention_heads or k.shape[-2] != self.num_gqa_groups:
            raise ValueError("head counts of q/k differ from the module's")
        if q.shape[-1] != self.kv_channels:
            raise ValueError("head dim of q differs from kv_channels")
        return dot_product_attention(
            q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
            max_seqlen_q or 0, max_seqlen_kv or 0, attn_mask_type or self.attn_mask_type,
            self.softmax_scale, fmt)
