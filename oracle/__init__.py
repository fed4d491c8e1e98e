"""CPU float64 oracle for packed variable-length (THD) attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may call it. It shares no code, headers, tables or helpers with
the CUDA path under ``bwd_packed_varlen_gb300/``.

Every function is the plain definition of scaled-dot-product attention written out
per sequence and per key/value head group, in numpy float64, with no tiling, no
online softmax and no fusion. The pages this follows (TransformerEngine issues on
packed-sequence attention) fix:

* real ``cu_seqlens_q/kv`` drive the masks and padded ``cu_seqlens_*_padded`` drive
  the memory offsets; the output keeps the padded layout ([2892], "Expected
  Behavior", items 1-3);
* GQA maps query head h to key/value head h // (hq // hkv) ([3216],
  ``fp32_reference`` with ``repeat_interleave``);
* the causal mask is the upper-left triangle, key j visible to query i iff j <= i
  ([3216], ``torch.triu(..., 1)`` filled with -inf); the lower-right variant
  (``padding_causal_bottom_right``, j <= i + Lk - Lq) is this package's own
  restatement of that mask name, pinned against torch's ``causal_lower_right``;
* rows that hold no token of any sequence get exactly-zero gradients ([2448],
  "Expected behavior": the first 4 tokens of dk/dv are zero when the first query
  sequence is empty).

Parity status of each function is stated in its docstring; all are pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle.py``.

Pages cited, by title (keys are the pages' issue numbers):
  [2448] "Inconsistent fused_attn_bwd results of dk, dv under THD layout + GQA on multiple calls"
  [3333] "[Bug] FusedAttention (cuDNN) THD backward produces wrong gradients on sm_120 (RTX 5090); forward is correct, Unfused is correct"
  [3216] "flash-attn-4 4.0.0b11: DotProductAttention batched backward returns wrong dQ/dK/dV at head_dim=256 on Blackwell (sm_100)"
  [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
"""

from .attention import (  # noqa: F401
    MASK_PADDING,
    MASK_PADDING_CAUSAL,
    MASK_PADDING_CAUSAL_BOTTOM_RIGHT,
    causal_diagonal,
    seq_spans,
    attn_group_fwd_bwd,
    attn_group_bwd_given,
    attn_group_error_scales,
    attn_error_scales_thd,
    attn_fwd_thd,
    attn_bwd_thd,
    attn_fwd_bwd_thd,
    attn_fwd_bwd_sbhd,
    attn_fwd_thd_e4m3,
    valid_row_masks,
    fwd_bwd_flops,
)
