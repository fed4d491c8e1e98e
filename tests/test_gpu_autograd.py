"""GPU tests of the autograd wrapper (DotProductAttention-like module).

Pages cited, by title (keys are the pages' issue numbers):
  [2448] "Inconsistent fused_attn_bwd results of dk, dv under THD layout + GQA on multiple calls"
  [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
"""

import numpy as np
import pytest
import torch

from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import check_against_oracle, np64, oracle_fwd_bwd, to_dev

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.view(torch.int32 if x.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("mask", [W.MASK_PADDING, W.MASK_PADDING_CAUSAL,
                                  W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT])
def test_autograd_matches_oracle(mask):
    """out.backward(dout) through the module gives the oracle's out, dq, dk, dv on a
    ragged GQA case with real != padded lengths ([2892] call shape)."""
    import bwd_packed_varlen_gb300 as ta
    w = W.random_varlen(70 + mask, 5, 400, 8, 2, 128, mask, "bf16")
    t = to_dev(w)
    q, k, v = (t[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    dpa = ta.DotProductAttention(8, 128, num_gqa_groups=2, attn_mask_type=mask,
                                 softmax_scale=w.attn_scale)
    out = dpa(q, k, v, cu_seqlens_q=t["cu_q"], cu_seqlens_kv=t["cu_kv"],
              cu_seqlens_q_padded=t["cu_q_pad"], cu_seqlens_kv_padded=t["cu_kv_pad"],
              max_seqlen_q=w.max_seqlen_q, max_seqlen_kv=w.max_seqlen_kv)
    assert out.shape == (q.shape[0], 8 * 128)
    out.backward(t["dout"].view(out.shape))
    # the lse the module stashed is the one the plain entry point returns
    _, lse = ta.fwd(t["q"], t["k"], t["v"], t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"],
                    w.attn_scale, mask)
    torch.cuda.synchronize()
    res = (out.detach().view(q.shape), lse, q.grad, k.grad, v.grad)
    check_against_oracle(w, res)


def test_autograd_allocator_churn_issue2448():
    """[2448] minimal repro through the module: GQA (4 query heads, 1 kv head),
    head dim 256, two packed sequences of 64, padding_causal, loss out.sum();
    between backward calls an nn.Linear(4096, 1024).bfloat16() frees and reallocates
    blocks, then torch.cuda.empty_cache(). dK stays finite and bit-identical across
    the three calls (the page saw NaN after the churn), and matches the oracle."""
    import bwd_packed_varlen_gb300 as ta
    dev, dt = "cuda", torch.bfloat16
    n_q, n_kv, hd = 4, 1, 256
    cu = torch.tensor([0, 64, 128], device=dev, dtype=torch.int32)
    g = torch.Generator().manual_seed(0)
    base = [torch.randn(128, h, hd, generator=g).to(dt) for h in (n_q, n_kv, n_kv)]
    dpa = ta.DotProductAttention(num_attention_heads=n_q, kv_channels=hd, num_gqa_groups=n_kv,
                                 qkv_format="thd", attn_mask_type="padding_causal",
                                 softmax_scale=hd ** -0.5)

    def grads():
        q, k, v = (x.to(dev).requires_grad_(True) for x in base)
        dpa(q, k, v, cu_seqlens_q=cu, cu_seqlens_kv=cu, max_seqlen_q=64,
            max_seqlen_kv=64).sum().backward()
        torch.cuda.synchronize()
        return q.grad, k.grad, v.grad

    first = grads()
    torch.nn.Linear(4096, 1024).to(dev).bfloat16()
    second = grads()
    torch.cuda.empty_cache()
    third = grads()
    for a, b, c in zip(first, second, third):
        assert torch.isfinite(a.float()).all()
        assert torch.equal(_bits(a), _bits(b)) and torch.equal(_bits(a), _bits(c))
    w = W.Workload(name="issue2448_churn", q=base[0], k=base[1], v=base[2],
                   dout=torch.ones(128, n_q, hd, dtype=dt), cu_seqlens_q=cu.cpu(),
                   cu_seqlens_kv=cu.cpu(), cu_seqlens_q_padded=cu.cpu(),
                   cu_seqlens_kv_padded=cu.cpu(), attn_scale=hd ** -0.5,
                   mask_type=W.MASK_PADDING_CAUSAL, dtype="bf16")
    ref = oracle_fwd_bwd(w)
    for got, r in zip(first, ref[2:]):
        rel = np.linalg.norm(np64(got) - r) / np.linalg.norm(r)
        assert rel <= 1e-2, rel


def test_bshd_is_packed_with_uniform_padding():
    """qkv_format="bshd" with real lengths below S equals the packed call with
    padded offsets b * S, bit for bit, in the output and all three gradients."""
    import bwd_packed_varlen_gb300 as ta
    B, S, hq, hkv, d = 3, 200, 4, 2, 64
    g = torch.Generator().manual_seed(7)
    mk = lambda h: torch.randn(B, S, h, d, generator=g).to(torch.bfloat16).cuda()
    qb, kb, vb, dob = mk(hq), mk(hkv), mk(hkv), mk(hq)
    cu = torch.tensor([0, 150, 350, 551], dtype=torch.int32, device="cuda")
    cu_pad = torch.tensor([0, S, 2 * S, 3 * S], dtype=torch.int32, device="cuda")

    def run(fmt):
        q, k, v = (x.clone().requires_grad_(True) for x in (qb, kb, vb))
        if fmt == "bshd":
            out = ta.dot_product_attention(q, k, v, cu, cu, attn_mask_type="padding_causal",
                                           qkv_format="bshd")
            out.backward(dob.view(out.shape))
        else:
            out = ta.dot_product_attention(q.view(B * S, hq, d), k.view(B * S, hkv, d),
                                           v.view(B * S, hkv, d), cu, cu, cu_pad, cu_pad,
                                           attn_mask_type="padding_causal")
            out.backward(dob.view(out.shape))
        torch.cuda.synchronize()
        return out.detach().reshape(-1), q.grad.reshape(-1), k.grad.reshape(-1), v.grad.reshape(-1)

    for a, b in zip(run("bshd"), run("thd")):
        assert torch.equal(_bits(a), _bits(b))
