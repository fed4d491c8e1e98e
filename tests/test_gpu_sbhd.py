"""GPU parity of the sequence-major ("sbhd") entry points against the oracle.

Pages cited, by title (keys are the pages' issue numbers):
  [3216] "flash-attn-4 4.0.0b11: DotProductAttention batched backward returns wrong dQ/dK/dV at head_dim=256 on Blackwell (sm_100)"
"""

import math

import numpy as np
import pytest
import torch

import oracle
from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import assert_close, LSE_TOL, np64, UNIT_ROUNDOFF

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.view(torch.int32 if x.dtype == torch.float32 else torch.int16)


def _sbhd_case(seed, S_q, S_kv, lq, lk, hq, hkv, d, dtype=torch.bfloat16):
    """[S, B, h, d] tensors; tokens at or past each entry's real length are pad
    slots filled with +-1e3 (they must not reach any real output)."""
    g = torch.Generator().manual_seed(seed)
    B = len(lq)
    q = torch.randn(S_q, B, hq, d, generator=g)
    k = torch.randn(S_kv, B, hkv, d, generator=g)
    v = torch.randn(S_kv, B, hkv, d, generator=g)
    do = torch.randn(S_q, B, hq, d, generator=g)
    for b in range(B):
        for x, n in ((q, lq[b]), (do, lq[b]), (k, lk[b]), (v, lk[b])):
            pad = x[n:, b]
            pad.copy_(torch.where(torch.rand(pad.shape, generator=g) < 0.5, -1e3, 1e3))
    cu = lambda ls: torch.tensor([0] + list(np.cumsum(ls)), dtype=torch.int32)
    return [t.to(dtype) for t in (q, k, v, do)], cu(lq), cu(lk)


def _run(q, k, v, do, cu_q, cu_kv, scale, mask):
    import bwd_packed_varlen_gb300 as ta
    dev = [t.cuda() for t in (q, k, v, do)]
    cq, ck = cu_q.cuda(), cu_kv.cuda()
    out, lse = ta.fwd_sbhd(dev[0], dev[1], dev[2], cq, ck, scale, mask)
    dq, dk, dv = ta.bwd_sbhd(dev[0], dev[1], dev[2], out, dev[3], lse, cq, ck, scale, mask)
    torch.cuda.synchronize()
    return out, lse, dq, dk, dv


def _scales(q, k, v, do, cu_q, cu_kv, scale, mask):
    """Oracle magnitude sums in the sequence-major layout: computed on the packed
    view of the same values (batch entry b at rows b * S ..) and laid back out."""
    S_q, B = q.shape[:2]
    S_kv = k.shape[0]
    packed = lambda x: np.ascontiguousarray(np.swapaxes(np64(x), 0, 1)).reshape((-1,) + tuple(x.shape[2:]))
    cp_q, cp_k = np.arange(B + 1) * S_q, np.arange(B + 1) * S_kv
    back = lambda x, S: np.swapaxes(x.reshape((B, S) + x.shape[1:]), 0, 1)
    res = []
    for norm in (1, 2):
        m = oracle.attn_error_scales_thd(packed(q), packed(k), packed(v), packed(do),
                                         cu_q.numpy(), cu_kv.numpy(), cp_q, cp_k, scale, mask,
                                         norm=norm)
        res.append((back(m[0], S_q), back(m[1], S_q), back(m[2], S_kv), back(m[3], S_kv)))
    return list(zip(*res))


def _check(res, ref, lq, lk, scales):
    out, lse, dq, dk, dv = (np64(x) for x in res)
    u = UNIT_ROUNDOFF[res[0].dtype]
    for name, a, b, m in zip(("out", "dq", "dk", "dv"), (out, dq, dk, dv),
                             (ref[0], ref[2], ref[3], ref[4]), scales):
        assert_close(name, a, b, m, u)
    fin = np.isfinite(ref[1])
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref[1]))
    assert np.abs(lse[fin] - ref[1][fin]).max() <= LSE_TOL
    for b in range(len(lq)):
        assert np.all(out[lq[b]:, b] == 0) and np.all(dq[lq[b]:, b] == 0)
        assert np.all(lse[lq[b]:, b] == 0)
        assert np.all(dk[lk[b]:, b] == 0) and np.all(dv[lk[b]:, b] == 0)


@pytest.mark.parametrize("mask", [W.MASK_PADDING, W.MASK_PADDING_CAUSAL,
                                  W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_sbhd_matches_oracle(mask, d):
    """Ragged real lengths inside [S, B, h, d] tensors (one entry empty, one full,
    one with more keys than queries), GQA, pad slots +-1e3, three masks."""
    lq, lk = [300, 0, 129, 333], [300, 77, 250, 100]
    (q, k, v, do), cu_q, cu_kv = _sbhd_case(80 + d + mask, 333, 300, lq, lk, 4, 2, d)
    scale = 1.0 / math.sqrt(d)
    res = _run(q, k, v, do, cu_q, cu_kv, scale, mask)
    ref = oracle.attn_fwd_bwd_sbhd(np64(q), np64(k), np64(v), np64(do), cu_q.numpy(),
                                   cu_kv.numpy(), scale, mask)
    _check(res, ref, lq, lk, _scales(q, k, v, do, cu_q, cu_kv, scale, mask))


def test_sbhd_equals_packed_bitwise():
    """The same values through the packed entry points (row b * S + s, padded
    offsets b * S) give bit-identical outputs: only the addressing differs."""
    import bwd_packed_varlen_gb300 as ta
    lq, lk = [200, 57, 256], [180, 256, 3]
    S_q, S_kv, hq, hkv, d = 256, 256, 8, 2, 128
    (q, k, v, do), cu_q, cu_kv = _sbhd_case(99, S_q, S_kv, lq, lk, hq, hkv, d)
    scale, mask = 0.1, W.MASK_PADDING_CAUSAL
    sb = _run(q, k, v, do, cu_q, cu_kv, scale, mask)
    packed = lambda x: x.transpose(0, 1).contiguous().view((-1,) + tuple(x.shape[2:])).cuda()
    B = len(lq)
    cp_q = torch.arange(0, (B + 1) * S_q, S_q, dtype=torch.int32).cuda()
    cp_k = torch.arange(0, (B + 1) * S_kv, S_kv, dtype=torch.int32).cuda()
    cq, ck = cu_q.cuda(), cu_kv.cuda()
    tq, tk, tv, tdo = (packed(x) for x in (q, k, v, do))
    out, lse = ta.fwd(tq, tk, tv, cq, ck, cp_q, cp_k, scale, mask)
    dq, dk, dv = ta.bwd(tq, tk, tv, out, tdo, lse, cq, ck, cp_q, cp_k, scale, mask)
    torch.cuda.synchronize()
    back = lambda x, S: x.view((B, S) + tuple(x.shape[1:])).transpose(0, 1).contiguous()
    th = (back(out, S_q), back(lse, S_q), back(dq, S_q), back(dk, S_kv), back(dv, S_kv))
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), sb, th):
        assert torch.equal(_bits(a), _bits(b)), name


def test_issue3216_native_layout():
    """[3216]'s shape in its own layout: sbhd [384, 2, 16, 256] with 2 kv heads,
    causal, lognormal channel scales and shared outlier channels (the packed
    stand-in of the same data passes the oracle too)."""
    w = W.gqa_d256()
    S, B = 384, 2
    to_sbhd = lambda x: x.view((B, S) + tuple(x.shape[1:])).transpose(0, 1).contiguous()
    q, k, v, do = (to_sbhd(x) for x in (w.q, w.k, w.v, w.dout))
    cu = torch.tensor([0, S, 2 * S], dtype=torch.int32)
    res = _run(q, k, v, do, cu, cu, w.attn_scale, W.MASK_PADDING_CAUSAL)
    ref = oracle.attn_fwd_bwd_sbhd(np64(q), np64(k), np64(v), np64(do), cu.numpy(), cu.numpy(),
                                   w.attn_scale, W.MASK_PADDING_CAUSAL)
    _check(res, ref, [S, S], [S, S],
           _scales(q, k, v, do, cu, cu, w.attn_scale, W.MASK_PADDING_CAUSAL))


def test_autograd_sbhd():
    """qkv_format="sbhd" through the module: out [S, B, hq * d] and the gradients
    equal the direct entry points' bit for bit."""
    import bwd_packed_varlen_gb300 as ta
    lq, lk = [120, 200], [200, 64]
    (q, k, v, do), cu_q, cu_kv = _sbhd_case(7, 200, 200, lq, lk, 4, 1, 64)
    ref = _run(q, k, v, do, cu_q, cu_kv, 0.125, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT)
    qg, kg, vg = (x.cuda().requires_grad_(True) for x in (q, k, v))
    dpa = ta.DotProductAttention(4, 64, 1, attn_mask_type="padding_causal_bottom_right",
                                 softmax_scale=0.125, qkv_format="sbhd")
    out = dpa(qg, kg, vg, cu_seqlens_q=cu_q.cuda(), cu_seqlens_kv=cu_kv.cuda())
    assert out.shape == (200, 2, 4 * 64)
    out.backward(do.cuda().view(out.shape))
    torch.cuda.synchronize()
    for a, b in zip((out.detach().view(q.shape), qg.grad, kg.grad, vg.grad),
                    (ref[0], ref[2], ref[3], ref[4])):
        assert torch.equal(_bits(a), _bits(b))
