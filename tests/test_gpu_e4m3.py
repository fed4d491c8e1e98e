"""GPU parity of the e4m3 forward (te_attn_fwd_thd_e4m3) against the oracle.

Pages cited, by title (keys are the pages' issue numbers):
  [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
"""

import numpy as np
import pytest
import torch

import oracle
from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import assert_close, LSE_TOL, np64, to_dev, UNIT_ROUNDOFF

pytestmark = pytest.mark.gpu

F8 = getattr(torch, "float8_e4m3fn", None)


def _quantise(x, real_rows):
    """Per-tensor e4m3: descale = amax(real rows) / 448; values clamped into the
    finite range first (pad slots of +-1e3 saturate, they must stay finite)."""
    amax = float(x[real_rows].abs().max()) if real_rows.any() else 1.0
    descale = max(amax, 1e-6) / 448.0
    q8 = (x.float() / descale).clamp(-448.0, 448.0).to(F8)
    return q8, descale


def _real_rows(cu, cp, T):
    m = torch.zeros(T, dtype=torch.bool)
    for b in range(len(cu) - 1):
        m[int(cp[b]):int(cp[b]) + int(cu[b + 1] - cu[b])] = True
    return m


def _run_and_check(w):
    import bwd_packed_varlen_gb300 as ta
    mq = _real_rows(w.cu_seqlens_q, w.cu_seqlens_q_padded, w.q.shape[0])
    mk = _real_rows(w.cu_seqlens_kv, w.cu_seqlens_kv_padded, w.k.shape[0])
    (q8, qd), (k8, kd), (v8, vd) = _quantise(w.q, mq), _quantise(w.k, mk), _quantise(w.v, mk)
    t = to_dev(w)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    out, lse = ta.fwd_e4m3(q8.cuda(), k8.cuda(), v8.cuda(), *cu, w.attn_scale, qd, kd, vd,
                           w.mask_type)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attn_fwd_thd_e4m3(
        np64(q8), np64(k8), np64(v8), qd, kd, vd, w.cu_seqlens_q.numpy(),
        w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(), w.cu_seqlens_kv_padded.numpy(),
        w.attn_scale, w.mask_type)
    qm, _ = oracle.valid_row_masks(
        w.cu_seqlens_q.numpy(), w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
        w.cu_seqlens_kv_padded.numpy(), w.q.shape[0], w.k.shape[0], w.mask_type)
    o, l = np64(out), np64(lse)
    assert out.dtype == torch.bfloat16 and out.shape == w.q.shape  # padded layout kept
    # magnitude sums of the dequantised inputs (widening V to bf16 adds one more
    # rounding of V, inside the factor 2 of the bound)
    args = (np64(q8) * qd, np64(k8) * kd, np64(v8) * vd, np.zeros(w.q.shape),
            w.cu_seqlens_q.numpy(), w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
            w.cu_seqlens_kv_padded.numpy(), w.attn_scale, w.mask_type)
    m_out = tuple(oracle.attn_error_scales_thd(*args, norm=n)[0] for n in (1, 2))
    assert_close("out", o, ref_out, m_out, UNIT_ROUNDOFF["bf16"])
    assert np.all(o[~qm] == 0), "out: nonzero pad row"
    assert np.array_equal(np.isneginf(l), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    assert np.abs(l[fin] - ref_lse[fin]).max() <= LSE_TOL
    assert np.all(l[~qm & ~np.isneginf(ref_lse).any(axis=1)] == 0)
    return out, lse, (q8, k8, v8, qd, kd, vd)


@pytest.mark.skipif(F8 is None, reason="torch without float8_e4m3fn")
@pytest.mark.parametrize("mask", [W.MASK_PADDING, W.MASK_PADDING_CAUSAL])
def test_e4m3_real_ne_padded_issue2892(mask):
    """[2892]'s shape in e4m3: real lengths [100, 150, 120, 130] inside padded slots
    [112, 160, 128, 144] (pad slots +-1e3, saturated to +-448 in e4m3), 32 heads,
    d = 48: no out-of-bounds access, the output keeps the padded layout, pad rows
    are exactly zero, real rows match the oracle on the dequantised inputs."""
    _run_and_check(W.real_ne_padded(mask_type=mask))


@pytest.mark.skipif(F8 is None, reason="torch without float8_e4m3fn")
@pytest.mark.parametrize("mask", [W.MASK_PADDING_CAUSAL, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT])
@pytest.mark.parametrize("d", [64, 128])
def test_e4m3_ragged_gqa(mask, d):
    """Ragged GQA packing with empty sequences, Lq != Lk and tails, bit-identical
    on a repeated call."""
    import bwd_packed_varlen_gb300 as ta
    w = W.random_varlen(90 + d + mask, 5, 500, 8, 2, d, mask, "bf16")
    out, lse, (q8, k8, v8, qd, kd, vd) = _run_and_check(w)
    t = to_dev(w)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    out2, lse2 = ta.fwd_e4m3(q8.cuda(), k8.cuda(), v8.cuda(), *cu, w.attn_scale, qd, kd, vd,
                             w.mask_type)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


@pytest.mark.skipif(F8 is None, reason="torch without float8_e4m3fn")
def test_e4m3_rejects_unsupported_head_dim():
    import bwd_packed_varlen_gb300 as ta
    q = torch.zeros(16, 2, 40, device="cuda").to(F8)
    cu = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    with pytest.raises(ta.TeAttnError) as e:
        ta.fwd_e4m3(q, q, q, cu, cu, cu, cu, 0.1, 1.0, 1.0, 1.0)
    assert e.value.code == -2
