"""Pins of the CPU float64 oracle against things other than itself.

Each test fixes the oracle to an independent fact: finite differences of the loss,
torch's own float64 SDPA + autograd, closed forms, algebraic invariants, and the
layouts and zero rows that the TransformerEngine pages state (tests/golden/).

Pages cited, by title (keys are the pages' issue numbers):
  [2448] "Inconsistent fused_attn_bwd results of dk, dv under THD layout + GQA on multiple calls"
  [3333] "[Bug] FusedAttention (cuDNN) THD backward produces wrong gradients on sm_120 (RTX 5090); forward is correct, Unfused is correct"
  [3216] "flash-attn-4 4.0.0b11: DotProductAttention batched backward returns wrong dQ/dK/dV at head_dim=256 on Blackwell (sm_100)"
  [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import MASK_PADDING, MASK_PADDING_CAUSAL, MASK_PADDING_CAUSAL_BOTTOM_RIGHT

ALL_MASKS = [MASK_PADDING, MASK_PADDING_CAUSAL, MASK_PADDING_CAUSAL_BOTTOM_RIGHT]
# torch's own constructions of the two causal alignments
_ALIGN = {MASK_PADDING: None, MASK_PADDING_CAUSAL: "tl", MASK_PADDING_CAUSAL_BOTTOM_RIGHT: "br"}

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed, lq, lk, pq, pk, hq, hkv, d, tail=2):
    """float64 THD tensors with the given real/padded lengths (pad slots random)."""
    rng = np.random.default_rng(seed)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int64)
    cp_q = np.concatenate([[0], np.cumsum(pq)]).astype(np.int64)
    cp_k = np.concatenate([[0], np.cumsum(pk)]).astype(np.int64)
    Tq, Tk = int(cp_q[-1]) + tail, int(cp_k[-1]) + tail
    q = rng.standard_normal((Tq, hq, d))
    k = rng.standard_normal((Tk, hkv, d))
    v = rng.standard_normal((Tk, hkv, d))
    do = rng.standard_normal((Tq, hq, d))
    return q, k, v, do, cu_q, cu_k, cp_q, cp_k


def _loss(q, k, v, do, cu_q, cu_k, cp_q, cp_k, scale, mask):
    out, _ = oracle.attn_fwd_thd(q, k, v, cu_q, cu_k, cp_q, cp_k, scale, mask)
    return float((out * do).sum())


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_finite_differences(mask):
    """Central differences of L = sum(dO * O) w.r.t. every element of q, k, v agree
    with the oracle's dq, dk, dv (float64, eps 1e-6), including the exact-zero
    derivative w.r.t. pad slots. Lq != Lk per sequence, padded offsets != real."""
    lq, lk, pq, pk = [3, 5], [4, 2], [4, 6], [5, 2]
    args = _rand_case(1, lq, lk, pq, pk, hq=2, hkv=1, d=3)
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = args
    scale = 0.7
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(
        q, k, v, do, cu_q, cu_k, cp_q, cp_k, scale, mask)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, do, cu_q, cu_k, cp_q, cp_k, scale, mask)
            x[idx] = old - eps
            lm = _loss(q, k, v, do, cu_q, cu_k, cp_q, cp_k, scale, mask)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(num - g) / np.linalg.norm(num)
        assert err < 1e-6, (name, err)
        assert np.array_equal(num == 0, g == 0) or np.all(np.abs(num[g == 0]) < 1e-9), name


def _torch_reference(q, k, v, do, cu_q, cu_k, cp_q, cp_k, scale, causal):
    """Per-sequence torch float64 SDPA (math) + autograd with repeat_interleave GQA,
    the reference construction of [3333] and [3216]. ``causal``: None, "tl" (a
    lower-triangular boolean mask) or "br" (torch's ``causal_lower_right`` bias,
    whose fully masked rows torch's math backend returns as zeros)."""
    hq, hkv = q.shape[1], k.shape[1]
    G = hq // hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    out = torch.zeros_like(tq)
    outs = []
    lses = []
    for b in range(len(cu_q) - 1):
        oq, Lq = int(cp_q[b]), int(cu_q[b + 1] - cu_q[b])
        ok, Lk = int(cp_k[b]), int(cu_k[b + 1] - cu_k[b])
        if Lq == 0 or Lk == 0:
            continue
        qi = tq[oq:oq + Lq].transpose(0, 1)
        ki = tk[ok:ok + Lk].transpose(0, 1).repeat_interleave(G, 0)
        vi = tv[ok:ok + Lk].transpose(0, 1).repeat_interleave(G, 0)
        mask = bias = None
        if causal == "tl":
            mask = bias = torch.ones(Lq, Lk, dtype=torch.bool).tril()
        elif causal == "br":
            import warnings
            from torch.nn.attention.bias import causal_lower_right
            with warnings.catch_warnings():
                warnings.simplefilter("ignore")  # it warns about rows with no key
                bias = causal_lower_right(Lq, Lk)
            mask = bias._materialize(device=qi.device)
        o = torch.nn.functional.scaled_dot_product_attention(
            qi, ki, vi, attn_mask=bias, scale=scale)
        s = scale * qi @ ki.transpose(-1, -2)
        if causal:
            s = s.masked_fill(~mask, float("-inf"))
        lses.append((oq, Lq, torch.logsumexp(s, -1).transpose(0, 1).detach()))
        outs.append((oq, Lq, o.transpose(0, 1)))
    for oq, Lq, o in outs:
        out = out.index_put((torch.arange(oq, oq + Lq),), o)
    out.backward(torch.tensor(do))
    lse = torch.zeros(q.shape[0], hq, dtype=torch.float64)
    for oq, Lq, l in lses:
        lse[oq:oq + Lq] = l
    return (out.detach().numpy(), lse.numpy(), tq.grad.numpy(), tk.grad.numpy(),
            tv.grad.numpy())


@pytest.mark.parametrize("mask", ALL_MASKS)
@pytest.mark.parametrize("seed", [2, 3])
def test_matches_torch_sdpa_autograd(mask, seed):
    """Oracle == torch.nn.functional.scaled_dot_product_attention (float64, CPU) +
    autograd, per sequence with repeat_interleave GQA (<= 1e-10 relative)."""
    lq, lk = [7, 0, 12, 5], [9, 4, 12, 3]
    pq, pk = [9, 3, 12, 8], [11, 4, 15, 3]
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(seed, lq, lk, pq, pk, 4, 2, 16)
    scale = 0.25
    mine = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k, scale, mask)
    ref = _torch_reference(q, k, v, do, cu_q, cu_k, cp_q, cp_k, scale, _ALIGN[mask])
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), mine, ref):
        # rows that see no key: -inf in both lse (lower-right, Lq > Lk)
        inf = np.isneginf(b)
        assert np.array_equal(np.isneginf(a), inf), name
        a, b = np.where(inf, 0.0, a), np.where(inf, 0.0, b)
        assert np.abs(a - b).max() <= 1e-10 * max(1.0, np.abs(b).max()), name
    given = oracle.attn_bwd_thd(q, k, v, mine[0], do, mine[1], cu_q, cu_k, cp_q, cp_k,
                                scale, mask)
    for name, a, b in zip(("dq", "dk", "dv"), given, ref[2:]):
        assert np.abs(a - b).max() <= 1e-10 * max(1.0, np.abs(b).max()), name


def test_hand_worked_two_keys():
    """d=1, one query q=1, keys (0, ln 3), values (4, 8), scale 1, dO = 1:
    P = (1/4, 3/4), O = 7, LSE = ln 4, dV = (1/4, 3/4), dP = (4, 8), D = 7,
    dS = (-3/4, 3/4), dQ = (3/4) ln 3, dK = (-3/4, 3/4)."""
    q = np.array([[[1.0]]])
    k = np.array([[[0.0]], [[math.log(3.0)]]])
    v = np.array([[[4.0]], [[8.0]]])
    do = np.array([[[1.0]]])
    cq, ck = [0, 1], [0, 2]
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, cq, ck, cq, ck, 1.0,
                                                   MASK_PADDING)
    assert out[0, 0, 0] == pytest.approx(7.0, abs=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(4.0), abs=1e-14)
    assert dv[:, 0, 0] == pytest.approx([0.25, 0.75], abs=1e-14)
    assert dq[0, 0, 0] == pytest.approx(0.75 * math.log(3.0), abs=1e-14)
    assert dk[:, 0, 0] == pytest.approx([-0.75, 0.75], abs=1e-14)


def test_hand_worked_transposes():
    """d=2 with distinct rows/columns so a transposed operand changes the result:
    q0 = (1, 0), q1 = (0, 2), k0 = (ln 2, 0), k1 = (0, 0), v0 = (1, 3), v1 = (5, 7),
    scale 1, padding. Row 0: scores (ln2, 0) -> P = (2/3, 1/3); row 1: scores (0, 0)
    -> P = (1/2, 1/2). O0 = (7/3, 13/3), O1 = (3, 5)."""
    q = np.array([[[1.0, 0.0]], [[0.0, 2.0]]])
    k = np.array([[[math.log(2.0), 0.0]], [[0.0, 0.0]]])
    v = np.array([[[1.0, 3.0]], [[5.0, 7.0]]])
    do = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    c = [0, 2]
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, c, c, c, c, 1.0,
                                                   MASK_PADDING)
    assert out[:, 0, :] == pytest.approx(np.array([[7 / 3, 13 / 3], [3.0, 5.0]]), abs=1e-13)
    assert lse[:, 0] == pytest.approx([math.log(3.0), math.log(2.0)], abs=1e-13)
    # dV_j = sum_i P_ij dO_i: dV0 = 2/3 (1,0) + 1/2 (0,1); dV1 = 1/3 (1,0) + 1/2 (0,1)
    assert dv[:, 0, :] == pytest.approx(np.array([[2 / 3, 0.5], [1 / 3, 0.5]]), abs=1e-13)
    # row 0: dP = dO0 . v_j = (1, 5); D0 = 2/3 + 5/3 = 7/3; dS0 = (2/3(-4/3), 1/3(8/3))
    # row 1: dP = (3, 7); D1 = 5; dS1 = (1/2(-2), 1/2(2)) = (-1, 1)
    ds = np.array([[-8 / 9, 8 / 9], [-1.0, 1.0]])
    kk = np.array([[math.log(2.0), 0.0], [0.0, 0.0]])
    qq = np.array([[1.0, 0.0], [0.0, 2.0]])
    assert dq[:, 0, :] == pytest.approx(ds @ kk, abs=1e-13)
    assert dk[:, 0, :] == pytest.approx(ds.T @ qq, abs=1e-13)
    assert dq[0, 0, :] == pytest.approx([-8 / 9 * math.log(2.0), 0.0], abs=1e-13)
    assert dk[:, 0, :] == pytest.approx(np.array([[-8 / 9, -2.0], [8 / 9, 2.0]]), abs=1e-13)


@pytest.mark.parametrize("mask", [MASK_PADDING, MASK_PADDING_CAUSAL])
def test_single_key_closed_form(mask):
    """Lk = 1: every valid query attends only to key 0, so O_i = V_0,
    LSE_i = scale q_i.k_0, dQ = 0, dK = 0, dV_0 = sum of dO over the group."""
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(4, [5], [1], [6], [3], 3, 1, 4)
    scale = 0.3
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k,
                                                   scale, mask)
    assert np.allclose(out[:5], np.broadcast_to(v[0, 0], (5, 3, 4)), atol=1e-14)
    assert np.allclose(lse[:5], scale * np.einsum("thd,d->th", q[:5], k[0, 0]), atol=1e-13)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    assert np.allclose(dv[0, 0], do[:5].sum(axis=(0, 1)), atol=1e-12)
    assert np.all(dv[1:] == 0)


def test_causal_first_row_and_zero_query():
    """Causal row 0 sees only key 0: O_0 = V_0, dQ_0 = 0. With q = 0 and the
    padding mask the softmax is uniform: O = mean(V), LSE = log Lk."""
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(5, [6], [6], [6], [6], 2, 2, 5, tail=0)
    out, lse, dq, _, _ = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k,
                                                 0.5, MASK_PADDING_CAUSAL)
    assert np.allclose(out[0], v[0], atol=1e-14)
    assert np.abs(dq[0]).max() < 1e-14
    q0 = np.zeros_like(q)
    out, lse, _, _, _ = oracle.attn_fwd_bwd_thd(q0, k, v, do, cu_q, cu_k, cp_q, cp_k,
                                                0.5, MASK_PADDING)
    assert np.allclose(out, np.broadcast_to(v.mean(axis=0), out.shape), atol=1e-14)
    assert np.allclose(lse, math.log(6.0), atol=1e-14)


def test_bottom_right_closed_forms():
    """Lower-right causal alignment: with Lq == Lk it is the upper-left triangle,
    bit for bit; a single query (Lq = 1) sees every key, as with the padding mask;
    with Lk = 1 only the last query sees the key (O = V_0, LSE = scale q.k_0) and
    the Lq - 1 queries before it see nothing (O = 0, LSE = -inf, dQ = 0)."""
    br, tl = MASK_PADDING_CAUSAL_BOTTOM_RIGHT, MASK_PADDING_CAUSAL
    args = _rand_case(21, [6, 4], [6, 4], [7, 4], [6, 5], 2, 1, 5)
    a = oracle.attn_fwd_bwd_thd(*args, 0.5, br)
    b = oracle.attn_fwd_bwd_thd(*args, 0.5, tl)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    args = _rand_case(22, [1], [7], [2], [9], 3, 1, 4)
    a = oracle.attn_fwd_bwd_thd(*args, 0.5, br)
    b = oracle.attn_fwd_bwd_thd(*args, 0.5, MASK_PADDING)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(23, [5], [1], [6], [3], 3, 1, 4)
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k,
                                                   0.3, br)
    assert np.all(out[:4] == 0) and np.all(dq[:4] == 0) and np.all(np.isneginf(lse[:4]))
    assert np.allclose(out[4], np.broadcast_to(v[0, 0], (3, 4)), atol=1e-14)
    assert np.allclose(lse[4], 0.3 * q[4] @ k[0, 0], atol=1e-13)
    assert np.abs(dq[4]).max() < 1e-13 and np.abs(dk).max() < 1e-13
    assert np.allclose(dv[0, 0], do[4].sum(axis=0), atol=1e-12)


@pytest.mark.parametrize("lq,lk", [(3, 8), (5, 5), (8, 3), (1, 4), (4, 1)])
def test_bottom_right_is_shifted_top_left(lq, lk):
    """The lower-right triangle puts query i at position Lk - Lq + i. So for
    Lq <= Lk it is the upper-left problem over Lk queries of which only the last
    Lq carry a gradient (the others get dO = 0 and change nothing in dK/dV); for
    Lq > Lk the last Lk queries form the upper-left problem and the first Lq - Lk
    see no key. Checked on out, lse, dq, dk, dv against the upper-left oracle."""
    br, tl = MASK_PADDING_CAUSAL_BOTTOM_RIGHT, MASK_PADDING_CAUSAL
    q, k, v, do, _, _, _, _ = _rand_case(30 + lq * 10 + lk, [lq], [lk], [lq], [lk], 4, 2, 6, tail=0)
    cq, ck = [0, lq], [0, lk]
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, cq, ck, cq, ck, 0.45, br)
    if lq <= lk:
        rng = np.random.default_rng(lq + 100 * lk)
        qx = np.concatenate([rng.standard_normal((lk - lq,) + q.shape[1:]), q])
        dox = np.concatenate([np.zeros((lk - lq,) + q.shape[1:]), do])
        c = [0, lk]
        o2, l2, dq2, dk2, dv2 = oracle.attn_fwd_bwd_thd(qx, k, v, dox, c, c, c, c, 0.45, tl)
        sl = slice(lk - lq, lk)
        pairs = ((out, o2[sl]), (lse, l2[sl]), (dq, dq2[sl]), (dk, dk2), (dv, dv2))
    else:
        c = [0, lk]
        o2, l2, dq2, dk2, dv2 = oracle.attn_fwd_bwd_thd(q[lq - lk:], k, v, do[lq - lk:], c, c,
                                                        c, c, 0.45, tl)
        n = lq - lk
        assert np.all(out[:n] == 0) and np.all(dq[:n] == 0) and np.all(np.isneginf(lse[:n]))
        pairs = ((out[n:], o2), (lse[n:], l2), (dq[n:], dq2), (dk, dk2), (dv, dv2))
    for a, b in pairs:
        assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_bottom_right_zero_rows():
    """Lower-right alignment with more queries than keys: the leading queries that
    see no key are exactly 0 in out and dq with lse -inf, and every real key row is
    seen (the last query sees them all)."""
    lq, lk, pq, pk = [7, 2, 3], [3, 5, 0], [8, 4, 3], [4, 5, 2]
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(24, lq, lk, pq, pk, 2, 2, 4, tail=1)
    br = MASK_PADDING_CAUSAL_BOTTOM_RIGHT
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k, 0.5, br)
    qm, km = oracle.valid_row_masks(cu_q, cu_k, cp_q, cp_k, q.shape[0], k.shape[0], br)
    # sequence 0: queries 0-3 see no key; sequence 2 has no key at all
    assert list(np.nonzero(qm)[0]) == [4, 5, 6, 8, 9]
    assert list(np.nonzero(km)[0]) == [0, 1, 2, 4, 5, 6, 7, 8]
    assert np.all(out[~qm] == 0) and np.all(dq[~qm] == 0)
    assert np.all(np.abs(out[qm]).sum(axis=(1, 2)) > 0)
    assert np.all(dk[~km] == 0) and np.all(dv[~km] == 0)
    assert np.all(np.abs(dv[km]).sum(axis=(1, 2)) > 0)
    assert np.all(np.isneginf(lse[[0, 1, 2, 3, 12, 13, 14]]))
    assert np.all(lse[[7, 10, 11, 15]] == 0)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_invariants(mask):
    """Softmax rows sum to 1 (O = 1 for V = 1); LSE = logsumexp of the scaled,
    masked scores (scipy); sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per sequence
    and kv head; sum_i <dQ_i, Q_i> = sum_j <dK_j, K_j> per sequence and kv group."""
    from scipy.special import logsumexp
    lq, lk, pq, pk = [6, 9, 4], [6, 9, 7], [8, 9, 4], [6, 12, 7]
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(6, lq, lk, pq, pk, 4, 2, 8)
    scale = 0.4
    causal = _ALIGN[mask]
    out1, _ = oracle.attn_fwd_thd(q, k, np.ones_like(v), cu_q, cu_k, cp_q, cp_k, scale, mask)
    qm, _ = oracle.valid_row_masks(cu_q, cu_k, cp_q, cp_k, q.shape[0], k.shape[0], mask)
    assert np.allclose(out1[qm], 1.0, atol=1e-14)
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k,
                                                   scale, mask)
    G = 2
    for b in range(3):
        oq, Lq, ok, Lk = cp_q[b], lq[b], cp_k[b], lk[b]
        for g in range(2):
            kk = k[ok:ok + Lk, g]
            for h in range(g * G, g * G + G):
                s = scale * q[oq:oq + Lq, h] @ kk.T
                if causal:
                    # query i sits at position i (upper-left) or Lk - Lq + i (lower-right)
                    pos = np.arange(Lq) + (Lk - Lq if causal == "br" else 0)
                    s = np.where(np.arange(Lk)[None, :] <= pos[:, None], s, -np.inf)
                assert np.allclose(lse[oq:oq + Lq, h], logsumexp(s, axis=1), atol=1e-12)
            assert np.abs(dk[ok:ok + Lk, g].sum(axis=0)).max() < 1e-11
            rows = slice(oq, oq + Lq)
            assert np.allclose(dv[ok:ok + Lk, g].sum(axis=0),
                               do[rows, g * G:g * G + G].sum(axis=(0, 1)), atol=1e-11)
            lhs = (dq[rows, g * G:g * G + G] * q[rows, g * G:g * G + G]).sum()
            rhs = (dk[ok:ok + Lk, g] * kk).sum()
            assert lhs == pytest.approx(rhs, rel=1e-11, abs=1e-11)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_gqa_identity(mask):
    """GQA dK/dV equal the MHA gradients with K/V repeat_interleaved over each
    group and summed back over the group; out/lse/dq are unchanged."""
    lq, lk, pq, pk = [5, 7], [6, 7], [5, 9], [8, 7]
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(7, lq, lk, pq, pk, 6, 2, 4)
    G = 3
    gqa = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k, 0.5, mask)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    mha = oracle.attn_fwd_bwd_thd(q, kr, vr, do, cu_q, cu_k, cp_q, cp_k, 0.5, mask)
    for a, b in zip(gqa[:3], mha[:3]):
        assert np.allclose(a, b, atol=1e-13)
    for a, b in zip(gqa[3:], mha[3:]):
        summed = b.reshape(b.shape[0], 2, G, b.shape[2]).sum(axis=2)
        assert np.allclose(a, summed, atol=1e-12)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_packed_equals_unpacked(mask):
    """THD packing with padded offsets gives, row for row, what each sequence gives
    on its own (offset 0, no padding, batch of 1); pad-slot contents are ignored."""
    lq, lk, pq, pk = [4, 8, 3], [5, 8, 6], [7, 8, 5], [5, 12, 6]
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(8, lq, lk, pq, pk, 2, 1, 6)
    packed = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k, 0.6, mask)
    for b in range(3):
        sq = slice(cp_q[b], cp_q[b] + lq[b])
        sk = slice(cp_k[b], cp_k[b] + lk[b])
        single = oracle.attn_fwd_bwd_thd(
            q[sq], k[sk], v[sk], do[sq], [0, lq[b]], [0, lk[b]], [0, lq[b]], [0, lk[b]],
            0.6, mask)
        for name, a, s in zip(("out", "lse", "dq"), packed[:3], single[:3]):
            assert np.array_equal(a[sq], s), name
        for name, a, s in zip(("dk", "dv"), packed[3:], single[3:]):
            assert np.array_equal(a[sk], s), name
    # changing every pad slot changes nothing
    qm = np.ones(q.shape[0], dtype=bool)
    for b in range(3):
        qm[cp_q[b]:cp_q[b] + lq[b]] = False
    km = np.ones(k.shape[0], dtype=bool)
    for b in range(3):
        km[cp_k[b]:cp_k[b] + lk[b]] = False
    q2, k2, v2, do2 = q.copy(), k.copy(), v.copy(), do.copy()
    q2[qm] = 1e3
    do2[qm] = -1e3
    k2[km] = -1e3
    v2[km] = 1e3
    again = oracle.attn_fwd_bwd_thd(q2, k2, v2, do2, cu_q, cu_k, cp_q, cp_k, 0.6, mask)
    for a, b in zip(packed, again):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_exact_zero_rows(mask):
    """Pad slots, tail rows, empty sequences and key rows no query sees are exactly
    zero in out/lse/dq/dk/dv; rows that may be nonzero are nonzero here."""
    lq, lk, pq, pk = [0, 5, 3, 6], [4, 7, 0, 6], [2, 6, 4, 6], [5, 7, 3, 9]
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(9, lq, lk, pq, pk, 2, 1, 4, tail=3)
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, cu_q, cu_k, cp_q, cp_k,
                                                   0.5, mask)
    qm, km = oracle.valid_row_masks(cu_q, cu_k, cp_q, cp_k, q.shape[0], k.shape[0], mask)
    assert np.all(out[~qm] == 0) and np.all(dq[~qm] == 0)
    assert np.all(dk[~km] == 0) and np.all(dv[~km] == 0)
    assert np.all(np.abs(out[qm]).sum(axis=(1, 2)) > 0)
    assert np.all(np.abs(dv[km]).sum(axis=(1, 2)) > 0)
    # sequence 2 has 3 queries but no key: lse -inf on its real rows, 0 on pad rows
    o2 = cp_q[2]
    assert np.all(np.isneginf(lse[o2:o2 + 3]))
    real_q = np.zeros(q.shape[0], dtype=bool)
    for b in range(4):
        real_q[cp_q[b]:cp_q[b] + lq[b]] = True
    assert np.all(lse[~real_q] == 0)
    if mask == MASK_PADDING_CAUSAL:
        # sequence 3: Lq = Lk = 6, every key seen; sequence 1: Lq 5 < Lk 7 -> keys 5,6 unseen
        o1 = cp_k[1]
        assert np.all(dk[o1 + 5:o1 + 7] == 0) and np.all(dv[o1 + 5:o1 + 7] == 0)


@pytest.mark.parametrize("mask", ALL_MASKS)
def test_sbhd_is_packed_layout_transposed(mask):
    """The sequence-major oracle ([3216]'s layout, q[s, b, h, d]) equals the packed
    oracle on the same values moved to rows b * S + s with padded offsets b * S,
    for ragged real lengths below S (pad slots zero in every output)."""
    rng = np.random.default_rng(11)
    Sq, Sk, B, hq, hkv, d = 9, 7, 3, 4, 2, 5
    q = rng.standard_normal((Sq, B, hq, d))
    k = rng.standard_normal((Sk, B, hkv, d))
    v = rng.standard_normal((Sk, B, hkv, d))
    do = rng.standard_normal((Sq, B, hq, d))
    lq, lk = [9, 4, 0], [5, 7, 3]
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    sb = oracle.attn_fwd_bwd_sbhd(q, k, v, do, cu_q, cu_k, 0.4, mask)
    packed = lambda x: np.ascontiguousarray(np.swapaxes(x, 0, 1)).reshape((-1,) + x.shape[2:])
    cp_q, cp_k = np.arange(B + 1) * Sq, np.arange(B + 1) * Sk
    th = oracle.attn_fwd_bwd_thd(packed(q), packed(k), packed(v), packed(do), cu_q, cu_k,
                                 cp_q, cp_k, 0.4, mask)
    for name, a, t in zip(("out", "lse", "dq", "dk", "dv"), sb, th):
        assert np.array_equal(packed(a), t), name
    assert np.all(sb[0][4:, 1] == 0) and np.all(sb[0][:, 2] == 0) and np.all(sb[3][5:, 0] == 0)


def test_e4m3_decoding_matches_the_format():
    """The e4m3 values the GPU tests hand to the oracle come from torch's
    float8_e4m3fn decoding; every one of the 254 finite codes equals the format's
    definition: sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals at
    exponent 0, and 0x7f / 0xff are NaN (no infinities)."""
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is None:
        pytest.skip("torch without float8_e4m3fn")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    got = codes.view(f8).to(torch.float64).numpy()
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert np.isnan(got[c])
            continue
        mag = 2.0 ** (e - 7) * (1 + m / 8) if e > 0 else 2.0 ** -6 * (m / 8)
        assert got[c] == (-mag if s else mag), c
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e4m3_forward_is_the_dequantised_forward():
    """The e4m3 forward of the oracle equals the float64 forward on the
    dequantised inputs (values times their per-tensor factors)."""
    q, k, v, do, cu_q, cu_k, cp_q, cp_k = _rand_case(31, [5, 9], [7, 4], [6, 9], [8, 4], 4, 2, 16)
    r8 = lambda x: np.round(x * 8) / 8  # any representable values will do here
    a = oracle.attn_fwd_thd_e4m3(r8(q), r8(k), r8(v), 0.5, 0.25, 2.0, cu_q, cu_k, cp_q, cp_k,
                                 0.3, MASK_PADDING_CAUSAL)
    b = oracle.attn_fwd_thd(r8(q) * 0.5, r8(k) * 0.25, r8(v) * 2.0, cu_q, cu_k, cp_q, cp_k, 0.3,
                            MASK_PADDING_CAUSAL)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_e4m3_forward_single_key_closed_form():
    """Closed form of the e4m3 forward with one key per sequence: every query sees
    only key 0, so P = 1, out = v8 * v_descale and
    lse = attn_scale * q_descale * k_descale * <q8, k8>. Distinct descale factors
    make a swapped factor (v's in place of q's or k's), a factor applied twice or
    a missing attn_scale fail."""
    rng = np.random.default_rng(77)
    lq = [3, 5]
    cu_q = np.array([0, 3, 8])
    cp_q = np.array([0, 4, 10])
    cu_k = np.array([0, 1, 2])
    cp_k = np.array([0, 2, 3])
    hq, hkv, d = 4, 2, 16
    q8 = np.round(rng.standard_normal((10, hq, d)) * 4) / 4
    k8 = np.round(rng.standard_normal((3, hkv, d)) * 4) / 4
    v8 = np.round(rng.standard_normal((3, hkv, d)) * 4) / 4
    qd, kd, vd, sc = 0.5, 0.125, 3.0, 0.7
    for mask in (MASK_PADDING, MASK_PADDING_CAUSAL):
        out, lse = oracle.attn_fwd_thd_e4m3(q8, k8, v8, qd, kd, vd, cu_q, cu_k, cp_q, cp_k, sc, mask)
        for b in range(2):
            for i in range(lq[b]):
                r = cp_q[b] + i
                for h in range(hq):
                    g = h // (hq // hkv)
                    kr = cp_k[b]
                    assert np.allclose(out[r, h], v8[kr, g] * vd, rtol=0, atol=1e-12)
                    want = sc * qd * kd * float(q8[r, h] @ k8[kr, g])
                    assert abs(lse[r, h] - want) <= 1e-12 * max(1.0, abs(want))
        assert np.all(out[3] == 0) and np.all(lse[3] == 0)  # pad slot of sequence 0


def test_flop_count_matches_the_mask():
    """The metric's pair count against a brute-force count of the kept (query, key)
    entries of the oracle's own score matrices: equal for the padding mask; for
    either causal mask the convention Lq*Lk/2 sits below the exact triangle
    count sum_i (keys of row i) by Lq/2 when Lq = Lk (it drops the diagonal's
    half), so 3.5 * 4 * d * hq * (count - Lq/2) per sequence reproduces it."""
    from oracle.attention import _scores, _is_causal
    lens = [5, 9, 1, 16]
    cu = np.concatenate([[0], np.cumsum(lens)])
    hq, d = 3, 8
    for mask in (MASK_PADDING, MASK_PADDING_CAUSAL, MASK_PADDING_CAUSAL_BOTTOM_RIGHT):
        kept = 0.0
        half_diag = 0.0
        for L in lens:
            s = _scores(np.ones((L, d)), np.ones((L, d)), 1.0, _is_causal(mask))
            kept += float(np.isfinite(s).sum())
            half_diag += L / 2.0 if mask != MASK_PADDING else 0.0
        want = 3.5 * 4.0 * d * hq * (kept - half_diag)
        assert oracle.fwd_bwd_flops(cu, cu, hq, d, mask) == want, mask


def test_golden_issue2448_zero_rows():
    """[2448] 'Expected behavior': on the second call (query lengths 0 and 3)
    the first 4 tokens of dk and dv are all zero; on the first they are not."""
    g = json.load(open(os.path.join(GOLDEN, "issue2448_expected_zero_rows.json")))
    rng = np.random.default_rng(0)
    T, hq, hkv, d = g["T"], g["hq"], g["hkv"], g["d"]
    q = rng.standard_normal((T, hq, d))
    k = rng.standard_normal((T, hkv, d))
    v = rng.standard_normal((T, hkv, d))
    do = rng.standard_normal((T, hq, d))
    res = {}
    for call, c in g["calls"].items():
        res[call] = oracle.attn_fwd_bwd_thd(
            q, k, v, do, c["cu_seqlens_q"], c["cu_seqlens_kv"], g["cu_seqlens_q_padded"],
            g["cu_seqlens_kv_padded"], g["attn_scale"], g["attn_mask_type"])
    rows = g["expected_zero_dk_dv_rows_call_B"]
    assert np.all(res["B"][3][rows] == 0) and np.all(res["B"][4][rows] == 0)
    assert np.all(np.abs(res["A"][4][0:3]).sum(axis=(1, 2)) > 0)
    assert np.all(res["A"][4][3] == 0)  # row 3 is a pad slot of sequence 0


def test_golden_issue2892_layout():
    """[2892] / TE docstring: real [0,3,5,9] in padded [0,4,8,13]; the output
    keeps the padded shape, real rows carry values, pad rows are zero."""
    g = json.load(open(os.path.join(GOLDEN, "issue2892_te_docstring_layout.json")))
    rng = np.random.default_rng(1)
    T = g["T"]
    q = rng.standard_normal((T, 2, 4))
    k = rng.standard_normal((T, 2, 4))
    v = rng.standard_normal((T, 2, 4))
    do = rng.standard_normal((T, 2, 4))
    cu, cp = g["cu_seqlens"], g["cu_seqlens_padded"]
    out, lse, dq, dk, dv = oracle.attn_fwd_bwd_thd(q, k, v, do, cu, cu, cp, cp, 0.5,
                                                   MASK_PADDING)
    assert out.shape == q.shape
    nz = lambda x: np.abs(x).reshape(T, -1).sum(axis=1) > 0  # noqa: E731
    assert sorted(np.nonzero(nz(out))[0].tolist()) == g["real_rows"]
    assert sorted(np.nonzero(~nz(dq))[0].tolist()) == g["pad_rows"]
    assert sorted(np.nonzero(nz(dv))[0].tolist()) == g["real_rows"]


def test_flop_count():
    """Causal-adjusted fwd+bwd FLOPs: 3.5 * 4 * d * hq * sum(Lq Lk / 2)."""
    f = oracle.fwd_bwd_flops([0, 128, 384], [0, 128, 384], 8, 128, MASK_PADDING_CAUSAL)
    assert f == 3.5 * 4 * 128 * 8 * (128 * 128 / 2 + 256 * 256 / 2)


def test_workloads_recipes():
    """The seeded recipes produce the shapes and layouts the pages describe."""
    from bwd_packed_varlen_gb300 import workloads as W
    w = W.tiny_gqa("B")
    assert tuple(w.q.shape) == (12, 2, 8) and w.q.dtype == torch.float16
    assert w.cu_seqlens_q.tolist() == [0, 0, 3]
    assert W.tiny_gqa("A").q.equal(w.q)
    assert W.throughput_lengths(5) == [5580, 6645, 435, 6668, 3977, 4346, 5117]
    w4 = W.real_ne_padded()
    assert w4.cu_seqlens_q_padded.tolist() == [0, 112, 272, 400, 544]
    assert w4.q[100:112].float().abs().min().item() == 1000.0
    w3 = W.gqa_d256()
    assert tuple(w3.q.shape) == (768, 16, 256) and tuple(w3.k.shape) == (768, 2, 256)
