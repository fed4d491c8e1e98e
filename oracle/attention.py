"""Plain float64 scaled-dot-product attention over packed (THD) sequences.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA path never imports it.

Notation follows the TransformerEngine pages this oracle restates:

* ``q, out, dout, dq`` are ``[T_q, hq, d]``; ``k, v, dk, dv`` are ``[T_kv, hkv, d]``;
  ``lse`` is ``[T_q, hq]`` ([2448], reproduction script: THD tensors
  ``(seqlen, heads, dim)`` and the softmax aux tensor ``(seqlen, hq, 1)``).
* Sequence b occupies rows ``cu_*_padded[b] .. cu_*_padded[b+1]`` of its tensor and
  holds ``cu_*[b+1] - cu_*[b]`` real tokens at the front of that span ([2892],
  "Expected Behavior": real boundaries mask, padded boundaries index memory).
* Query head h reads key/value head ``h // G`` with ``G = hq // hkv`` ([3216],
  ``fp32_reference``: ``repeat_interleave`` of K/V over the group), so dK/dV of a
  key/value head are sums over the G query heads of its group.
* ``attn_scale`` multiplies ``q k^T`` inside the softmax ([2448] passes
  ``attn_scale=0.1``; [3216] divides by sqrt(d)); ``lse`` is the natural log of
  the softmax denominator of the *scaled* scores.
* ``padding_causal`` keeps key j for query i iff ``j <= i`` (upper-left alignment,
  [3216] ``torch.triu(ones, 1)`` masked to -inf).
* ``padding_causal_bottom_right`` keeps key j for query i iff ``j <= i + Lk - Lq``:
  the causal triangle aligned to the last query and the last key. The pages use
  only equal lengths, where the two alignments agree; this variant is the mask
  name TransformerEngine gives the lower-right alignment, restated from its
  definition (query i sits at absolute position ``Lk - Lq + i``).

Readings where the pages are silent:

* A valid query that sees no key (its sequence has no valid key, or the
  bottom-right triangle leaves it none when ``Lq > Lk``) gets ``out = 0``,
  ``lse = -inf`` and ``dq = 0`` (empty-sum convention).
* Every row that is not a real token (pad slots, tails, rows of empty sequences) is
  exactly 0 in ``out, dq`` and ``lse``; key/value rows that are not real tokens, or
  that no valid query sees, are exactly 0 in ``dk, dv``.
* The backward entry takes ``out`` and ``lse`` as inputs, as TransformerEngine's
  ``fused_attn_bwd`` does ([2448] passes ``out`` and ``[lse, rng]``), and forms
  ``P = exp(S - lse)`` and ``D = rowsum(dout * out)`` from them.

Pages cited, by title (keys are the pages' issue numbers):
  [2448] "Inconsistent fused_attn_bwd results of dk, dv under THD layout + GQA on multiple calls"
  [3333] "[Bug] FusedAttention (cuDNN) THD backward produces wrong gradients on sm_120 (RTX 5090); forward is correct, Unfused is correct"
  [3216] "flash-attn-4 4.0.0b11: DotProductAttention batched backward returns wrong dQ/dK/dV at head_dim=256 on Blackwell (sm_100)"
  [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
"""

from __future__ import annotations

import numpy as np

MASK_PADDING = 1
MASK_PADDING_CAUSAL = 2
MASK_PADDING_CAUSAL_BOTTOM_RIGHT = 3

# mask type -> causal alignment: None (no triangle), "tl" (upper-left), "br" (lower-right)
_MASKS = {MASK_PADDING: None, MASK_PADDING_CAUSAL: "tl", MASK_PADDING_CAUSAL_BOTTOM_RIGHT: "br",
          "padding": None, "padding_causal": "tl", "padding_causal_bottom_right": "br"}


def _is_causal(mask_type):
    """Causal alignment of a mask type: None, ``"tl"`` or ``"br"``."""
    if mask_type not in _MASKS:
        raise ValueError(f"unknown mask_type {mask_type!r}")
    return _MASKS[mask_type]


def causal_diagonal(causal, lq, lk):
    """Offset c of the causal boundary: query i keeps key j iff ``j <= i + c``
    (0 for the upper-left triangle, ``Lk - Lq`` for the lower-right one)."""
    return lk - lq if causal == "br" else 0


def seq_spans(cu_seqlens, cu_seqlens_padded):
    """Per sequence ``(offset, real_length)``: offset from the padded prefix sums,
    length from the real ones ([2892], "Expected Behavior", items 1-2)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cp = np.asarray(cu_seqlens_padded, dtype=np.int64)
    if cu.shape != cp.shape or cu.ndim != 1 or cu.size < 2:
        raise ValueError("cu_seqlens and cu_seqlens_padded must both be [B+1]")
    lens = np.diff(cu)
    plens = np.diff(cp)
    if np.any(lens < 0) or np.any(lens > plens):
        raise ValueError("real lengths must be >= 0 and <= padded lengths")
    return [(int(cp[b]), int(lens[b])) for b in range(lens.size)]


def _scores(qh, kg, scale, causal):
    """S = scale * q k^T for one query head, -inf where the mask removes a key."""
    s = scale * (qh @ kg.T)
    if causal:
        lq, lk = s.shape
        c = causal_diagonal(causal, lq, lk)
        s[np.arange(lk)[None, :] > np.arange(lq)[:, None] + c] = -np.inf
    return s


def _softmax_rows(s):
    """``(P, lse)`` of score rows; a row without any kept key gets P = 0 and
    lse = -inf (empty-sum convention)."""
    m = s.max(axis=1)
    seen = np.isfinite(m)
    ms = np.where(seen, m, 0.0)
    e = np.where(seen[:, None], np.exp(s - ms[:, None]), 0.0)
    l = e.sum(axis=1)
    p = np.divide(e, l[:, None], out=np.zeros_like(e), where=seen[:, None])
    with np.errstate(divide="ignore"):
        lse = np.where(seen, ms + np.log(np.where(seen, l, 1.0)), -np.inf)
    return p, lse


def attn_group_fwd_bwd(qg, kg, vg, dog, scale, causal):
    """Forward and exact gradient for one sequence and one key/value head group.

    ``qg, dog``: ``[Lq, G, d]``; ``kg, vg``: ``[Lk, d]``. Returns
    ``(out [Lq,G,d], lse [Lq,G], dq [Lq,G,d], dk [Lk,d], dv [Lk,d])``.

    Forward is the softmax-attention definition ([3216] ``fp32_reference``:
    ``softmax(q k^T / sqrt(d)) v`` with the causal triangle). Backward is the
    gradient of ``sum(dout * out)`` ([3333] and [3216] obtain their reference
    gradients by autograd of this loss): ``dV = P^T dO``, ``dP = dO V^T``,
    ``D_i = sum_j P_ij dP_ij``, ``dS = P (dP - D)``, ``dQ = scale dS K``,
    ``dK = scale dS^T Q``, summed over the G query heads for dK and dV.
    Parity: pinned (finite differences, torch autograd, closed forms, invariants).
    """
    qg = np.asarray(qg, dtype=np.float64)
    kg = np.asarray(kg, dtype=np.float64)
    vg = np.asarray(vg, dtype=np.float64)
    dog = np.asarray(dog, dtype=np.float64)
    lq, G, d = qg.shape
    lk = kg.shape[0]
    out = np.zeros((lq, G, d))
    lse = np.zeros((lq, G))
    dq = np.zeros((lq, G, d))
    dk = np.zeros((lk, d))
    dv = np.zeros((lk, d))
    if lq == 0:
        return out, lse, dq, dk, dv
    if lk == 0:
        lse[:] = -np.inf
        return out, lse, dq, dk, dv
    for j in range(G):
        s = _scores(qg[:, j, :], kg, scale, causal)
        p, lse[:, j] = _softmax_rows(s)
        out[:, j, :] = p @ vg
        do = dog[:, j, :]
        dv += p.T @ do
        dp = do @ vg.T
        dsum = (p * dp).sum(axis=1)
        ds = p * (dp - dsum[:, None])
        dq[:, j, :] = scale * (ds @ kg)
        dk += scale * (ds.T @ qg[:, j, :])
    return out, lse, dq, dk, dv


def attn_group_bwd_given(qg, kg, vg, outg, dog, lseg, scale, causal):
    """Backward for one sequence and key/value group from a supplied ``out``/``lse``.

    This is the interface TransformerEngine's ``fused_attn_bwd`` exposes (issue
    [2448] reproduction: ``q, k, v, out, dout`` plus the aux tensor ``lse``):
    ``P = exp(S - lse)``, ``D = rowsum(dout * out)``, then the same products as
    :func:`attn_group_fwd_bwd`. When ``out, lse`` are the exact forward results the
    two functions agree (``sum_j P_ij dP_ij = dO_i . O_i``).
    Parity: pinned against :func:`attn_group_fwd_bwd` and torch autograd.
    """
    qg = np.asarray(qg, dtype=np.float64)
    kg = np.asarray(kg, dtype=np.float64)
    vg = np.asarray(vg, dtype=np.float64)
    outg = np.asarray(outg, dtype=np.float64)
    dog = np.asarray(dog, dtype=np.float64)
    lseg = np.asarray(lseg, dtype=np.float64)
    lq, G, d = qg.shape
    lk = kg.shape[0]
    dq = np.zeros((lq, G, d))
    dk = np.zeros((lk, d))
    dv = np.zeros((lk, d))
    if lq == 0 or lk == 0:
        return dq, dk, dv
    for j in range(G):
        s = _scores(qg[:, j, :], kg, scale, causal)
        # a row without kept keys contributes nothing (its lse is -inf)
        keep = np.isfinite(s)
        p = np.where(keep, np.exp(np.where(keep, s, 0.0) - np.where(keep, lseg[:, j][:, None], 0.0)), 0.0)
        do = dog[:, j, :]
        dv += p.T @ do
        dp = do @ vg.T
        dsum = (do * outg[:, j, :]).sum(axis=1)
        ds = p * (dp - dsum[:, None])
        dq[:, j, :] = scale * (ds @ kg)
        dk += scale * (ds.T @ qg[:, j, :])
    return dq, dk, dv


def attn_group_error_scales(qg, kg, vg, dog, scale, causal, norm=1):
    """Magnitude sums that bound the rounding error of each output element of one
    sequence and key/value group (test helper for the GPU comparisons).

    An implementation that rounds a product's operand to 16 bits (P before P V and
    P^T dO, dS before dS K and dS^T Q) changes the product by at most u times the
    sum of the absolute values of its terms; one that forms D = rowsum(dout * out)
    from a rounded ``out`` changes D_i by at most u a_i, and with it dS_ij by
    P_ij u a_i. With ``norm=1`` (worst case) this returns, in float64 and the shapes
    of :func:`attn_group_fwd_bwd`'s outputs:
      m_out = |P| |V|
      m_dq  = scale (|dS| |K| + (P * a) |K|)
      m_dk  = scale sum_h (|dS|^T |Q| + (P * a)^T |Q|)
      m_dv  = sum_h |P|^T |dout|
    with a_i = sum_c |dout_ic| (|out_ic| + m_out_ic). With ``norm=2`` the terms of
    each sum are combined as a root of the sum of squares instead (the size of a sum
    of independent rounding errors), except that the D term of a dq row stays
    |a_i| (P |K|): one D_i perturbs every term of that row alike. The products are
    the same ones :func:`attn_group_fwd_bwd` forms, on absolute values.
    Parity: pinned (norm=1 equals the plain products on nonnegative data and bounds
    them from above elementwise; norm=2 lies between the largest term and norm=1)."""
    if norm not in (1, 2):
        raise ValueError("norm must be 1 or 2")
    qg = np.asarray(qg, dtype=np.float64)
    kg = np.asarray(kg, dtype=np.float64)
    vg = np.asarray(vg, dtype=np.float64)
    dog = np.asarray(dog, dtype=np.float64)
    lq, G, d = qg.shape
    lk = kg.shape[0]
    m_out = np.zeros((lq, G, d))
    m_dq = np.zeros((lq, G, d))
    m_dk = np.zeros((lk, d))
    m_dv = np.zeros((lk, d))
    if lq == 0 or lk == 0:
        return m_out, m_dq, m_dk, m_dv
    pw = (lambda x: np.abs(x)) if norm == 1 else (lambda x: x * x)  # per-term power
    root = (lambda x: x) if norm == 1 else np.sqrt
    ak, av = pw(kg), pw(vg)
    for j in range(G):
        s = _scores(qg[:, j, :], kg, scale, causal)
        p, _ = _softmax_rows(s)
        do = dog[:, j, :]
        out = p @ vg
        dp = do @ vg.T
        ds = p * (dp - (p * dp).sum(axis=1)[:, None])
        mo = root(pw(p) @ av)
        m_out[:, j, :] = mo
        a = root(pw(do * (np.abs(out) + mo)).sum(axis=1))
        pa = p * a[:, None]
        d_term = pa @ np.abs(kg)  # one D_i moves the whole row alike
        m_dq[:, j, :] = scale * (root(pw(ds) @ ak) + d_term)
        aq = pw(qg[:, j, :])
        m_dk += pw(scale) * (pw(ds).T @ aq + pw(pa).T @ aq)
        m_dv += pw(p).T @ pw(do)
    if norm == 2:
        m_dk = np.sqrt(m_dk)
        m_dv = np.sqrt(m_dv)
    return m_out, m_dq, m_dk, m_dv


def attn_error_scales_thd(q, k, v, dout, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                          cu_seqlens_kv_padded, attn_scale, mask_type, norm=1):
    """:func:`attn_group_error_scales` over packed sequences: ``(m_out, m_dq, m_dk,
    m_dv)`` in the padded layout of ``(out, dq, dk, dv)``, 0 on rows that are not
    computed; ``norm`` as there. Parity: pinned with :func:`attn_group_error_scales`."""
    causal = _is_causal(mask_type)
    hq, hkv, G = _check_heads(q, k)
    qs = seq_spans(cu_seqlens_q, cu_seqlens_q_padded)
    ks = seq_spans(cu_seqlens_kv, cu_seqlens_kv_padded)
    Tq, _, d = q.shape
    Tk = k.shape[0]
    res = [np.zeros((Tq, hq, d)), np.zeros((Tq, hq, d)), np.zeros((Tk, hkv, d)),
           np.zeros((Tk, hkv, d))]
    for (oq, lq), (ok, lk) in zip(qs, ks):
        for g in range(hkv):
            hs = slice(g * G, (g + 1) * G)
            mo, mq, mk, mv = attn_group_error_scales(
                q[oq:oq + lq, hs], k[ok:ok + lk, g], v[ok:ok + lk, g], dout[oq:oq + lq, hs],
                attn_scale, causal, norm)
            res[0][oq:oq + lq, hs] = mo
            res[1][oq:oq + lq, hs] = mq
            res[2][ok:ok + lk, g] = mk
            res[3][ok:ok + lk, g] = mv
    return tuple(res)


def _check_heads(q, k):
    hq, hkv = q.shape[1], k.shape[1]
    if hkv < 1 or hq % hkv != 0:
        raise ValueError("hq must be a positive multiple of hkv")
    return hq, hkv, hq // hkv


def attn_fwd_bwd_thd(q, k, v, dout, cu_seqlens_q, cu_seqlens_kv,
                     cu_seqlens_q_padded, cu_seqlens_kv_padded, attn_scale,
                     mask_type):
    """THD forward + backward: ``(out, lse, dq, dk, dv)`` in float64, padded layout.

    Loops over sequences and key/value heads and calls :func:`attn_group_fwd_bwd`
    on the real rows; every other row stays exactly 0 ([2448] "Expected
    behavior"; [2892]: output keeps the padded shape of Q).
    Parity: pinned.
    """
    causal = _is_causal(mask_type)
    hq, hkv, G = _check_heads(q, k)
    qs = seq_spans(cu_seqlens_q, cu_seqlens_q_padded)
    ks = seq_spans(cu_seqlens_kv, cu_seqlens_kv_padded)
    if len(qs) != len(ks):
        raise ValueError("q and kv cu_seqlens describe different batch sizes")
    Tq, _, d = q.shape
    Tk = k.shape[0]
    out = np.zeros((Tq, hq, d))
    lse = np.zeros((Tq, hq))
    dq = np.zeros((Tq, hq, d))
    dk = np.zeros((Tk, hkv, d))
    dv = np.zeros((Tk, hkv, d))
    for (oq, lq), (ok, lk) in zip(qs, ks):
        if oq + lq > Tq or ok + lk > Tk:
            raise ValueError("padded offsets run past the tensors")
        for g in range(hkv):
            hs = slice(g * G, (g + 1) * G)
            o, l, a, b_, c = attn_group_fwd_bwd(
                q[oq:oq + lq, hs], k[ok:ok + lk, g], v[ok:ok + lk, g],
                dout[oq:oq + lq, hs], attn_scale, causal)
            out[oq:oq + lq, hs] = o
            lse[oq:oq + lq, hs] = l
            dq[oq:oq + lq, hs] = a
            dk[ok:ok + lk, g] = b_
            dv[ok:ok + lk, g] = c
    return out, lse, dq, dk, dv


def attn_fwd_thd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                 cu_seqlens_kv_padded, attn_scale, mask_type):
    """THD forward only: ``(out, lse)``. Same arithmetic as the forward half of
    :func:`attn_fwd_bwd_thd` (called with a zero upstream gradient).
    Parity: pinned."""
    zero = np.zeros(q.shape)
    out, lse, _, _, _ = attn_fwd_bwd_thd(
        q, k, v, zero, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
        cu_seqlens_kv_padded, attn_scale, mask_type)
    return out, lse


def attn_bwd_thd(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_kv,
                 cu_seqlens_q_padded, cu_seqlens_kv_padded, attn_scale, mask_type):
    """THD backward from supplied ``out`` and ``lse``: ``(dq, dk, dv)`` float64.

    The interface of TransformerEngine's ``fused_attn_bwd`` ([2448]
    reproduction). Rows that are not real tokens, and key/value rows that no valid
    query sees, are exactly 0.
    Parity: pinned."""
    causal = _is_causal(mask_type)
    hq, hkv, G = _check_heads(q, k)
    qs = seq_spans(cu_seqlens_q, cu_seqlens_q_padded)
    ks = seq_spans(cu_seqlens_kv, cu_seqlens_kv_padded)
    if len(qs) != len(ks):
        raise ValueError("q and kv cu_seqlens describe different batch sizes")
    Tq, _, d = q.shape
    Tk = k.shape[0]
    dq = np.zeros((Tq, hq, d))
    dk = np.zeros((Tk, hkv, d))
    dv = np.zeros((Tk, hkv, d))
    for (oq, lq), (ok, lk) in zip(qs, ks):
        for g in range(hkv):
            hs = slice(g * G, (g + 1) * G)
            a, b_, c = attn_group_bwd_given(
                q[oq:oq + lq, hs], k[ok:ok + lk, g], v[ok:ok + lk, g],
                out[oq:oq + lq, hs], dout[oq:oq + lq, hs], lse[oq:oq + lq, hs],
                attn_scale, causal)
            dq[oq:oq + lq, hs] = a
            dk[ok:ok + lk, g] = b_
            dv[ok:ok + lk, g] = c
    return dq, dk, dv


def attn_fwd_thd_e4m3(q8, k8, v8, q_descale, k_descale, v_descale, cu_seqlens_q,
                      cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, attn_scale,
                      mask_type):
    """Forward from 8-bit e4m3 inputs with per-tensor dequantisation factors:
    ``q8, k8, v8`` are the e4m3 values already decoded to numbers (the stored byte's
    value), and the attention runs on ``q8 * q_descale`` etc. exactly as
    :func:`attn_fwd_thd` does. The pages give no FP8 arithmetic beyond [2892]'s
    failing forward with real != padded lengths; the per-tensor factors are this
    package's reading. Returns ``(out, lse)`` float64.
    Parity: pinned by the one-key closed form (out = v8 * v_descale, lse =
    attn_scale * q_descale * k_descale * <q8, k8>) and through :func:`attn_fwd_thd`;
    the e4m3 decoding it relies on is pinned code by code against the format's
    definition in the tests."""
    q = np.asarray(q8, dtype=np.float64) * float(q_descale)
    k = np.asarray(k8, dtype=np.float64) * float(k_descale)
    v = np.asarray(v8, dtype=np.float64) * float(v_descale)
    return attn_fwd_thd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                        cu_seqlens_kv_padded, attn_scale, mask_type)


def attn_fwd_bwd_sbhd(q, k, v, dout, cu_seqlens_q, cu_seqlens_kv, attn_scale, mask_type):
    """Sequence-major forward + backward: ``q, dout [S_q, B, hq, d]``, ``k, v
    [S_kv, B, hkv, d]`` (the layout of [3216]'s reproduction, whose
    ``fp32_reference`` indexes ``q[s, b, hq, d]``). Batch entry b holds
    ``cu_seqlens_*[b+1] - cu_seqlens_*[b]`` real tokens at its front; the rest are
    pad slots. Returns ``(out, lse [S_q, B, hq], dq, dk, dv)`` float64, exactly 0 on
    pad slots (lse 0; -inf on real queries that see no key), computed per batch
    entry and key/value head by :func:`attn_group_fwd_bwd`.
    Parity: pinned (equals :func:`attn_fwd_bwd_thd` on the same data laid out as
    packed sequences)."""
    causal = _is_causal(mask_type)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    Sq, B, hq, d = q.shape
    Sk, Bk, hkv, _ = k.shape
    if Bk != B:
        raise ValueError("q and k hold different batch sizes")
    if hkv < 1 or hq % hkv != 0:
        raise ValueError("hq must be a positive multiple of hkv")
    G = hq // hkv
    lq = np.diff(np.asarray(cu_seqlens_q, dtype=np.int64))
    lk = np.diff(np.asarray(cu_seqlens_kv, dtype=np.int64))
    if lq.size != B or lk.size != B:
        raise ValueError("cu_seqlens must be [B+1]")
    if np.any(lq < 0) or np.any(lk < 0) or np.any(lq > Sq) or np.any(lk > Sk):
        raise ValueError("real lengths must lie in [0, S]")
    out = np.zeros((Sq, B, hq, d))
    lse = np.zeros((Sq, B, hq))
    dq = np.zeros((Sq, B, hq, d))
    dk = np.zeros((Sk, B, hkv, d))
    dv = np.zeros((Sk, B, hkv, d))
    for b in range(B):
        nq, nk = int(lq[b]), int(lk[b])
        for g in range(hkv):
            hs = slice(g * G, (g + 1) * G)
            o, l, a, b_, c = attn_group_fwd_bwd(q[:nq, b, hs], k[:nk, b, g], v[:nk, b, g],
                                                dout[:nq, b, hs], attn_scale, causal)
            out[:nq, b, hs] = o
            lse[:nq, b, hs] = l
            dq[:nq, b, hs] = a
            dk[:nk, b, g] = b_
            dv[:nk, b, g] = c
    return out, lse, dq, dk, dv


def valid_row_masks(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                    cu_seqlens_kv_padded, T_q, T_kv, mask_type):
    """Which rows may be nonzero: ``(q_rows [T_q], kv_rows [T_kv])`` booleans.

    A query row may be nonzero iff it is a real token that sees at least one real
    key; a key/value row may be nonzero in dk/dv iff it is a real token that some
    real query sees (padding: the sequence has a query; padding_causal: also its
    index is below the query length, since query i sees keys j <= i;
    padding_causal_bottom_right: every real key, since the last query sees all).
    Every other row must be exactly 0 ([2448] "Expected behavior").
    Parity: pinned by the golden fixtures of [2448] and [2892].
    """
    causal = _is_causal(mask_type)
    qs = seq_spans(cu_seqlens_q, cu_seqlens_q_padded)
    ks = seq_spans(cu_seqlens_kv, cu_seqlens_kv_padded)
    qm = np.zeros(T_q, dtype=bool)
    km = np.zeros(T_kv, dtype=bool)
    for (oq, lq), (ok, lk) in zip(qs, ks):
        if lk > 0:
            # query i sees key 0 iff 0 <= i + c
            first = max(0, -causal_diagonal(causal, lq, lk)) if causal else 0
            qm[oq + min(first, lq):oq + lq] = True
        if lq > 0:
            seen = min(lk, lq + causal_diagonal(causal, lq, lk)) if causal else lk
            km[ok:ok + max(seen, 0)] = True
    return qm, km


def fwd_bwd_flops(cu_seqlens_q, cu_seqlens_kv, hq, d, mask_type):
    """Causal-adjusted algorithmic FLOPs of forward + backward (test helper).

    Per (sequence, query head): ``F_fwd = 4 d pairs`` with ``pairs = Lq Lk``
    (padding) or ``Lq Lk / 2`` (either causal alignment); forward + backward is ``3.5 F_fwd``
    (2 GEMMs forward, 5 backward).
    Parity: pinned against a brute-force count of the kept entries of the score
    matrices."""
    causal = _is_causal(mask_type)
    lq = np.diff(np.asarray(cu_seqlens_q, dtype=np.int64)).astype(np.float64)
    lk = np.diff(np.asarray(cu_seqlens_kv, dtype=np.int64)).astype(np.float64)
    pairs = lq * lk * (0.5 if causal else 1.0)
    return float(3.5 * 4.0 * d * hq * pairs.sum())
