"""Helpers shared by the GPU tests: run the CUDA path through the C ABI binding,
run the CPU oracle on the same inputs, and compare with the stated tolerances."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from bwd_packed_varlen_gb300 import workloads as W

# Tolerances of the GPU path against the float64 oracle (bf16/fp16 inputs):
# relative Frobenius error <= 1e-2 on out/dq/dk/dv, cosine >= 0.9999,
# |lse - ref| <= 1e-3 on real query rows; rows that must be zero are exactly 0.
REL_TOL = 1e-2
COS_TOL = 0.9999
LSE_TOL = 1e-3
# Element by element and row by row (a row is one token's d values of one head):
#   |x_e - ref_e|   <= ERR_C * u * (m1_e + |ref_e|)            every element,
#   ||x_r - ref_r|| <= ROW_C * u * ||m2_r + |ref_r|||          every row,
# with u the unit roundoff of the storage type (2^-8 bf16, 2^-11 fp16) and m1, m2
# the oracle's magnitude sums (oracle.attn_group_error_scales, norm 1 and 2): |P||V|
# for out, scale (|dS||K| + (P a)|K|) for dq, and so on. Rounding an operand of a
# product to 16 bits (P, dS) moves each term by at most u times its size, rounding
# the result moves it by at most u |x|, and D = rowsum(dO * out) from a rounded out
# moves dS through a; so u (m1 + |ref|) bounds the kernels' roundings in the worst
# case, and u (m2 + |ref|) is the size of the same errors when they are independent
# (added in quadrature). A numpy emulation of those rounding steps reaches 0.95 of
# the first and 0.98 of the second (tests/test_checker.py); ERR_C = 2 and ROW_C = 3
# leave room for the fp32 accumulation and exp2 approximation on top. The row check
# is the one that sees a systematic mistake in a row whose terms cancel (a dk row
# scaled by 10 %), which the worst-case element bound cannot.
ERR_C = 2.0
ROW_C = 3.0
UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11,
                 torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


def to_dev(w, dev="cuda"):
    return {
        "q": w.q.to(dev), "k": w.k.to(dev), "v": w.v.to(dev), "dout": w.dout.to(dev),
        "cu_q": w.cu_seqlens_q.to(dev), "cu_kv": w.cu_seqlens_kv.to(dev),
        "cu_q_pad": w.cu_seqlens_q_padded.to(dev), "cu_kv_pad": w.cu_seqlens_kv_padded.to(dev),
    }


def gpu_fwd_bwd(w, t=None, **kw):
    import bwd_packed_varlen_gb300 as ta
    t = t or to_dev(w)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    out, lse = ta.fwd(t["q"], t["k"], t["v"], *cu, w.attn_scale, w.mask_type,
                      w.max_seqlen_q, w.max_seqlen_kv, **kw.get("fwd", {}))
    dq, dk, dv = ta.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, w.attn_scale,
                        w.mask_type, w.max_seqlen_q, w.max_seqlen_kv, **kw.get("bwd", {}))
    torch.cuda.synchronize()
    return out, lse, dq, dk, dv


def np64(x):
    return x.detach().to("cpu", torch.float64).numpy()


def oracle_fwd_bwd(w):
    return oracle.attn_fwd_bwd_thd(
        np64(w.q), np64(w.k), np64(w.v), np64(w.dout), w.cu_seqlens_q.numpy(),
        w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
        w.cu_seqlens_kv_padded.numpy(), w.attn_scale, w.mask_type)


def rel_cos(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    nb = np.linalg.norm(b)
    na = np.linalg.norm(a)
    if nb == 0:
        return (0.0 if na == 0 else np.inf), 1.0 if na == 0 else 0.0
    return float(np.linalg.norm(a - b) / nb), float(a @ b / (na * nb)) if na > 0 else 0.0


def row_elem_check(got, ref, ms, u):
    """Worst element ratio to ERR_C * u * (m1 + |ref|) and worst row ratio to
    ROW_C * u * ||m2 + |ref||| (<= 1 passes); ms = (m1, m2)."""
    m1, m2 = ms
    a = np.asarray(got, dtype=np.float64)
    b = np.asarray(ref, dtype=np.float64)
    assert a.shape == b.shape == np.shape(m1) == np.shape(m2), (a.shape, b.shape)
    d = b.shape[-1]
    a2, b2 = a.reshape(-1, d), b.reshape(-1, d)
    m1 = np.asarray(m1, dtype=np.float64).reshape(-1, d)
    m2 = np.asarray(m2, dtype=np.float64).reshape(-1, d)
    diff = np.abs(a2 - b2)
    bound = ERR_C * u * (m1 + np.abs(b2))
    rb = ROW_C * u * np.linalg.norm(m2 + np.abs(b2), axis=1)
    rd = np.linalg.norm(diff, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, diff / bound, np.where(diff > 0, np.inf, 0.0))
        row_ratio = np.where(rb > 0, rd / rb, np.where(rd > 0, np.inf, 0.0))
    if ratio.size == 0:
        return {"elem_ratio": 0.0, "row_ratio": 0.0, "elem": (0, 0), "row": 0}
    e = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    r = int(np.argmax(row_ratio))
    return {"elem_ratio": float(ratio[e]), "elem": tuple(int(x) for x in e),
            "elem_got": float(a2[e]), "elem_ref": float(b2[e]), "elem_m": float(m1[e]),
            "row_ratio": float(row_ratio[r]), "row": r, "row_err": float(rd[r]),
            "row_norm": float(np.linalg.norm(b2[r]))}


def assert_close(name, got, ref, ms, u):
    """Whole tensor (relative Frobenius error and cosine), then every element and
    every row against the bounds above; ms = (m1, m2) magnitude sums of this tensor."""
    rel, cos = rel_cos(got, ref)
    assert rel <= REL_TOL and cos >= COS_TOL, f"{name}: rel={rel:.3e} cos={cos:.6f}"
    c = row_elem_check(got, ref, ms, u)
    assert c["elem_ratio"] <= 1.0, (
        f"{name}: element {c['elem']} = {c['elem_got']:.6g}, oracle {c['elem_ref']:.6g}, "
        f"magnitude sum {c['elem_m']:.4g}: {c['elem_ratio']:.2f}x its bound")
    assert c["row_ratio"] <= 1.0, (
        f"{name}: row {c['row']} error {c['row_err']:.4g} (row norm {c['row_norm']:.4g}): "
        f"{c['row_ratio']:.2f}x its bound")
    return rel, cos


def error_scales(w):
    """Oracle magnitude sums of a workload: ``[(m1, m2)]`` for out, dq, dk, dv."""
    args = (np64(w.q), np64(w.k), np64(w.v), np64(w.dout), w.cu_seqlens_q.numpy(),
            w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
            w.cu_seqlens_kv_padded.numpy(), w.attn_scale, w.mask_type)
    m1 = oracle.attn_error_scales_thd(*args, norm=1)
    m2 = oracle.attn_error_scales_thd(*args, norm=2)
    return list(zip(m1, m2))


def check_against_oracle(w, res, ref=None):
    """Compare GPU (out, lse, dq, dk, dv) to the oracle; returns a metrics dict."""
    ref = ref if ref is not None else oracle_fwd_bwd(w)
    out, lse, dq, dk, dv = (np64(x) for x in res)
    r_out, r_lse, r_dq, r_dk, r_dv = ref
    qm, km = oracle.valid_row_masks(
        w.cu_seqlens_q.numpy(), w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
        w.cu_seqlens_kv_padded.numpy(), w.q.shape[0], w.k.shape[0], w.mask_type)
    scales = error_scales(w)
    u = UNIT_ROUNDOFF[w.dtype]
    m = {}
    for name, a, b, ms in zip(("out", "dq", "dk", "dv"), (out, dq, dk, dv),
                              (r_out, r_dq, r_dk, r_dv), scales):
        m[name] = assert_close(name, a, b, ms, u)
    # exact zeros where nothing may be nonzero
    assert np.all(out[~qm] == 0), "out: nonzero pad row"
    assert np.all(dq[~qm] == 0), "dq: nonzero pad row"
    assert np.all(dk[~km] == 0), "dk: nonzero pad/unseen row"
    assert np.all(dv[~km] == 0), "dv: nonzero pad/unseen row"
    fin = np.isfinite(r_lse)
    assert np.array_equal(np.isneginf(lse), np.isneginf(r_lse)), "lse: -inf rows differ"
    err = np.abs(lse[fin] - r_lse[fin]).max() if fin.any() else 0.0
    assert err <= LSE_TOL, f"lse: max abs err {err:.3e}"
    m["lse"] = float(err)
    return m


def random_configs(n=16, seed=2026):
    """Seeded draws over the supported parameter space: head dim any multiple of 8
    in [8, 256], 1-4 query heads per kv head, every mask, both 16-bit types, 1-6
    sequences of 0-350 rows with independent query and key lengths."""
    rng = np.random.default_rng(seed)
    masks = [W.MASK_PADDING, W.MASK_PADDING_CAUSAL, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT]
    out = []
    for i in range(n):
        d = 8 * int(rng.integers(1, 33))
        hkv = int(rng.choice([1, 2, 4]))
        hq = hkv * int(rng.integers(1, 5))
        out.append((100 + i, int(rng.integers(1, 7)), int(rng.integers(1, 351)), hq, hkv, d,
                    masks[int(rng.integers(0, 3))], ["bf16", "fp16"][int(rng.integers(0, 2))]))
    return out
