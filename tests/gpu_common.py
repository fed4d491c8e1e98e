"""Helpers shared by the GPU tests: run the CUDA path through the C ABI binding,
run the CPU oracle on the same inputs, and compare with the stated tolerances."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the GPU path against the float64 oracle (bf16/fp16 inputs):
# relative Frobenius error <= 1e-2 on out/dq/dk/dv, cosine >= 0.9999,
# |lse - ref| <= 1e-3 on real query rows; rows that must be zero are exactly 0.
REL_TOL = 1e-2
COS_TOL = 0.9999
LSE_TOL = 1e-3
# Row by row and element by element (a row is one token's d values of one head):
#   |x_r - ref_r|   <= ROW_TOL  * (|ref_r| + rms)      for every row r,
#   |x_e - ref_e|   <= ELEM_TOL * (|ref_e| + (|ref_r| + rms) / sqrt(d)) for every element,
# rms = root-mean-square norm of the reference's nonzero rows. ROW_TOL is 8 bf16
# unit roundoffs (8 * 2^-8): the 16-bit roundings a row goes through (P or dS before
# the second product, the output, and D from the stored output) each add at most
# one unit relative to the row's scale; the rms term keeps rows that are small
# because of cancellation (dQ rows sum dS_ij K_j with sum_j dS_ij = 0) on the
# tensor's scale. ELEM_TOL adds the same allowance per element on the element's
# own size plus its row's typical element size.
ROW_TOL = 8.0 * 2.0 ** -8
ELEM_TOL = 8.0 * 2.0 ** -8


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


def row_elem_check(got, ref):
    """Worst row and element ratios to their bounds (<= 1 passes); see ROW_TOL."""
    a = np.asarray(got, dtype=np.float64)
    b = np.asarray(ref, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    d = b.shape[-1]
    a2, b2 = a.reshape(-1, d), b.reshape(-1, d)
    rn = np.linalg.norm(b2, axis=1)
    nz = rn > 0
    rms = float(np.sqrt(np.mean(rn[nz] ** 2))) if nz.any() else 0.0
    err = np.linalg.norm(a2 - b2, axis=1)
    row_bound = ROW_TOL * (rn + rms)
    with np.errstate(divide="ignore", invalid="ignore"):
        row_ratio = np.where(row_bound > 0, err / row_bound, np.where(err > 0, np.inf, 0.0))
        elem_bound = ELEM_TOL * (np.abs(b2) + ((rn + rms) / np.sqrt(d))[:, None])
        ediff = np.abs(a2 - b2)
        elem_ratio = np.where(elem_bound > 0, ediff / elem_bound, np.where(ediff > 0, np.inf, 0.0))
    r = int(np.argmax(row_ratio)) if row_ratio.size else 0
    e = np.unravel_index(int(np.argmax(elem_ratio)), elem_ratio.shape) if elem_ratio.size else (0, 0)
    return {"row_ratio": float(row_ratio.max()) if row_ratio.size else 0.0, "row": r,
            "row_err": float(err[r]) if err.size else 0.0, "row_norm": float(rn[r]) if rn.size else 0.0,
            "elem_ratio": float(elem_ratio.max()) if elem_ratio.size else 0.0,
            "elem": tuple(int(x) for x in e), "rms": rms}


def assert_close(name, got, ref):
    """Whole tensor (rel. Frobenius, cosine), then every row and every element."""
    rel, cos = rel_cos(got, ref)
    assert rel <= REL_TOL and cos >= COS_TOL, f"{name}: rel={rel:.3e} cos={cos:.6f}"
    m = row_elem_check(got, ref)
    assert m["row_ratio"] <= 1.0, (
        f"{name}: row {m['row']} error {m['row_err']:.3e} exceeds {ROW_TOL:.3g} * (|ref_r| "
        f"{m['row_norm']:.3e} + rms {m['rms']:.3e}) by {m['row_ratio']:.2f}x")
    assert m["elem_ratio"] <= 1.0, (
        f"{name}: element {m['elem']} exceeds its bound by {m['elem_ratio']:.2f}x")
    return rel, cos


def check_against_oracle(w, res, ref=None):
    """Compare GPU (out, lse, dq, dk, dv) to the oracle; returns a metrics dict."""
    ref = ref if ref is not None else oracle_fwd_bwd(w)
    out, lse, dq, dk, dv = (np64(x) for x in res)
    r_out, r_lse, r_dq, r_dk, r_dv = ref
    qm, km = oracle.valid_row_masks(
        w.cu_seqlens_q.numpy(), w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
        w.cu_seqlens_kv_padded.numpy(), w.q.shape[0], w.k.shape[0], w.mask_type)
    m = {}
    for name, a, b in (("out", out, r_out), ("dq", dq, r_dq), ("dk", dk, r_dk), ("dv", dv, r_dv)):
        m[name] = assert_close(name, a, b)
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
