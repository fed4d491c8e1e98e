"""The parity checker of the GPU tests, checked on the CPU.

The bounds of tests/gpu_common.py (every element within ERR_C * u * (m1 + |ref|),
every row within ROW_C * u * ||m2 + |ref|||) are derived from the arithmetic the
kernels do: 16-bit rounding of P before P V and P^T dO, of dS before dS K and
dS^T Q, of the outputs, and D formed from the rounded out. Here those steps are
emulated in numpy on top of the oracle's float64 values; the emulated results must
stay within the bounds with their factors ERR_C and ROW_C taken out, on the pages'
workloads (peaked outlier softmax, pad slots of +-1e3, fp16, d = 8). The checker
must also accept the oracle's result rounded to 16 bits and reject the single-row
mistakes a wrong kernel makes -- a sign flip, a row scaled by 10 %, a row taken
from the neighbouring token, one element off by a typical element's size -- which
the whole-tensor norms alone can hide.
"""

import numpy as np
import pytest
import torch

import oracle
from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import ERR_C, ROW_C, UNIT_ROUNDOFF, assert_close, row_elem_check
from oracle.attention import _is_causal, _scores


def _r16(x, dt):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dt).double().numpy()


def _emulate_group(qg, kg, vg, dog, scale, causal, dt):
    """The kernels' rounding steps for one sequence and key/value group: forward
    with unnormalised P rounded to 16 bits before P V, O divided by the fp32 sum
    and rounded; backward with P = exp(S - lse), D from the rounded O, P and dS
    rounded before their products, outputs rounded."""
    lq, G, d = qg.shape
    lk = kg.shape[0]
    out = np.zeros((lq, G, d))
    dq = np.zeros((lq, G, d))
    dk = np.zeros((lk, d))
    dv = np.zeros((lk, d))
    for j in range(G):
        s = _scores(qg[:, j], kg, scale, causal)
        m = s.max(axis=1)
        seen = np.isfinite(m)
        ms = np.where(seen, m, 0.0)
        pt = np.where(seen[:, None], np.exp(s - ms[:, None]), 0.0)
        l = pt.sum(axis=1)
        o = _r16((_r16(pt, dt) @ vg) / np.where(l > 0, l, 1.0)[:, None], dt)
        lse = np.where(seen, ms + np.log(np.where(l > 0, l, 1.0)), 0.0)
        out[:, j] = o
        keep = np.isfinite(s)
        p = np.where(keep, np.exp(np.where(keep, s, 0.0) - lse[:, None]), 0.0)
        do = dog[:, j]
        dv += _r16(p, dt).T @ do
        ds = p * (do @ vg.T - (do * o).sum(axis=1)[:, None])
        dq[:, j] = scale * (_r16(ds, dt) @ kg)
        dk += scale * (_r16(ds, dt).T @ qg[:, j])
    return tuple(_r16(x, dt) for x in (out, dq, dk, dv))


EMULATED = {
    "gqa_d256_set": lambda: W.gqa_d256(),
    "gqa_d256_mul": lambda: W.gqa_d256(outlier_mode="mul"),
    "real_ne_padded_causal": lambda: W.real_ne_padded(mask_type=W.MASK_PADDING_CAUSAL, H=8),
    "packings_128_96": lambda: W.packings([128, 96]),
    "ragged_fp16_d128": lambda: W.random_varlen(13, 3, 260, 6, 3, 128, W.MASK_PADDING_CAUSAL, "fp16"),
    "ragged_fp16_d8": lambda: W.random_varlen(14, 4, 200, 2, 1, 8, W.MASK_PADDING, "fp16"),
    "ragged_bottom_right": lambda: W.random_varlen(22, 6, 500, 4, 2, 64,
                                                   W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT, "bf16"),
}


@pytest.mark.parametrize("name", sorted(EMULATED))
def test_emulated_kernel_rounding_within_the_bound(name):
    w = EMULATED[name]()
    dt = w.q.dtype
    u = UNIT_ROUNDOFF[w.dtype]
    q, k, v, do = (x.double().numpy() for x in (w.q, w.k, w.v, w.dout))
    causal = _is_causal(w.mask_type)
    G = w.hq // w.hkv
    cq, ck = w.cu_seqlens_q.numpy(), w.cu_seqlens_kv.numpy()
    pq, pk = w.cu_seqlens_q_padded.numpy(), w.cu_seqlens_kv_padded.numpy()
    worst = 0.0
    for b in range(w.batch):
        oq, lq, ok, lk = pq[b], cq[b + 1] - cq[b], pk[b], ck[b + 1] - ck[b]
        if lq == 0 or lk == 0:
            continue
        for g in range(w.hkv):
            hs = slice(g * G, g * G + G)
            args = (q[oq:oq + lq, hs], k[ok:ok + lk, g], v[ok:ok + lk, g], do[oq:oq + lq, hs],
                    w.attn_scale, causal)
            ref = oracle.attn_group_fwd_bwd(*args)
            ms = zip(*(oracle.attn_group_error_scales(*args, norm=n) for n in (1, 2)))
            emu = _emulate_group(*args, dt)
            for e, r, m in zip(emu, (ref[0], ref[2], ref[3], ref[4]), ms):
                c = row_elem_check(e, r, m, u)
                # the emulation must stay within the bounds without their factors
                worst = max(worst, c["elem_ratio"] * ERR_C, c["row_ratio"] * ROW_C)
    assert worst <= 1.0, worst


def _case(seed=5, L=(300, 180, 77), hq=4, hkv=2, d=64):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(L)])
    T = int(cu[-1])
    q = rng.standard_normal((T, hq, d))
    k = rng.standard_normal((T, hkv, d))
    v = rng.standard_normal((T, hkv, d))
    do = rng.standard_normal((T, hq, d))
    args = (q, k, v, do, cu, cu, cu, cu, d ** -0.5, oracle.MASK_PADDING_CAUSAL)
    ref = oracle.attn_fwd_bwd_thd(*args)
    m = list(zip(*(oracle.attn_error_scales_thd(*args, norm=n) for n in (1, 2))))
    return (ref[0], ref[2], ref[3], ref[4]), m


def _bf16(x):
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


U = UNIT_ROUNDOFF["bf16"]


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_rounded_result_passes(idx):
    refs, ms = _case()
    assert_close("rounded", _bf16(refs[idx]), refs[idx], ms[idx], U)


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
@pytest.mark.parametrize("mistake", ["sign", "scale", "shift", "element"])
def test_single_row_mistakes_fail(idx, mistake):
    refs, ms = _case()
    ref, m = refs[idx], ms[idx]
    got = _bf16(ref).copy()
    flat = got.reshape(-1, got.shape[-1])
    rn = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    r = int(np.argsort(rn)[len(rn) // 2 + 7])  # a row of median size
    if mistake == "sign":
        flat[r] = -flat[r]
    elif mistake == "scale":
        flat[r] = 1.1 * flat[r]
    elif mistake == "shift":
        flat[r] = flat[r + 1]
    else:
        flat[r, 3] += rn.mean() / np.sqrt(flat.shape[1])  # one typical element size
    with pytest.raises(AssertionError):
        assert_close(mistake, got, ref, m, U)


def test_error_scales_are_the_products_on_nonnegative_data():
    """With nonnegative q, k, v and dout the magnitude sum of out is out itself,
    and every magnitude sum bounds its plain product from above."""
    rng = np.random.default_rng(9)
    cu = np.array([0, 7, 19])
    q, k, v = (np.abs(rng.standard_normal((19, h, 8))) for h in (4, 2, 2))
    do = np.abs(rng.standard_normal((19, 4, 8)))
    args = (q, k, v, do, cu, cu, cu, cu, 0.3, oracle.MASK_PADDING_CAUSAL)
    out, _, dq, dk, dv = oracle.attn_fwd_bwd_thd(*args)
    m_out, m_dq, m_dk, m_dv = oracle.attn_error_scales_thd(*args)
    assert np.allclose(m_out, out, rtol=1e-13, atol=0)
    assert np.allclose(m_dv, dv, rtol=1e-13, atol=0)
    q2, k2, v2, do2 = (rng.standard_normal(x.shape) for x in (q, k, v, do))
    args2 = (q2, k2, v2, do2, cu, cu, cu, cu, 0.3, oracle.MASK_PADDING)
    out, _, dq, dk, dv = oracle.attn_fwd_bwd_thd(*args2)
    m1 = oracle.attn_error_scales_thd(*args2)
    m2 = oracle.attn_error_scales_thd(*args2, norm=2)
    for x, a, b in zip((out, dq, dk, dv), m1, m2):
        assert np.all(np.abs(x) <= a * (1 + 1e-12) + 1e-15)
        assert np.all(b <= a * (1 + 1e-12) + 1e-15)  # root of squares <= sum of sizes
