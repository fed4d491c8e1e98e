"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on the
workloads of the TransformerEngine pages, ragged edge cases, and the determinism
requirements (call order, buffer contents, allocator churn).

Pages cited, by title (keys are the pages' issue numbers):
  [2448] "Inconsistent fused_attn_bwd results of dk, dv under THD layout + GQA on multiple calls"
  [3333] "[Bug] FusedAttention (cuDNN) THD backward produces wrong gradients on sm_120 (RTX 5090); forward is correct, Unfused is correct"
  [3216] "flash-attn-4 4.0.0b11: DotProductAttention batched backward returns wrong dQ/dK/dV at head_dim=256 on Blackwell (sm_100)"
  [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
"""

import numpy as np
import pytest
import torch

import oracle
from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import (
    UNIT_ROUNDOFF,
    assert_close,
    row_elem_check,
    check_against_oracle,
    error_scales,
    gpu_fwd_bwd,
    np64,
    oracle_fwd_bwd,
    random_configs,
    to_dev,
)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import bwd_packed_varlen_gb300 as ta
    ta.library()


# --------------------------------------------------------------------- configs


def test_tiny_gqa_call_order_and_zero_rows():
    """[2448]: calls A then B and B then A give identical results, and in call B
    (empty first query sequence) dk/dv rows 0-3 are exactly zero."""
    wa, wb = W.tiny_gqa("A"), W.tiny_gqa("B")
    ta, tb = to_dev(wa), to_dev(wb)
    ab = [gpu_fwd_bwd(wa, ta), gpu_fwd_bwd(wb, tb)]
    ba = [gpu_fwd_bwd(wb, tb), gpu_fwd_bwd(wa, ta)]
    for x, y in zip(ab[0], ba[1]):
        assert torch.equal(x, y)
    for x, y in zip(ab[1], ba[0]):
        assert torch.equal(x, y)
    _, _, _, dk, dv = ab[1]
    assert torch.all(dk[0:4] == 0) and torch.all(dv[0:4] == 0)
    assert torch.any(ab[0][4][0:3] != 0)
    check_against_oracle(wa, ab[0])
    check_against_oracle(wb, ab[1])


@pytest.mark.parametrize("lengths", W.PACKINGS, ids=lambda x: "_".join(map(str, x)))
def test_packings(lengths):
    """[3333] packings: bf16, 8 heads, d=128, padding_causal, sum loss."""
    w = W.packings(list(lengths))
    check_against_oracle(w, gpu_fwd_bwd(w))


def test_gqa_d256_peaked():
    """[3216] shape: 2 x 384 causal, hq=16, hkv=2, d=256, peaked softmax."""
    w = W.gqa_d256()
    check_against_oracle(w, gpu_fwd_bwd(w))


@pytest.mark.parametrize("mask", [W.MASK_PADDING, W.MASK_PADDING_CAUSAL])
def test_real_ne_padded(mask):
    """[2892]: real lengths inside larger padded slots filled with +-1e3; the
    output keeps the padded layout and pad rows are exactly zero."""
    w = W.real_ne_padded(mask_type=mask)
    res = gpu_fwd_bwd(w)
    check_against_oracle(w, res)
    assert res[0].shape == w.q.shape


GIVEN = {
    "real_ne_padded_causal_d64": lambda: W.real_ne_padded(mask_type=W.MASK_PADDING_CAUSAL, H=8, d=64),
    "gqa_d256_mul_outliers": lambda: W.gqa_d256(outlier_mode="mul"),
}


@pytest.mark.parametrize("name", sorted(GIVEN))
def test_backward_from_given_out_lse(name):
    """The backward alone: both sides take the same out (rounded to the storage
    dtype) and lse (fp32) produced by the oracle, as TransformerEngine's
    fused_attn_bwd takes them. The harsher outlier variant of the d=256 workload is
    checked here: there the rounding of out itself (D = rowsum(dO * out)) moves dQ
    by more than 1e-2 from the exact gradient, for any implementation of this
    interface, so the kernel is held to the interface's own definition."""
    import bwd_packed_varlen_gb300 as ta
    w = GIVEN[name]()
    r_out, r_lse, _, _, _ = oracle_fwd_bwd(w)
    out = torch.from_numpy(r_out).to(w.q.dtype)
    lse = torch.from_numpy(r_lse).to(torch.float32)
    ref = oracle.attn_bwd_thd(np64(w.q), np64(w.k), np64(w.v), np64(out), np64(w.dout),
                              lse.double().numpy(), w.cu_seqlens_q.numpy(),
                              w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
                              w.cu_seqlens_kv_padded.numpy(), w.attn_scale, w.mask_type)
    t = to_dev(w)
    dq, dk, dv = ta.bwd(t["q"], t["k"], t["v"], out.cuda(), t["dout"], lse.cuda(), t["cu_q"],
                        t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"], w.attn_scale, w.mask_type)
    scales = error_scales(w)
    for nm, a, b, m in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, scales[1:]):
        assert_close(nm, np64(a), b, m, UNIT_ROUNDOFF[w.dtype])


# ----------------------------------------------------------------- edge cases

EDGE = [
    # seed, batch, max_len, hq, hkv, d, mask, dtype
    (11, 5, 300, 4, 2, 64, W.MASK_PADDING, "bf16"),
    (12, 5, 300, 4, 2, 64, W.MASK_PADDING_CAUSAL, "bf16"),
    (13, 3, 260, 6, 3, 128, W.MASK_PADDING_CAUSAL, "fp16"),
    (14, 4, 200, 2, 1, 8, W.MASK_PADDING, "fp16"),
    (15, 4, 200, 4, 4, 48, W.MASK_PADDING_CAUSAL, "bf16"),
    (16, 3, 150, 2, 1, 96, W.MASK_PADDING, "bf16"),
    (17, 2, 300, 4, 1, 256, W.MASK_PADDING_CAUSAL, "bf16"),
    (18, 2, 200, 2, 2, 256, W.MASK_PADDING, "fp16"),
    (19, 6, 129, 8, 2, 32, W.MASK_PADDING_CAUSAL, "bf16"),
    (20, 4, 400, 8, 8, 16, W.MASK_PADDING_CAUSAL, "bf16"),
    (21, 3, 400, 4, 2, 192, W.MASK_PADDING_CAUSAL, "bf16"),
    (22, 6, 500, 4, 2, 64, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT, "bf16"),
    (23, 5, 400, 6, 3, 128, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT, "fp16"),
    (24, 3, 400, 4, 1, 256, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT, "bf16"),
    (25, 4, 300, 4, 4, 48, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT, "bf16"),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"s{c[0]}_d{c[5]}_m{c[6]}_{c[7]}")
def test_ragged_edge_cases(case):
    """Zero-length sequences, Lq != Lk, ragged tails spanning several tiles, pad
    slots, tail rows, head dims 8..256 and both 16-bit types."""
    seed, batch, max_len, hq, hkv, d, mask, dtype = case
    w = W.random_varlen(seed, batch, max_len, hq, hkv, d, mask, dtype)
    check_against_oracle(w, gpu_fwd_bwd(w))


@pytest.mark.parametrize("case", random_configs(), ids=lambda c: f"s{c[0]}_d{c[5]}_h{c[3]}x{c[4]}_m{c[6]}_{c[7]}")
def test_random_configurations(case):
    """Seeded random shapes beyond the hand-picked edge cases, each element checked
    against the oracle (forward and backward)."""
    seed, batch, max_len, hq, hkv, d, mask, dtype = case
    w = W.random_varlen(seed, batch, max_len, hq, hkv, d, mask, dtype)
    check_against_oracle(w, gpu_fwd_bwd(w))


def _same_bits(x, y):
    view = torch.int32 if x.dtype == torch.float32 else torch.int16
    return torch.equal(x.view(view), y.view(view))


def _lengths_case(lq, lk, hq, hkv, d, mask, seed, pad=9):
    """THD workload with the given real query/key lengths per sequence."""
    import math
    rng = np.random.default_rng(seed)
    lq, lk = np.asarray(lq), np.asarray(lk)
    pq = lq + rng.integers(0, pad + 1, size=lq.size)
    pk = lk + rng.integers(0, pad + 1, size=lk.size)
    cu = lambda x: torch.tensor([0] + list(np.cumsum(x)), dtype=torch.int32)
    g = torch.Generator().manual_seed(seed)
    mk = lambda T, h: torch.randn(T, h, d, generator=g).to(torch.bfloat16)
    Tq, Tk = int(pq.sum()) + 3, int(pk.sum()) + 3
    return W.Workload(name=f"lengths_{seed}", q=mk(Tq, hq), k=mk(Tk, hkv), v=mk(Tk, hkv),
                      dout=mk(Tq, hq), cu_seqlens_q=cu(lq), cu_seqlens_kv=cu(lk),
                      cu_seqlens_q_padded=cu(pq), cu_seqlens_kv_padded=cu(pk),
                      attn_scale=1.0 / math.sqrt(d), mask_type=mask, dtype="bf16")


@pytest.mark.parametrize("d", [128, 256])
def test_bottom_right_causal(d):
    """Lower-right causal alignment: more queries than keys (whole query tiles and
    forward tile pairs before the triangle see no key: out 0, lse -inf, dq 0),
    fewer queries than keys (every key row seen), equal lengths (bit-identical to
    the upper-left mask), bit-identical on a repeated call."""
    lq, lk = [700, 130, 384, 1, 300], [150, 900, 384, 77, 0]
    w = _lengths_case(lq, lk, 4, 2, d, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT, 50 + d)
    t = to_dev(w)
    a = gpu_fwd_bwd(w, t)
    check_against_oracle(w, a)
    b = gpu_fwd_bwd(w, t)
    for x, y in zip(a, b):
        assert _same_bits(x, y)
    # first sequence: queries 0..549 see no key
    o0 = int(w.cu_seqlens_q_padded[0])
    assert torch.all(a[0][o0:o0 + 550] == 0) and torch.all(a[2][o0:o0 + 550] == 0)
    assert torch.all(torch.isneginf(a[1][o0:o0 + 550]))
    eq = _lengths_case([384, 200], [384, 200], 4, 2, d, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT, 60 + d)
    te = to_dev(eq)
    br = gpu_fwd_bwd(eq, te)
    eq.mask_type = W.MASK_PADDING_CAUSAL
    tl = gpu_fwd_bwd(eq, te)
    for x, y in zip(br, tl):
        assert _same_bits(x, y)



@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mask", [W.MASK_PADDING_CAUSAL, W.MASK_PADDING])
def test_running_max_raised_between_key_tiles(d, dtype, mask):
    """Odd query rows whose scores climb by more than 2^8 per key tile, even rows
    flat: the forward raises the running max (scaling O and l, and redoing the
    tile's exponentials) on most tiles for half the rows of every warp. The forward
    is held to the oracle. The backward is held to the interface's definition from
    the oracle's out (rounded to the storage dtype) and lse, element by element and
    row by row. A raise means later keys outweigh earlier ones by more than 2^8, so
    these rows are peaked: dS = P (dP - D) cancels, and rounding dS to bf16 before
    dS K -- which any tensor-core backward does -- moves dQ by 1-2 % of its norm
    (the arithmetic, emulated in float64 on the CPU, gives the same). The
    whole-tensor 1e-2 bar is therefore applied to dQ only in fp16."""
    import bwd_packed_varlen_gb300 as ta
    w = W.growing_scores(d=d, dtype=dtype, mask_type=mask)
    t = to_dev(w)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    out, lse = ta.fwd(t["q"], t["k"], t["v"], *cu, w.attn_scale, w.mask_type)
    r_out, r_lse, _, _, _ = oracle_fwd_bwd(w)
    scales = error_scales(w)
    u = UNIT_ROUNDOFF[w.dtype]
    assert_close("out", np64(out), r_out, scales[0], u)
    got_lse, fin = np64(lse), np.isfinite(r_lse)
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(r_lse))
    assert np.abs(got_lse[fin] - r_lse[fin]).max() <= 1e-3

    o16 = torch.from_numpy(r_out).to(w.q.dtype)
    l32 = torch.from_numpy(r_lse).to(torch.float32)
    ref = oracle.attn_bwd_thd(np64(w.q), np64(w.k), np64(w.v), np64(o16), np64(w.dout),
                              l32.double().numpy(), w.cu_seqlens_q.numpy(),
                              w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
                              w.cu_seqlens_kv_padded.numpy(), w.attn_scale, w.mask_type)
    dq, dk, dv = ta.bwd(t["q"], t["k"], t["v"], o16.cuda(), t["dout"], l32.cuda(), *cu,
                        w.attn_scale, w.mask_type)
    for nm, a, b, m in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, scales[1:]):
        if nm == "dq" and dtype == "bf16":
            c = row_elem_check(np64(a), b, m, u)
            assert c["elem_ratio"] <= 1.0 and c["row_ratio"] <= 1.0, c
        else:
            assert_close(nm, np64(a), b, m, u)


@pytest.mark.parametrize("lengths", [[1024] * 8, [1024] * 8 + [100], [1024] * 16 + [129, 1]],
                         ids=["64_key_tiles", "65_key_tiles", "131_key_tiles"])
def test_key_tile_list_band_boundaries(lengths):
    """dK/dV items come in bands of 64 sorted key tiles (kv-head-major inside a
    band), except the last full band and the remainder, which go pair-major: exactly
    one full band (all pair-major), one full band plus one tile (all pair-major), and
    two full bands plus three tiles (one band, then 67 tiles pair-major) must each
    cover every (key tile, kv head) once."""
    rng = np.random.default_rng(len(lengths))
    T, hq, hkv, d = sum(lengths), 4, 2, 32
    q, k, v, do = (torch.from_numpy(rng.standard_normal((T, h, d), dtype=np.float32)).to(torch.bfloat16)
                   for h in (hq, hkv, hkv, hq))
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)
    w = W.Workload(name="bands", q=q, k=k, v=v, dout=do, cu_seqlens_q=cu, cu_seqlens_kv=cu,
                   cu_seqlens_q_padded=cu.clone(), cu_seqlens_kv_padded=cu.clone(),
                   attn_scale=d ** -0.5, mask_type=W.MASK_PADDING_CAUSAL, dtype="bf16")
    check_against_oracle(w, gpu_fwd_bwd(w))

def test_all_sequences_empty_and_keyless():
    """A batch where every query sequence is empty, and one where queries exist but
    no keys: outputs are exact zeros (lse -inf on real keyless queries)."""
    w = W.random_varlen(30, 3, 50, 2, 1, 64, W.MASK_PADDING, "bf16")
    w.cu_seqlens_q = torch.zeros_like(w.cu_seqlens_q)
    res = gpu_fwd_bwd(w)
    for x in res[:1] + res[2:]:
        assert torch.all(x == 0)
    w = W.random_varlen(31, 3, 50, 2, 1, 64, W.MASK_PADDING, "bf16", allow_empty=False)
    w.cu_seqlens_kv = torch.zeros_like(w.cu_seqlens_kv)
    res = gpu_fwd_bwd(w)
    check_against_oracle(w, res)


# ---------------------------------------------------------------- determinism


def test_bitwise_repeatable_and_poisoned_buffers():
    """Outputs are bit-identical across repeated calls, with output and workspace
    buffers pre-filled with NaN bytes, and after allocator churn between calls
    (the workspace-reuse failure of [2448])."""
    import bwd_packed_varlen_gb300 as ta
    w = W.random_varlen(40, 4, 700, 8, 2, 128, W.MASK_PADDING_CAUSAL, "bf16")
    t = to_dev(w)
    base = gpu_fwd_bwd(w, t)
    again = gpu_fwd_bwd(w, t)
    for x, y in zip(base, again):
        assert torch.equal(x, y)
    Tq, hq, d = w.q.shape
    Tk, hkv, _ = w.k.shape
    B = w.batch

    def nanfill(x):
        x.view(torch.uint8).fill_(0xFF)
        return x

    out = nanfill(torch.empty_like(t["q"]))
    lse = nanfill(torch.empty((Tq, hq), dtype=torch.float32, device="cuda"))
    dq, dk, dv = (nanfill(torch.empty_like(x)) for x in (t["q"], t["k"], t["v"]))
    wsf = torch.full((ta.fwd_workspace_size(B, Tq, Tk, hq, hkv, d),), 0xFF, dtype=torch.uint8,
                     device="cuda")
    wsb = torch.full((ta.bwd_workspace_size(B, Tq, Tk, hq, hkv, d),), 0xFF, dtype=torch.uint8,
                     device="cuda")
    churn = [torch.empty(4096 * 1024 + 17 * i, dtype=torch.float32, device="cuda")
             for i in range(3)]
    del churn
    poisoned = gpu_fwd_bwd(w, t, fwd={"out": out, "lse": lse, "workspace": wsf},
                           bwd={"dq": dq, "dk": dk, "dv": dv, "workspace": wsb})
    for x, y in zip(base, poisoned):
        assert torch.equal(x, y)
    assert ta.read_status(wsf) == 0 and ta.read_status(wsb) == 0
    check_against_oracle(w, base)


# ------------------------------------------------------------------- boundary


def test_invalid_arguments_return_errors():
    """Host-detectable errors return codes and launch nothing."""
    import bwd_packed_varlen_gb300 as ta
    w = W.packings([128])
    t = to_dev(w)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    with pytest.raises(ta.TeAttnError) as e:
        ta.fwd(t["q"], t["k"][:, :3].contiguous(), t["v"][:, :3].contiguous(), *cu, 0.1, 1)
    assert e.value.code == -1
    with pytest.raises(ta.TeAttnError) as e:
        ta.fwd(t["q"][..., :12].contiguous(), t["k"][..., :12].contiguous(),
               t["v"][..., :12].contiguous(), *cu, 0.1, 1)
    assert e.value.code == -2
    with pytest.raises(ta.TeAttnError) as e:
        ta.fwd(t["q"], t["k"], t["v"], *cu, 0.1, 4)
    assert e.value.code == -2
    with pytest.raises(ta.TeAttnError) as e:
        ta.fwd(t["q"], t["k"], t["v"], *cu, 0.1, 1,
               workspace=torch.empty(8, dtype=torch.uint8, device="cuda"))
    assert e.value.code == -3


def test_inconsistent_seqlens_flagged():
    """Real length above padded length is reported in the device status word and
    nothing outside the tensors is touched."""
    import bwd_packed_varlen_gb300 as ta
    w = W.packings([128, 96])
    t = to_dev(w)
    bad = torch.tensor([0, 130, 224], dtype=torch.int32, device="cuda")
    ws = torch.empty(ta.fwd_workspace_size(2, 224, 224, 8, 8, 128), dtype=torch.uint8,
                     device="cuda")
    ta.fwd(t["q"], t["k"], t["v"], bad, t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"], 0.1, 2,
           workspace=ws)
    assert ta.read_status(ws) & 1


# --------------------------------------------------------------- full size


def test_many_short_sequences_unsorted_lists():
    """16000 sequences of 1-3 queries and 0-3 keys: about 12000 (sequence, tile)
    pairs, more than the scheduler sorts in shared memory (8192), so the lists keep
    their natural order; results and zero rows still match the oracle, for both
    causal alignments and GQA."""
    rng = np.random.default_rng(16000)
    B = 16000
    lq = rng.integers(1, 4, size=B)
    lk = rng.integers(0, 4, size=B)
    assert int(((lq > 0) & (lk > 0)).sum()) > 8192
    for mask in (W.MASK_PADDING_CAUSAL, W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT):
        w = _lengths_case(lq, lk, 2, 1, 64, mask, 77, pad=2)
        check_against_oracle(w, gpu_fwd_bwd(w))


@pytest.mark.slow
def test_throughput_workload_sampled():
    """The large packed workload (32768 real tokens, hq=32, hkv=8, d=128, causal) in
    the configuration the benchmark times; the oracle checks every output of a
    sample of (sequence, kv-head group) pairs plus all zero rows."""
    w = W.throughput()
    res = gpu_fwd_bwd(w)
    out, lse, dq, dk, dv = (np64(x) for x in res)
    qm, km = oracle.valid_row_masks(
        w.cu_seqlens_q.numpy(), w.cu_seqlens_kv.numpy(), w.cu_seqlens_q_padded.numpy(),
        w.cu_seqlens_kv_padded.numpy(), w.q.shape[0], w.k.shape[0], w.mask_type)
    assert np.all(out[~qm] == 0) and np.all(dq[~qm] == 0)
    assert np.all(dk[~km] == 0) and np.all(dv[~km] == 0)
    G = w.hq // w.hkv
    cq, cp = w.cu_seqlens_q.numpy(), w.cu_seqlens_q_padded.numpy()
    for b, g in ((2, 0), (3, 7), (0, 3)):
        oq, L = int(cp[b]), int(cq[b + 1] - cq[b])
        hs = slice(g * G, g * G + G)
        q = np64(w.q[oq:oq + L, hs])
        k = np64(w.k[oq:oq + L, g])
        v = np64(w.v[oq:oq + L, g])
        do = np64(w.dout[oq:oq + L, hs])
        r = oracle.attn_group_fwd_bwd(q, k, v, do, w.attn_scale, "tl")
        m = list(zip(*(oracle.attn_group_error_scales(q, k, v, do, w.attn_scale, "tl", norm=n)
                       for n in (1, 2))))
        u = UNIT_ROUNDOFF[w.dtype]
        assert_close(f"out[{b},{g}]", out[oq:oq + L, hs], r[0], m[0], u)
        assert np.abs(lse[oq:oq + L, hs] - r[1]).max() <= 1e-3
        assert_close(f"dq[{b},{g}]", dq[oq:oq + L, hs], r[2], m[1], u)
        assert_close(f"dk[{b},{g}]", dk[oq:oq + L, g], r[3], m[2], u)
        assert_close(f"dv[{b},{g}]", dv[oq:oq + L, g], r[4], m[3], u)


def test_issue3333_reference_norms_from_page_rng():
    """[3333] "Reproduction" / "Results": q, k, v drawn exactly as the page's script
    draws them (torch.manual_seed(42), three bf16 torch.randn(total, 8, 128) on the
    GPU), per-sequence causal attention, loss = sum(out). The page prints the norm
    of the fp32 reference query gradient to two decimals: 74.97, 101.93, 104.96,
    126.25. The oracle's dQ norm must print the same for the packings of up to 256
    tokens, and the CUDA path's must match the oracle for all four. For the 512-token
    packing the generator's stream appears to depend on the GPU, so a
    different norm there is reported, not failed; if even the first packing does not
    reproduce, this GPU's generator differs and the pin is skipped."""
    import json
    import os

    import bwd_packed_varlen_gb300 as ta

    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "issue3333_qgrad_norms.json")))
    results = []
    for lengths, ref_norm in zip(fx["lengths"], fx["ref_qgrad_norm"]):
        total = sum(lengths)
        torch.manual_seed(42)
        q, k, v = (torch.randn(total, 8, 128, device="cuda", dtype=torch.bfloat16) for _ in range(3))
        dout = torch.ones_like(q)
        offs = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        cu = torch.tensor(offs, dtype=torch.int32).cuda()
        scale = 1.0 / np.sqrt(128.0)
        _, _, dq_ref, _, _ = oracle.attn_fwd_bwd_thd(
            np64(q), np64(k), np64(v), np64(dout), offs, offs, offs, offs, scale, W.MASK_PADDING_CAUSAL)
        norm = float(np.linalg.norm(dq_ref))
        out, lse = ta.fwd(q, k, v, cu, cu, cu, cu, scale, W.MASK_PADDING_CAUSAL, max(lengths), max(lengths))
        dq, _, _ = ta.bwd(q, k, v, out, dout, lse, cu, cu, cu, cu, scale, W.MASK_PADDING_CAUSAL,
                          max(lengths), max(lengths))
        torch.cuda.synchronize()
        gnorm = float(np.linalg.norm(np64(dq)))
        assert abs(gnorm - norm) <= 1e-2 * norm, (lengths, gnorm, norm)
        results.append((lengths, total, norm, ref_norm, abs(norm - ref_norm) <= 0.006))
    if not results[0][4]:
        pytest.skip(f"this GPU's generator does not reproduce the page's stream: {results}")
    bad = [r for r in results if r[1] <= 256 and not r[4]]
    assert not bad, f"page norms not reproduced: {bad} (all: {results})"
    print("issue 3333 norms (lengths, tokens, oracle, page, reproduced):", results)


def test_bwd_dq_event_handover():
    """te_attn_bwd_thd_ev: the same bits as te_attn_bwd_thd, and dq copied on a second
    stream as soon as the recorded event fires already equals the final dq (the
    backward computes dq before dk/dv)."""
    import bwd_packed_varlen_gb300 as ta

    w = W.random_varlen(11, batch=6, max_len=700, hq=8, hkv=2, d=128, mask_type=W.MASK_PADDING_CAUSAL)
    t = to_dev(w)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    args = (w.attn_scale, w.mask_type, w.max_seqlen_q, w.max_seqlen_kv)
    out, lse = ta.fwd(t["q"], t["k"], t["v"], *cu, *args)
    ref = ta.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, *args)
    ev = torch.cuda.Event()
    side = torch.cuda.Stream()
    got = ta.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, *args, dq_done=ev)
    side.wait_event(ev)
    with torch.cuda.stream(side):
        early_dq = got[0].clone()
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    assert torch.equal(early_dq, got[0])
