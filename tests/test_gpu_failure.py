"""Failure detection on the GPU without a GPU fault.

* Bounded waits: te_attn_selftest_wait_timeout makes one pipeline wait run out on
  purpose (a barrier nothing arrives on, a 1 ms limit). The kernel must return, the
  status word must carry TE_STATUS_TIMEOUT, the block's second wait (4 s limit) must
  have given up early on seeing the bit, the block must have reached its end (TMEM
  freed), and a normal call on the same workspace afterwards must be clean and
  bit-identical to a call on a fresh workspace.
* Debug build: libteattn_debug.so checks every computed global offset and records a
  bad one as TE_STATUS_OUT_OF_BOUNDS. On a ragged case with pad slots, empty
  sequences and tails it must report nothing and give the release build's bits.
"""

import pytest
import torch

from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import check_against_oracle, gpu_fwd_bwd, random_configs, to_dev

pytestmark = pytest.mark.gpu

STATUS_TIMEOUT = 2
STATUS_OUT_OF_BOUNDS = 4


def _bits(x):
    return x.view(torch.int32 if x.dtype == torch.float32 else torch.int16)


def test_bounded_wait_runs_out_and_unwinds():
    import bwd_packed_varlen_gb300 as ta
    w = W.random_varlen(70, 4, 400, 4, 2, 64, W.MASK_PADDING_CAUSAL, "bf16")
    t = to_dev(w)
    Tq, hq, d = w.q.shape
    Tk, hkv, _ = w.k.shape
    wsb = torch.zeros(ta.bwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d), dtype=torch.uint8,
                      device="cuda")
    ta.selftest_wait_timeout(wsb, limit_us=1000)
    status = ta.read_status(wsb)
    hdr = wsb[:256].view(torch.int32).cpu()
    first_ok, first_us, second_us, done = (int(x) for x in hdr[8:12])
    assert status & STATUS_TIMEOUT, status
    assert first_ok == 0 and done == 1, hdr[8:12].tolist()
    assert 1000 <= first_us < 1_000_000, first_us
    assert second_us < 1_000_000, second_us  # gave up on the bit, long before its 4 s
    # the context is intact and the workspace is rewritten by the next call
    fresh = gpu_fwd_bwd(w, t)
    reused = gpu_fwd_bwd(w, t, bwd={"workspace": wsb})
    assert ta.read_status(wsb) == 0
    for a, b in zip(fresh, reused):
        assert torch.equal(_bits(a), _bits(b))
    check_against_oracle(w, reused)


def test_selftest_rejects_bad_arguments():
    import bwd_packed_varlen_gb300 as ta
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ta.TeAttnError) as e:
        ta.selftest_wait_timeout(small, limit_us=10)
    assert e.value.code == -3
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ta.TeAttnError) as e:
        ta.selftest_wait_timeout(ws, limit_us=0)
    assert e.value.code == -1


@pytest.mark.parametrize("mask", [W.MASK_PADDING, W.MASK_PADDING_CAUSAL,
                                  W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT])
def test_debug_build_reports_no_out_of_bounds(mask):
    import bwd_packed_varlen_gb300 as ta
    w = W.random_varlen(71, 6, 520, 8, 2, 128, mask, "bf16")
    t = to_dev(w)
    Tq, hq, d = w.q.shape
    Tk, hkv, _ = w.k.shape
    release = gpu_fwd_bwd(w, t)
    wsf = torch.empty(ta.fwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d), dtype=torch.uint8,
                      device="cuda")
    wsb = torch.empty(ta.bwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d), dtype=torch.uint8,
                      device="cuda")
    with ta.debug_build():
        debug = gpu_fwd_bwd(w, t, fwd={"workspace": wsf}, bwd={"workspace": wsb})
        assert ta.read_status(wsf) == 0 and ta.read_status(wsb) == 0
    for a, b in zip(release, debug):
        assert torch.equal(_bits(a), _bits(b))
    check_against_oracle(w, debug)


def test_debug_build_d256_and_sbhd():
    """The d = 256 kernels and the sequence-major layout under the bounds checks."""
    import bwd_packed_varlen_gb300 as ta
    w = W.random_varlen(72, 3, 300, 4, 2, 256, W.MASK_PADDING_CAUSAL, "bf16")
    t = to_dev(w)
    Tq, hq, d = w.q.shape
    Tk, hkv, _ = w.k.shape
    wsb = torch.empty(ta.bwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d), dtype=torch.uint8,
                      device="cuda")
    with ta.debug_build():
        res = gpu_fwd_bwd(w, t, bwd={"workspace": wsb})
        assert ta.read_status(wsb) == 0
    check_against_oracle(w, res)
    S, B = 200, 3
    g = torch.Generator().manual_seed(73)
    q = torch.randn(S, B, 4, 64, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(S, B, 2, 64, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(S, B, 2, 64, generator=g).to(torch.bfloat16).cuda()
    do = torch.randn(S, B, 4, 64, generator=g).to(torch.bfloat16).cuda()
    cu = torch.tensor([0, 200, 331, 331], dtype=torch.int32, device="cuda")
    ws = torch.empty(ta.bwd_workspace_size(B, S * B, S * B, 4, 2, 64), dtype=torch.uint8,
                     device="cuda")
    out, lse = ta.fwd_sbhd(q, k, v, cu, cu, 0.125, "padding_causal")
    ref = ta.bwd_sbhd(q, k, v, out, do, lse, cu, cu, 0.125, "padding_causal")
    with ta.debug_build():
        out_d, lse_d = ta.fwd_sbhd(q, k, v, cu, cu, 0.125, "padding_causal")
        got = ta.bwd_sbhd(q, k, v, out_d, do, lse_d, cu, cu, 0.125, "padding_causal", workspace=ws)
        assert ta.read_status(ws) == 0
    for a, b in zip((out, lse) + tuple(ref), (out_d, lse_d) + tuple(got)):
        assert torch.equal(_bits(a), _bits(b))


def test_debug_build_fused_backward_and_e4m3_forward():
    """The opt-in paths under the bounds checks -- the fused backward (ordered fp32
    dQ accumulation, then the conversion kernel) and the e4m3 forward (V widened in
    the workspace) -- and the default backward on a packing whose key tiles fill
    more than one 64-tile band of the dK/dV item order; each bit-identical to the
    release build."""
    import bwd_packed_varlen_gb300 as ta
    w = W.random_varlen(74, 14, 1200, 4, 2, 128, W.MASK_PADDING_CAUSAL, "bf16")  # 106 key tiles
    t = to_dev(w)
    Tq, hq, d = w.q.shape
    Tk, hkv, _ = w.k.shape
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    out, lse = ta.fwd(t["q"], t["k"], t["v"], *cu, w.attn_scale, w.mask_type)
    release = ta.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, w.attn_scale,
                     w.mask_type, fused=True)
    two_kernel = ta.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, w.attn_scale,
                        w.mask_type)
    f8 = torch.float8_e4m3fn
    q8, k8, v8 = (x.to(f8) for x in (t["q"], t["k"], t["v"]))
    rel_e4 = ta.fwd_e4m3(q8, k8, v8, *cu, w.attn_scale, 1.0, 1.0, 1.0, w.mask_type)
    wsb = torch.empty(ta.bwd_fused_workspace_size(w.batch, Tq, Tk, hq, hkv, d),
                      dtype=torch.uint8, device="cuda")
    with ta.debug_build():
        debug = ta.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, w.attn_scale,
                       w.mask_type, workspace=wsb, fused=True)
        assert ta.read_status(wsb) == 0
        dbg_e4 = ta.fwd_e4m3(q8, k8, v8, *cu, w.attn_scale, 1.0, 1.0, 1.0, w.mask_type)
        ws2 = torch.empty(ta.bwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d),
                          dtype=torch.uint8, device="cuda")
        dbg_two = ta.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, w.attn_scale,
                         w.mask_type, workspace=ws2)
        assert ta.read_status(ws2) == 0
    torch.cuda.synchronize()
    for a, b in zip(tuple(release) + tuple(rel_e4) + tuple(two_kernel),
                    tuple(debug) + tuple(dbg_e4) + tuple(dbg_two)):
        assert torch.equal(_bits(a), _bits(b))


@pytest.mark.parametrize("case", random_configs(), ids=lambda c: f"s{c[0]}_d{c[5]}_h{c[3]}x{c[4]}_m{c[6]}_{c[7]}")
def test_debug_build_random_configurations(case):
    """The seeded random configurations of the parity tests under the bounds checks:
    no out-of-bounds offset, a clean status word, and the release build's bits."""
    import bwd_packed_varlen_gb300 as ta
    seed, batch, max_len, hq, hkv, d, mask, dtype = case
    w = W.random_varlen(seed, batch, max_len, hq, hkv, d, mask, dtype)
    t = to_dev(w)
    Tq, hq, d = w.q.shape
    Tk, hkv, _ = w.k.shape
    release = gpu_fwd_bwd(w, t)
    wsf = torch.empty(ta.fwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d), dtype=torch.uint8,
                      device="cuda")
    wsb = torch.empty(ta.bwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d), dtype=torch.uint8,
                      device="cuda")
    with ta.debug_build():
        debug = gpu_fwd_bwd(w, t, fwd={"workspace": wsf}, bwd={"workspace": wsb})
        assert ta.read_status(wsf) == 0 and ta.read_status(wsb) == 0
    for a, b in zip(release, debug):
        assert torch.equal(_bits(a), _bits(b))

