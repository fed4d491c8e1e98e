"""The backward entry point for callers that cannot allocate device memory.

te_attn_bwd_thd_noalloc serves callers with no way to obtain scratch memory (plugin
hosts that own all device allocations, runtimes that forbid allocating after
start-up, foreign-language callers without a CUDA allocator): it runs the same
backward pass with a scratch array built into the library. These tests call it
through the C ABI on two different problems in a row, in both orders, so that each
call starts from the other problem's leftovers in the shared array, and require the
bits of te_attn_bwd_thd with a caller-provided workspace (both run the same kernels
on the same inputs, and results never depend on what a workspace held before). A
call with inconsistent cu_seqlens must be reported through the array's status
word. The file sorts last so a run that stops at the first failure has already run
every other test.
"""

import ctypes

import pytest
import torch

from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import gpu_fwd_bwd, to_dev

pytestmark = pytest.mark.gpu


def _problems():
    return [W.random_varlen(60, 5, 700, 8, 2, 128, W.MASK_PADDING_CAUSAL, "bf16"),
            W.real_ne_padded(mask_type=W.MASK_PADDING, H=8, d=64)]


def _run(w, t, ref):
    import bwd_packed_varlen_gb300 as ta
    out, lse, dq, dk, dv = ref
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    got = ta.bwd_noalloc(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, w.attn_scale,
                         w.mask_type, w.max_seqlen_q, w.max_seqlen_kv)
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv"), got, (dq, dk, dv)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{name}: bits differ"
    assert ta.read_status_noalloc() == 0


def test_noalloc_matches_workspace_entry_in_both_orders():
    ws = _problems()
    ts = [to_dev(w) for w in ws]
    refs = [gpu_fwd_bwd(w, t) for w, t in zip(ws, ts)]
    for order in ((0, 1), (1, 0), (0, 1)):
        for i in order:
            _run(ws[i], ts[i], refs[i])


def test_noalloc_reports_bad_seqlens_in_status():
    """A real length above its padded length (a host-side input mistake, not a GPU
    fault): the scheduler treats the sequence as empty and raises the status bit,
    which the caller reads back with te_attn_read_status_noalloc."""
    import bwd_packed_varlen_gb300 as ta
    w = W.packings([128, 96])
    t = to_dev(w)
    out, lse, _, _, _ = gpu_fwd_bwd(w, t)
    bad = torch.tensor([0, 130, 224], dtype=torch.int32, device="cuda")
    ta.bwd_noalloc(t["q"], t["k"], t["v"], out, t["dout"], lse, bad, t["cu_kv"], t["cu_q_pad"],
                   t["cu_kv_pad"], w.attn_scale, w.mask_type)
    assert ta.read_status_noalloc() & 1
    # and the next clean call clears it
    _run(w, t, gpu_fwd_bwd(w, t))


def test_noalloc_rejects_too_large_problem():
    import bwd_packed_varlen_gb300 as ta
    w = W.tiny_gqa("A")
    t = to_dev(w)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    big = 1 << 20  # claimed token count whose workspace exceeds the built-in scratch
    L = ta.library()
    rc = L.te_attn_bwd_thd_noalloc(
        t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["q"].data_ptr(),
        t["dout"].data_ptr(), t["q"].data_ptr(), t["q"].data_ptr(), t["k"].data_ptr(),
        t["v"].data_ptr(), *(c.data_ptr() for c in cu), 2, big, 12, 0, 0, 64, 1, 8, 0.1, 1, 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -3
    assert b"more than the built-in" in L.te_attn_last_error()
