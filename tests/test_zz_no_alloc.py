"""The backward entry point for callers that cannot allocate device memory.

te_attn_bwd_thd_noalloc serves callers with no way to obtain scratch memory (plugin
hosts that own all device allocations, runtimes that forbid allocating after
start-up, foreign-language callers without a CUDA allocator): it runs the same
backward pass with a scratch array built into the library. This test calls it
through the C ABI twice in a row, on two different problems so that the second call
starts from the first call's leftovers in the shared array, and checks each result
against te_attn_bwd_thd with a caller-provided workspace, at the tolerances of the
other GPU tests. The file sorts last so a run that stops at the first failure has
already run every other test.
"""

import pytest
import torch

from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import assert_close, gpu_fwd_bwd, np64, to_dev

pytestmark = pytest.mark.gpu


def _run(w):
    import bwd_packed_varlen_gb300 as ta
    t = to_dev(w)
    out, lse, dq, dk, dv = gpu_fwd_bwd(w, t)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    got = ta.bwd_noalloc(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, w.attn_scale,
                         w.mask_type, w.max_seqlen_q, w.max_seqlen_kv)
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv"), got, (dq, dk, dv)):
        assert_close(name, np64(a), np64(b))
        assert torch.equal(a == 0, b == 0), f"{name}: zero rows differ"


def test_noalloc_matches_workspace_entry_twice():
    _run(W.random_varlen(60, 5, 700, 8, 2, 128, W.MASK_PADDING_CAUSAL, "bf16"))
    _run(W.real_ne_padded(mask_type=W.MASK_PADDING, H=8, d=64))


def test_noalloc_rejects_too_large_problem():
    import bwd_packed_varlen_gb300 as ta
    w = W.tiny_gqa("A")
    t = to_dev(w)
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    big = 1 << 20  # claimed token count whose workspace exceeds the built-in scratch
    L = ta.library()
    import ctypes
    rc = L.te_attn_bwd_thd_noalloc(
        t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["q"].data_ptr(),
        t["dout"].data_ptr(), None, t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
        *(c.data_ptr() for c in cu), 2, big, 12, 0, 0, 64, 1, 8, 0.1, 1, 0, None)
    assert rc == -3
    assert b"more than the built-in" in L.te_attn_last_error()
