"""CUDA graphs: the forward and backward entry points capture into one graph.

Every launch of the library is asynchronous on the caller's stream, with no host
synchronisation and no allocation inside a call (the caller passes the workspace),
so a training step that calls forward and backward can be captured once and
replayed. Replays must give the same bits as eager calls on the same inputs,
including after the inputs were overwritten in place (the graph reads whatever
its buffers hold at replay time) and with the ragged packings and masks of the
pages' configurations.
"""

import dataclasses

import pytest
import torch

import bwd_packed_varlen_gb300 as ta
from bwd_packed_varlen_gb300 import workloads as W
from gpu_common import check_against_oracle, oracle_fwd_bwd, to_dev

pytestmark = pytest.mark.gpu


def _buffers(w, t):
    Tq, hq, d = w.q.shape
    Tk, hkv, _ = w.k.shape
    dev = t["q"].device
    return {
        "out": torch.empty_like(t["q"]), "lse": torch.empty((Tq, hq), dtype=torch.float32, device=dev),
        "dq": torch.empty_like(t["q"]), "dk": torch.empty_like(t["k"]), "dv": torch.empty_like(t["v"]),
        "wsf": torch.empty(max(1, ta.fwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d)),
                           dtype=torch.uint8, device=dev),
        "wsb": torch.empty(max(1, ta.bwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d)),
                           dtype=torch.uint8, device=dev),
    }


def _step(w, t, b):
    cu = (t["cu_q"], t["cu_kv"], t["cu_q_pad"], t["cu_kv_pad"])
    ta.fwd(t["q"], t["k"], t["v"], *cu, w.attn_scale, w.mask_type, w.max_seqlen_q,
           w.max_seqlen_kv, out=b["out"], lse=b["lse"], workspace=b["wsf"])
    ta.bwd(t["q"], t["k"], t["v"], b["out"], t["dout"], b["lse"], *cu, w.attn_scale,
           w.mask_type, w.max_seqlen_q, w.max_seqlen_kv, dq=b["dq"], dk=b["dk"], dv=b["dv"],
           workspace=b["wsb"])


def _results(b):
    return [b[n].clone() for n in ("out", "lse", "dq", "dk", "dv")]


def _same_bits(a, b):
    return all(torch.equal(x.view(torch.uint8), y.view(torch.uint8)) for x, y in zip(a, b))


CASES = {
    "packings_128_96": lambda: W.packings([128, 96]),
    "real_ne_padded_causal": lambda: W.real_ne_padded(mask_type=W.MASK_PADDING_CAUSAL, H=8),
    "ragged_bottom_right": lambda: W.random_varlen(22, 6, 500, 4, 2, 64,
                                                   W.MASK_PADDING_CAUSAL_BOTTOM_RIGHT, "bf16"),
    "ragged_fp16_d128": lambda: W.random_varlen(13, 3, 260, 6, 3, 128, W.MASK_PADDING_CAUSAL,
                                                "fp16"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_captured_step_matches_eager_bits(name):
    w = CASES[name]()
    t = to_dev(w)
    b = _buffers(w, t)
    _step(w, t, b)  # eager reference (and kernel attributes set before capture)
    torch.cuda.synchronize()
    eager = _results(b)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(w, t, b)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step(w, t, b)
    for n in ("out", "lse", "dq", "dk", "dv"):
        b[n].fill_(float("nan"))  # what the replay writes must not depend on this
    g.replay()
    torch.cuda.synchronize()
    assert _same_bits(_results(b), eager)
    assert ta.read_status(b["wsb"]) == 0 and ta.read_status(b["wsf"]) == 0

    # new inputs, same buffers: the replay computes on them, as eager calls would
    gen = torch.Generator().manual_seed(7)
    for n in ("q", "k", "v", "dout"):
        t[n].copy_(torch.randn(t[n].shape, generator=gen).to(t[n].dtype))
    g.replay()
    torch.cuda.synchronize()
    replayed = _results(b)
    _step(w, t, b)
    torch.cuda.synchronize()
    assert _same_bits(replayed, _results(b))
    w2 = dataclasses.replace(w, q=t["q"].cpu(), k=t["k"].cpu(), v=t["v"].cpu(),
                             dout=t["dout"].cpu())
    check_against_oracle(w2, replayed, oracle_fwd_bwd(w2))
