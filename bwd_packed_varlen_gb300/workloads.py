"""Seeded synthetic inputs for packed variable-length attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic. Both the CUDA path's tests/bench and the CPU oracle consume
what it returns, so it is the one module the two sides share.

Every tensor is drawn on the host with ``numpy.random.default_rng(seed)`` in
float32, rounded once to the storage dtype, and returned as CPU torch tensors, so a
given seed yields the same bits on any machine. The recipes restate the workloads
of the TransformerEngine issues this library addresses:

``tiny_gqa``      [2448] reproduction (THD + GQA, fp16, d=8, padded to [0,4,12]).
``packings``      [3333] reproduction (bf16 H=8 d=128 padding_causal, sum loss).
``gqa_d256``      [3216] shape ([384,2,16,256] sbhd == 2 x 384 THD, hq=16,
                  hkv=2, causal), with a synthetic peaked-softmax stand-in for the
                  captured activations that page attaches.
``real_ne_padded`` [2892] reproduction (real [100,150,120,130] in padded
                  [112,160,128,144] slots, 32 heads, d=48), pad slots +-1e3.
``throughput``    32768 real tokens in seeded lengths in [256, 8192] padded to a
                  multiple of 64; hq=32, hkv=8, d=128, padding_causal.

Pages cited, by title (keys are the pages' issue numbers):
  [2448] "Inconsistent fused_attn_bwd results of dk, dv under THD layout + GQA on multiple calls"
  [3333] "[Bug] FusedAttention (cuDNN) THD backward produces wrong gradients on sm_120 (RTX 5090); forward is correct, Unfused is correct"
  [3216] "flash-attn-4 4.0.0b11: DotProductAttention batched backward returns wrong dQ/dK/dV at head_dim=256 on Blackwell (sm_100)"
  [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

MASK_PADDING = 1
MASK_PADDING_CAUSAL = 2
MASK_PADDING_CAUSAL_BOTTOM_RIGHT = 3

_DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor
    cu_seqlens_q: torch.Tensor
    cu_seqlens_kv: torch.Tensor
    cu_seqlens_q_padded: torch.Tensor
    cu_seqlens_kv_padded: torch.Tensor
    attn_scale: float
    mask_type: int
    dtype: str
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.cu_seqlens_q.numel() - 1)

    @property
    def hq(self) -> int:
        return int(self.q.shape[1])

    @property
    def hkv(self) -> int:
        return int(self.k.shape[1])

    @property
    def d(self) -> int:
        return int(self.q.shape[2])

    @property
    def max_seqlen_q(self) -> int:
        return int((self.cu_seqlens_q[1:] - self.cu_seqlens_q[:-1]).max().item())

    @property
    def max_seqlen_kv(self) -> int:
        return int((self.cu_seqlens_kv[1:] - self.cu_seqlens_kv[:-1]).max().item())

    def algorithmic_flops(self) -> float:
        """Causal-adjusted fwd+bwd FLOPs: per (sequence, query head)
        ``3.5 * 4 * d * pairs``, pairs = Lq*Lk (padding) or Lq*Lk/2 (either causal
        alignment)."""
        lq = (self.cu_seqlens_q[1:] - self.cu_seqlens_q[:-1]).double()
        lk = (self.cu_seqlens_kv[1:] - self.cu_seqlens_kv[:-1]).double()
        f = 0.5 if self.mask_type in (MASK_PADDING_CAUSAL, MASK_PADDING_CAUSAL_BOTTOM_RIGHT) else 1.0
        return float(3.5 * 4.0 * self.d * self.hq * (lq * lk * f).sum().item())


def _cu(lengths):
    return torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def _to(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(_DT[dtype])


def tiny_gqa(call: str = "A", seed: int = 42) -> Workload:
    """[2448]: 12 token slots padded as [0,4,12]; call A has query lengths
    (1, 2) and key lengths (3, 6); call B has query lengths (0, 3). The same q, k,
    v, dout feed both calls, so A;B versus B;A isolates call-order effects."""
    rng = np.random.default_rng(seed)
    T, hq, hkv, d = 12, 2, 1, 8
    q = _normal(rng, (T, hq, d))
    k = _normal(rng, (T, hkv, d))
    v = _normal(rng, (T, hkv, d))
    do = _normal(rng, (T, hq, d))
    cu_q = {"A": [0, 1, 3], "B": [0, 0, 3]}[call]
    pad = torch.tensor([0, 4, 12], dtype=torch.int32)
    return Workload(
        name=f"tiny_gqa_{call}", q=_to(q, "fp16"), k=_to(k, "fp16"),
        v=_to(v, "fp16"), dout=_to(do, "fp16"),
        cu_seqlens_q=torch.tensor(cu_q, dtype=torch.int32),
        cu_seqlens_kv=torch.tensor([0, 3, 9], dtype=torch.int32),
        cu_seqlens_q_padded=pad.clone(), cu_seqlens_kv_padded=pad.clone(),
        attn_scale=0.1, mask_type=MASK_PADDING, dtype="fp16")


PACKINGS = ([128], [128, 96], [128, 128], [256, 256])


def packings(lengths=(128,), seed: int = 42, H: int = 8, d: int = 128) -> Workload:
    """[3333]: bf16, H=8 heads (MHA), d=128, padding_causal, cu == cu_padded,
    upstream gradient of the sum loss (dout = ones)."""
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    q, k, v = (_normal(rng, (T, H, d)) for _ in range(3))
    cu = _cu(lengths)
    return Workload(
        name=f"packings_{'_'.join(map(str, lengths))}", q=_to(q, "bf16"),
        k=_to(k, "bf16"), v=_to(v, "bf16"),
        dout=torch.ones((T, H, d), dtype=torch.bfloat16),
        cu_seqlens_q=cu.clone(), cu_seqlens_kv=cu.clone(),
        cu_seqlens_q_padded=cu.clone(), cu_seqlens_kv_padded=cu.clone(),
        attn_scale=1.0 / math.sqrt(d), mask_type=MASK_PADDING_CAUSAL, dtype="bf16")


def gqa_d256(seed: int = 3216, seq: int = 384, batch: int = 2, hq: int = 16,
             hkv: int = 2, d: int = 256, outlier: float = 20.0,
             outlier_mode: str = "set") -> Workload:
    """[3216] shape as THD: ``batch`` causal sequences of ``seq`` tokens,
    hq=16, hkv=2, d=256, scale 1/sqrt(d). q and k are N(0,1) times a per-channel
    lognormal(0,1) scale (drawn separately for q and k); the same 4 seeded outlier
    channels get scale ``outlier`` (20, i.e. 20x the median channel scale of 1) in
    both, so q.k peaks and the softmax is sharp; v and dout are N(0,1).
    ``outlier_mode="mul"`` multiplies the lognormal scale by ``outlier`` instead
    (a harsher, heavier-tailed variant)."""
    rng = np.random.default_rng(seed)
    T = seq * batch
    sq = rng.lognormal(0.0, 1.0, size=d).astype(np.float32)
    sk = rng.lognormal(0.0, 1.0, size=d).astype(np.float32)
    outl = rng.choice(d, size=4, replace=False)
    if outlier_mode == "mul":
        sq[outl] *= outlier
        sk[outl] *= outlier
    else:
        sq[outl] = outlier
        sk[outl] = outlier
    q = _normal(rng, (T, hq, d)) * sq
    k = _normal(rng, (T, hkv, d)) * sk
    v = _normal(rng, (T, hkv, d))
    do = _normal(rng, (T, hq, d))
    cu = _cu([seq] * batch)
    return Workload(
        name=f"gqa_d256_{outlier_mode}", q=_to(q, "bf16"), k=_to(k, "bf16"), v=_to(v, "bf16"),
        dout=_to(do, "bf16"), cu_seqlens_q=cu.clone(), cu_seqlens_kv=cu.clone(),
        cu_seqlens_q_padded=cu.clone(), cu_seqlens_kv_padded=cu.clone(),
        attn_scale=1.0 / math.sqrt(d), mask_type=MASK_PADDING_CAUSAL, dtype="bf16",
        meta={"outlier_channels": sorted(int(c) for c in outl)})


def real_ne_padded(seed: int = 2892, mask_type: int = MASK_PADDING,
                   real=(100, 150, 120, 130), padded=(112, 160, 128, 144),
                   H: int = 32, d: int = 48, pad_value: float = 1e3) -> Workload:
    """[2892]: real lengths [100,150,120,130] inside padded slots
    [112,160,128,144] (544 rows), 32 heads, d=48, hq=hkv. Real tokens are N(0,1);
    pad slots of q, k, v and dout hold +-pad_value with a seeded random sign, so any
    leak of a pad slot into a real output is large."""
    rng = np.random.default_rng(seed)
    T = int(sum(padded))
    cu = _cu(real)
    cp = _cu(padded)
    valid = np.zeros(T, dtype=bool)
    for b in range(len(real)):
        valid[int(cp[b]):int(cp[b]) + real[b]] = True

    def draw():
        x = _normal(rng, (T, H, d))
        sign = np.where(rng.random(size=(T, H, d)) < 0.5, -1.0, 1.0).astype(np.float32)
        x[~valid] = (pad_value * sign)[~valid]
        return x

    q, k, v, do = draw(), draw(), draw(), draw()
    return Workload(
        name="real_ne_padded" + ("_causal" if mask_type == MASK_PADDING_CAUSAL else ""),
        q=_to(q, "bf16"), k=_to(k, "bf16"), v=_to(v, "bf16"), dout=_to(do, "bf16"),
        cu_seqlens_q=cu.clone(), cu_seqlens_kv=cu.clone(),
        cu_seqlens_q_padded=cp.clone(), cu_seqlens_kv_padded=cp.clone(),
        attn_scale=1.0 / math.sqrt(d), mask_type=mask_type, dtype="bf16")


def throughput_lengths(seed: int = 5, total: int = 32768, lo: int = 256,
                       hi: int = 8192):
    """Seeded sequence lengths: draw uniform integers in [lo, hi] until ``total``
    real tokens are used; the last length takes the remainder, and a draw that would
    leave fewer than ``lo`` tokens is shortened so the remainder stays >= lo."""
    rng = np.random.default_rng(seed)
    rem, out = total, []
    while rem > 0:
        x = int(rng.integers(lo, hi + 1))
        if x >= rem:
            x = rem
        elif rem - x < lo:
            x = rem - lo
        out.append(x)
        rem -= x
    return out


def throughput(seed: int = 5, tensor_seed: int = 55, hq: int = 32, hkv: int = 8,
               d: int = 128, total: int = 32768, align: int = 64) -> Workload:
    """Large packed workload: 32768 real tokens in lengths from
    :func:`throughput_lengths`, each padded up to a multiple of ``align`` rows in
    memory; GQA hq=32, hkv=8, d=128, padding_causal, scale 1/sqrt(d); every slot of
    q, k, v, dout (pad slots included) is N(0,1)."""
    lengths = throughput_lengths(seed, total)
    padded = [((x + align - 1) // align) * align for x in lengths]
    rng = np.random.default_rng(tensor_seed)
    T = int(sum(padded))
    q = _normal(rng, (T, hq, d))
    k = _normal(rng, (T, hkv, d))
    v = _normal(rng, (T, hkv, d))
    do = _normal(rng, (T, hq, d))
    return Workload(
        name="throughput", q=_to(q, "bf16"), k=_to(k, "bf16"), v=_to(v, "bf16"),
        dout=_to(do, "bf16"), cu_seqlens_q=_cu(lengths), cu_seqlens_kv=_cu(lengths),
        cu_seqlens_q_padded=_cu(padded), cu_seqlens_kv_padded=_cu(padded),
        attn_scale=1.0 / math.sqrt(d), mask_type=MASK_PADDING_CAUSAL, dtype="bf16",
        meta={"lengths": lengths, "padded": padded})


def growing_scores(seed: int = 11, lengths=(700, 513, 300), hq: int = 4, hkv: int = 2,
                   d: int = 64, mask_type: int = MASK_PADDING_CAUSAL, dtype: str = "bf16",
                   growth: float = 1.5):
    """Scores that rise along the key axis for every other query row: key j gets
    growth * (j / 128) times a fixed direction u (|u|^2 = d) added to its N(0,1)
    entries, odd query rows get u added. With scale 1/sqrt(d), an odd row's score
    against key j then carries growth * sqrt(d) * j / 128, i.e. it grows by
    growth * sqrt(d) per 128 keys (12 for the defaults, over 17 in log2 units): a
    running row maximum moves by more than 2^8 from one key tile to the next, while
    even rows stay nearly flat. Packed, padded by 0-5 rows per sequence."""
    rng = np.random.default_rng(seed)
    lens = list(lengths)
    pads = [x + int(rng.integers(0, 6)) for x in lens]
    T = int(sum(pads))
    u = rng.standard_normal(d).astype(np.float32)
    u *= np.float32(math.sqrt(d) / np.linalg.norm(u))
    q = _normal(rng, (T, hq, d))
    k = _normal(rng, (T, hkv, d))
    v = _normal(rng, (T, hkv, d))
    do = _normal(rng, (T, hq, d))
    off = 0
    for L, P in zip(lens, pads):
        j = np.arange(P, dtype=np.float32)
        k[off:off + P] += (growth * j / 128.0)[:, None, None] * u[None, None, :]
        q[off + 1:off + P:2] += u[None, None, :]
        off += P
    return Workload(
        name=f"growing_scores_{seed}", q=_to(q, dtype), k=_to(k, dtype), v=_to(v, dtype),
        dout=_to(do, dtype), cu_seqlens_q=_cu(lens), cu_seqlens_kv=_cu(lens),
        cu_seqlens_q_padded=_cu(pads), cu_seqlens_kv_padded=_cu(pads),
        attn_scale=1.0 / math.sqrt(d), mask_type=mask_type, dtype=dtype)


def random_varlen(seed: int, batch: int, max_len: int, hq: int, hkv: int, d: int,
                  mask_type: int, dtype: str = "bf16", pad_max: int = 17,
                  allow_empty: bool = True, tail: int = 5, kv_differs: bool = True):
    """Small random ragged case for edge coverage: per-sequence real lengths in
    [0, max_len] (zero allowed), padded by 0..pad_max extra rows, extra tail rows
    after the last sequence, and independent query and key lengths."""
    rng = np.random.default_rng(seed)
    lo = 0 if allow_empty else 1
    lq = rng.integers(lo, max_len + 1, size=batch)
    lk = rng.integers(lo, max_len + 1, size=batch) if kv_differs else lq.copy()
    pq = lq + rng.integers(0, pad_max + 1, size=batch)
    pk = lk + rng.integers(0, pad_max + 1, size=batch)
    Tq = int(pq.sum()) + tail
    Tk = int(pk.sum()) + tail
    q = _normal(rng, (Tq, hq, d))
    k = _normal(rng, (Tk, hkv, d))
    v = _normal(rng, (Tk, hkv, d))
    do = _normal(rng, (Tq, hq, d))
    return Workload(
        name=f"random_varlen_{seed}", q=_to(q, dtype), k=_to(k, dtype), v=_to(v, dtype),
        dout=_to(do, dtype), cu_seqlens_q=_cu(lq.tolist()),
        cu_seqlens_kv=_cu(lk.tolist()), cu_seqlens_q_padded=_cu(pq.tolist()),
        cu_seqlens_kv_padded=_cu(pk.tolist()), attn_scale=1.0 / math.sqrt(d),
        mask_type=mask_type, dtype=dtype)
