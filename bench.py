#!/usr/bin/env python
"""Throughput of THD attention forward + backward on GB300.

One step = te_attn_fwd_thd + te_attn_bwd_thd over the large packed workload:
32768 real tokens in seeded lengths in [256, 8192] (each padded to a multiple of
64 rows in memory), GQA hq=32 / hkv=8, head_dim 128, padding_causal, bf16.
The metric is causal-adjusted algorithmic fwd+bwd TFLOPS: per (sequence, query
head) 3.5 * 4 * d * Lq*Lk/2 FLOPs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --configs      # every configuration, GPU beside the CPU oracle

Under torchrun every rank runs its own replica of the workload on its own GPU
(the path needs no collective); rank 0 prints one JSON line. ``--impl reference``
times the CPU float64 oracle on a bounded sample of the same workload instead.
``--configs`` prints one JSON line per configuration of the pages' workloads (the
tiny GQA pair, the four packings, the d=256 GQA batch, real != padded, the large
packed workload): GPU fwd+bwd time and TFLOPS, and the oracle's wall time for the
same fwd+bwd on the host cores (the large workload's oracle time is extrapolated
from a timed sample, as stated in its line).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "THD attn fwd+bwd TFLOPS (causal-adj) & % GB300 dense BF16 peak, 1 GPU"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the timings of the e4m3 forward and the sequence-major layout")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["throughput", "small"], default="throughput",
                    help="small: the same recipe with 8192 real tokens (for ncu captures)")
    ap.add_argument("--head-dim", type=int, default=128,
                    help="head dim of the workload (a multiple of 8 in [8, 256]; default 128)")
    ap.add_argument("--bwd", choices=["two-kernel", "fused"], default="two-kernel",
                    help="backward of the timed step: te_attn_bwd_thd (dQ and dK/dV kernels) "
                         "or te_attn_bwd_thd_fused (one pass)")
    ap.add_argument("--configs", action="store_true",
                    help="time every configuration beside the CPU oracle (one line each)")
    args = ap.parse_args()
    if not (8 <= args.head_dim <= 256 and args.head_dim % 8 == 0):
        ap.error("--head-dim must be a multiple of 8 in [8, 256]")
    return args


# ----------------------------------------------------------------- helpers


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            raw = json.load(open(path))

            def find(*keys):
                for k in keys:
                    if k in raw and isinstance(raw[k], (int, float)):
                        return float(raw[k])
                return None
            out = {"hbm_gbs": find("hbm_gbs"), "bf16_tflops": find("bf16_tflops"),
                   "bf16_tflops_sustained": find("bf16_tflops_sustained")}
            if all(v is not None for v in out.values()):
                out["source"] = "measured"
                return out
        except Exception:
            pass
    out = dict(FALLBACK)
    out["source"] = "fallback"
    return out


class ClockSampler:
    """nvidia-smi sampled every 100 ms by a reader thread that stamps each line on
    arrival; only samples taken between ``mark_start()`` and ``mark_end()`` (the
    timed region) are summarised."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None
        self.thread = None

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line))

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True,
                bufsize=1)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except Exception:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        t0 = self.t0 if self.t0 is not None else -math.inf
        t1 = self.t1 if self.t1 is not None else math.inf
        sm, smax, pw, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for stamp, line in list(self.lines):
            # a line arrives at most one sampling period after it was taken
            if not (t0 < stamp <= t1 + 0.1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            if self.uuid and f[0] != self.uuid:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                pw.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in timed region"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "sm_min_mhz": min(sm), "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(pw)}


def gpu_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# Sources each kernel's code comes from (its file and the headers it includes).
_HEADERS = ["common.cuh", "sm103_ptx.cuh", "row_store.cuh", "work_queue.cuh", "tmap.h"]
KERNEL_SOURCES = {"fwd": ["attn_fwd_pair.cu"] + _HEADERS, "dkdv": ["attn_bwd.cu"] + _HEADERS,
                  "dq": ["attn_bwd.cu"] + _HEADERS, "bwd_fused": ["attn_bwd_fused.cu"] + _HEADERS}


def code_only(text):
    """C++ source without comments and with whitespace collapsed: edits to comments
    leave a kernel's hash (and so its traffic record) unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bwd_packed_varlen_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu record, if it was
    taken on the kernel's current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    try:
        k = json.load(open(path)).get("kernels", {}).get(kernel, {})
        if k.get("source_hash") != kernel_source_hash(kernel):
            return None
        return k.get("dram_bytes_per_launch_full")
    except Exception:
        return None


def causal_pairs(w):
    import numpy as np
    lq = np.diff(w.cu_seqlens_q.numpy()).astype(np.float64)
    lk = np.diff(w.cu_seqlens_kv.numpy()).astype(np.float64)
    f = 0.5 if w.mask_type in (2, 3) else 1.0
    return float((lq * lk * f).sum())


def workload_config(w):
    lengths = w.meta.get("lengths")
    return {
        "workload": (f"packed THD fwd+bwd: {sum(lengths)} real tokens in {len(lengths)} seeded "
                     f"sequences {lengths} padded to multiples of 64 (T={w.q.shape[0]}), "
                     f"hq={w.hq}, hkv={w.hkv}, d={w.d}, padding_causal, bf16"),
        "global_batch": len(lengths),
        "seq_len": max(lengths),
        "total_tokens": int(sum(lengths)),
        "padded_rows": int(w.q.shape[0]),
        "hq": w.hq, "hkv": w.hkv, "head_dim": w.d,
        "parallelism": "replicas (one independent workload per GPU)",
        "l2": ("device-resident value: flushed between timed steps (256 MiB write); "
               "e2e: inputs copied in from the host every step, larger than L2, no flush"),
    }


# ------------------------------------------------------------ oracle sample


def oracle_sample(w, seqs, groups):
    """Run the CPU float64 oracle on (sequence, kv-group) pairs of the workload;
    returns (seconds, algorithmic FLOPs of the sample)."""
    import numpy as np
    import oracle
    G = w.hq // w.hkv
    cq, cp = w.cu_seqlens_q.numpy(), w.cu_seqlens_q_padded.numpy()
    flops = 0.0
    args = []
    for b in seqs:
        o, L = int(cp[b]), int(cq[b + 1] - cq[b])
        for g in groups:
            hs = slice(g * G, g * G + G)
            args.append((w.q[o:o + L, hs].double().numpy(), w.k[o:o + L, g].double().numpy(),
                         w.v[o:o + L, g].double().numpy(), w.dout[o:o + L, hs].double().numpy()))
            flops += 3.5 * 4.0 * w.d * G * L * L / 2.0
    t0 = time.perf_counter()
    for q, k, v, do in args:
        oracle.attn_group_fwd_bwd(q, k, v, do, w.attn_scale, True)
    return time.perf_counter() - t0, flops


def blas_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


# ------------------------------------------------------------------ ranks


def max_over_ranks(x, world, device="cpu"):
    """Largest value of x over all ranks: the slowest replica sets the step time.
    (No-op for one rank; uses the default process group otherwise.)"""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_replica, ms_per_step, world):
    """Throughput of all replicas together: each rank processes one workload per
    step, and a step lasts as long as the slowest rank's."""
    return world * flops_per_replica / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------ variants


def time_calls(fn, flush, steps, warmup):
    """Mean device time (ms) of fn() over `steps` calls after `warmup`, with L2
    flushed before each call and CUDA events on the current stream."""
    import torch
    for _ in range(warmup):
        flush.fill_(1)
        fn()
    st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i & 0xFF)
        st[i].record()
        fn()
        en[i].record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in zip(st, en)) / steps


def measure_variants(ta, w, t, flops, fwd_flops, flush, dev, steps=20, warmup=5):
    """Device-resident timings of the library's other entry points on the same
    sequences: the e4m3 forward (inputs quantised once with per-tensor factors
    amax / 448) and forward + backward in the sequence-major layout (each sequence
    the front of one [S, B, h, d] batch entry, S = the longest length)."""
    import numpy as np
    import torch
    out = {}
    f8 = getattr(torch, "float8_e4m3fn", None)
    cu = (t["cu_seqlens_q"], t["cu_seqlens_kv"], t["cu_seqlens_q_padded"], t["cu_seqlens_kv_padded"])
    if f8 is not None and w.d % 16 == 0 and w.d <= 128:  # the e4m3 forward's head dims
        def quant(x):
            descale = float(x.float().abs().amax()) / 448.0
            return (x.float() / descale).clamp(-448.0, 448.0).to(f8), descale
        (q8, qd), (k8, kd), (v8, vd) = quant(t["q"]), quant(t["k"]), quant(t["v"])
        o = torch.empty_like(t["q"])
        l = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=dev)
        Tq, hq, d = t["q"].shape
        Tk, hkv, _ = t["k"].shape
        ws = torch.empty(int(ta.library().te_attn_fwd_e4m3_workspace_size(w.batch, Tq, Tk, hq, hkv, d)),
                         dtype=torch.uint8, device=dev)
        ms = time_calls(lambda: ta.fwd_e4m3(q8, k8, v8, *cu, w.attn_scale, qd, kd, vd,
                                            w.mask_type, out=o, lse=l, workspace=ws),
                        flush, steps, warmup)
        out["e4m3_forward"] = {"ms": ms, "tflops": fwd_flops / (ms * 1e-3) / 1e12,
                               "note": "Q K^T on the e4m3 tensor path, V widened to bf16 once "
                                       "per call, P V in bf16; includes the widening"}
    lens = [int(x) for x in w.meta["lengths"]]
    S, B = max(lens), len(lens)
    offs = [int(x) for x in w.cu_seqlens_q_padded[:-1]]

    def to_sbhd(x):
        y = torch.zeros((S, B) + tuple(x.shape[1:]), dtype=x.dtype, device=dev)
        for b in range(B):
            y[:lens[b], b] = x[offs[b]:offs[b] + lens[b]]
        return y
    qs, ks, vs, dos = (to_sbhd(t[n]) for n in ("q", "k", "v", "dout"))
    cus = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
    os_, ls = torch.empty_like(qs), torch.empty((S, B, qs.shape[2]), dtype=torch.float32, device=dev)
    dq_, dk_, dv_ = torch.empty_like(qs), torch.empty_like(ks), torch.empty_like(vs)
    wsf = torch.empty(ta.fwd_workspace_size(B, S * B, S * B, qs.shape[2], ks.shape[2], qs.shape[3]),
                      dtype=torch.uint8, device=dev)
    wsb = torch.empty(ta.bwd_workspace_size(B, S * B, S * B, qs.shape[2], ks.shape[2], qs.shape[3]),
                      dtype=torch.uint8, device=dev)

    def sbhd_step():
        ta.fwd_sbhd(qs, ks, vs, cus, cus, w.attn_scale, w.mask_type, out=os_, lse=ls, workspace=wsf)
        ta.bwd_sbhd(qs, ks, vs, os_, dos, ls, cus, cus, w.attn_scale, w.mask_type, dq=dq_, dk=dk_,
                    dv=dv_, workspace=wsb)
    ms = time_calls(sbhd_step, flush, steps, warmup)
    out["sbhd_fwd_bwd"] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                           "shape": f"[{S}, {B}, h, d] with the workload's real lengths"}
    # A/B of the backward: the default two-kernel path (separate dQ kernel recomputing
    # S and dP) against the fused one (one pass, ordered fp32 dQ accumulation).
    Tq, hq, d = t["q"].shape
    Tk, hkv, _ = t["k"].shape
    o = torch.empty_like(t["q"])
    l = torch.empty((Tq, hq), dtype=torch.float32, device=dev)
    ta.fwd(t["q"], t["k"], t["v"], *cu, w.attn_scale, w.mask_type, out=o, lse=l)
    g = [torch.empty_like(t[n]) for n in ("q", "k", "v")]
    for name, fused in (("bwd_default", False), ("bwd_fused", True)):
        size = (ta.bwd_fused_workspace_size if fused else ta.bwd_workspace_size)(
            w.batch, Tq, Tk, hq, hkv, d)
        ws = torch.empty(size, dtype=torch.uint8, device=dev)
        ms = time_calls(lambda: ta.bwd(t["q"], t["k"], t["v"], o, t["dout"], l, *cu, w.attn_scale,
                                       w.mask_type, dq=g[0], dk=g[1], dv=g[2], workspace=ws,
                                       fused=fused),
                        flush, steps, warmup)
        out[name] = {"ms": ms, "tflops": 2.5 * fwd_flops / (ms * 1e-3) / 1e12,
                     "workspace_bytes": size}
    return out


# ------------------------------------------------------------------ arms


def run_reference(args, rank, world):
    if rank != 0:
        return
    from bwd_packed_varlen_gb300 import workloads as W
    w = (W.throughput(d=args.head_dim) if args.workload == "throughput"
         else W.throughput(total=8192, d=args.head_dim))
    seqs, groups = [min(4, w.batch - 1)], [0]
    for _ in range(args.warmup):
        oracle_sample(w, seqs, groups)
    times, fl = [], 0.0
    for _ in range(args.steps):
        t, fl = oracle_sample(w, seqs, groups)
        times.append(t)
    mean = sum(times) / len(times)
    val = fl / mean / 1e12
    b = seqs[0]
    sample = (f"sequence {b} ({int(w.cu_seqlens_q[b + 1] - w.cu_seqlens_q[b])} tokens) x kv-group 0 "
              f"({w.hq // w.hkv} query heads) of the workload, fwd+bwd")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import bwd_packed_varlen_gb300 as ta
    from bwd_packed_varlen_gb300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    ta.library()
    w = (W.throughput(d=args.head_dim) if args.workload == "throughput"
         else W.throughput(total=8192, d=args.head_dim))
    # the committed DRAM counts were taken on the default workload only
    default_workload = args.workload == "throughput" and args.head_dim == 128
    flops = w.algorithmic_flops()
    pairs_h = causal_pairs(w) * w.hq  # sum over (sequence, query head) of Lq*Lk/2
    t = {k: getattr(w, k).to(dev) for k in ("q", "k", "v", "dout", "cu_seqlens_q",
                                             "cu_seqlens_kv", "cu_seqlens_q_padded",
                                             "cu_seqlens_kv_padded")}
    Tq, hq, d = w.q.shape
    Tk, hkv, _ = w.k.shape
    B = w.batch
    out = torch.empty_like(t["q"])
    lse = torch.empty((Tq, hq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    wsf = torch.empty(ta.fwd_workspace_size(B, Tq, Tk, hq, hkv, d), dtype=torch.uint8, device=dev)
    fused = args.bwd == "fused"
    wsb = torch.empty((ta.bwd_fused_workspace_size if fused else ta.bwd_workspace_size)(
        B, Tq, Tk, hq, hkv, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cu = (t["cu_seqlens_q"], t["cu_seqlens_kv"], t["cu_seqlens_q_padded"], t["cu_seqlens_kv_padded"])

    def step(q, k, v, do, cus):
        ta.fwd(q, k, v, *cus, w.attn_scale, w.mask_type, w.max_seqlen_q, w.max_seqlen_kv,
               out=out, lse=lse, workspace=wsf)
        ta.bwd(q, k, v, out, do, lse, *cus, w.attn_scale, w.mask_type, w.max_seqlen_q,
               w.max_seqlen_kv, dq=dq, dk=dk, dv=dv, workspace=wsb, fused=fused)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        flush.fill_(1)
        step(t["q"], t["k"], t["v"], t["dout"], cu)
    torch.cuda.synchronize()
    ta.profile_read()  # clear

    # ------------------------------------------------ device-resident timed region
    ta.profile_enable(True)
    clocks = ClockSampler(gpu_uuid(dev))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    clocks.mark_start()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record()
        step(t["q"], t["k"], t["v"], t["dout"], cu)
        ends[i].record()
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier()
    clk = clocks.stop()
    ta.profile_enable(False)
    kprof = ta.profile_read()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    value = whole_job_tflops(flops, ms, world)
    launches = sum(c for _, c in kprof.values())

    # ------------------------------------------------ end to end from host buffers
    e2e = None
    if not args.no_e2e:
        host_in = {k: v.pin_memory() for k, v in
                   (("q", w.q), ("k", w.k), ("v", w.v), ("dout", w.dout),
                    ("cu_seqlens_q", w.cu_seqlens_q), ("cu_seqlens_kv", w.cu_seqlens_kv),
                    ("cu_seqlens_q_padded", w.cu_seqlens_q_padded),
                    ("cu_seqlens_kv_padded", w.cu_seqlens_kv_padded))}
        # two device copies of the inputs: step i+1's inputs arrive while step i runs
        dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host_in.items()}
                  for _ in range(2)]
        host_out = [torch.empty_like(x, device="cpu").pin_memory() for x in (out, lse, dq, dk, dv)]
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(x.numel() * x.element_size() for x in host_out)
        # Every step copies its own inputs in from pinned host memory and its own
        # results out, all inside the timed region (one pair of events around the
        # K steps, divided by K). The copies run on two copy streams and overlap
        # compute the way a training loop's prefetch does: step i's inputs go into
        # one of two device buffers while step i-1 computes on the other; out/lse
        # travel back while the backward runs, dq while dk/dv are computed (the
        # backward's dq hand-over event), dk/dv while the next step's forward runs.
        # Events order every reuse of a buffer after the copy that reads it. The
        # inputs copied each step exceed L2, so no flush runs in this region.
        main = torch.cuda.current_stream(dev)
        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)
        fwd_in = ("q", "k", "v", "cu_seqlens_q", "cu_seqlens_kv", "cu_seqlens_q_padded",
                  "cu_seqlens_kv_padded")
        ev = lambda: torch.cuda.Event()

        def e2e_steps(n):
            """n steps of the overlapped loop, then both copy streams joined into main."""
            in_free = [None, None]       # backward of the last step that read buffer j
            out_copied = dq_copied = dkdv_copied = None
            first = ev()
            first.record(main)
            s_in.wait_event(first)
            s_out.wait_event(first)
            for i in range(n):
                buf = dev_in[i % 2]
                with torch.cuda.stream(s_in):
                    if in_free[i % 2] is not None:
                        s_in.wait_event(in_free[i % 2])
                    for k_ in fwd_in:
                        buf[k_].copy_(host_in[k_], non_blocking=True)
                    ev_fwd_in = ev()
                    ev_fwd_in.record(s_in)
                    buf["dout"].copy_(host_in["dout"], non_blocking=True)
                    ev_bwd_in = ev()
                    ev_bwd_in.record(s_in)
                cus_d = (buf["cu_seqlens_q"], buf["cu_seqlens_kv"], buf["cu_seqlens_q_padded"],
                         buf["cu_seqlens_kv_padded"])
                main.wait_event(ev_fwd_in)
                if out_copied is not None:
                    main.wait_event(out_copied)
                ta.fwd(buf["q"], buf["k"], buf["v"], *cus_d, w.attn_scale, w.mask_type,
                       w.max_seqlen_q, w.max_seqlen_kv, out=out, lse=lse, workspace=wsf)
                ev_fwd = ev()
                ev_fwd.record(main)
                main.wait_event(ev_bwd_in)
                if dq_copied is not None:
                    main.wait_event(dq_copied)
                    main.wait_event(dkdv_copied)
                ev_dq = ev()
                ta.bwd(buf["q"], buf["k"], buf["v"], out, buf["dout"], lse, *cus_d,
                       w.attn_scale, w.mask_type, w.max_seqlen_q, w.max_seqlen_kv, dq=dq, dk=dk, dv=dv,
                       workspace=wsb, dq_done=None if fused else ev_dq, fused=fused)
                if fused:
                    ev_dq.record(main)
                ev_bwd = ev()
                ev_bwd.record(main)
                in_free[i % 2] = ev_bwd
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_fwd)
                    host_out[0].copy_(out, non_blocking=True)
                    host_out[1].copy_(lse, non_blocking=True)
                    out_copied = ev()
                    out_copied.record(s_out)
                    s_out.wait_event(ev_dq)
                    host_out[2].copy_(dq, non_blocking=True)
                    dq_copied = ev()
                    dq_copied.record(s_out)
                    s_out.wait_event(ev_bwd)
                    host_out[3].copy_(dk, non_blocking=True)
                    host_out[4].copy_(dv, non_blocking=True)
                    dkdv_copied = ev()
                    dkdv_copied.record(s_out)
            main.wait_stream(s_out)
            main.wait_stream(s_in)

        # untimed warm-up steps of the same loop, as for the device-resident region
        e2e_steps(max(args.warmup, 3))
        torch.cuda.synchronize()
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e_start.record(main)
        e2e_steps(args.steps)
        e_end.record(main)
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(e_start.elapsed_time(e_end) / args.steps, world, dev)
        # the results that came back are the device results of the last step
        for got, ref in zip(host_out, (out, lse, dq, dk, dv)):
            if not torch.equal(got.view(torch.uint8), ref.cpu().view(torch.uint8)):
                raise RuntimeError("end-to-end copies returned other bytes than the device holds")
        e2e = {"value": whole_job_tflops(flops, ems, world), "unit": "TFLOPS",
               "ms_per_step": ems, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "overlap": "double-buffered input prefetch; outputs copied as they become final"}

    variants = None
    if not args.no_variants:
        variants = measure_variants(ta, w, t, flops, 4.0 * d * pairs_h, flush, dev)

    if rank != 0:
        return

    # ------------------------------------------------ roofline of the dominant kernel
    peaks = load_peaks()
    credited = {"fwd": 4.0 * d * pairs_h, "dkdv": 8.0 * d * pairs_h, "dq": 2.0 * d * pairs_h,
                "bwd_fused": 10.0 * d * pairs_h}
    executed = {"fwd": 4.0 * d * pairs_h, "dkdv": 8.0 * d * pairs_h, "dq": 6.0 * d * pairs_h,
                "bwd_fused": 10.0 * d * pairs_h}
    kernels = {}
    for name, (tot, cnt) in kprof.items():
        if cnt == 0:
            continue
        avg = tot / cnt
        ent = {"launches": cnt, "total_ms": tot, "avg_ms": avg, "share": tot / max(1e-9, sum(
            x for x, _ in kprof.values()))}
        if name in credited:
            ent["tflops_credited"] = credited[name] / (avg * 1e-3) / 1e12
            ent["tflops_executed"] = executed[name] / (avg * 1e-3) / 1e12
            ent["frac_credited"] = ent["tflops_credited"] / peaks["bf16_tflops"]
            ent["frac_executed"] = ent["tflops_executed"] / peaks["bf16_tflops"]
        kernels[name] = ent
    dom = max(("fwd", "dkdv", "dq", "bwd_fused"),
              key=lambda n: kernels.get(n, {}).get("total_ms", 0.0))
    # The dominant kernel runs for a few ms at a time inside a step of a fraction of
    # a second of timed work: the burst figure is its denominator.
    peak = peaks["bf16_tflops"]
    ach = kernels[dom]["tflops_credited"]
    roofline = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak,
                "traffic": ncu_traffic(dom) if default_workload else None,
                "peak_kind": f"bf16 dense burst ({peaks['source']})",
                "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                "flops_per_launch": credited[dom]}
    if "delta" in kernels:
        dbytes = 2 * Tq * hq * d * 2 + Tq * hq * 4
        kernels["delta"]["gbs"] = dbytes / (kernels["delta"]["avg_ms"] * 1e-3) / 1e9
        kernels["delta"]["hbm_frac"] = kernels["delta"]["gbs"] / peaks["hbm_gbs"]
    if "dq_convert" in kernels:
        # reads the fp32 accumulator of every real row and head, writes 16-bit dq
        real = int(w.cu_seqlens_q[-1])
        cbytes = real * hq * d * (4 + 2)
        kernels["dq_convert"]["gbs"] = cbytes / (kernels["dq_convert"]["avg_ms"] * 1e-3) / 1e9
        kernels["dq_convert"]["hbm_frac"] = kernels["dq_convert"]["gbs"] / peaks["hbm_gbs"]

    cpu = None
    if not args.no_cpu_baseline and world == 1 and args.workload == "throughput":
        secs, fl = oracle_sample(w, [3, 4], [0, 1, 2])
        cpu = {"value": fl / secs / 1e12, "unit": "TFLOPS", "cores": blas_threads(),
               "kind": "oracle", "seconds": secs,
               "sample": "sequences 3 and 4 (6668 and 3977 tokens) x kv-groups 0-2 (4 query "
                         "heads each) of the workload, fwd+bwd, numpy float64"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": dict(workload_config(w), backward=(
            "te_attn_bwd_thd_fused" if fused else "te_attn_bwd_thd (dQ, dK/dV kernels)")),
        "pct_peak": {"burst": value / world / peaks["bf16_tflops"],
                     "sustained": value / world / peaks["bf16_tflops_sustained"],
                     "source": peaks["source"]},
        "flops_per_step": flops * world,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clk, "kernels": kernels, "variants": variants,
        "step_ms_median": statistics.median(step_ms), "step_ms_min": min(step_ms),
        "step_ms_max": max(step_ms),
    }
    print(json.dumps(line), flush=True)


def median_calls(fn, flush, steps, warmup):
    """Median device time (ms) of fn() over `steps` calls after `warmup`, L2 flushed
    before each call, CUDA events on the current stream."""
    import torch
    for _ in range(warmup):
        flush.fill_(1)
        fn()
    st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i & 0xFF)
        st[i].record()
        fn()
        en[i].record()
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in zip(st, en))


def run_configs(args):
    """One line per configuration: GPU fwd+bwd median (20 timed calls after 5
    warm-ups, L2 flushed) and the CPU oracle's wall time for the same fwd+bwd."""
    import torch
    import bwd_packed_varlen_gb300 as ta
    import oracle
    from bwd_packed_varlen_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ta.library()
    peaks = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cases = [("C1 tiny GQA, call A", W.tiny_gqa("A")), ("C1 tiny GQA, call B", W.tiny_gqa("B"))]
    cases += [(f"C2 packing {list(p)}", W.packings(list(p))) for p in W.PACKINGS]
    cases += [("C3 GQA d=256, 2 x 384 causal", W.gqa_d256()),
              ("C4 real != padded, d=48", W.real_ne_padded()),
              ("C5 large packed workload", W.throughput())]
    for name, w in cases:
        t = {k: getattr(w, k).to(dev) for k in ("q", "k", "v", "dout", "cu_seqlens_q",
                                                 "cu_seqlens_kv", "cu_seqlens_q_padded",
                                                 "cu_seqlens_kv_padded")}
        cu = (t["cu_seqlens_q"], t["cu_seqlens_kv"], t["cu_seqlens_q_padded"],
              t["cu_seqlens_kv_padded"])
        Tq, hq, d = w.q.shape
        Tk, hkv, _ = w.k.shape
        out = torch.empty_like(t["q"])
        lse = torch.empty((Tq, hq), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
        wsf = torch.empty(max(1, ta.fwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d)),
                          dtype=torch.uint8, device=dev)
        wsb = torch.empty(max(1, ta.bwd_workspace_size(w.batch, Tq, Tk, hq, hkv, d)),
                          dtype=torch.uint8, device=dev)

        def step():
            ta.fwd(t["q"], t["k"], t["v"], *cu, w.attn_scale, w.mask_type, out=out, lse=lse,
                   workspace=wsf)
            ta.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, *cu, w.attn_scale, w.mask_type,
                   dq=dq, dk=dk, dv=dv, workspace=wsb)
        ms = median_calls(step, flush, 20, 5)
        flops = w.algorithmic_flops()
        line = {"config": name, "gpu_ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                "pct_of_bf16_burst": flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                "flops": flops, "dtype": w.dtype, "cores": blas_threads()}
        if name.startswith("C5"):
            secs, fl = oracle_sample(w, [3, 4], [0, 1, 2])
            line["oracle_s"] = secs * flops / fl
            line["oracle_note"] = ("extrapolated from a timed sample (sequences 3 and 4 x kv "
                                   "groups 0-2) by FLOPs")
        else:
            np64 = lambda x: x.double().numpy()  # noqa: E731
            t0 = time.perf_counter()
            oracle.attn_fwd_bwd_thd(np64(w.q), np64(w.k), np64(w.v), np64(w.dout),
                                    w.cu_seqlens_q.numpy(), w.cu_seqlens_kv.numpy(),
                                    w.cu_seqlens_q_padded.numpy(),
                                    w.cu_seqlens_kv_padded.numpy(), w.attn_scale, w.mask_type)
            line["oracle_s"] = time.perf_counter() - t0
        line["oracle_tflops"] = flops / line["oracle_s"] / 1e12
        print(json.dumps(line), flush=True)
        del t, out, lse, dq, dk, dv, wsf, wsb


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.configs:
        if rank == 0:
            run_configs(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
