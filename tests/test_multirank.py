"""The N > 1 host logic of bench.py on CPU: two gloo ranks (world size 2).

The path needs no collective (every sequence and key/value head is independent),
so several GPUs run independent replicas; what the ranks share is the step time
(the slowest rank's), the whole-job throughput, and rank 0 alone printing.
"""

import io
import contextlib
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        worst = bench.max_over_ranks(ms[rank], world)
        value = bench.whole_job_tflops(1.0e12, worst, world)
        dist.barrier()
        # the reference arm prints on rank 0 only; other ranks return at once
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(None, rank, world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"worst": worst, "value": value, "printed": buf.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step(tmp_path):
    ms = [4.0, 5.0]
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, ms, str(tmp_path)))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["worst"] == 5.0
        # 2 replicas x 1 TFLOP each per 5 ms step
        assert r["value"] == pytest.approx(2 * 1.0e12 / 5e-3 / 1e12)
    assert res[1]["printed"] == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(5.0e12, 5.0, 1) == pytest.approx(1000.0)


def test_kernel_source_hash_ignores_comments_only():
    """The traffic record stays valid across comment edits and goes stale on any
    code edit: the hash covers the sources with comments and whitespace removed."""
    sys.path.insert(0, ROOT)
    import bench
    code = "int f(int x) {  // doubles x\n  return 2 * x; /* no overflow check */\n}\n"
    recommented = "// f: twice x\nint f(int x) {\n  return 2 * x;   // same code\n}\n"
    changed = "int f(int x) {  // doubles x\n  return 3 * x;\n}\n"
    assert bench.code_only(code) == bench.code_only(recommented)
    assert bench.code_only(code) != bench.code_only(changed)
    assert bench.code_only('asm("mov.b32 %0, %1;");') == 'asm("mov.b32 %0, %1;");'
    for k in bench.KERNEL_SOURCES:
        assert len(bench.kernel_source_hash(k)) == 16


def test_head_dim_option_is_checked(monkeypatch):
    """`--head-dim` takes the library's head dims only (multiples of 8 in [8, 256]);
    anything else stops at argument parsing, before any workload is built."""
    sys.path.insert(0, ROOT)
    import bench
    for good in ("8", "64", "256"):
        monkeypatch.setattr(sys, "argv", ["bench.py", "--head-dim", good])
        assert bench.parse().head_dim == int(good)
    for bad in ("0", "12", "264"):
        monkeypatch.setattr(sys, "argv", ["bench.py", "--head-dim", bad])
        with pytest.raises(SystemExit):
            bench.parse()
