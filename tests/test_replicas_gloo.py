"""The N > 1 bench path on CPU: one process per rank over gloo (world size 2).

The GEMM shards trivially and this build runs one GEMM per GPU with no
exchange ("replicas only"), so the only multi-rank logic is the bench's:
the step time is the maximum over ranks and the job's throughput counts
every rank's work over that time.  The reference arm prints from rank 0
only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    my_ms = [2.0, 3.5][rank]                       # rank 1 is the slow one
    agreed = bench.slowest_rank_ms(my_ms, world)
    rate = bench.job_throughput(1e12, world, agreed)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, agreed, rate))


def test_step_time_is_max_over_ranks_and_throughput_counts_all_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, agreed, rate in out:
        assert agreed == 3.5                       # both ranks report the slowest time
        assert rate == pytest.approx(2 * 1e12 / 3.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod1", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.slowest_rank_ms(1.25, 1) == 1.25
    assert bench.job_throughput(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_prints_only_on_rank_zero():
    # rank 1 of a reference run exits 0 without work or output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "c1", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
