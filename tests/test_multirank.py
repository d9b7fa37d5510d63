"""The benchmark's multi-rank path on the CPU: two gloo ranks (no GPU).

Every rank runs an independent replica (the decode step has no exchange), so what is shared is
host logic: the slowest rank's timed span (max over ranks), the whole-job throughput from it,
and the reference arm running on rank 0 alone."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, spans, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup(None)
        assert (w, r, local) == (world, rank, rank)
        dist.barrier()
        slowest = bench.max_over_ranks(dist, spans[rank], "cpu")
        out.put((rank, slowest, bench.job_throughput(w, 10, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_span_and_sum_the_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    spans = [0.25, 0.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, spans, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 0.5, 40.0), (1, 0.5, 40.0)]  # 2 replicas x 10 steps in 0.5 s


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(None, 1.5, "cpu") == 1.5
    assert bench.job_throughput(1, 4, 2.0) == 2.0


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
