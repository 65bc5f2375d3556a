"""The bench's N>1 path on CPU: two gloo ranks (no GPU).

Each rank verifies its own batch (weak scaling, no collective on the data
path); the job's time is the slowest rank's, its throughput the tokens of all
ranks over that time, and only rank 0 prints a line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        got = bench.job_elapsed_ms(10.0 * (rank + 1), world, "cpu", torch)
        tok = bench.job_tokens_per_s(8, 16, 100, world, got)
        out.put((rank, got, tok))
    finally:
        dist.destroy_process_group()


def test_job_time_is_max_over_ranks_and_value_counts_all_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's 20 ms; 2 ranks x 8 x 16 tokens x 100 steps / 20 ms
    assert [r[1] for r in res] == [20.0, 20.0]
    assert res[0][2] == pytest.approx(2 * 8 * 16 * 100 / 0.020)


def test_only_rank0_prints_the_reference_line():
    """Under torchrun the reference arm runs on rank 0 alone; the other ranks
    exit 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_single_rank_reference_line_without_gpu():
    """Rank 0 of the reference arm prints one JSON line (here: unavailable, no
    CUDA device to prepare the inputs)."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"


def test_steps_per_graph_divides_the_timed_steps():
    import bench
    for R in (1, 2, 3, 4, 8):
        for K in (1, 2, 3, 5, 7, 12, 2000, 2001):
            P = bench.steps_per_graph(R, K)
            assert 1 <= P <= min(R, 4, K) and K % P == 0, (R, K, P)
    assert bench.steps_per_graph(4, 2000) == 4
    assert bench.steps_per_graph(2, 5) == 1
