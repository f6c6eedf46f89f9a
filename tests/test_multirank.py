"""The multi-rank paths of bench.py on CPU: two gloo ranks (no GPU).

bench.py --gpus N runs one replica per rank (the block has no exchange step);
`value` is all ranks' tokens over the slowest rank's time, and the reference
arm runs on rank 0 alone while the other ranks exit without work.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's 5 timed steps sum to 10 (r + 1) ms
        ms = bench.slowest_rank_ms(10.0 * (rank + 1), 5, world)
        out[rank] = (ms, bench.whole_job_rate(4096, ms, world))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_whole_job_rate_over_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, rate = res[rank]
        assert ms == 4.0  # the slowest rank: 20 ms over 5 steps
        assert rate == 2 * 4096 / 0.004


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(12.0, 4, 1) == 3.0
    assert bench.whole_job_rate(100, 2.0, 1) == 50_000.0


def test_reference_arm_runs_on_rank_zero_only():
    """torchrun with two CPU ranks: one JSON line, from rank 0, both exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--gpus", "2", "--impl", "reference", "--workload", "tiny", "--steps", "1",
           "--warmup", "3", "--reference-tokens", "4"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert lines[0]["impl"] == "reference" and lines[0]["value"] > 0
