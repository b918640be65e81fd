"""bench.py's multi-rank path on the CPU: two gloo ranks, as torchrun would start them.
Each rank shards its own trees (distinct seeds), the ranks meet at the barrier, the
step time is the maximum over ranks, and the reported rate counts every rank's rows.
The reference arm prints from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench

    w, r, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    elapsed_ms = 10.0 + 5.0 * r  # rank 1 is the slow one
    slowest = bench.max_over_ranks(elapsed_ms, w, "cpu")
    rate = bench.whole_job_rate(w, 3840, 100, slowest)
    seeds = [None] * w
    torch.distributed.all_gather_object(seeds, bench.shard_seed(20261202, r))
    bench.barrier(w)
    torch.distributed.destroy_process_group()
    queue.put((r, slowest, rate, seeds))


def test_two_gloo_ranks_shard_and_reduce():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, slowest, rate, seeds in results:
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 3840 * 100 / 15e-3)
        assert len(set(seeds)) == 2


def _reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--gpus", str(world), "--workload", "eagle10_v32000", "--steps", "4",
                           "--warmup", "1"], env=env, cwd=ROOT, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_prints_from_rank_zero_only():
    other = _reference(1, 2)
    assert other.returncode == 0, other.stderr
    assert other.stdout.strip() == ""
    lead = _reference(0, 2)
    assert lead.returncode == 0, lead.stderr
    lines = [ln for ln in lead.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
