"""The multi-replica path of bench.py on CPU (world size 2, gloo, 127.0.0.1):
rank discovery from the launcher's environment, the barrier, the time taken
as the maximum over ranks, and the reference arm that only rank 0 runs.
The hot path does not shard across GPUs here (replicas only), so these
host-side pieces are the whole N > 1 path."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, ws = bench._dist(backend="gloo")
    bench._barrier(dist)
    slowest = bench._max_over_ranks(dist, 1.5 * (rank + 1))
    bench._barrier(dist)
    q.put((r, ws, slowest))
    dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 for g in got)
    assert all(g[2] == 3.0 for g in got)          # max over ranks, seen by both


@pytest.mark.timeout(600)
def test_reference_arm_runs_on_rank_zero_only():
    """bench.py --impl reference under a 2-rank launcher environment: rank 1
    exits 0 at once without work or output; rank 0 prints the JSON line."""
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()),
               WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
            "--steps", "1", "--warmup", "1"]
    r1 = subprocess.run(args, env=dict(env, RANK="1", LOCAL_RANK="1"), capture_output=True,
                        text=True, timeout=120)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = subprocess.run(args, env=dict(env, RANK="0", LOCAL_RANK="0"), capture_output=True,
                        text=True, timeout=600)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
