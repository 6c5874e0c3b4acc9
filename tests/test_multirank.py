"""The bench's multi-GPU path (one replica per GPU, no data-path collective) on CPU ranks.

Each request is independent and all c shards of a request live on one GPU, so N GPUs run N
replicas: the ranks meet at a barrier around the timed region, the step time is the maximum over
ranks, and the whole-job value counts every rank's bytes.  These tests run two gloo ranks on CPU:
the barrier and max-over-ranks helpers, the aggregate, and the reference arm under torchrun
(rank 0 alone runs and prints; the other rank exits 0 without work).
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


def _rank_main(rank, ws, port, local_ms, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(ws),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    got_ws, got_rank, got_local = bench.dist_env()
    bench.barrier(got_ws)
    ms = bench.max_over_ranks(local_ms[rank], got_ws)
    value = bench.whole_job_gbs(1e9, ms, got_ws)
    bench.barrier(got_ws)
    dist.destroy_process_group()
    q.put((rank, got_ws, got_rank, got_local, ms, value))


def test_two_gloo_ranks_take_the_slowest_step_and_count_every_replica():
    ws, port = 2, _free_port()
    local_ms = [0.5, 0.8]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, local_ms, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got_ws, got_rank, got_local, ms, value in res:
        assert (got_ws, got_rank, got_local) == (ws, rank, rank)
        assert ms == max(local_ms)                      # every rank sees the slowest step
        # two replicas of 1 GB each in 0.8 ms: 2 GB / 0.8 ms = 2500 GB/s
        assert value == pytest.approx(2500.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--config", "tiny", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
