"""The N > 1 host path of bench.py on CPU: world-size-2 gloo ranks.

bench.py runs one independent replica per GPU (the path has no exchange
step); across ranks it needs only a barrier, max-over-ranks of the timed
region and the sum of the work done.  These tests run that logic on two gloo
ranks, and the reference arm under torchrun, where rank 0 alone prints.
"""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local, pg = bench.dist_setup(world)
    assert (r, w) == (rank, world) and pg is not None
    bench.barrier(pg)
    mx = bench.max_over_ranks(pg, 10.0 + rank)       # slowest rank's time
    sm = bench.sum_over_ranks(pg, 1000.0 * (rank + 1))  # bytes from all ranks
    out.put((rank, mx, sm))
    pg.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 11.0, 3000.0), (1, 11.0, 3000.0)]


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # the same metric and workload as the CUDA arm's default line
    sys.path.insert(0, ROOT)
    import bench
    assert d["metric"] == bench.LM_HEAD_METRIC and d["higher_is_better"] is True
    assert d["config"] == dict(bench.lm_head_config(152064, 4096, [1, 4, 8, 16]), parallelism="replicas x2")
