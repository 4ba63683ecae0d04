"""The N > 1 plumbing of bench.py on CPU: two ranks over gloo.

The layer does not shard (every GPU runs an independent replica), so the
only multi-rank logic is the timing harness: the barrier around the timed
region, the maximum over ranks of the measured time, and the reference arm,
which rank 0 alone runs while the other ranks exit without work.
"""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r, local = bench.dist_init(None)
    bench.barrier(ws)
    v = bench.max_over_ranks(1.5 + 2.0 * rank, ws)
    bench.barrier(ws)
    dist.destroy_process_group()
    q.put((r, ws, v))


def test_barrier_and_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")  # a fresh interpreter per rank
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("rank did not finish")
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    # every rank sees world size 2 and the maximum of (1.5, 3.5)
    assert got == [(0, 2, 3.5), (1, 2, 3.5)]


def test_reference_arm_two_ranks_rank0_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["n_gpus"] == 2 and rec["value"] > 0 and rec["steps"] == 1
