"""The N>1 path of bench.py on CPU: two gloo ranks through torch.distributed.

bench.py runs one process per GPU; the method's ranks are virtual shards
inside each process, so the processes are independent replicas and the only
cross-rank traffic is the timing protocol: a barrier around the timed region
and the maximum of the ranks' times.  These tests run that protocol on CPU,
and check that under --impl reference only rank 0 prints a line.
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


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench

    r, w = bench._dist()
    assert (r, w) == (rank, world)
    assert dist.get_backend() == "gloo"
    bench._barrier()
    got = bench.max_over_ranks(10.0 + rank)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 11.0, 1: 11.0}


def test_reference_arm_under_torchrun_prints_one_line():
    # --impl reference on CPU: the oracle on a small sample; rank 1 exits quietly
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
           "--workload", "tiny-noncausal-B1H2S256D64P4", "--steps", "1", "--warmup", "3",
           "--ref-rows", "8"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
