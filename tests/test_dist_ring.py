"""The multi-rank exchange of ring_attention_02_b300.dist on CPU: gloo ranks
(world 2 and 3) run the ring's point-to-point schedule and the head-sharded
all-to-all on CPU tensors, without kernels.  At ring step t rank r must hold
the block of shard (r - t) mod P ("Tiefer Einblick": blocks pass from rank to
rank), and the accumulators that travel with the blocks must return to their
owner after P hops."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from ring_attention_02_b300.dist import RingComm

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        comm = RingComm()
        assert (comm.rank, comm.world) == (rank, world)
        # block identities along the ring, double-buffered like ring_fwd
        held = torch.full((3, 5), float(rank))
        bufs = [torch.empty(3, 5), torch.empty(3, 5)]
        seen = [int(held[0, 0])]
        for t in range(world - 1):
            nxt = bufs[t % 2]
            h = comm.start([held], [nxt])
            comm.finish(h)
            held = nxt
            seen.append(int(held[0, 0]))
        # accumulators travelling with their block: each rank adds 10^rank
        acc = [torch.zeros(4), torch.zeros(4)]
        for t in range(world):
            cur, other = acc[t % 2], acc[(t + 1) % 2]
            cur += 10 ** rank
            comm.finish(comm.start([cur], [other], tag=1))
        final = acc[world % 2]
        # the head-sharded all-to-all: block i of rank j's input lands as block j
        # of rank i's output
        inp = torch.arange(world * 6, dtype=torch.float32).view(world, 6) + 100 * rank
        out = comm.all_to_all(torch.empty_like(inp), inp)
        q.put((rank, seen, final.tolist(), out.tolist()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_schedule_and_all_to_all_on_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, seen, final, out = q.get(timeout=180)
        res[rank] = (seen, final, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    total = float(sum(10 ** r for r in range(world)))
    for r in range(world):
        seen, final, out = res[r]
        assert seen == [(r - t) % world for t in range(world)]
        # the accumulators that came back to rank r have met every rank once
        assert final == [total] * 4
        for j in range(world):
            assert out[j] == [100 * j + 6 * r + c for c in range(6)]
