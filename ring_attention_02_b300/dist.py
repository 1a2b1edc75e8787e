"""Ring attention across ranks: one process per GPU, one shard per rank.

The pages' setting ("Sequenzparallelitaet und Ringaufmerksamkeit", "Tiefer
Einblick"; "Context parallelism and zig-zag ring attention", "Zig Zag Ring
Attention"): rank r keeps the queries of shard r, its key/value block travels
around the ring (sent to rank r+1, received from rank r-1), and every rank
computes the partial attention of each arriving block and folds it into its
running result.  The next block's transfer is started before the current
block's products, so communication overlaps compute.

The backward lets each block's dk/dv accumulators travel with it: at step t
rank r holds block s = (r - t) mod P and its accumulators, adds its own
queries' contribution and passes both on; after P steps the accumulators have
met every query shard and one last hop returns them to their owner.

The SP/EP page names Ulysses beside Ring Attention: an all-to-all gives every
rank the whole sequence of H/P heads, each rank runs attention on its head
group, and a second all-to-all returns the sequence shards (``ulysses_fwd``,
``ulysses_bwd``).

Every computation runs in the library's kernels (``api``); this module only
moves blocks between ranks with ``torch.distributed``.  NCCL process groups
exchange the device tensors directly.  Other backends (gloo) carry CPU tensors
only: the blocks are staged through pinned host buffers, which serves tests
that run several ranks without a GPU each.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


class RingComm:
    """The ring's point-to-point exchange: send to rank (r+1) mod P, receive
    from (r-1) mod P, several tensors at a time, started and finished apart so
    that compute can run in between."""

    def __init__(self, group=None):
        if not dist.is_initialized():
            raise RuntimeError("torch.distributed is not initialized")
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.backend = dist.get_backend(group)
        self.staged = self.backend != "nccl"
        nxt, prv = (self.rank + 1) % self.world, (self.rank - 1) % self.world
        self.next = dist.get_global_rank(group, nxt) if group is not None else nxt
        self.prev = dist.get_global_rank(group, prv) if group is not None else prv
        self._pinned = {}

    def _host(self, key, like):
        buf = self._pinned.get(key)
        if buf is None or buf.shape != like.shape or buf.dtype != like.dtype:
            buf = torch.empty(like.shape, dtype=like.dtype,
                              pin_memory=torch.cuda.is_available())
            self._pinned[key] = buf
        return buf

    def start(self, send, recv, tag: int = 0):
        """Starts sending each tensor of `send` to the next rank and receiving
        each of `recv` (same shapes) from the previous one.  Returns a handle
        for finish().  Device tensors must be complete on the current stream."""
        if self.world == 1:
            raise RuntimeError("a ring of one rank exchanges nothing")
        if not self.staged:
            ops = [dist.P2POp(dist.isend, t, self.next, self.group) for t in send]
            ops += [dist.P2POp(dist.irecv, t, self.prev, self.group) for t in recv]
            return dist.batch_isend_irecv(ops), None
        if any(t.is_cuda for t in send):
            torch.cuda.current_stream().synchronize()
        hs = [self._host(("s", tag, i), t) for i, t in enumerate(send)]
        hr = [self._host(("r", tag, i), t) for i, t in enumerate(recv)]
        for h, t in zip(hs, send):
            h.copy_(t)
        works = [dist.isend(h, self.next, self.group, tag=100 * tag + i) for i, h in enumerate(hs)]
        works += [dist.irecv(h, self.prev, self.group, tag=100 * tag + i)
                  for i, h in enumerate(hr)]
        return works, (hr, recv)

    def finish(self, handle):
        """Waits for a start()ed exchange; the received tensors are then ready
        on the current stream."""
        works, staged = handle
        for w in works:
            w.wait()
        if staged is not None:
            for h, t in zip(*staged):
                t.copy_(h)

    def all_to_all(self, out, inp):
        """out[i] = block i of rank i's `inp` (both [world, ...], contiguous)."""
        if not self.staged:
            dist.all_to_all_single(out, inp, group=self.group)
            return out
        if inp.is_cuda:
            torch.cuda.current_stream().synchronize()
        hi = self._host(("a2a_in",), inp)
        ho = self._host(("a2a_out",), out)
        hi.copy_(inp)
        dist.all_to_all_single(ho, hi, group=self.group)
        out.copy_(ho)
        return out


def _scale(D, scale):
    return D ** -0.5 if scale is None else float(scale)


class HopTimeline:
    """Per-hop timings of one rank's ring: for each step t the block s it
    computed on, the device time of that hop's kernels and the time the rank
    then spent waiting for the next block to arrive.  The pages' overlap
    condition ("Zig Zag Ring Attention": compute per hop at least the transfer
    per hop) holds where the waits stay near zero.  CUDA events on the current
    stream; read the numbers with hops() after a synchronize."""

    def __init__(self):
        self._rec = []

    def mark(self, t, s):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record()
        self._rec.append((t, s, ev))
        return ev

    def hops(self):
        out = []
        for t, s, ev in self._rec:
            out.append({"step": t, "block": s, "compute_ms": ev[0].elapsed_time(ev[1]),
                        "wait_ms": ev[1].elapsed_time(ev[2])})
        return out


def ring_fwd(q, k, v, S: int, layout, causal: bool = True, scale: float | None = None,
             comm: RingComm | None = None, out_dtype=torch.bfloat16,
             timeline: HopTimeline | None = None):
    """Forward on rank r of a P-rank ring (P = the group size).

    q [B, n, H, D], k/v [B, n, Hkv, D]: this rank's shard r in local-slot order
    (bf16), n = S / P, shard contents fixed by `layout`.  Returns this shard's
    (out [B, n, H, D] in out_dtype (bf16 or fp32), lse [B, H, n] fp32).
    With a HopTimeline (device tensors only), each hop's compute and wait
    times are recorded in it.
    """
    comm = comm or RingComm()
    P, r = comm.world, comm.rank
    B, n, H, D = q.shape
    scale = _scale(D, scale)
    if n * P != S:
        raise ValueError(f"shard of {n} rows on {P} ranks does not make S={S}")
    acc_o = torch.empty((B, n, H, D), dtype=torch.float32, device=q.device)
    acc_l = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
    if P > 1:
        part_o, part_l = torch.empty_like(acc_o), torch.empty_like(acc_l)
        bufs = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]
    held = (k, v)
    for t in range(P):
        s = (r - t) % P
        pend = None
        if t < P - 1:
            nxt = bufs[t % 2]
            pend = comm.start(list(held), list(nxt))      # block s moves on while it is used
        ev = timeline.mark(t, s) if timeline is not None else None
        if t == 0:
            api.step(q, held[0], held[1], S, P, layout, r, s, causal, scale, out=acc_o, lse=acc_l)
        else:
            api.step(q, held[0], held[1], S, P, layout, r, s, causal, scale, out=part_o,
                     lse=part_l)
            api.merge(acc_o, acc_l, part_o, part_l)
        if ev is not None:
            ev[1].record()
        if pend is not None:
            comm.finish(pend)
            held = nxt
        if ev is not None:
            ev[2].record()
    out = api.finalize(acc_o) if out_dtype == torch.bfloat16 else acc_o
    return out, acc_l


def ring_bwd(q, k, v, out, lse, dout, S: int, layout, causal: bool = True,
             scale: float | None = None, comm: RingComm | None = None):
    """Backward on rank r of a P-rank ring.

    q, out, dout [B, n, H, D] and k, v [B, n, Hkv, D]: shard r (bf16, local
    order); lse [B, H, n] fp32 from ring_fwd.  Returns fp32 (dq [B, n, H, D],
    dk, dv [B, n, Hkv, D]) of shard r.
    """
    comm = comm or RingComm()
    P, r = comm.world, comm.rank
    B, n, H, D = q.shape
    Hkv = k.shape[2]
    scale = _scale(D, scale)
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.empty((B, n, H, D), **f32)
    acc = [(torch.empty((B, n, Hkv, D), **f32), torch.empty((B, n, Hkv, D), **f32))
           for _ in range(2)]
    if P > 1:
        bufs = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]
    held = (k, v)
    for t in range(P):
        s = (r - t) % P
        dk_s, dv_s = acc[t % 2]
        pend = None
        if t < P - 1:
            nxt = bufs[t % 2]
            pend = comm.start(list(held), list(nxt), tag=0)
        # t = 0: dq and this rank's own block's accumulators start here
        api.step_bwd(q, held[0], held[1], out, lse, dout, S, P, layout, r, s, causal, scale,
                     dq=dq, dk=dk_s, dv=dv_s, accumulate=t > 0)
        if P > 1:
            # block s's accumulators follow it to the next rank
            pend_acc = comm.start([dk_s, dv_s], list(acc[(t + 1) % 2]), tag=1)
        if pend is not None:
            comm.finish(pend)
            held = nxt
        if P > 1:
            comm.finish(pend_acc)
    # after the last hop rank r holds its own block's complete accumulators
    dk, dv = acc[P % 2] if P > 1 else acc[0]
    return dq, dk, dv


# ---------------------------------------------------------------- Ulysses

def _seq_to_heads(x, S, layout, comm):
    """[B, n, Hx, D] sequence shard of all heads -> [B, S, Hx/P, D] whole
    sequence (natural order) of this rank's head group."""
    P = comm.world
    B, n, Hx, D = x.shape
    send = api.head_split(x, B * n, P).view(P, B, n, Hx // P, D)
    recv = comm.all_to_all(torch.empty_like(send), send)
    full = torch.empty((B, S, Hx // P, D), dtype=x.dtype, device=x.device)
    return api.permute_shards(recv, S, P, layout, inverse=True, out=full)


def _heads_to_seq(x, S, layout, comm):
    """Inverse of _seq_to_heads: [B, S, Hg, D] -> [B, n, Hg*P, D]."""
    P = comm.world
    B, _, Hg, D = x.shape
    n = S // P
    blocks = api.permute_shards(x, S, P, layout).view(P, B, n, Hg, D)
    recv = comm.all_to_all(torch.empty_like(blocks), blocks)
    out = torch.empty((B, n, Hg * P, D), dtype=x.dtype, device=x.device)
    return api.head_split(recv, B * n, P, inverse=True, out=out)


def _lse_to_heads(lse, S, layout, comm):
    """[B, H, n] -> [B, H/P, S] (this rank's head group, natural order)."""
    P = comm.world
    B, H, n = lse.shape
    send = api.head_split(lse, B, P).view(P, B * (H // P), n)
    recv = comm.all_to_all(torch.empty_like(send), send)
    full = torch.empty((B, H // P, S), dtype=lse.dtype, device=lse.device)
    return api.permute_shards(recv, S, P, layout, inverse=True, out=full)


def _lse_to_seq(lse, S, layout, comm):
    """[B, Hg, S] -> [B, Hg*P, n]."""
    P = comm.world
    B, Hg, _ = lse.shape
    n = S // P
    blocks = api.permute_shards(lse.view(B * Hg, S), S, P, layout).view(P, B, Hg, n)
    recv = comm.all_to_all(torch.empty_like(blocks), blocks)
    out = torch.empty((B, Hg * P, n), dtype=lse.dtype, device=lse.device)
    return api.head_split(recv, B, P, inverse=True, out=out)


def _check_heads(H, Hkv, P):
    if H % P or Hkv % P:
        raise ValueError(f"head-sharded attention needs H={H} and Hkv={Hkv} divisible by the "
                         f"{P} ranks")


def ulysses_fwd(q, k, v, S: int, layout, causal: bool = True, scale: float | None = None,
                comm: RingComm | None = None):
    """Head-sharded forward on rank r: same shard inputs and outputs as
    ring_fwd (bf16 out [B, n, H, D], lse [B, H, n]); H and Hkv divisible by P.
    The all-to-all gives this rank heads [r*H/P, (r+1)*H/P) of the whole
    sequence, the fused forward runs on them, and a second all-to-all returns
    the sequence shard."""
    comm = comm or RingComm()
    B, n, H, D = q.shape
    _check_heads(H, k.shape[2], comm.world)
    scale = _scale(D, scale)
    qf, kf, vf = (_seq_to_heads(t, S, layout, comm) for t in (q, k, v))
    of, lf = api.fwd(qf, kf, vf, 1, "contiguous", causal, scale=scale)
    return _heads_to_seq(of, S, layout, comm), _lse_to_seq(lf, S, layout, comm)


def ulysses_bwd(q, k, v, out, lse, dout, S: int, layout, causal: bool = True,
                scale: float | None = None, comm: RingComm | None = None):
    """Head-sharded backward on rank r: bf16 (dq [B, n, H, D], dk, dv
    [B, n, Hkv, D]) of shard r, from the shard tensors ulysses_fwd (or
    ring_fwd) took and gave."""
    comm = comm or RingComm()
    B, n, H, D = q.shape
    _check_heads(H, k.shape[2], comm.world)
    scale = _scale(D, scale)
    qf, kf, vf, of, dof = (_seq_to_heads(t, S, layout, comm) for t in (q, k, v, out, dout))
    lf = _lse_to_heads(lse, S, layout, comm)
    dqf, dkf, dvf = api.bwd(qf, kf, vf, of, lf, dof, 1, "contiguous", causal, scale=scale)
    return tuple(_heads_to_seq(t, S, layout, comm) for t in (dqf, dkf, dvf))
