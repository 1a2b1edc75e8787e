"""GPU parity of the per-hop backward (ring_attn_step_bwd) against the CPU
oracle (fp64).

A P-rank ring runs P hops per rank: rank r keeps its queries, the key/value
block of shard s = (r - t) mod P arrives at step t, and the block's dk/dv
accumulators travel with it.  Here the P ranks are virtual: every (r, s) hop is
one call, dq is accumulated per query shard and dk/dv per key block, and the
sums are compared with the oracle's full gradients.  Tolerance per gradient
tensor as in the fused backward's tests: max-abs <= 5e-2, relative L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from ring_attention_02_b300 import api
from ring_attention_02_b300.inputs import make_dout, make_qkv

from helpers import max_abs, rel_l2, to64

pytestmark = pytest.mark.gpu

ABS_TOL = 5e-2
REL_TOL = 1e-2
LAYOUTS = ["contiguous", "striped", "zigzag"]


def _shards(x, S, P, layout):
    """[B, S, heads, D] natural order -> list of P shard tensors [B, n, heads, D]."""
    B, n = x.shape[0], S // P
    xs = api.permute(x, S, P, layout).view(B, P, n, *x.shape[2:])
    return [xs[:, r].contiguous() for r in range(P)]


def _lse_shards(lse, S, P, layout):
    B, H = lse.shape[0], lse.shape[1]
    ls = api.permute(lse.reshape(B * H, S).contiguous(), S, P, layout).view(B, H, P, S // P)
    return [ls[:, :, r].contiguous() for r in range(P)]


def _unshard(parts, S, P, layout):
    B = parts[0].shape[0]
    x = torch.stack(parts, dim=1).reshape(B, S, *parts[0].shape[2:]).contiguous()
    return api.permute(x, S, P, layout, inverse=True)


def _ring_of_hops(q, k, v, out, lse, do, P, layout, causal, scale):
    S = q.shape[1]
    qs, ks, vs = (_shards(t, S, P, layout) for t in (q, k, v))
    os_, dos = _shards(out, S, P, layout), _shards(do, S, P, layout)
    ls = _lse_shards(lse, S, P, layout)
    f32 = lambda t: torch.zeros(t.shape, dtype=torch.float32, device=t.device)
    dq = [f32(qs[r]) for r in range(P)]
    dk = [f32(ks[r]) for r in range(P)]
    dv = [f32(vs[r]) for r in range(P)]
    for r in range(P):
        for t in range(P):
            s = (r - t) % P
            api.step_bwd(qs[r], ks[s], vs[s], os_[r], ls[r], dos[r], S, P, layout, r, s, causal,
                         scale, dq=dq[r], dk=dk[s], dv=dv[s], accumulate=True)
    api.check_status()
    return (_unshard(dq, S, P, layout), _unshard(dk, S, P, layout), _unshard(dv, S, P, layout))


def _compare(q, k, v, do, grads, causal, scale, pairs):
    H, Hkv = q.shape[2], k.shape[2]
    G = H // Hkv
    rq, rk, rv = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, scale, pairs)
    gq, gk, gv = (to64(t) for t in grads)
    ours_q = np.stack([np.stack([gq[b, :, g * G + e] for e in range(G)]) for b, g in pairs])
    ours_k = np.stack([gk[b, :, g] for b, g in pairs])
    ours_v = np.stack([gv[b, :, g] for b, g in pairs])
    errs = {n: (max_abs(o, r), rel_l2(o, r))
            for n, o, r in (("dq", ours_q, rq), ("dk", ours_k, rk), ("dv", ours_v, rv))}
    print(f"PARITY hops S{q.shape[1]} H{H} Hkv{Hkv} D{q.shape[3]}: "
          + " ".join(f"{n} max|d|={a:.3e} relL2={r:.3e}" for n, (a, r) in errs.items()))
    for name, (ea, er) in errs.items():
        assert ea <= ABS_TOL and er <= REL_TOL, (name, errs)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_ring_of_backward_hops_matches_oracle(layout, causal, D):
    # S = 1536, P = 4: shards of 384 slots; zig-zag chunks of 192 (ragged tiles)
    B, H, Hkv, S, P = 2, 4, 2, 1536, 4
    scale = D ** -0.5
    q, k, v = make_qkv(B, H, Hkv, S, D, seed=41, device="cuda")
    do = make_dout(B, H, S, D, seed=41, device="cuda")
    out, lse = api.fwd(q, k, v, P, layout, causal)
    grads = _ring_of_hops(q, k, v, out, lse, do, P, layout, causal, scale)
    _compare(q, k, v, do, grads, causal, scale, [(b, g) for b in range(B) for g in range(Hkv)])


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("S,P", [(24, 4), (640, 5), (130, 1)])
def test_ring_of_backward_hops_ragged_shards(layout, S, P):
    if layout == "zigzag" and S % (2 * P):
        pytest.skip("zig-zag needs S % 2P == 0")
    scale = 128 ** -0.5
    q, k, v = make_qkv(1, 2, 1, S, 128, seed=42, device="cuda")
    do = make_dout(1, 2, S, 128, seed=42, device="cuda")
    out, lse = api.fwd(q, k, v, P, layout, True)
    grads = _ring_of_hops(q, k, v, out, lse, do, P, layout, True, scale)
    _compare(q, k, v, do, grads, True, scale, [(0, 0)])


def test_hop_overwrite_and_hidden_block():
    # accumulate = False overwrites every element: a visible hop equals the same
    # hop added onto zeros bit for bit, and a hop whose keys all come after the
    # queries (contiguous shards, r < s, causal) is exactly zero
    B, H, Hkv, S, D, P, layout = 1, 4, 2, 2048, 128, 4, "contiguous"
    q, k, v = make_qkv(B, H, Hkv, S, D, seed=43, device="cuda")
    do = make_dout(B, H, S, D, seed=43, device="cuda")
    out, lse = api.fwd(q, k, v, P, layout, True)
    qs, ks, vs = (_shards(t, S, P, layout) for t in (q, k, v))
    os_, dos, ls = _shards(out, S, P, layout), _shards(do, S, P, layout), \
        _lse_shards(lse, S, P, layout)
    for r, s in ((2, 1), (2, 2), (1, 3)):
        fill = lambda t: torch.full(t.shape, float("nan"), dtype=torch.float32, device="cuda")
        a = api.step_bwd(qs[r], ks[s], vs[s], os_[r], ls[r], dos[r], S, P, layout, r, s, True,
                         dq=fill(qs[r]), dk=fill(ks[s]), dv=fill(vs[s]), accumulate=False)
        zero = lambda t: torch.zeros(t.shape, dtype=torch.float32, device="cuda")
        b = api.step_bwd(qs[r], ks[s], vs[s], os_[r], ls[r], dos[r], S, P, layout, r, s, True,
                         dq=zero(qs[r]), dk=zero(ks[s]), dv=zero(vs[s]), accumulate=True)
        api.check_status()
        for x, y in zip(a, b):
            assert torch.equal(x, y), (r, s)
            if r < s:
                assert torch.count_nonzero(x).item() == 0, (r, s)
