"""GPU parity of the backward (dq, dk, dv) against the CPU oracle (fp64).

The forward's own outputs (bf16 out, fp32 lse) feed the backward, as in
training.  Tolerance per gradient tensor: max-abs <= 5e-2 and relative L2
<= 1e-2 against the fp64 gradients of the same bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from ring_attention_02_b300 import api
from ring_attention_02_b300.inputs import TRAIN_32K, make_dout, make_qkv

from helpers import max_abs, rel_l2, to64

pytestmark = pytest.mark.gpu

ABS_TOL = 5e-2
REL_TOL = 1e-2
LAYOUTS = ["contiguous", "striped", "zigzag"]


def _run(B, H, Hkv, S, D, P, layout, causal, seed, scale=None):
    scale = D ** -0.5 if scale is None else scale
    q, k, v = make_qkv(B, H, Hkv, S, D, seed=seed, device="cuda")
    do = make_dout(B, H, S, D, seed=seed, device="cuda")
    out, lse = api.fwd(q, k, v, P, layout, causal, scale=scale)
    dq, dk, dv = api.bwd(q, k, v, out, lse, do, P, layout, causal, scale=scale)
    api.check_status()
    return q, k, v, do, dq, dk, dv, scale


def _compare(q, k, v, do, dq, dk, dv, causal, scale, pairs):
    """Oracle gradients for the (b, kv head) pairs, compared tensor by tensor."""
    H, Hkv = q.shape[2], k.shape[2]
    G = H // Hkv
    rq, rk, rv = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, scale, pairs)
    gq, gk, gv = to64(dq), to64(dk), to64(dv)
    ours_q = np.stack([np.stack([gq[b, :, g * G + e] for e in range(G)]) for b, g in pairs])
    ours_k = np.stack([gk[b, :, g] for b, g in pairs])
    ours_v = np.stack([gv[b, :, g] for b, g in pairs])
    errs = {}
    for name, ours, ref in (("dq", ours_q, rq), ("dk", ours_k, rk), ("dv", ours_v, rv)):
        errs[name] = (max_abs(ours, ref), rel_l2(ours, ref))
    print(f"PARITY bwd B{q.shape[0]} S{q.shape[1]} H{H} Hkv{Hkv} D{q.shape[3]} pairs={pairs}: "
          + " ".join(f"{n} max|d|={a:.3e} relL2={r:.3e}" for n, (a, r) in errs.items()))
    for name, (ea, er) in errs.items():
        assert ea <= ABS_TOL and er <= REL_TOL, (name, errs)
    return errs


def _all_pairs(B, Hkv):
    return [(b, g) for b in range(B) for g in range(Hkv)]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_small_all_layouts(layout, causal, D):
    # S = 1536, P = 4: shards of 384 slots; zig-zag chunks of 192 (ragged tiles).
    B, H, Hkv, S, P = 2, 4, 2, 1536, 4
    q, k, v, do, dq, dk, dv, scale = _run(B, H, Hkv, S, D, P, layout, causal, seed=11)
    _compare(q, k, v, do, dq, dk, dv, causal, scale, _all_pairs(B, Hkv))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("S,P", [(8, 8), (24, 4), (200, 2), (640, 5), (130, 1)])
def test_ragged_and_tiny_shards(layout, S, P):
    if layout == "zigzag" and S % (2 * P):
        pytest.skip("zig-zag needs S % 2P == 0")
    q, k, v, do, dq, dk, dv, scale = _run(1, 2, 1, S, 128, P, layout, True, seed=12)
    _compare(q, k, v, do, dq, dk, dv, True, scale, [(0, 0)])


def test_grouped_heads_sum_over_the_group():
    # four query heads per key/value head: dk and dv sum the four heads' terms
    q, k, v, do, dq, dk, dv, scale = _run(1, 8, 2, 2048, 128, 8, "zigzag", True, seed=13)
    _compare(q, k, v, do, dq, dk, dv, True, scale, _all_pairs(1, 2))


def test_negative_scale():
    q, k, v, do, dq, dk, dv, scale = _run(1, 2, 2, 512, 64, 4, "striped", True, seed=14,
                                          scale=-0.2)
    _compare(q, k, v, do, dq, dk, dv, True, scale, _all_pairs(1, 2))


def test_zero_dout_gives_zero_gradients():
    B, H, S, D = 1, 2, 1024, 128
    q, k, v = make_qkv(B, H, H, S, D, seed=15, device="cuda")
    out, lse = api.fwd(q, k, v, 4, "zigzag", True)
    do = torch.zeros_like(q)
    dq, dk, dv = api.bwd(q, k, v, out, lse, do, 4, "zigzag", True)
    api.check_status()
    for t in (dq, dk, dv):
        assert torch.count_nonzero(t).item() == 0


def test_training_step_32k_two_heads_in_full():
    # The training workload at full size: every gradient of (b=0, kv head 0) and
    # (b=1, kv head 15) against the oracle (its forward half is checked on
    # sampled rows in test_gpu_fwd.py).
    w = TRAIN_32K
    q, k, v, do, dq, dk, dv, scale = _run(w.B, w.H, w.Hkv, w.S, w.D, w.P, w.layout, True,
                                          seed=0)
    _compare(q, k, v, do, dq, dk, dv, True, scale, [(0, 0), (1, w.Hkv - 1)])


def test_deterministic():
    args = (1, 4, 2, 4096, 128, 8, "zigzag", True)
    r1 = _run(*args, seed=16)
    r2 = _run(*args, seed=16)
    for a, b in zip(r1[4:7], r2[4:7]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
