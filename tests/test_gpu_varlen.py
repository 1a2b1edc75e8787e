"""GPU parity of the packed-sequence forward: each sequence of the pack must
equal the plain attention (fp64 oracle) of that sequence alone; tolerances as
for the forward (out max-abs 2e-2, lse max-abs 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
from ring_attention_02_b300 import api
from ring_attention_02_b300.inputs import make_qkv

from helpers import max_abs, to64

pytestmark = pytest.mark.gpu

LAYOUTS = ["contiguous", "striped", "zigzag"]


def _pack(lengths, H, Hkv, D, seed):
    total = int(sum(lengths))
    q, k, v = make_qkv(1, H, Hkv, total, D, seed=seed, device="cuda")
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q[0], k[0], v[0], cu


def _check(lengths, H, Hkv, D, P, layout, causal, seed, out_dtype=torch.bfloat16):
    q, k, v, cu = _pack(lengths, H, Hkv, D, seed)
    out, lse = api.fwd_varlen(q, k, v, cu, P, layout, causal, out_dtype=out_dtype)
    api.check_status()
    eo = el = 0.0
    for i in range(len(lengths)):
        a, b = int(cu[i]), int(cu[i + 1])
        ro, rl = oracle.attn_fwd(to64(q[a:b])[None], to64(k[a:b])[None], to64(v[a:b])[None],
                                 causal, D ** -0.5)
        eo = max(eo, max_abs(to64(out[a:b]), ro[0]))
        el = max(el, max_abs(to64(lse[:, a:b]), rl[0]))
    print(f"PARITY varlen {lengths} H{H} Hkv{Hkv} D{D} P{P} {layout} causal={causal}: "
          f"max|out|={eo:.3e} max|lse|={el:.3e}")
    assert eo <= 2e-2 and el <= 1e-3, (eo, el)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_pack_of_four(layout, causal, D):
    _check([1024, 2048, 512, 3072], 4, 2, D, 4, layout, causal, seed=41)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_ragged_and_tiny_sequences(layout):
    # shards of 8..200 slots: ragged tiles inside every sequence
    _check([16, 400, 8, 1600, 96], 2, 1, 128, 4 if layout != "zigzag" else 4, layout, True,
           seed=42)


def test_single_sequence_equals_dense_forward():
    S, H, Hkv, D, P = 4096, 8, 2, 128, 8
    q, k, v = make_qkv(1, H, Hkv, S, D, seed=43, device="cuda")
    dense_o, dense_l = api.fwd(q, k, v, P, "zigzag", True)
    vo, vl = api.fwd_varlen(q[0], k[0], v[0], [0, S], P, "zigzag", True)
    api.check_status()
    assert torch.equal(vo.view(torch.int16), dense_o[0].view(torch.int16))
    assert torch.equal(vl, dense_l[0])


def test_rejects_lengths_the_layout_cannot_split():
    q, k, v, cu = _pack([1024, 1020], 2, 2, 64, seed=44)
    with pytest.raises(api.RingAttnError):
        api.fwd_varlen(q, k, v, cu, 4, "zigzag", True)       # 1020 % 8 != 0


# ---------------------------------------------------------------- backward

def _check_bwd(lengths, H, Hkv, D, P, layout, causal, seed):
    q, k, v, cu = _pack(lengths, H, Hkv, D, seed)
    from ring_attention_02_b300.inputs import make_dout
    do = make_dout(1, H, int(cu[-1]), D, seed=seed, device="cuda")[0]
    out, lse = api.fwd_varlen(q, k, v, cu, P, layout, causal)
    dq, dk, dv = api.bwd_varlen(q, k, v, out, lse, do, cu, P, layout, causal)
    api.check_status()
    G = H // Hkv
    worst = {"dq": (0.0, 0.0), "dk": (0.0, 0.0), "dv": (0.0, 0.0)}
    for i in range(len(lengths)):
        a, b = int(cu[i]), int(cu[i + 1])
        pairs = [(0, g) for g in range(Hkv)]
        rq, rk, rv = oracle.attn_bwd(to64(q[a:b])[None], to64(k[a:b])[None], to64(v[a:b])[None],
                                     to64(do[a:b])[None], causal, D ** -0.5, pairs)
        gq, gk, gv = to64(dq[a:b]), to64(dk[a:b]), to64(dv[a:b])
        ours_q = np.stack([np.stack([gq[:, g * G + e] for e in range(G)]) for _, g in pairs])
        ours_k = np.stack([gk[:, g] for _, g in pairs])
        ours_v = np.stack([gv[:, g] for _, g in pairs])
        for name, ours, ref in (("dq", ours_q, rq), ("dk", ours_k, rk), ("dv", ours_v, rv)):
            ea = max_abs(ours, ref)
            er = float(np.linalg.norm(ours - ref) / max(np.linalg.norm(ref), 1e-300))
            worst[name] = (max(worst[name][0], ea), max(worst[name][1], er))
    print(f"PARITY varlen bwd {lengths} H{H} Hkv{Hkv} D{D} P{P} {layout} causal={causal}: "
          + " ".join(f"{n} max|d|={a:.3e} relL2={r:.3e}" for n, (a, r) in worst.items()))
    for name, (ea, er) in worst.items():
        assert ea <= 5e-2 and er <= 1e-2, (name, worst)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
def test_backward_pack_of_four(layout, causal):
    _check_bwd([1024, 2048, 512, 3072], 4, 2, 128, 4, layout, causal, seed=45)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_backward_ragged_sequences_d64(layout):
    _check_bwd([16, 400, 8, 1600, 96], 2, 1, 64, 4, layout, True, seed=46)


def test_backward_single_sequence_equals_dense():
    S, H, Hkv, D, P = 4096, 8, 2, 128, 8
    from ring_attention_02_b300.inputs import make_dout
    q, k, v = make_qkv(1, H, Hkv, S, D, seed=47, device="cuda")
    do = make_dout(1, H, S, D, seed=47, device="cuda")
    out, lse = api.fwd(q, k, v, P, "zigzag", True)
    dense = api.bwd(q, k, v, out, lse, do, P, "zigzag", True)
    packed = api.bwd_varlen(q[0], k[0], v[0], out[0], lse[0], do[0], [0, S], P, "zigzag", True)
    api.check_status()
    for a, b in zip(packed, dense):
        assert torch.equal(a.view(torch.int16), b[0].view(torch.int16))
