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
