"""Every output element is written: each call runs twice, once into output
buffers filled with NaN and once into buffers filled with zeros, and the two
results must be bit-identical (a row or column a kernel skipped would keep
its NaN, or its zero).  Parity of the values themselves against the oracle
is covered by the other GPU tests; these shapes include ones whose work items
are dealt by the balanced schedule, ragged zig-zag chunks whose last tile
pair has one tile, and a launch small enough to overlap the call before it.
"""
import pytest
import torch

from ring_attention_02_b300 import api
from ring_attention_02_b300.inputs import make_dout, make_qkv

pytestmark = pytest.mark.gpu

LAYOUTS = ["contiguous", "striped", "zigzag"]
SHAPES = [
    # B, H, Hkv, S, D, P, causal
    (1, 16, 4, 4096, 128, 8, True),     # 256+ work items: scheduled
    (1, 4, 2, 3072, 64, 4, True),       # zig-zag chunks of 3 tiles: a one-tile pair
    (1, 2, 2, 256, 64, 4, False),       # 8 items: the small-launch path
]


def _twice(run, shapes_dtypes):
    """run(bufs) fills the given buffers; returns (NaN-started, zero-started)."""
    outs = []
    for fill in (float("nan"), 0.0):
        bufs = [torch.full(s, fill, dtype=d, device="cuda") for s, d in shapes_dtypes]
        run(bufs)
        outs.append(bufs)
    torch.cuda.synchronize()
    api.check_status()
    return outs


def _same(a, b, what):
    for x, y in zip(a, b):
        assert not torch.isnan(x).any(), f"{what}: NaN left in an output"
        assert torch.equal(x, y), f"{what}: result depends on the buffer's prior contents"


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"S{s[3]}H{s[1]}D{s[4]}")
def test_forward_and_backward_write_every_element(layout, shape):
    B, H, Hkv, S, D, P, causal = shape
    if layout == "zigzag" and S % (2 * P):
        pytest.skip("zig-zag needs S % 2P == 0")
    q, k, v = make_qkv(B, H, Hkv, S, D, seed=51, device="cuda")
    for odt in (torch.bfloat16, torch.float32):
        a, b = _twice(lambda bufs: api.fwd(q, k, v, P, layout, causal, out=bufs[0], lse=bufs[1]),
                      [((B, S, H, D), odt), ((B, H, S), torch.float32)])
        _same(a, b, f"fwd {layout} {odt}")
    out, lse = api.fwd(q, k, v, P, layout, causal)
    do = make_dout(B, H, S, D, seed=51, device="cuda")
    a, b = _twice(lambda bufs: api.bwd(q, k, v, out, lse, do, P, layout, causal, dq=bufs[0],
                                       dk=bufs[1], dv=bufs[2]),
                  [(q.shape, torch.bfloat16), (k.shape, torch.bfloat16),
                   (v.shape, torch.bfloat16)])
    _same(a, b, f"bwd {layout}")


@pytest.mark.parametrize("layout", LAYOUTS)
def test_every_hop_writes_every_element(layout):
    B, H, Hkv, S, D, P = 1, 8, 2, 2048, 128, 4
    n = S // P
    q, k, v = make_qkv(B, H, Hkv, S, D, seed=52, device="cuda")
    pos = api.index_map(S, P, layout).cuda()
    for r in range(P):
        qr = q[:, pos[r]].contiguous()
        for s_ in range(P):
            ks, vs = k[:, pos[s_]].contiguous(), v[:, pos[s_]].contiguous()
            a, b = _twice(lambda bufs: api.step(qr, ks, vs, S, P, layout, r, s_, True,
                                                out=bufs[0], lse=bufs[1]),
                          [((B, n, H, D), torch.float32), ((B, H, n), torch.float32)])
            _same(a, b, f"step r={r} s={s_}")


def test_decode_and_packed_forward_write_every_element():
    B, H, Hkv, S, D, P, T = 1, 16, 4, 8192, 128, 8, 5
    q_all, k, v = make_qkv(B, H, Hkv, S, D, seed=53, device="cuda")
    q = q_all[:, S - T:].contiguous()
    a, b = _twice(lambda bufs: api.decode(q, k, v, P, "zigzag", out=bufs[0], lse=bufs[1]),
                  [((B, T, H, D), torch.bfloat16), ((B, H, T), torch.float32)])
    _same(a, b, "decode")
    lengths = [1024, 3072, 512, 2048]
    total = sum(lengths)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    qp, kp, vp = (t[0, :total].contiguous() for t in make_qkv(1, H, Hkv, total, D, seed=54,
                                                                   device="cuda"))
    a, b = _twice(lambda bufs: api.fwd_varlen(qp, kp, vp, cu, P, "zigzag", out=bufs[0],
                                              lse=bufs[1]),
                  [((total, H, D), torch.bfloat16), ((H, total), torch.float32)])
    _same(a, b, "fwd_varlen")
