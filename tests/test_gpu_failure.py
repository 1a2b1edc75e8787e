"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies gives up, the device status word records it, ring_attn_check_status
reports RA_ERR_DEVICE_TIMEOUT once, and the context keeps working."""
import numpy as np
import pytest

import oracle
from ring_attention_02_b300 import api
from ring_attention_02_b300.inputs import make_dout, make_qkv

from helpers import max_abs, rel_l2, to64

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_survives():
    api.check_status()                      # start from a clean status word
    waited = api.wait_selfcheck(50)
    assert 50e6 <= waited < 1e9, waited     # gave up after the 50 ms limit
    with pytest.raises(api.RingAttnError) as ei:
        api.check_status()
    assert ei.value.status == 7             # RA_ERR_DEVICE_TIMEOUT
    api.check_status()                      # reported once, then cleared
    # the library keeps computing correct results afterwards
    q, k, v = make_qkv(1, 2, 2, 512, 128, seed=31, device="cuda")
    out, lse = api.fwd(q, k, v, 4, "zigzag", True)
    api.check_status()
    ro, rl = oracle.attn_fwd(to64(q), to64(k), to64(v), True, 128 ** -0.5)
    assert max_abs(to64(out), ro) <= 2e-2 and max_abs(to64(lse), rl) <= 1e-3


def test_selfcheck_rejects_bad_limits():
    with pytest.raises(api.RingAttnError):
        api.wait_selfcheck(0)
    with pytest.raises(api.RingAttnError):
        api.wait_selfcheck(5000)


def _expect_timeout():
    with pytest.raises(api.RingAttnError) as ei:
        api.check_status()
    assert ei.value.status == 7             # RA_ERR_DEVICE_TIMEOUT


def test_production_kernels_give_up_and_the_next_calls_are_correct():
    # The forward and backward kernels with a 1 us wait limit: their waits for
    # tensor-core products and the other roles run out, every CTA gives up,
    # waits for its own loads and products in flight, frees its tensor memory
    # and returns.  The status reports the timeout once; with the default limit
    # back, the same calls (and a decode) match the oracle.
    B, H, Hkv, S, D, P = 1, 8, 4, 4096, 128, 8
    scale = D ** -0.5
    q, k, v = make_qkv(B, H, Hkv, S, D, seed=61, device="cuda")
    do = make_dout(B, H, S, D, seed=61, device="cuda")
    api.check_status()
    out0, lse0 = api.fwd(q, k, v, P, "zigzag", True)
    api.check_status()
    try:
        api.set_wait_limit(1000)
        api.fwd(q, k, v, P, "zigzag", True)
        _expect_timeout()
        api.bwd(q, k, v, out0, lse0, do, P, "zigzag", True)
        _expect_timeout()
    finally:
        api.set_wait_limit(0)
    api.check_status()                      # reported once, then cleared
    out, lse = api.fwd(q, k, v, P, "zigzag", True)
    dq, dk, dv = api.bwd(q, k, v, out, lse, do, P, "zigzag", True)
    od, ld = api.decode(q[:, S - 2:].contiguous(), k, v, P, "zigzag")
    api.check_status()
    q64, k64, v64 = to64(q), to64(k), to64(v)
    ro, rl = oracle.attn_fwd(q64, k64, v64, True, scale)
    assert max_abs(to64(out), ro) <= 2e-2 and max_abs(to64(lse), rl) <= 1e-3
    assert max_abs(to64(od), ro[:, S - 2:]) <= 2e-2 and max_abs(to64(ld), rl[:, :, S - 2:]) <= 1e-3
    rq, rk, rv = oracle.attn_bwd(q64, k64, v64, to64(do), True, scale, [(0, 1)])
    G = H // Hkv
    ours = (np.stack([to64(dq)[0, :, G + e] for e in range(G)]), to64(dk)[0, :, 1],
            to64(dv)[0, :, 1])
    for o, r in zip(ours, (rq[0], rk[0], rv[0])):
        assert max_abs(o, r) <= 5e-2 and rel_l2(o, r) <= 1e-2


def test_wait_limit_rejects_bad_values():
    with pytest.raises(api.RingAttnError):
        api.set_wait_limit(-1)
