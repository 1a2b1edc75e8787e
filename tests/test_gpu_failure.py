"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies gives up, the device status word records it, ring_attn_check_status
reports RA_ERR_DEVICE_TIMEOUT once, and the context keeps working."""
import numpy as np
import pytest

import oracle
from ring_attention_02_b300 import api
from ring_attention_02_b300.inputs import make_qkv

from helpers import max_abs, to64

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
