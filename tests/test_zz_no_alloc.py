"""ring_attn_bwd_noalloc: the backward for callers that cannot allocate GPU
memory while they run (a framework that has reserved the whole device for its
own caching allocator, or a program that forbids allocation after start-up).
Its scratch is the library's fixed device array instead of a cudaMallocAsync
workspace; its results must match ring_attn_bwd.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

from ring_attention_02_b300 import api
from ring_attention_02_b300.inputs import make_dout, make_qkv

from helpers import max_abs, rel_l2, to64

# the tolerance the backward parity tests use, per gradient tensor
ABS_TOL = 5e-2
REL_TOL = 1e-2


def _inputs(B, H, Hkv, S, D, P, layout, seed):
    q, k, v = make_qkv(B, H, Hkv, S, D, seed=seed, device="cuda")
    do = make_dout(B, H, S, D, seed=seed, device="cuda")
    out, lse = api.fwd(q, k, v, P, layout, True)
    return q, k, v, out, lse, do


@pytest.mark.gpu
def test_noalloc_matches_allocating_backward_two_calls_in_a_row():
    # The second call is smaller than the first, so the fixed array still holds
    # the first call's values beyond the second call's range.
    cases = [(2, 4, 2, 4096, 128, 8, "zigzag", 31), (1, 2, 1, 640, 64, 5, "striped", 32)]
    for B, H, Hkv, S, D, P, layout, seed in cases:
        q, k, v, out, lse, do = _inputs(B, H, Hkv, S, D, P, layout, seed)
        ref = api.bwd(q, k, v, out, lse, do, P, layout, True)
        got = api.bwd_noalloc(q, k, v, out, lse, do, P, layout, True)
        api.check_status()
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            ea, er = max_abs(to64(a), to64(b)), rel_l2(to64(a), to64(b))
            assert ea <= ABS_TOL and er <= REL_TOL, (layout, name, ea, er)


def test_noalloc_rejects_problems_beyond_the_fixed_workspace():
    # B*H*P*T*128 = 1*32*16*64*128 = 4194304 > 2097152: refused on the host
    # before any GPU work (the pointers are never dereferenced).
    L = api.lib()
    buf = ctypes.c_void_p(0x1000)
    rc = L.ring_attn_bwd_noalloc(buf, buf, buf, buf, buf, buf, buf, buf, buf, 1, 32, 8, 131072,
                                 128, 16, 2, 1, 0.088, None)
    assert rc == 2
    assert b"fixed workspace" in L.ring_attn_last_error()
