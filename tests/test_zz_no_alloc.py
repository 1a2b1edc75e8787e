"""ring_attn_bwd_noalloc: the backward for callers that cannot allocate GPU
memory while they run (a framework that has reserved the whole device for its
own caching allocator, or a program that forbids allocation after start-up).
Its scratch is the library's fixed device array instead of a cudaMallocAsync
workspace; its results must match ring_attn_bwd.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

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
    # The two entry points run the same kernels on the same inputs; only the
    # scratch address differs, so the gradients must agree bit for bit.  The
    # second call is smaller than the first, so the fixed array still holds
    # the first call's values beyond the second call's range: stale scratch
    # that leaked into a result would show up as a bit difference.
    cases = [(2, 4, 2, 4096, 128, 8, "zigzag", 31), (1, 2, 1, 640, 64, 5, "striped", 32)]
    for B, H, Hkv, S, D, P, layout, seed in cases:
        q, k, v, out, lse, do = _inputs(B, H, Hkv, S, D, P, layout, seed)
        ref = api.bwd(q, k, v, out, lse, do, P, layout, True)
        got = api.bwd_noalloc(q, k, v, out, lse, do, P, layout, True)
        api.check_status()
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (layout, name)
    # and the last call's gradients against the fp64 oracle, at the tolerance
    # of the backward parity tests
    G = H // Hkv
    rq, rk, rv = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), True, D ** -0.5, [(0, 0)])
    gq, gk, gv = (to64(t) for t in got)
    ours = (np.stack([gq[0, :, e] for e in range(G)]), gk[0, :, 0], gv[0, :, 0])
    for name, a, r in zip(("dq", "dk", "dv"), ours, (rq[0], rk[0], rv[0])):
        ea, er = max_abs(a, r), rel_l2(a, r)
        assert ea <= ABS_TOL and er <= REL_TOL, (name, ea, er)


def test_noalloc_rejects_problems_beyond_the_fixed_workspace():
    # B*H*P*T*128 = 1*32*16*64*128 = 4194304 > 2097152: refused on the host
    # before any GPU work (the pointers are never dereferenced).
    L = api.lib()
    buf = ctypes.c_void_p(0x1000)
    rc = L.ring_attn_bwd_noalloc(buf, buf, buf, buf, buf, buf, buf, buf, buf, 1, 32, 8, 131072,
                                 128, 16, 2, 1, 0.088, None)
    assert rc == 2
    assert b"fixed workspace" in L.ring_attn_last_error()
