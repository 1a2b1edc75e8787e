"""GPU parity of ring_attn_decode: T new query tokens against a key/value
cache that the P ring ranks hold by layout.  The oracle is the plain
definition at the query positions S-T .. S-1 (causal over the cache);
tolerances as for the forward: out max-abs 2e-2, lse max-abs 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from ring_attention_02_b300 import api
from ring_attention_02_b300.inputs import make_qkv

from helpers import max_abs, to64

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3
LAYOUTS = ["contiguous", "striped", "zigzag"]


def _case(B, H, Hkv, S, D, P, layout, T, seed, out_dtype=torch.bfloat16, scale=None):
    scale = D ** -0.5 if scale is None else scale
    q_all, k, v = make_qkv(B, H, Hkv, S, D, seed=seed, device="cuda")
    q = q_all[:, S - T:].contiguous()               # the new tokens' queries
    out, lse = api.decode(q, k, v, P, layout, scale=scale, out_dtype=out_dtype)
    api.check_status()
    rows = np.arange(S - T, S, dtype=np.int64)
    ro, rl = oracle.attn_fwd_rows(to64(q), rows, to64(k), to64(v), True, scale)
    eo, el = max_abs(to64(out), ro), max_abs(to64(lse), rl)
    print(f"PARITY decode B{B} S{S} H{H} Hkv{Hkv} D{D} P{P} {layout} T{T}: "
          f"max|out|={eo:.3e} max|lse|={el:.3e}")
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    return q_all, k, v, out, lse


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("T", [1, 3])
def test_small_all_layouts(layout, D, T):
    # S = 3072, P = 4: shards of 768 slots; zig-zag chunks of 384 (3 tiles each)
    _case(2, 8, 2, 3072, D, 4, layout, T, seed=21)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("S,P,T", [(8, 8, 1), (24, 4, 5), (200, 2, 2), (640, 5, 16), (130, 1, 7)])
def test_ragged_and_tiny(layout, S, P, T):
    if layout == "zigzag" and S % (2 * P):
        pytest.skip("zig-zag needs S % 2P == 0")
    _case(1, 2, 2, S, 128, P, layout, T, seed=22)


def test_fp32_out_and_negative_scale():
    _case(1, 4, 4, 1024, 64, 4, "striped", 2, seed=23, out_dtype=torch.float32, scale=-0.3)


def test_equals_the_fused_forward_rows():
    # the decode of the last T tokens is those rows of the whole-sequence forward
    B, H, Hkv, S, D, P, T = 1, 16, 4, 4096, 128, 8, 4
    q_all, k, v, out, lse = _case(B, H, Hkv, S, D, P, "zigzag", T, seed=24)
    fo, fl = api.fwd(q_all, k, v, P, "zigzag", True, out_dtype=torch.float32)
    assert max_abs(to64(out), to64(fo[:, S - T:])) <= OUT_TOL
    assert max_abs(to64(lse), to64(fl[:, :, S - T:])) <= LSE_TOL


def test_million_token_cache():
    # the million-token shapes: B=1, H=8, Hkv=1, S=2^20, P=32 zig-zag, one new token
    _case(1, 8, 1, 1 << 20, 128, 32, "zigzag", 1, seed=25)


def test_gqa_128k_cache_four_tokens():
    _case(1, 32, 8, 131072, 128, 16, "zigzag", 4, seed=26)


@pytest.mark.parametrize("T", [64, 128])
def test_gqa_128k_cache_chunked_prefill(T):
    # T new tokens at once (G*T = 256 or 512 query rows per kv head: 16 or 32
    # row groups per cache chunk) on the 128k GQA cache
    _case(1, 32, 8, 131072, 128, 16, "zigzag", T, seed=27)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_row_groups_with_a_ragged_last_group(layout):
    # G*T = 4*9 = 36 rows: groups of 16, 16 and 4
    _case(2, 8, 2, 2048, 128, 4, layout, 9, seed=28)


def test_append_then_decode():
    # append T new tokens' keys and values into a cache that holds S-T of them,
    # compare the cache bit for bit with a host-side copy, then decode them
    B, H, Hkv, S, D, P, T = 2, 8, 2, 4096, 128, 8, 16
    q_all, k_all, v_all = make_qkv(B, H, Hkv, S, D, seed=29, device="cuda")
    kc, vc = torch.zeros_like(k_all), torch.zeros_like(v_all)
    kc[:, :S - T] = k_all[:, :S - T]
    vc[:, :S - T] = v_all[:, :S - T]
    k_new, v_new = k_all[:, S - T:].contiguous(), v_all[:, S - T:].contiguous()
    host_k = kc.view(torch.int16).cpu().clone()
    host_k[:, S - T:] = k_new.view(torch.int16).cpu()
    api.cache_append(kc, vc, k_new, v_new, S - T)
    api.check_status()
    assert torch.equal(kc.view(torch.int16).cpu(), host_k)
    assert torch.equal(vc.view(torch.int16), v_all.view(torch.int16))
    q = q_all[:, S - T:].contiguous()
    out, lse = api.decode(q, kc, vc, P, "zigzag")
    api.check_status()
    rows = np.arange(S - T, S, dtype=np.int64)
    ro, rl = oracle.attn_fwd_rows(to64(q), rows, to64(k_all), to64(v_all), True, D ** -0.5)
    assert max_abs(to64(out), ro) <= OUT_TOL and max_abs(to64(lse), rl) <= LSE_TOL
