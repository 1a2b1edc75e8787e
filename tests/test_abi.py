"""CPU checks of the C ABI: the library loads, exports what the header
declares, its host-side functions agree with the oracle, and argument errors
come back as status codes before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from ring_attention_02_b300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ring_attn.h")
LAYOUTS = ["contiguous", "striped", "zigzag"]


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:ra_status|const char\*)\s+(ring_attn_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ring_attn_fwd", "ring_attn_bwd", "ring_attn_step", "ring_attn_merge",
                     "ring_attn_permute", "ring_attn_index_map", "ring_attn_check_status",
                     "ring_attn_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol():
    L = api.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert api.version().startswith("ring_attn")


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("S,P", [(256, 4), (8192, 8), (131072, 16), (64, 1), (96, 3)])
def test_index_map_bit_exact_vs_oracle(layout, S, P):
    if layout == "zigzag" and S % (2 * P):
        pytest.skip("zig-zag needs S % 2P == 0")
    ours = api.index_map(S, P, layout).numpy()
    ref = oracle.layout_positions(S, P, layout)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S,P", [(1024, 4), (768, 4), (512, 8), (2048, 2), (96, 3), (4096, 8),
                                 (3072, 8)])
def test_census_matches_brute_force(layout, causal, S, P):
    if layout == "zigzag" and S % (2 * P):
        pytest.skip("zig-zag needs S % 2P == 0")
    pairs, tiles = api.census(S, P, layout, causal)
    # the library's tiles never straddle a zig-zag chunk: the brute force cuts
    # its tiles at the chunk boundaries too (run = C)
    run = S // (2 * P) if layout == "zigzag" else 0
    bp, bt = oracle.work_census(S, P, layout, causal, tile=128, run=run)
    assert np.array_equal(pairs.numpy(), bp)
    assert np.array_equal(tiles.numpy(), bt)


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_census_matches_brute_force_at_the_headline_size(layout):
    # the sizes bench.py reports its shard imbalance at: S = 131072, P = 16
    S, P = 131072, 16
    pairs, tiles = api.census(S, P, layout, True)
    run = S // (2 * P) if layout == "zigzag" else 0
    bp, bt = oracle.work_census(S, P, layout, True, tile=128, run=run)
    assert np.array_equal(pairs.numpy(), bp)
    assert np.array_equal(tiles.numpy(), bt)


def test_census_balance_closed_forms_at_full_sizes():
    # zig-zag: every shard identical; contiguous at P=32: imbalance (P-1)/P.
    S, P = 1048576, 32
    pz, tz = api.census(S, P, "zigzag", True)
    assert len(set(pz.tolist())) == 1 and len(set(tz.tolist())) == 1
    pc, tc = api.census(S, P, "contiguous", True)
    n = S // P
    assert pc.tolist() == [n * (r * n) + n * (n + 1) // 2 for r in range(P)]
    imb = tc.max().item() / tc.float().mean().item() - 1
    assert abs(imb - (P - 1) / P) < 0.01
    ps, ts = api.census(131072, 16, "striped", True)
    assert len(set(ts.tolist())) == 1
    assert (ps.max() - ps.min()).item() == (16 - 1) * (131072 // 16)


def _status(fn, *args):
    rc = fn(*args)
    return rc, api.lib().ring_attn_last_error().decode()


def test_argument_errors_return_codes_without_gpu():
    L = api.lib()
    vp = ctypes.c_void_p
    buf = vp(0x1000)  # never dereferenced: every case below fails validation first
    cases = [
        ((None, buf, buf, buf, 0, None, 1, 2, 2, 256, 64, 4, 0, 0, 0.1, None), 1),   # null q
        ((buf, buf, buf, buf, 0, None, 1, 3, 2, 256, 64, 4, 0, 0, 0.1, None), 2),    # H % Hkv
        ((buf, buf, buf, buf, 0, None, 1, 2, 2, 256, 96, 4, 0, 0, 0.1, None), 4),    # D
        ((buf, buf, buf, buf, 0, None, 1, 2, 2, 250, 64, 4, 0, 0, 0.1, None), 3),    # S % P
        ((buf, buf, buf, buf, 0, None, 1, 2, 2, 258, 64, 2, 2, 0, 0.1, None), 3),    # S % 2P
        ((buf, buf, buf, buf, 0, None, 1, 2, 2, 256, 64, 4, 7, 0, 0.1, None), 3),    # layout
        ((buf, buf, buf, buf, 0, None, 1, 2, 2, 256, 64, 4, 0, 0, float("nan"), None), 4),
        ((vp(0x1001), buf, buf, buf, 0, None, 1, 2, 2, 256, 64, 4, 0, 0, 0.1, None), 5),
        ((buf, buf, buf, buf, 0, None, 0, 2, 2, 256, 64, 4, 0, 0, 0.1, None), 2),    # B = 0
    ]
    for args, want in cases:
        rc, msg = _status(L.ring_attn_fwd, *args)
        assert rc == want, (args, rc, msg)
        assert msg
    rc, _ = _status(L.ring_attn_step, buf, buf, buf, buf, buf, 1, 2, 2, 256, 64, 4, 0, 4, 0, 1,
                    0.1, None)
    assert rc == 2   # r outside [0, P)
    rc, _ = _status(L.ring_attn_merge, buf, buf, buf, None, 1, 2, 64, 64, None)
    assert rc == 1
    rc, _ = _status(L.ring_attn_permute, buf, buf, 1, 256, 6, 4, 0, 0, None)
    assert rc == 2   # row_bytes not a multiple of 4
    rc, _ = _status(L.ring_attn_permute, buf, buf, 1, 256, 512, 4, 0, 0, None)
    assert rc == 2   # src and dst overlap
    # decode: (H/Hkv)*T above 4096, and T above S
    rc, _ = _status(L.ring_attn_decode, buf, buf, buf, buf, 0, None, 1, 8, 1, 600, 1024, 64, 4, 0,
                    0.1, None)
    assert rc == 4
    rc, _ = _status(L.ring_attn_decode, buf, buf, buf, buf, 0, None, 1, 2, 2, 300, 256, 64, 4, 0,
                    0.1, None)
    assert rc == 2
    rc, _ = _status(L.ring_attn_index_map, 12, 4, 2, None)
    assert rc == 1
    pos = (ctypes.c_int64 * 12)()
    rc, _ = _status(L.ring_attn_index_map, 12, 4, 2, pos)
    assert rc == 3   # 12 % 8 != 0


def test_missing_library_is_an_error(monkeypatch):
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "LIB_PATH", "/nonexistent/libringattn.so")
    with pytest.raises(RuntimeError):
        api.lib()
