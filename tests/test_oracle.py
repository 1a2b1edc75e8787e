"""Pins for the CPU oracle, independent of the oracle's own code.

Each check ties the oracle to something it does not compute itself: the
worked example a page prints, hand enumeration of a definition, closed forms,
a library routine on a special case (torch's float64 scaled_dot_product_attention
and autograd), finite differences, or an invariant the pages state.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LAYOUTS = ["contiguous", "striped", "zigzag"]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, causal, scale, mask=None):
    """torch float64 SDPA on natural-order [B,S,H,D] arrays; grouped heads expanded."""
    qt = torch.from_numpy(np.ascontiguousarray(q)).permute(0, 2, 1, 3)
    kt = torch.from_numpy(np.ascontiguousarray(k)).permute(0, 2, 1, 3)
    vt = torch.from_numpy(np.ascontiguousarray(v)).permute(0, 2, 1, 3)
    G = qt.shape[1] // kt.shape[1]
    kt = kt.repeat_interleave(G, dim=1)
    vt = vt.repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask, is_causal=causal and mask is None, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


def _lse_lib(q, k, causal, scale):
    """lse via torch.logsumexp over the materialised score matrix (float64)."""
    qt = torch.from_numpy(np.ascontiguousarray(q)).permute(0, 2, 1, 3)
    kt = torch.from_numpy(np.ascontiguousarray(k)).permute(0, 2, 1, 3)
    G = qt.shape[1] // kt.shape[1]
    kt = kt.repeat_interleave(G, dim=1)
    s = torch.einsum("bhid,bhjd->bhij", qt, kt) * scale
    if causal:
        S = s.shape[-1]
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    return torch.logsumexp(s, dim=-1).numpy()


# ---------------------------------------------------------------- layout maps

def test_striped_matches_page_example():
    with open(os.path.join(GOLDEN, "striped_p4_example.txt")) as f:
        lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    P = int(lines[0][1])
    pos = oracle.layout_positions(64, P, "striped")
    for row in lines[1:]:
        r, first = int(row[0]), [int(x) for x in row[1:]]
        assert list(pos[r, :len(first)]) == first
        stride = first[1] - first[0]
        assert np.all(np.diff(pos[r]) == stride)


def test_zigzag_hand_enumeration():
    # 2P = 4 chunks of 2 tokens: [0 1] [2 3] [4 5] [6 7]; shard 0 holds chunks 0 and 3,
    # shard 1 holds chunks 1 and 2.
    assert oracle.layout_positions(8, 2, "zigzag").tolist() == [[0, 1, 6, 7], [2, 3, 4, 5]]
    # P = 4, S = 16: chunks of 2, shard r holds chunk r and chunk 7 - r.
    assert oracle.layout_positions(16, 4, "zigzag").tolist() == [
        [0, 1, 14, 15], [2, 3, 12, 13], [4, 5, 10, 11], [6, 7, 8, 9]]


def test_contiguous_hand_enumeration():
    assert oracle.layout_positions(8, 2, "contiguous").tolist() == [[0, 1, 2, 3], [4, 5, 6, 7]]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("S,P", [(8, 1), (16, 2), (48, 3), (64, 4), (96, 8), (256, 16)])
def test_layout_is_bijection_and_increasing(layout, S, P):
    pos = oracle.layout_positions(S, P, layout)
    assert sorted(pos.ravel().tolist()) == list(range(S))
    assert np.all(np.diff(pos, axis=1) > 0)
    if P == 1:
        assert pos.ravel().tolist() == list(range(S))


def test_layout_rejects_bad_sizes():
    with pytest.raises(ValueError):
        oracle.layout_positions(10, 4, "striped")
    with pytest.raises(ValueError):
        oracle.layout_positions(12, 4, "zigzag")   # 12 % 8 != 0
    with pytest.raises(ValueError):
        oracle.layout_positions(8, 0, "contiguous")


@pytest.mark.parametrize("layout", LAYOUTS)
def test_permute_roundtrip_and_gather(layout):
    S, P = 32, 4
    src = np.arange(3 * S * 5, dtype=np.int16).reshape(3, S, 5)
    dst = oracle.permute(src, S, P, layout)
    pos = oracle.layout_positions(S, P, layout).ravel()
    assert np.array_equal(dst, src[:, pos])
    assert np.array_equal(oracle.permute(dst, S, P, layout, inverse=True), src)


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Hkv,S,D", [(1, 2, 2, 7, 4), (2, 4, 2, 13, 8), (1, 6, 1, 9, 5)])
def test_fwd_matches_library_sdpa(causal, B, H, Hkv, S, D):
    q, k, v = _rand((B, S, H, D), 1), _rand((B, S, Hkv, D), 2), _rand((B, S, Hkv, D), 3)
    scale = 0.37
    out, lse = oracle.attn_fwd(q, k, v, causal, scale)
    assert np.allclose(out, _sdpa(q, k, v, causal, scale), rtol=0, atol=1e-12)
    assert np.allclose(lse, _lse_lib(q, k, causal, scale), rtol=0, atol=1e-12)


def test_fwd_row_sampling_matches_full():
    q, k, v = _rand((2, 40, 4, 8), 4), _rand((2, 40, 2, 8), 5), _rand((2, 40, 2, 8), 6)
    full_o, full_l = oracle.attn_fwd(q, k, v, True, 0.3)
    rows = np.array([0, 39, 17, 5])
    o, l = oracle.attn_fwd(q, k, v, True, 0.3, rows=rows)
    assert np.array_equal(o, full_o[:, rows])
    assert np.array_equal(l, full_l[:, :, rows])


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    B, S, H, D = 1, 11, 2, 4
    q = np.zeros((B, S, H, D))
    k, v = _rand((B, S, H, D), 7), _rand((B, S, H, D), 8)
    out, lse = oracle.attn_fwd(q, k, v, causal, 0.5)
    for i in range(S):
        last = i + 1 if causal else S
        assert np.allclose(out[0, i], v[0, :last].mean(axis=0), atol=1e-13)
        assert np.allclose(lse[0, :, i], math.log(last), atol=1e-13)


def test_zero_scale_gives_mean_of_visible_values():
    B, S, H, D = 1, 9, 1, 3
    q, k, v = _rand((B, S, H, D), 9), _rand((B, S, H, D), 10), _rand((B, S, H, D), 11)
    out, lse = oracle.attn_fwd(q, k, v, True, 0.0)
    for i in range(S):
        assert np.allclose(out[0, i, 0], v[0, :i + 1, 0].mean(axis=0), atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-13


def test_causal_row_zero_is_first_value():
    B, S, H, Hkv, D = 2, 10, 4, 2, 6
    q, k, v = _rand((B, S, H, D), 12), _rand((B, S, Hkv, D), 13), _rand((B, S, Hkv, D), 14)
    scale = 0.21
    out, lse = oracle.attn_fwd(q, k, v, True, scale)
    for b in range(B):
        for h in range(H):
            g = h // (H // Hkv)
            assert np.array_equal(out[b, 0, h], v[b, 0, g])
            assert abs(lse[b, h, 0] - scale * float(q[b, 0, h] @ k[b, 0, g])) < 1e-13


def test_single_key_returns_value():
    q, k, v = _rand((1, 1, 3, 5), 15), _rand((1, 1, 3, 5), 16), _rand((1, 1, 3, 5), 17)
    for causal in (False, True):
        out, _ = oracle.attn_fwd(q, k, v, causal, 1.0)
        assert np.array_equal(out, v)


def test_grouped_heads_use_floor_mapping():
    # Query heads 0,1 share kv head 0 and heads 2,3 share kv head 1.  Giving the
    # two kv heads very different values makes a wrong mapping visible.
    B, S, H, Hkv, D = 1, 6, 4, 2, 3
    q, k = _rand((B, S, H, D), 18), _rand((B, S, Hkv, D), 19)
    v = np.zeros((B, S, Hkv, D))
    v[:, :, 0] = 1.0
    v[:, :, 1] = -1.0
    out, _ = oracle.attn_fwd(q, k, v, False, 1.0)
    assert np.allclose(out[0, :, :2], 1.0) and np.allclose(out[0, :, 2:], -1.0)


# ---------------------------------------------------------------- blockwise ring == full

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_blockwise_equals_full_attention(layout, P, causal):
    # "Online softmax ... makes the blockwise computation numerically identical to
    # full attention" -- exact in real arithmetic, 1e-12 in fp64.
    S = 48
    B, H, Hkv, D = 1, 4, 2, 8
    q, k, v = _rand((B, S, H, D), 20), _rand((B, S, Hkv, D), 21) * 3, _rand((B, S, Hkv, D), 22)
    full_o, full_l = oracle.attn_fwd(q, k, v, causal, 0.4)
    ring_o, ring_l = oracle.ring_fwd(q, k, v, P, layout, causal, 0.4)
    assert np.max(np.abs(ring_o - full_o)) < 1e-12
    assert np.max(np.abs(ring_l - full_l)) < 1e-12


# ---------------------------------------------------------------- step and merge

def _shard(x, pos_r):
    return np.ascontiguousarray(x[:, pos_r])


@pytest.mark.parametrize("layout", LAYOUTS)
def test_step_matches_masked_library_sdpa(layout):
    S, P, B, H, Hkv, D = 32, 4, 1, 2, 1, 8
    q, k, v = _rand((B, S, H, D), 23), _rand((B, S, Hkv, D), 24), _rand((B, S, Hkv, D), 25)
    pos = oracle.layout_positions(S, P, layout)
    for r in range(P):
        for s in range(P):
            o, l = oracle.step(_shard(q, pos[r]), _shard(k, pos[s]), _shard(v, pos[s]),
                               S, P, layout, r, s, True, 0.5)
            vis = pos[s][None, :] <= pos[r][:, None]          # [n_q, n_k]
            rows = vis.any(axis=1)
            if rows.any():
                ref = _sdpa(_shard(q, pos[r][rows]), _shard(k, pos[s]), _shard(v, pos[s]),
                            False, 0.5, mask=torch.from_numpy(vis[rows]))
                assert np.allclose(o[:, rows], ref, atol=1e-12)
            assert np.all(o[:, ~rows] == 0.0)
            assert np.all(np.isneginf(l[:, :, ~rows]))
            assert np.all(np.isfinite(l[:, :, rows]))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_ring_of_steps_and_merges_equals_full(layout, causal):
    S, P, B, H, Hkv, D = 48, 4, 2, 2, 2, 8
    q, k, v = _rand((B, S, H, D), 26), _rand((B, S, Hkv, D), 27), _rand((B, S, Hkv, D), 28)
    full_o, full_l = oracle.attn_fwd(q, k, v, causal, 0.3)
    pos = oracle.layout_positions(S, P, layout)
    for r in range(P):
        acc_o = acc_l = None
        for t in range(P):
            s = (r - t) % P
            o, l = oracle.step(_shard(q, pos[r]), _shard(k, pos[s]), _shard(v, pos[s]),
                               S, P, layout, r, s, causal, 0.3)
            if acc_o is None:
                acc_o, acc_l = o, l
            else:
                acc_o, acc_l = oracle.merge(acc_o, acc_l, o, l)
        assert np.max(np.abs(acc_o - full_o[:, pos[r]])) < 1e-12
        assert np.max(np.abs(acc_l - full_l[:, :, pos[r]])) < 1e-12


def test_merge_identity_commutativity_and_union():
    B, n, H, D = 1, 5, 2, 4
    q, k, v = _rand((B, n, H, D), 29), _rand((B, 12, H, D), 30), _rand((B, 12, H, D), 31)
    # two disjoint key sets; partials by the library, merged by the oracle
    def part(ks):
        o = _sdpa(q, k[:, ks], v[:, ks], False, 0.7)
        l = _lse_lib(q, k[:, ks], False, 0.7)
        return o, l
    o1, l1 = part(slice(0, 7))
    o2, l2 = part(slice(7, 12))
    mo, ml = oracle.merge(o1, l1, o2, l2)
    assert np.allclose(mo, _sdpa(q, k, v, False, 0.7), atol=1e-13)
    assert np.allclose(ml, _lse_lib(q, k, False, 0.7), atol=1e-13)
    mo2, ml2 = oracle.merge(o2, l2, o1, l1)
    assert np.allclose(mo, mo2, atol=1e-15) and np.allclose(ml, ml2, atol=1e-15)
    empty_o, empty_l = np.zeros_like(o1), np.full_like(l1, -np.inf)
    io, il = oracle.merge(o1, l1, empty_o, empty_l)
    assert np.array_equal(io, o1) and np.array_equal(il, l1)
    io, il = oracle.merge(empty_o, empty_l, o1, l1)
    assert np.array_equal(io, o1) and np.array_equal(il, l1)
    zo, zl = oracle.merge(empty_o, empty_l, empty_o, empty_l)
    assert np.all(zo == 0) and np.all(np.isneginf(zl))


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Hkv,S,D", [(1, 2, 2, 9, 4), (2, 4, 2, 7, 3)])
def test_bwd_matches_autograd(causal, B, H, Hkv, S, D):
    q, k, v = _rand((B, S, H, D), 32), _rand((B, S, Hkv, D), 33), _rand((B, S, Hkv, D), 34)
    do = _rand((B, S, H, D), 35)
    scale = 0.45
    qt, kt, vt = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    G = H // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.permute(0, 2, 1, 3), kt.permute(0, 2, 1, 3).repeat_interleave(G, 1),
        vt.permute(0, 2, 1, 3).repeat_interleave(G, 1), is_causal=causal, scale=scale)
    (o * torch.from_numpy(do).permute(0, 2, 1, 3)).sum().backward()
    pairs = [(b, g) for b in range(B) for g in range(Hkv)]
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, scale, pairs)
    for t, (b, g) in enumerate(pairs):
        for e in range(G):
            assert np.allclose(dq[t, e], qt.grad[b, :, g * G + e].numpy(), atol=1e-12)
        assert np.allclose(dk[t], kt.grad[b, :, g].numpy(), atol=1e-12)
        assert np.allclose(dv[t], vt.grad[b, :, g].numpy(), atol=1e-12)


def test_bwd_matches_finite_differences():
    B, S, H, Hkv, D = 1, 6, 2, 1, 3
    q, k, v = _rand((B, S, H, D), 36), _rand((B, S, Hkv, D), 37), _rand((B, S, Hkv, D), 38)
    do = _rand((B, S, H, D), 39)
    scale = 0.8
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, True, scale, [(0, 0)])

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd(q_, k_, v_, True, scale)
        return float(np.sum(o * do))

    eps = 1e-6
    rng = np.random.default_rng(40)
    for _ in range(12):
        which = rng.integers(3)
        x = [q, k, v][which]
        idx = tuple(rng.integers(s) for s in x.shape)
        xp, xm = x.copy(), x.copy()
        xp[idx] += eps
        xm[idx] -= eps
        args_p = [q, k, v]
        args_m = [q, k, v]
        args_p[which], args_m[which] = xp, xm
        fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        if which == 0:
            an = dq[0, idx[2], idx[1], idx[3]]
        elif which == 1:
            an = dk[0, idx[1], idx[3]]
        else:
            an = dv[0, idx[1], idx[3]]
        assert abs(fd - an) < 1e-7, (which, idx, fd, an)


# ---------------------------------------------------------------- work census

@pytest.mark.parametrize("P", [2, 4, 8])
def test_census_pairs_closed_forms(P):
    S = 32 * P
    n, C = S // P, S // (2 * P)
    pc, _ = oracle.work_census(S, P, "contiguous", True, tile=16)
    pz, _ = oracle.work_census(S, P, "zigzag", True, tile=16)
    ps, _ = oracle.work_census(S, P, "striped", True, tile=16)
    for r in range(P):
        assert pc[r] == n * (r * n) + n * (n + 1) // 2
        assert pz[r] == C * C * (2 * P - 1) + C * (C + 1)
        assert ps[r] == n * (r + 1) + P * n * (n - 1) // 2
    assert pc.sum() == pz.sum() == ps.sum() == S * (S + 1) // 2


def test_census_tiles_balance():
    S, P, tile = 512, 4, 16
    nt = S // P // tile
    _, tz = oracle.work_census(S, P, "zigzag", True, tile=tile)
    _, ts = oracle.work_census(S, P, "striped", True, tile=tile)
    _, tc = oracle.work_census(S, P, "contiguous", True, tile=tile)
    assert len(set(tz.tolist())) == 1
    assert np.all(ts == P * nt * (nt + 1) // 2)
    # contiguous: shard r sees r full shards plus its own triangle
    assert tc.tolist() == [r * nt * nt + nt * (nt + 1) // 2 for r in range(P)]
    pairs, tiles = oracle.work_census(S, P, "contiguous", False, tile=tile)
    assert np.all(pairs == (S // P) * S) and np.all(tiles == P * nt * nt)


def test_census_run_cut_tiles():
    # tiles that may not straddle a run of `run` slots
    S, P = 96, 4
    C = S // (2 * P)                                   # 12
    for layout in ("contiguous", "striped", "zigzag"):
        # tile = 1: every visible pair is its own block
        p1, t1 = oracle.work_census(S, P, layout, True, tile=1, run=C)
        assert np.array_equal(p1, t1)
        # runs that the tiles never reach across change nothing
        a = oracle.work_census(S, P, layout, True, tile=4, run=0)
        b = oracle.work_census(S, P, layout, True, tile=4, run=C)
        c = oracle.work_census(S, P, layout, True, tile=4, run=S // P)
        assert np.array_equal(a[1], b[1]) and np.array_equal(a[1], c[1])
        assert np.array_equal(a[0], b[0])
    # zig-zag with one tile per chunk: query chunk a sees key chunks 0..a, and
    # shard r holds chunks r and 2P-1-r, so (r+1) + (2P-r) = 2P+1 blocks
    _, tz = oracle.work_census(S, P, "zigzag", True, tile=C, run=C)
    assert np.all(tz == 2 * P + 1)
    # a ragged cut: chunks of 12 slots in tiles of 8 -> 2 tiles per chunk
    # (8 + 4), 4 per shard; without the cut the shard's 24 slots make 3 tiles
    _, tr = oracle.work_census(S, P, "zigzag", False, tile=8, run=C)
    _, tn = oracle.work_census(S, P, "zigzag", False, tile=8, run=0)
    assert np.all(tr == P * 4 * 4) and np.all(tn == P * 3 * 3)
