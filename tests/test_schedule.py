"""CPU checks of the persistent kernels' work schedules (ring_attn_work_schedule).

Every work item must be dealt to exactly one CTA, and each CTA must take its
items in list order (the order that keeps the tiles running CTAs share in L2).
The balance is checked with a cost written here from the shard positions the
oracle gives: the key tiles a query tile multiplies are those whose first
position is at or before its last one (causal), the query tiles a key tile
meets are those whose last position is at or after its first, plus a fixed
cost per item.  The item numbering restated here is the kernels' documented
order: the forward's items are grouped by (b, kv head), longest unit first,
the G heads of a kv head side by side; the backward's item i is unit i mod U
of (b, kv head) or (b, head) number i div U.
"""
import numpy as np
import pytest

import oracle
from ring_attention_02_b300 import api

TILE = 128
ITEM_COST = 2.0
L2 = 126 * 1024 * 1024


def _tiles(S, P, layout):
    """[(shard, seg, tile, first position, last position)] in the kernels' tiling:
    128-slot tiles of one run of consecutive slots (a zig-zag chunk, else the shard)."""
    pos = oracle.layout_positions(S, P, layout)
    n = S // P
    seglen = n // 2 if layout == "zigzag" else n
    out = []
    for r in range(P):
        for seg in range(n // seglen):
            for t in range((seglen + TILE - 1) // TILE):
                sl = pos[r, seg * seglen + t * TILE: seg * seglen + min((t + 1) * TILE, seglen)]
                out.append((r, seg, t, int(sl.min()), int(sl.max())))
    return out, seglen


def _unit_order(S, P, layout, pair):
    """The units of one (b, head) in the kernels' order: longest first for the
    query side (decreasing position), increasing position for key tiles."""
    tiles, seglen = _tiles(S, P, layout)
    nt = (seglen + TILE - 1) // TILE
    nseg = S // P // seglen
    key = {(r, s, t): (lo, hi) for r, s, t, lo, hi in tiles}
    step = 2 if pair else 1
    units = []
    if layout == "zigzag":
        chunks = [(c, 0) if c < P else (2 * P - 1 - c, 1) for c in range(2 * P)]
    elif layout == "striped":
        chunks = None
    else:
        chunks = [(r, 0) for r in range(P)]
    if chunks is not None:
        for r, s in chunks:
            for t in range(0, nt, step):
                units.append((r, s, t))
    else:
        for t in range(0, nt, step):
            for r in range(P):
                units.append((r, 0, t))
    return units, key, nseg


def _fwd_costs(B, H, Hkv, S, P, layout, causal, kv_group):
    units, key, _ = _unit_order(S, P, layout, pair=True)
    units = units[::-1]                       # the query side runs longest first
    keys = list(key.values())
    cost = []
    for r, s, t in units:
        last = key.get((r, s, t + 1), key[(r, s, t)])[1]
        cost.append(sum(1 for lo, _ in keys if lo <= last) if causal else len(keys))
    G, BK, U = H // Hkv, B * Hkv, len(units)
    items = []
    for grp in range((BK + kv_group - 1) // kv_group):
        hg = min(kv_group, BK - grp * kv_group)
        for u in range(U):
            items += [cost[u]] * (hg * G)
    return np.array(items, dtype=float)


def _bwd_costs(B, H, Hkv, S, P, layout, causal, dkdv):
    units, key, _ = _unit_order(S, P, layout, pair=False)
    G = H // Hkv
    vals = list(key.values())
    if dkdv:
        cost = [G * (sum(1 for _, hi in vals if hi >= key[u][0]) if causal else len(vals))
                for u in units]
        reps = B * Hkv
    else:
        units = units[::-1]
        cost = [sum(1 for lo, _ in vals if lo <= key[u][1]) if causal else len(vals)
                for u in units]
        reps = B * H
    return np.array(cost * reps, dtype=float)


def _kv_group(B, H, Hkv, S, D, P, layout, sms=148):
    """The forward's (b, kv head) pairs per group: all, unless their keys and
    values overflow 3/4 of L2 and a smaller group still spans 8 grid rounds."""
    BK = B * Hkv
    pair_bytes = S * D * 4
    if pair_bytes * BK <= L2 * 3 // 4:
        return BK
    hg = max(1, (L2 * 3 // 4) // pair_bytes)
    units = len(_unit_order(S, P, layout, pair=True)[0])
    if hg * (H // Hkv) * units < 8 * sms:
        return BK
    return min(hg, BK)


def _loads(lists, cost):
    return np.array([cost[l].sum() + ITEM_COST * len(l) for l in lists])


def _snake_loads(n, cost, G=148):
    load = np.zeros(G)
    k = 0
    while k * G < n:
        for c in range(G):
            i = k * G + ((G - 1 - c) if k & 1 else c)
            if i < n:
                load[c] += cost[i] + ITEM_COST
        k += 1
    return load


CASES = [
    # B, H, Hkv, S, D, P, layout, causal
    (1, 32, 8, 131072, 128, 16, "zigzag", True),     # the 128k GQA forward
    (2, 16, 16, 32768, 128, 8, "zigzag", True),      # the 32k training step
    (1, 16, 16, 16384, 128, 8, "zigzag", True),
    (1, 8, 2, 24576, 64, 6, "striped", True),
    (1, 8, 8, 8192, 128, 4, "contiguous", True),
    (1, 12, 4, 6144, 128, 3, "zigzag", False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[6]}-S{c[3]}-H{c[1]}")
@pytest.mark.parametrize("kind", ["fwd", "dkdv", "dq"])
def test_schedule_deals_every_item_once_in_order_and_balances(kind, case):
    B, H, Hkv, S, D, P, layout, causal = case
    lists = api.work_schedule(kind, B, H, Hkv, S, D, P, layout, causal, sms=148, l2_bytes=L2)
    if kind == "fwd":
        cost = _fwd_costs(B, H, Hkv, S, P, layout, causal, _kv_group(B, H, Hkv, S, D, P, layout))
    else:
        cost = _bwd_costs(B, H, Hkv, S, P, layout, causal, kind == "dkdv")
    n = len(cost)
    assert lists is not None and len(lists) == 148
    flat = np.concatenate([np.array(l, dtype=np.int64) for l in lists])
    assert np.array_equal(np.sort(flat), np.arange(n))          # each item exactly once
    assert all(np.all(np.diff(l) > 0) for l in lists if len(l) > 1)   # in list order
    loads = _loads([np.array(l, dtype=np.int64) for l in lists], cost)
    snake = _snake_loads(n, cost)
    eff, eff_snake = loads.mean() / loads.max(), snake.mean() / snake.max()
    print(f"{kind} {case}: balance {eff:.3f} (snake {eff_snake:.3f}), {n} items")
    assert eff >= eff_snake - 1e-9
    # list scheduling's bound: the last item placed lands on the least-loaded
    # CTA, so the maximum exceeds the mean by at most one item's cost
    assert loads.max() <= loads.mean() + cost.max() + ITEM_COST + 1e-6


def test_short_lists_run_unscheduled():
    # 2 heads x 8 tile pairs: no more items than SMs
    assert api.work_schedule("fwd", 1, 2, 2, 4096, 128, 4, "zigzag", True) is None
    assert api.work_schedule("dq", 1, 1, 1, 1024, 64, 2, "striped", True, sms=148) is None


def test_schedule_argument_errors():
    with pytest.raises(api.RingAttnError):
        api.work_schedule("fwd", 1, 3, 2, 4096, 128, 4, "zigzag", True)   # H % Hkv
    with pytest.raises(api.RingAttnError):
        api.work_schedule("fwd", 1, 2, 2, 4100, 128, 4, "zigzag", True)   # S % 2P
    with pytest.raises(api.RingAttnError):
        api.work_schedule("dq", 1, 2, 2, 4096, 128, 4, "zigzag", True, sms=0)
