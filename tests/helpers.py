"""Shared test helpers: tensor conversion and error metrics (no attention math)."""
import numpy as np
import torch


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isneginf(a) & np.isneginf(b)
    d = np.abs(np.where(both_inf, 0.0, a) - np.where(both_inf, 0.0, b))
    return float(np.max(d)) if d.size else 0.0


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def sample_rows(S: int, P: int, layout: str, count: int, seed: int = 0) -> np.ndarray:
    """Query positions for sampled checks: first/last rows, shard and chunk
    boundaries +-1, 128-tile boundaries, and seeded uniform rows."""
    rows = {0, 1, S - 1, S - 2}
    n = S // P
    step = n if layout != "zigzag" else S // (2 * P)
    for b in range(0, S, step):
        rows.update({b - 1, b, b + 1})
    for b in range(0, S, max(S // 16, 128)):
        rows.update({b + 127, b + 128})
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, S, size=count).tolist())
    rows = sorted(r for r in rows if 0 <= r < S)
    return np.array(rows, dtype=np.int64)
