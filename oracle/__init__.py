"""CPU oracle for blockwise ring attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
library (``ring_attention_02_b300``) never does, and this package never
imports the product library: the two share no code.  The only module both
sides use is ``ring_attention_02_b300.inputs`` (seeded input generators, no
attention arithmetic), and this package does not import even that.

Every routine is plain fp64 with scalar loops, in ``oracle.c``.  This module
only marshals numpy arrays through ctypes.

Sources are web pages on sequence parallelism and ring attention:
  * "Context parallelism and zig-zag ring attention" (Khang Pham, Chinese
    translation), section "Zig Zag Ring Attention": the ring workflow, causal
    masking, the interleaved (striped) shard map and load balance.
  * "Sequenzparallelitaet und Ringaufmerksamkeit", sections "Tiefer Einblick"
    and FAQ: contiguous shards, the K/V ring, online softmax, exactness.
  * "Sequence Parallelism and Ring Attention" (Thai edition), section
    "technical insight": running maximum and normaliser, rescaling.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

CONTIGUOUS, STRIPED, ZIGZAG = 0, 1, 2
LAYOUTS = {"contiguous": CONTIGUOUS, "striped": STRIPED, "zigzag": ZIGZAG}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, -O2, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
                           "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        vp = ctypes.c_void_p
        lib.oracle_layout_positions.argtypes = [i64, i32, i32, vp]
        lib.oracle_attn_fwd_rows.argtypes = [vp, vp, vp, i32, i32, i32, i64, i32, i32, dbl,
                                             vp, i64, vp, vp, i32]
        lib.oracle_ring_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i64, i32, i32, i32, i32,
                                        dbl, vp, vp, i32]
        lib.oracle_step.argtypes = [vp, vp, vp, i32, i32, i32, i64, i32, i32, i32, i32, i32,
                                    i32, dbl, vp, vp, i32]
        lib.oracle_merge.argtypes = [vp, vp, vp, vp, i32, i32, i64, i32]
        lib.oracle_merge.restype = None
        lib.oracle_attn_bwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i64, i32, i32, dbl,
                                        vp, i32, vp, vp, vp, i32]
        lib.oracle_work_census.argtypes = [i64, i32, i32, i32, i32, i64, vp, vp, i32]
        lib.oracle_permute.argtypes = [vp, vp, i64, i64, i64, i32, i32, i32]
        _lib = lib
    return _lib


def _threads(nthreads):
    if nthreads:
        return int(nthreads)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _layout_id(layout):
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def layout_positions(S: int, P: int, layout) -> np.ndarray:
    """[P, S//P] int64: global token position held by (shard r, local slot j)."""
    pos = np.empty(S, dtype=np.int64)
    if _load().oracle_layout_positions(S, P, _layout_id(layout), _ptr(pos)) != 0:
        raise ValueError(f"bad layout arguments S={S} P={P} layout={layout}")
    return pos.reshape(P, S // P)


def attn_fwd(q, k, v, causal: bool, scale: float, rows=None, nthreads=None):
    """Plain attention (fp64).  q [B,S,H,D], k/v [B,S,Hkv,D] (natural order).

    ``rows``: query positions to evaluate (default all).  Returns
    ``out [B,len(rows),H,D]`` and ``lse [B,H,len(rows)]`` as float64.
    """
    q = np.asarray(q)
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    rows = np.arange(S, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    qrows = _f64(q[:, rows])
    k, v = _f64(k), _f64(v)
    nr = len(rows)
    out = np.empty((B, nr, H, D))
    lse = np.empty((B, H, nr))
    rc = _load().oracle_attn_fwd_rows(_ptr(qrows), _ptr(k), _ptr(v), B, H, Hkv, S, D,
                                      int(bool(causal)), float(scale), _ptr(rows), nr,
                                      _ptr(out), _ptr(lse), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_rows: bad arguments")
    return out, lse


def attn_fwd_rows(qrows, rows, k, v, causal: bool, scale: float, nthreads=None):
    """Like attn_fwd for the queries at positions ``rows`` only, given just
    those query rows: qrows [B, len(rows), H, D]; k/v [B, S, Hkv, D]."""
    qrows = _f64(qrows)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    k, v = _f64(k), _f64(v)
    B, nr, H, D = qrows.shape
    S, Hkv = k.shape[1], k.shape[2]
    out = np.empty((B, nr, H, D))
    lse = np.empty((B, H, nr))
    rc = _load().oracle_attn_fwd_rows(_ptr(qrows), _ptr(k), _ptr(v), B, H, Hkv, S, D,
                                      int(bool(causal)), float(scale), _ptr(rows), nr,
                                      _ptr(out), _ptr(lse), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_rows: bad arguments")
    return out, lse


def ring_fwd(q, k, v, P: int, layout, causal: bool, scale: float, nthreads=None):
    """Ring-order blockwise attention with online softmax (fp64, natural order)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    out = np.empty((B, S, H, D))
    lse = np.empty((B, H, S))
    rc = _load().oracle_ring_fwd(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, S, D, P,
                                 _layout_id(layout), int(bool(causal)), float(scale),
                                 _ptr(out), _ptr(lse), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_ring_fwd: bad arguments")
    return out, lse


def step(q_shard, k_shard, v_shard, S: int, P: int, layout, r: int, s: int, causal: bool,
         scale: float, nthreads=None):
    """Partial attention of shard r (queries) against block s (keys), shard-local order."""
    q, k, v = _f64(q_shard), _f64(k_shard), _f64(v_shard)
    B, n, H, D = q.shape
    Hkv = k.shape[2]
    out = np.empty((B, n, H, D))
    lse = np.empty((B, H, n))
    rc = _load().oracle_step(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, S, D, P, _layout_id(layout),
                             r, s, int(bool(causal)), float(scale), _ptr(out), _ptr(lse),
                             _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_step: bad arguments")
    return out, lse


def merge(out_acc, lse_acc, out_part, lse_part):
    """LSE-combine two partials; returns new (out, lse) without touching inputs."""
    oa, la = _f64(out_acc).copy(), _f64(lse_acc).copy()
    op, lp = _f64(out_part), _f64(lse_part)
    B, n, H, D = oa.shape
    _load().oracle_merge(_ptr(oa), _ptr(la), _ptr(op), _ptr(lp), B, H, n, D)
    return oa, la


def attn_bwd(q, k, v, dout, causal: bool, scale: float, bg_pairs, nthreads=None):
    """fp64 gradients for the listed (b, kv-head g) pairs.

    Returns ``dq [T,G,S,D]``, ``dk [T,S,D]``, ``dv [T,S,D]`` with T = len(bg_pairs),
    G = H // Hkv (query head g*G+e at index e).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    G = H // Hkv
    bg = np.ascontiguousarray(np.asarray(bg_pairs, dtype=np.int32).reshape(-1, 2))
    T = bg.shape[0]
    dq = np.empty((T, G, S, D))
    dk = np.empty((T, S, D))
    dv = np.empty((T, S, D))
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, H, Hkv, S, D,
                                 int(bool(causal)), float(scale), _ptr(bg), T, _ptr(dq),
                                 _ptr(dk), _ptr(dv), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_bwd: bad arguments")
    return dq, dk, dv


def work_census(S: int, P: int, layout, causal: bool, tile: int = 128, run: int = 0,
                nthreads=None):
    """Brute-force per-shard (visible pairs, computed tiles); O(S^2).

    Tiles are ``tile`` consecutive local slots of a shard; with ``run`` > 0 no
    tile straddles two runs of ``run`` slots (``run`` = S/(2P) keeps every tile
    inside one zig-zag chunk).
    """
    pairs = np.zeros(P, dtype=np.int64)
    tiles = np.zeros(P, dtype=np.int64)
    rc = _load().oracle_work_census(S, P, _layout_id(layout), int(bool(causal)), tile, int(run),
                                    _ptr(pairs), _ptr(tiles), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_work_census: bad arguments")
    return pairs, tiles


def permute(src: np.ndarray, S: int, P: int, layout, inverse: bool = False) -> np.ndarray:
    """Byte-level row gather (or scatter) by the layout map; src is [outer, S, ...]."""
    src = np.ascontiguousarray(src)
    outer = src.shape[0]
    row_bytes = src.nbytes // (outer * S)
    dst = np.empty_like(src)
    rc = _load().oracle_permute(_ptr(src), _ptr(dst), outer, S, row_bytes, P,
                                _layout_id(layout), int(bool(inverse)))
    if rc != 0:
        raise ValueError("oracle_permute: bad arguments")
    return dst
