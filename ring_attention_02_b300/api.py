"""Python binding of libringattn.so (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI of ``include/ring_attn.h``.  torch supplies device
memory and streams.  If the shared library is missing the first call raises:
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libringattn.so")

LAYOUTS = {"contiguous": 0, "striped": 1, "zigzag": 2}
RA_BF16, RA_F32 = 0, 1
STATUS = {0: "RA_OK", 1: "RA_ERR_NULL", 2: "RA_ERR_SHAPE", 3: "RA_ERR_LAYOUT",
          4: "RA_ERR_UNSUPPORTED", 5: "RA_ERR_ALIGN", 6: "RA_ERR_CUDA",
          7: "RA_ERR_DEVICE_TIMEOUT", 8: "RA_ERR_ALLOC"}

_lock = threading.Lock()
_lib = None


class RingAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} not built; run __graft_entry__.build() "
                                   "or python ring_attention_02_b300/build.py")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            L.ring_attn_fwd.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i64, i32, i32,
                                        i32, i32, f32, vp]
            L.ring_attn_fwd_varlen.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                               i32, i32, i32, f32, vp]
            L.ring_attn_fwd_counted.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i64, i32,
                                                i32, i32, i32, f32, vp, vp]
            L.ring_attn_fwd_traced.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i64, i32,
                                               i32, i32, i32, f32, vp, i64, vp, vp]
            L.ring_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i64,
                                        i32, i32, i32, i32, f32, vp]
            L.ring_attn_bwd_noalloc.argtypes = L.ring_attn_bwd.argtypes
            L.ring_attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                               i32, i32, i32, i32, i32, f32, vp]
            L.ring_attn_decode.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64,
                                           i32, i32, i32, f32, vp]
            L.ring_attn_cache_append.argtypes = [vp, vp, vp, vp, i32, i32, i64, i64, i32, i32, vp]
            L.ring_attn_step.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, i32, i32,
                                         i32, i32, i32, f32, vp]
            L.ring_attn_step_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                             i64, i32, i32, i32, i32, i32, i32, f32, i32, vp]
            L.ring_attn_merge.argtypes = [vp, vp, vp, vp, i32, i32, i64, i32, vp]
            L.ring_attn_permute.argtypes = [vp, vp, i64, i64, i64, i32, i32, i32, vp]
            L.ring_attn_permute_shards.argtypes = [vp, vp, i64, i64, i64, i32, i32, i32, vp]
            L.ring_attn_head_split.argtypes = [vp, vp, i64, i32, i64, i32, vp]
            L.ring_attn_finalize.argtypes = [vp, vp, i64, vp]
            L.ring_attn_index_map.argtypes = [i64, i32, i32, vp]
            L.ring_attn_census.argtypes = [i64, i32, i32, i32, vp, vp]
            L.ring_attn_work_schedule.argtypes = [i32, i32, i32, i32, i64, i32, i32, i32, i32,
                                                  i32, i64, vp, i64, vp]
            L.ring_attn_check_status.argtypes = [vp]
            L.ring_attn_wait_selfcheck.argtypes = [i32, vp, vp]
            L.ring_attn_set_wait_limit.argtypes = [i64]
            L.ring_attn_last_error.restype = ctypes.c_char_p
            L.ring_attn_version.restype = ctypes.c_char_p
            for name in ("ring_attn_fwd", "ring_attn_fwd_varlen", "ring_attn_fwd_counted",
                         "ring_attn_fwd_traced",
                         "ring_attn_bwd",
                         "ring_attn_bwd_noalloc", "ring_attn_decode", "ring_attn_bwd_varlen",
                         "ring_attn_step", "ring_attn_step_bwd", "ring_attn_merge",
                         "ring_attn_cache_append",
                         "ring_attn_permute", "ring_attn_permute_shards",
                         "ring_attn_head_split", "ring_attn_finalize",
                         "ring_attn_index_map", "ring_attn_census", "ring_attn_check_status",
                         "ring_attn_wait_selfcheck", "ring_attn_set_wait_limit"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
        return _lib


def _check(status: int):
    if status != 0:
        raise RingAttnError(status, lib().ring_attn_last_error().decode())


def _layout(layout) -> int:
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def fwd(q, k, v, P: int, layout, causal: bool = True, scale: float | None = None,
        out_dtype=torch.bfloat16, out=None, lse=None, want_lse: bool = True, stream=None):
    """Ring attention forward.  q [B,S,H,D], k/v [B,S,Hkv,D] bf16 (natural order).

    Returns (out [B,S,H,D] in out_dtype, lse [B,H,S] fp32 or None).
    """
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, nm)
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, S, H, D), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    odt = RA_F32 if out.dtype == torch.float32 else RA_BF16
    _check(lib().ring_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), odt, _ptr(lse), B, H, Hkv,
                               S, D, P, _layout(layout), int(bool(causal)), float(scale),
                               _stream(stream)))
    return out, lse


def fwd_varlen(q, k, v, cu_seqlens, P: int, layout, causal: bool = True,
               scale: float | None = None, out_dtype=torch.bfloat16, out=None, lse=None,
               want_lse: bool = True, stream=None):
    """Forward over packed sequences.  q [total,H,D], k/v [total,Hkv,D] bf16;
    cu_seqlens: host int64 offsets (list or CPU tensor) of nseq+1 entries.

    Returns (out [total,H,D], lse [H,total] fp32 or None).
    """
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, nm)
    total, H, D = q.shape
    Hkv = k.shape[1]
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int64).contiguous().cpu()
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((total, H, D), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    odt = RA_F32 if out.dtype == torch.float32 else RA_BF16
    _check(lib().ring_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), odt, _ptr(lse),
                                      ctypes.c_void_p(cu.data_ptr()), len(cu) - 1, H, Hkv, D, P,
                                      _layout(layout), int(bool(causal)), float(scale),
                                      _stream(stream)))
    return out, lse


def fwd_counted(q, k, v, P: int, layout, causal: bool = True, scale: float | None = None,
                out_dtype=torch.bfloat16, stream=None):
    """fwd plus the per-shard count of multiplied (query tile, key tile) blocks,
    summed over batch and heads."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = D ** -0.5
    out = torch.empty((B, S, H, D), dtype=out_dtype, device=q.device)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    tiles = torch.zeros(P, dtype=torch.int64, device=q.device)
    odt = RA_F32 if out_dtype == torch.float32 else RA_BF16
    _check(lib().ring_attn_fwd_counted(_ptr(q), _ptr(k), _ptr(v), _ptr(out), odt, _ptr(lse), B,
                                       H, Hkv, S, D, P, _layout(layout), int(bool(causal)),
                                       float(scale), _ptr(tiles), _stream(stream)))
    return out, lse, tiles


def fwd_traced(q, k, v, P: int, layout, causal: bool = True, scale: float | None = None,
               out_dtype=torch.bfloat16, stream=None):
    """fwd plus the per-work-item timeline: (out, lse, records) with records a
    CPU int64 tensor [items, 4] of (start ns, end ns, shard << 32 | CTA, key
    tiles multiplied)."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = D ** -0.5
    out = torch.empty((B, S, H, D), dtype=out_dtype, device=q.device)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    n = ctypes.c_int64(0)
    L = lib()
    # the number of items first (a call with no room fails before any launch)
    L.ring_attn_fwd_traced(_ptr(q), _ptr(k), _ptr(v), _ptr(out), 0, _ptr(lse), B, H, Hkv, S, D,
                           P, _layout(layout), int(bool(causal)), float(scale),
                           ctypes.c_void_p(8), 0, ctypes.byref(n), _stream(stream))
    rec = torch.empty((max(n.value, 1), 4), dtype=torch.int64, device=q.device)
    odt = RA_F32 if out_dtype == torch.float32 else RA_BF16
    _check(L.ring_attn_fwd_traced(_ptr(q), _ptr(k), _ptr(v), _ptr(out), odt, _ptr(lse), B, H,
                                  Hkv, S, D, P, _layout(layout), int(bool(causal)), float(scale),
                                  _ptr(rec), n.value, ctypes.byref(n), _stream(stream)))
    return out, lse, rec[:n.value].cpu()


def bwd(q, k, v, out, lse, dout, P: int, layout, causal: bool = True,
        scale: float | None = None, dq=None, dk=None, dv=None, stream=None):
    """Gradients (dq, dk, dv), bf16, natural order (written into dq, dk, dv
    when given)."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = D ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().ring_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, S, D, P,
                               _layout(layout), int(bool(causal)), float(scale),
                               _stream(stream)))
    return dq, dk, dv


def bwd_varlen(q, k, v, out, lse, dout, cu_seqlens, P: int, layout, causal: bool = True,
               scale: float | None = None, stream=None):
    """Gradients of fwd_varlen: (dq [total,H,D], dk, dv [total,Hkv,D]) bf16."""
    total, H, D = q.shape
    Hkv = k.shape[1]
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int64).contiguous().cpu()
    if scale is None:
        scale = D ** -0.5
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    _check(lib().ring_attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                      _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                      ctypes.c_void_p(cu.data_ptr()), len(cu) - 1, H, Hkv, D, P,
                                      _layout(layout), int(bool(causal)), float(scale),
                                      _stream(stream)))
    return dq, dk, dv


def bwd_noalloc(q, k, v, out, lse, dout, P: int, layout, causal: bool = True,
                scale: float | None = None, dq=None, dk=None, dv=None, stream=None):
    """bwd through ring_attn_bwd_noalloc: the library's scratch is its fixed
    device array, so the call itself allocates nothing.  Pass dq, dk and dv to
    keep this wrapper from allocating the outputs as well."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = D ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().ring_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                       _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, S,
                                       D, P, _layout(layout), int(bool(causal)), float(scale),
                                       _stream(stream)))
    return dq, dk, dv


def decode(q, k_cache, v_cache, P: int, layout, scale: float | None = None,
           out_dtype=torch.bfloat16, out=None, lse=None, want_lse: bool = True, stream=None):
    """Decode step: q [B,T,H,D] (positions S-T..S-1) against caches [B,S,Hkv,D].

    Returns (out [B,T,H,D] in out_dtype, lse [B,H,T] fp32 or None).
    """
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, nm)
    B, T, H, D = q.shape
    S, Hkv = k_cache.shape[1], k_cache.shape[2]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, T, H, D), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    odt = RA_F32 if out.dtype == torch.float32 else RA_BF16
    _check(lib().ring_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), odt,
                                  _ptr(lse), B, H, Hkv, T, S, D, P, _layout(layout),
                                  float(scale), _stream(stream)))
    return out, lse


def cache_append(k_cache, v_cache, k_new, v_new, pos: int, stream=None):
    """Writes k_new, v_new [B,T,Hkv,D] into the caches [B,S_cap,Hkv,D] at
    positions pos .. pos+T-1 (in place)."""
    for t, nm in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, nm)
    B, S_cap, Hkv, D = k_cache.shape
    T = k_new.shape[1]
    _check(lib().ring_attn_cache_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                        B, Hkv, S_cap, int(pos), T, D, _stream(stream)))
    return k_cache, v_cache


def step(q_shard, k_shard, v_shard, S: int, P: int, layout, r: int, s: int,
         causal: bool = True, scale: float | None = None, out=None, lse=None, stream=None):
    """One ring hop in shard-local order: (out_part fp32 [B,n,H,D], lse_part [B,H,n]),
    written into `out` and `lse` when given."""
    B, n, H, D = q_shard.shape
    Hkv = k_shard.shape[2]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, n, H, D), dtype=torch.float32, device=q_shard.device)
    if lse is None:
        lse = torch.empty((B, H, n), dtype=torch.float32, device=q_shard.device)
    _check(lib().ring_attn_step(_ptr(q_shard), _ptr(k_shard), _ptr(v_shard), _ptr(out),
                                _ptr(lse), B, H, Hkv, S, D, P, _layout(layout), r, s,
                                int(bool(causal)), float(scale), _stream(stream)))
    return out, lse


def step_bwd(q_shard, k_shard, v_shard, out_shard, lse_shard, dout_shard, S: int, P: int,
             layout, r: int, s: int, causal: bool = True, scale: float | None = None,
             dq=None, dk=None, dv=None, accumulate: bool = False, stream=None):
    """One hop of the backward in shard-local order: fp32 (dq_part [B,n,H,D],
    dk_part, dv_part [B,n,Hkv,D]) of shard r's queries against block s, written
    into (or, accumulate=True, added to) dq, dk, dv when given."""
    B, n, H, D = q_shard.shape
    Hkv = k_shard.shape[2]
    if scale is None:
        scale = D ** -0.5
    dev = q_shard.device
    if dq is None:
        dq = torch.empty((B, n, H, D), dtype=torch.float32, device=dev)
    if dk is None:
        dk = torch.empty((B, n, Hkv, D), dtype=torch.float32, device=dev)
    if dv is None:
        dv = torch.empty((B, n, Hkv, D), dtype=torch.float32, device=dev)
    _check(lib().ring_attn_step_bwd(_ptr(q_shard), _ptr(k_shard), _ptr(v_shard), _ptr(out_shard),
                                    _ptr(lse_shard), _ptr(dout_shard), _ptr(dq), _ptr(dk),
                                    _ptr(dv), B, H, Hkv, S, D, P, _layout(layout), r, s,
                                    int(bool(causal)), float(scale), int(bool(accumulate)),
                                    _stream(stream)))
    return dq, dk, dv


def merge(out_acc, lse_acc, out_part, lse_part, stream=None):
    """In-place LSE fold of (out_part, lse_part) into (out_acc, lse_acc)."""
    B, n, H, D = out_acc.shape
    _check(lib().ring_attn_merge(_ptr(out_acc), _ptr(lse_acc), _ptr(out_part), _ptr(lse_part),
                                 B, H, n, D, _stream(stream)))
    return out_acc, lse_acc


def permute(src, S: int, P: int, layout, inverse: bool = False, out=None, stream=None):
    """Rows of src [outer, S, ...] to shard-major order (or back, inverse=True)."""
    outer = src.shape[0]
    row_bytes = src.numel() * src.element_size() // (outer * S)
    dst = torch.empty_like(src) if out is None else out
    _check(lib().ring_attn_permute(_ptr(src), _ptr(dst), outer, S, row_bytes, P,
                                   _layout(layout), int(bool(inverse)), _stream(stream)))
    return dst


def permute_shards(src, S: int, P: int, layout, inverse: bool = False, out=None, stream=None):
    """Natural order [outer, S, ...] <-> shard-outer blocks [P, outer, S//P, ...]
    (inverse=True scatters the blocks back).  Returns the destination; its
    shape is src's (the caller views it as it needs)."""
    outer = src.shape[1] if inverse else src.shape[0]
    row_bytes = src.numel() * src.element_size() // (outer * S)
    dst = torch.empty_like(src) if out is None else out
    _check(lib().ring_attn_permute_shards(_ptr(src), _ptr(dst), outer, S, row_bytes, P,
                                          _layout(layout), int(bool(inverse)), _stream(stream)))
    return dst


def head_split(src, rows: int, parts: int, inverse: bool = False, out=None, stream=None):
    """[rows, parts, chunk] <-> [parts, rows, chunk] (bytes of src split evenly)."""
    chunk_bytes = src.numel() * src.element_size() // (rows * parts)
    dst = torch.empty_like(src) if out is None else out
    _check(lib().ring_attn_head_split(_ptr(src), _ptr(dst), rows, parts, chunk_bytes,
                                      int(bool(inverse)), _stream(stream)))
    return dst


def finalize(acc, out=None, stream=None):
    """bf16 copy of an fp32 accumulator (same shape)."""
    out = torch.empty(acc.shape, dtype=torch.bfloat16, device=acc.device) if out is None else out
    _check(lib().ring_attn_finalize(_ptr(acc), _ptr(out), acc.numel(), _stream(stream)))
    return out


def index_map(S: int, P: int, layout):
    """Host-side map, torch int64 [P, S//P] of global positions."""
    pos = torch.empty(S, dtype=torch.int64)
    _check(lib().ring_attn_index_map(S, P, _layout(layout), ctypes.c_void_p(pos.data_ptr())))
    return pos.view(P, S // P)


def census(S: int, P: int, layout, causal: bool = True):
    """Host-side per-shard (visible pairs, computed 128x128 tiles) for one (b, h)."""
    pairs = torch.empty(P, dtype=torch.int64)
    tiles = torch.empty(P, dtype=torch.int64)
    _check(lib().ring_attn_census(S, P, _layout(layout), int(bool(causal)),
                                  ctypes.c_void_p(pairs.data_ptr()),
                                  ctypes.c_void_p(tiles.data_ptr())))
    return pairs, tiles


SCHEDULE_KINDS = {"fwd": 0, "dkdv": 1, "dq": 2}


def work_schedule(kind: str, B: int, H: int, Hkv: int, S: int, D: int, P: int, layout,
                  causal: bool = True, sms: int = 148, l2_bytes: int = 126 * 1024 * 1024):
    """Host-side: the per-CTA work-item lists the persistent forward ("fwd")
    or backward pass ("dkdv", "dq") of a ring-mode call of this shape runs by,
    as a list of G int lists (None when the call runs unscheduled)."""
    n = ctypes.c_int64(0)
    args = (SCHEDULE_KINDS[kind], B, H, Hkv, S, D, P, _layout(layout), int(bool(causal)), sms,
            l2_bytes)
    _check(lib().ring_attn_work_schedule(*args, None, 0, ctypes.byref(n)))
    if n.value == 0:
        return None
    buf = (ctypes.c_int * n.value)()
    _check(lib().ring_attn_work_schedule(*args, buf, n.value, ctypes.byref(n)))
    flat = list(buf)
    off, items = flat[:sms + 1], flat[sms + 1:]   # scheduled calls have more items than SMs
    return [items[off[c]:off[c + 1]] for c in range(sms)]


def check_status(stream=None):
    """Synchronises the stream and raises if a kernel reported a timeout."""
    _check(lib().ring_attn_check_status(_stream(stream)))


def wait_selfcheck(limit_ms: int = 50, stream=None) -> int:
    """Runs one bounded wait that is never satisfied (limit_ms milliseconds);
    returns the nanoseconds it waited.  check_status() then raises
    RingAttnError(RA_ERR_DEVICE_TIMEOUT) once."""
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check(lib().ring_attn_wait_selfcheck(int(limit_ms), _ptr(waited), _stream(stream)))
    return int(waited.item())


def set_wait_limit(limit_ns: int = 0):
    """Sets the kernels' bounded-wait limit on the current device (0: the
    default of about two seconds)."""
    _check(lib().ring_attn_set_wait_limit(int(limit_ns)))


def version() -> str:
    return lib().ring_attn_version().decode()
