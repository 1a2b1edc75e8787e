// attn_bwd.cuh -- gradients of the ring-attention forward on tcgen05 tensor
// cores (sm_103a).
//
// The pages describe the forward only; the gradients are the textbook ones of
// out = softmax(scale q k^T + causal mask) v, recomputing P from the forward's
// log-sum-exp instead of storing it:
//   P = exp(scale q k^T - lse),  delta_i = sum_d dout_id out_id,
//   dv = P^T dout,  dP = dout v^T,  dS = P * (dP - delta),
//   dq = scale dS k,  dk = scale dS^T q,
// with dk and dv summed over the H/Hkv query heads that share a key/value head.
// The causal mask compares global positions ("Zig Zag Ring Attention"), and the
// key/value blocks meet the query shards in ring order: block s visits shard
// (s + t) mod P at step t ("Tiefer Einblick": blocks hop from rank to rank).
//
// Three kernels:
//   bwd_prep_kernel       delta and -lse*log2(e) per query row, written in
//                         tile order (one 128-float slab per 128-slot query
//                         tile, ragged tails padded so they contribute 0);
//   attn_bwd_dkdv_kernel  one 128-key tile per work unit; loops over the
//                         visible query tiles of every head of its group;
//                         S^T = K Q^T and dP^T = V dO^T into TMEM, P^T and
//                         dS^T (bf16) back into TMEM, dV += P^T dO and
//                         dK += dS^T Q accumulated in TMEM;
//   attn_bwd_dq_kernel    one 128-query tile per work unit; loops over the
//                         visible key tiles; S = Q K^T, dP = dO V^T, dS (bf16)
//                         into TMEM, dQ += dS K accumulated in TMEM.
// dQ is produced by its own pass, so nothing is accumulated with atomics and
// the result is deterministic; S and dP are computed twice for it.
//
// The same kernels also run one ring hop (kMode = BWD_STEP): the queries of
// shard r against the key/value block of shard s only, on shard-local
// tensors, writing or adding fp32 contributions: dq to shard r, dk / dv to
// block s.  A ring of P ranks sums them hop by hop while the block's dk / dv
// accumulators travel with the block.
//
// Roles in both tensor-core kernels (384 threads, one persistent CTA per SM):
//   warp 0       TMA producer,
//   warps 1, 3   tcgen05 issuers, one thread each (see each kernel); warp 1
//                owns the TMEM allocation,
//   warps 4..7   "half 0": columns [0, 64) of every S / dP tile,
//   warps 8..11  "half 1": columns [64, 128).
// The S / dP products are issued per half (N = 64), so half 0's elementwise
// work overlaps the tensor core computing half 1, and the accumulating
// products of one tile overlap the elementwise work of the next.
//
// Tensor memory (512 columns): S or S^T [0,128), dP or dP^T [128,256),
// accumulators from 256 (dK/dV pass: dV [256,256+D), dK [384,384+D);
// dQ pass: dQ [256,256+D)).  The bf16 P / dS of half x overwrite columns
// [64x, 64x+32) of their own fp32 region after it has been read.  The dQ pass
// also keeps its unit's Q [384,384+D/2) and dO [448,448+D/2) in tensor
// memory as the A operands of S and dP, so those products read only the key
// or value tile from shared memory.
#pragma once
#include "geometry.cuh"
#include "sm103_ptx.cuh"

namespace ra {

// What a launch covers (the kernels' kMode template argument):
//   BWD_RING    the whole ring on natural-order tensors, bf16 gradients;
//   BWD_VARLEN  the same over packed sequences;
//   BWD_STEP    one ring hop: the queries of shard step_r against the key /
//               value block of shard step_s, on shard-local tensors
//               ([B][n][heads][D], local-slot order), fp32 gradients written
//               or added (accumulate) into dq32 (the hop's dq contribution to
//               shard r) and dk32 / dv32 (its dk, dv contribution to block s).
enum { BWD_RING = 0, BWD_VARLEN = 1, BWD_STEP = 2 };

struct BwdParams {
  Geo g;
  float scale;         // multiplies dq and dk
  float scale_log2;    // scale * log2(e)
  const float* nlse2;  // tile order: -lse * log2(e); padded rows -inf
  const float* ndelta; // tile order: -delta; padded rows 0
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int64_t num_items;
  const int* sched;           // may be null: per-CTA item lists (see cta_items)
  // packed sequences (BWD_VARLEN only):
  const int4* units;          // (sequence, shard, segment, tile) per unit, longest first
  const int64_t* cu_seqlens;  // token offset of each sequence, and the total
  const int64_t* vbase;       // first element of each sequence in the tile-order vectors
  int total;                  // tokens in the pack
  // one ring hop (BWD_STEP only):
  int step_r, step_s;
  int accumulate;             // add into dq32 / dk32 / dv32 instead of overwriting
  float* dq32;
  float* dk32;
  float* dv32;
};

// Tile-order vectors: slab (b, h, shard, seg, tile) holds 128 floats, one per
// slot of that query tile.  A hop (BWD_STEP) holds shard step_r's slabs only.
__host__ __device__ inline int64_t vec_tile(const Geo& g, int b, int h, int shard, int seg,
                                            int tile) {
  return ((((int64_t)b * g.H + h) * g.P + shard) * g.nseg + seg) * g.ntile + tile;
}
__host__ __device__ inline int64_t vec_elems(const Geo& g) {
  return (int64_t)g.B * g.H * g.P * g.nseg * g.ntile * kTile;
}
__host__ __device__ inline int64_t vec_tile_step(const Geo& g, int b, int h, int seg, int tile) {
  return (((int64_t)b * g.H + h) * g.nseg + seg) * g.ntile + tile;
}
__host__ __device__ inline int64_t vec_elems_step(const Geo& g) {
  return (int64_t)g.B * g.H * g.nseg * g.ntile * kTile;
}
template <int kMode>
__device__ __forceinline__ int64_t vec_slab(const Geo& g, int b, int h, int shard, int seg,
                                            int tile) {
  if constexpr (kMode == BWD_STEP) return vec_tile_step(g, b, h, seg, tile);
  else return vec_tile(g, b, h, shard, seg, tile);
}

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kSubTiles = D / 64;
  static constexpr int kStages = D == 128 ? 2 : 4;   // streamed tile pairs in flight
  static constexpr int kVecBytes = kTile * 4;
};

constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 384;
constexpr uint32_t kColQA = 384, kColDOA = 448;   // dQ pass: Q and dO as A operands

// TMA coordinates (phase, row) of the tile at offset `off` of the segment
// (starting at position pos0 and local slot local0) of shard `shard`.  Ring
// modes: natural order, the batch entry or sequence's position 0 at token row
// row_base (a multiple of P).  Hop mode: shard-local order, the batch entry's
// slot 0 at row row_base (= b * n).
template <int kMode>
__device__ __forceinline__ void bwd_coords(const Geo& g, int shard, int pos0, int local0, int off,
                                           int row_base, int& phase, int& row) {
  if constexpr (kMode == BWD_STEP) {
    phase = 0;
    row = row_base + local0 + off;
  } else if (g.layout == LAYOUT_STRIPED) {
    phase = shard;
    row = row_base / g.P + off;
  } else {
    phase = 0;
    row = row_base + pos0 + off;
  }
}

// ---------------------------------------------------------------- prep
// delta = rowsum(dout * out) and -lse * log2(e) for every query row, in tile
// order.  D/8 lanes share a row (16 bytes of dout and of out each).
// Packed sequences (BWD_VARLEN): blockIdx.y is the sequence; its elements
// start at vbase[seq], its tokens at cu_seqlens[seq], lse is [H][total].
// One hop (BWD_STEP): the rows of shard step_r only; out and dout are
// [B][n][H][D] and lse [B][H][n] in shard-local order.
template <int D, int kMode>
__global__ void bwd_prep_kernel(const __nv_bfloat16* __restrict__ out,
                                const __nv_bfloat16* __restrict__ dout,
                                const float* __restrict__ lse, float* __restrict__ nlse2,
                                float* __restrict__ ndelta, Geo g, const int64_t* cu_seqlens,
                                const int64_t* vbase_arr, int total, int step_r) {
  constexpr int kLanes = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanes;
  const int lane = threadIdx.x % 32;
  const int sub = lane / kLanes, piece = lane % kLanes;
  int64_t tok0 = 0, vbase = 0;
  if constexpr (kMode == BWD_VARLEN) {
    const int seq = blockIdx.y;
    tok0 = cu_seqlens[seq];
    vbase = vbase_arr[seq];
    g = make_geo(1, g.H, g.Hkv, cu_seqlens[seq + 1] - tok0, g.P, g.layout, g.causal);
  }
  const int64_t rows = kMode == BWD_STEP ? vec_elems_step(g) : vec_elems(g);
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  for (int64_t base = warp0 * kRowsPerWarp; base < rows; base += warps_total * kRowsPerWarp) {
    const int64_t e = base + sub;
    float acc = 0.f;
    bool real = false;
    int64_t lidx = 0;
    if (e < rows) {
      int64_t t = e / kTile;
      const int i = (int)(e % kTile);
      const int tile = (int)(t % g.ntile); t /= g.ntile;
      const int seg = (int)(t % g.nseg); t /= g.nseg;
      int shard = step_r;
      if constexpr (kMode != BWD_STEP) {
        shard = (int)(t % g.P);
        t /= g.P;
      }
      const int h = (int)(t % g.H);
      const int b = (int)(t / g.H);
      const QTile qt = make_qtile(g, shard, seg, tile);
      if (i < qt.valid) {
        real = true;
        const int64_t pos = qt.pos0 + (int64_t)qt.stride * (qt.off + i);
        const int64_t slot = qt.local0 + qt.off + i;
        int64_t tok;
        if constexpr (kMode == BWD_STEP) tok = (int64_t)b * g.n + slot;
        else tok = kMode == BWD_VARLEN ? tok0 + pos : (int64_t)b * g.S + pos;
        const int64_t off = (tok * g.H + h) * D + piece * 8;
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(out + off));
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(dout + off));
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[j]));
          const float2 fc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cv[j]));
          acc = fmaf(fa.x, fc.x, acc);
          acc = fmaf(fa.y, fc.y, acc);
        }
        if constexpr (kMode == BWD_STEP) lidx = ((int64_t)b * g.H + h) * g.n + slot;
        else lidx = kMode == BWD_VARLEN ? (int64_t)h * total + tok : ((int64_t)b * g.H + h) * g.S + pos;
      }
    }
#pragma unroll
    for (int o = kLanes / 2; o > 0; o /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (e < rows && piece == 0) {
      ndelta[vbase + e] = real ? -acc : 0.f;
      nlse2[vbase + e] = real ? -__ldg(lse + lidx) * 1.4426950408889634f : -INFINITY;
    }
  }
}

// ---------------------------------------------------------------- schedule
// dK/dV pass: work item -> (b, kv head, key tile).  Within a (b, kv head) the
// key tiles come in increasing position, so under a causal mask the tiles
// that see the most queries come first.
struct KUnit {
  int b, hkv, shard, seg, tile;
  int row_base;     // token row of position 0 of this batch entry or sequence
  int64_t vbase;    // first element of this batch entry or sequence in the vectors
};

__host__ __device__ __forceinline__ KUnit kunit_of(const Geo& g, int64_t item) {
  const int64_t U = (int64_t)g.P * g.nseg * g.ntile;
  const int64_t bg = item / U;
  const int64_t u = item % U;
  KUnit w;
  w.b = (int)(bg / g.Hkv);
  w.hkv = (int)(bg % g.Hkv);
  if (g.layout == LAYOUT_STRIPED) {
    w.tile = (int)(u / g.P);
    w.shard = (int)(u % g.P);
    w.seg = 0;
  } else if (g.layout == LAYOUT_ZIGZAG) {
    const int chunk = (int)(u / g.ntile);
    w.tile = (int)(u % g.ntile);
    if (chunk < g.P) { w.shard = chunk; w.seg = 0; }
    else { w.shard = 2 * g.P - 1 - chunk; w.seg = 1; }
  } else {
    w.shard = (int)(u / g.ntile);
    w.tile = (int)(u % g.ntile);
    w.seg = 0;
  }
  return w;
}

// dQ pass: work item -> (b, h, query tile), decreasing position within (b, h).
struct QUnit {
  int b, h, shard, seg, tile;
  int row_base;
  int64_t vbase;
};

__host__ __device__ __forceinline__ QUnit qunit_of(const Geo& g, int64_t item) {
  const int64_t U = (int64_t)g.P * g.nseg * g.ntile;
  const int64_t bh = item / U;
  const int64_t u = item % U;
  QUnit w;
  w.b = (int)(bh / g.H);
  w.h = (int)(bh % g.H);
  if (g.layout == LAYOUT_STRIPED) {
    w.tile = g.ntile - 1 - (int)(u / g.P);
    w.shard = g.P - 1 - (int)(u % g.P);
    w.seg = 0;
  } else if (g.layout == LAYOUT_ZIGZAG) {
    const int chunk = 2 * g.P - 1 - (int)(u / g.ntile);
    w.tile = g.ntile - 1 - (int)(u % g.ntile);
    if (chunk < g.P) { w.shard = chunk; w.seg = 0; }
    else { w.shard = 2 * g.P - 1 - chunk; w.seg = 1; }
  } else {
    w.shard = g.P - 1 - (int)(u / g.ntile);
    w.tile = g.ntile - 1 - (int)(u % g.ntile);
    w.seg = 0;
  }
  return w;
}

// One hop: the key tiles of block step_s, resp. the query tiles of shard
// step_r, per (b, kv head) or (b, head); keys in increasing and queries in
// decreasing position.
__host__ __device__ __forceinline__ KUnit kunit_step(const Geo& g, int s, int64_t item) {
  const int64_t U = (int64_t)g.nseg * g.ntile;
  const int64_t bg = item / U;
  const int64_t u = item % U;
  KUnit w;
  w.b = (int)(bg / g.Hkv);
  w.hkv = (int)(bg % g.Hkv);
  w.shard = s;
  w.seg = (int)(u / g.ntile);
  w.tile = (int)(u % g.ntile);
  return w;
}

__host__ __device__ __forceinline__ QUnit qunit_step(const Geo& g, int r, int64_t item) {
  const int64_t U = (int64_t)g.nseg * g.ntile;
  const int64_t bh = item / U;
  const int64_t u = item % U;
  QUnit w;
  w.b = (int)(bh / g.H);
  w.h = (int)(bh % g.H);
  w.shard = r;
  w.seg = g.nseg - 1 - (int)(u / g.ntile);
  w.tile = g.ntile - 1 - (int)(u % g.ntile);
  return w;
}

// The unit of a work item and the geometry it runs in: the call's geometry,
// or for packed sequences the unit's sequence's (B = 1, S = its length; items
// are unit * Hkv + kv head, resp. unit * H + head, over the host's list).
// row_base is the token row of the unit's batch entry or sequence: position 0
// in the ring modes, local slot 0 (b * n) in the hop mode.
template <int kMode>
__device__ __forceinline__ const Geo& kunit_get(const BwdParams& p, int64_t item, KUnit& w,
                                                Geo& gv) {
  if constexpr (kMode == BWD_VARLEN) {
    const int64_t unit = item / p.g.Hkv;
    w.hkv = (int)(item % p.g.Hkv);
    w.b = 0;
    const int4 u4 = __ldg(p.units + unit);
    const int64_t t0 = __ldg(p.cu_seqlens + u4.x), t1 = __ldg(p.cu_seqlens + u4.x + 1);
    gv = make_geo(1, p.g.H, p.g.Hkv, t1 - t0, p.g.P, p.g.layout, p.g.causal);
    w.shard = u4.y;
    w.seg = u4.z;
    w.tile = u4.w;
    w.row_base = (int)t0;
    w.vbase = __ldg(p.vbase + u4.x);
    return gv;
  } else if constexpr (kMode == BWD_STEP) {
    w = kunit_step(p.g, p.step_s, item);
    w.row_base = w.b * p.g.n;
    w.vbase = 0;
    return p.g;
  } else {
    w = kunit_of(p.g, item);
    w.row_base = w.b * p.g.S;
    w.vbase = 0;
    return p.g;
  }
}

template <int kMode>
__device__ __forceinline__ const Geo& qunit_get(const BwdParams& p, int64_t item, QUnit& w,
                                                Geo& gv) {
  if constexpr (kMode == BWD_VARLEN) {
    const int64_t unit = item / p.g.H;
    w.h = (int)(item % p.g.H);
    w.b = 0;
    const int4 u4 = __ldg(p.units + unit);
    const int64_t t0 = __ldg(p.cu_seqlens + u4.x), t1 = __ldg(p.cu_seqlens + u4.x + 1);
    gv = make_geo(1, p.g.H, p.g.Hkv, t1 - t0, p.g.P, p.g.layout, p.g.causal);
    w.shard = u4.y;
    w.seg = u4.z;
    w.tile = u4.w;
    w.row_base = (int)t0;
    w.vbase = __ldg(p.vbase + u4.x);
    return gv;
  } else if constexpr (kMode == BWD_STEP) {
    w = qunit_step(p.g, p.step_r, item);
    w.row_base = w.b * p.g.n;
    w.vbase = 0;
    return p.g;
  } else {
    w = qunit_of(p.g, item);
    w.row_base = w.b * p.g.S;
    w.vbase = 0;
    return p.g;
  }
}

// Query tiles a key tile meets, in ring order: for each query head of the
// group, steps t = 0..P-1 visit shard r = (s + t) mod P; in each segment of r
// the tiles holding a position >= kmin (all tiles without a causal mask) are a
// suffix [a, ntile).  A hop visits shard r0 only (t_end = 1).
struct QIter {
  int e, t, t_end, sq, a, a_end;
  int r, r0, h, hkv, s, kmin;
  Seg seg;
};

__device__ __forceinline__ void qiter_range(const Geo& g, QIter& it) {
  it.seg = segment_of(g, it.r, it.sq);
  const int first = g.causal ? count_le(it.seg, it.kmin - 1) : 0;
  if (first >= it.seg.len) {
    it.a = 0;
    it.a_end = 0;
  } else {
    it.a = first / kTile;
    it.a_end = g.ntile;
  }
}

// Ring modes: r0 = s, t_end = P.  Hop mode: r0 = step_r, t_end = 1.
__device__ __forceinline__ void qiter_setup(const Geo& g, QIter& it, int hkv, int s, int kmin,
                                            int r0, int t_end) {
  it.e = 0; it.t = 0; it.t_end = t_end; it.sq = 0;
  it.hkv = hkv; it.s = s; it.kmin = kmin;
  it.h = hkv * (g.H / g.Hkv);
  it.r0 = r0;
  it.r = r0;
  qiter_range(g, it);
}

__device__ __forceinline__ bool qiter_next(const Geo& g, QIter& it) {
  while (it.a >= it.a_end) {
    if (++it.sq >= g.nseg) {
      it.sq = 0;
      if (++it.t >= it.t_end) {
        it.t = 0;
        if (++it.e >= g.H / g.Hkv) return false;
        it.h = it.hkv * (g.H / g.Hkv) + it.e;
      }
      it.r = (it.r0 + it.t) % g.P;
    }
    qiter_range(g, it);
  }
  return true;
}

// Key tiles a query tile meets, in ring order s = (r - t) mod P; the visible
// tiles of each key segment are a prefix (positions <= qmax).  A hop visits
// block s0 only (t_end = 1).
struct KIterB {
  int t, t_end, sk, bt, nk, s, r, qmax;
  Seg seg;
};

// Ring modes: s0 = r, t_end = P.  Hop mode: s0 = step_s, t_end = 1.
__device__ __forceinline__ void kiterb_setup(const Geo& g, KIterB& it, int r, int qmax, int s0,
                                             int t_end) {
  it.t = 0; it.t_end = t_end; it.sk = 0; it.bt = 0; it.r = r; it.qmax = qmax;
  it.s = s0;
  it.seg = segment_of(g, it.s, 0);
  it.nk = visible_tiles(g, it.seg, qmax);
}

__device__ __forceinline__ bool kiterb_next(const Geo& g, KIterB& it) {
  while (it.bt >= it.nk) {
    it.bt = 0;
    if (++it.sk >= g.nseg) {
      it.sk = 0;
      if (++it.t >= it.t_end) return false;
      it.s = ring_block(g, it.r, it.t);
    }
    it.seg = segment_of(g, it.s, it.sk);
    it.nk = visible_tiles(g, it.seg, it.qmax);
  }
  return true;
}

// Iterator set-up for a launch's mode.
template <int kMode>
__device__ __forceinline__ void qiter_start(const BwdParams& p, const Geo& g, QIter& it, int hkv,
                                            int s, int kmin) {
  if constexpr (kMode == BWD_STEP) qiter_setup(g, it, hkv, s, kmin, p.step_r, 1);
  else qiter_setup(g, it, hkv, s, kmin, s, g.P);
}
template <int kMode>
__device__ __forceinline__ void kiterb_start(const BwdParams& p, const Geo& g, KIterB& it, int r,
                                             int qmax) {
  if constexpr (kMode == BWD_STEP) kiterb_setup(g, it, r, qmax, p.step_s, 1);
  else kiterb_setup(g, it, r, qmax, r, g.P);
}

// Stores 32 fp32 accumulator columns of one row as fp32, times `mul`, added
// to what the row holds when `acc` is set (one hop's contribution).
__device__ __forceinline__ void store_row32_f32(float* dst, const uint32_t (&r)[32], float mul,
                                                bool acc) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 v = make_float4(__uint_as_float(r[4 * i]) * mul, __uint_as_float(r[4 * i + 1]) * mul,
                           __uint_as_float(r[4 * i + 2]) * mul,
                           __uint_as_float(r[4 * i + 3]) * mul);
    if (acc) {
      const float4 o = d4[i];
      v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
    }
    d4[i] = v;
  }
}

// ---------------------------------------------------------------- shared memory
template <int D>
struct __align__(1024) DkdvSmem {
  uint8_t k[BwdCfg<D>::kTileBytes];
  uint8_t v[BwdCfg<D>::kTileBytes];
  uint8_t q[BwdCfg<D>::kStages][BwdCfg<D>::kTileBytes];
  uint8_t dO[BwdCfg<D>::kStages][BwdCfg<D>::kTileBytes];
  float nlse2[BwdCfg<D>::kStages][kTile];
  float ndelta[BwdCfg<D>::kStages][kTile];
  uint64_t kv_full, kv_empty;
  uint64_t st_full[BwdCfg<D>::kStages], st_empty[BwdCfg<D>::kStages];
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full, acc_empty;
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
struct __align__(1024) DqSmem {
  uint8_t q[BwdCfg<D>::kTileBytes];
  uint8_t dO[BwdCfg<D>::kTileBytes];
  uint8_t k[BwdCfg<D>::kStages][BwdCfg<D>::kTileBytes];
  uint8_t v[BwdCfg<D>::kStages][BwdCfg<D>::kTileBytes];
  uint64_t q_full, q_empty;
  uint64_t qt_full;   // the unit's Q and dO are in tensor memory (one arrival per warp)
  uint64_t st_full[BwdCfg<D>::kStages], st_empty[BwdCfg<D>::kStages];
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full, acc_empty;
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort_flag;
};

// S_x = A B_x^T with A (128 rows x D) in tensor memory as bf16 pairs, B_x the
// 64 rows of a K-major tile in shared memory starting at row 64x.
template <int D>
__device__ __forceinline__ void issue_half_product_ta(uint32_t d_tmem, uint32_t a_tmem,
                                                      uint32_t b_base, int x) {
  constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * (kTile * 128) + (kk % 4) * 32;
    mma_ts(d_tmem, a_tmem + kk * 8, sdesc_sw128(b_base + x * (64 * 128) + off, 16, 1024), id,
           kk > 0 ? 1u : 0u);
  }
}

// Row `row` of a 128 x D bf16 tile that TMA laid out with 128-byte swizzle
// (D/64 sub-tiles; 16-byte chunk c of row r at chunk position c ^ (r % 8)),
// into this thread's tensor-memory lane as D/2 columns of bf16 pairs: the
// layout of an M = 128 MMA's A operand.
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t* src, int row, uint32_t t_dst) {
#pragma unroll
  for (int st = 0; st < D / 64; ++st) {
    uint32_t r[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + st * (kTile * 128) + row * 128 +
                                                      ((c ^ (row & 7)) << 4));
      r[4 * c] = v.x;
      r[4 * c + 1] = v.y;
      r[4 * c + 2] = v.z;
      r[4 * c + 3] = v.w;
    }
    tmem_st32(t_dst + 32 * st, r);
  }
}

// S_x (or S^T_x) = A B_x^T over the D contraction, N = 64 rows of B starting
// at row 64x; both operands K-major (128-byte swizzle, D/64 sub-tiles).
template <int D>
__device__ __forceinline__ void issue_half_product(uint32_t d_tmem, uint32_t a_base,
                                                   uint32_t b_base, int x) {
  constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * (kTile * 128) + (kk % 4) * 32;
    mma_ss(d_tmem, sdesc_sw128(a_base + off, 16, 1024),
           sdesc_sw128(b_base + x * (64 * 128) + off, 16, 1024), id, kk > 0 ? 1u : 0u);
  }
}

// acc += A_x B[64x .. 64x+64, :] with A_x (bf16, 128 lanes x 64 values) in
// TMEM and B a 128 x D tile in shared memory read MN-major.
template <int D>
__device__ __forceinline__ void issue_half_accumulate(uint32_t acc_tmem, uint32_t a_tmem,
                                                      uint32_t b_base, int x, bool first) {
  constexpr uint32_t id = idesc_bf16(128, D, false, true);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts(acc_tmem, a_tmem + kk * 8,
           sdesc_sw128(b_base + (4 * x + kk) * 2048, kTile * 128, 1024), id,
           (first && kk == 0) ? 0u : 1u);
}

// Stores 32 fp32 accumulator columns of one row as bf16, times `mul`.
__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16* dst, const uint32_t (&r)[32],
                                                 float mul) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d4[i] = make_uint4(
        pack_bf16x2(__uint_as_float(r[8 * i + 0]) * mul, __uint_as_float(r[8 * i + 1]) * mul),
        pack_bf16x2(__uint_as_float(r[8 * i + 2]) * mul, __uint_as_float(r[8 * i + 3]) * mul),
        pack_bf16x2(__uint_as_float(r[8 * i + 4]) * mul, __uint_as_float(r[8 * i + 5]) * mul),
        pack_bf16x2(__uint_as_float(r[8 * i + 6]) * mul, __uint_as_float(r[8 * i + 7]) * mul));
}

// dK/dV pass, one half of a tile, one key row per thread: reads S^T and dP^T
// (64 query columns starting at col0 of the tile), writes P^T and dS^T as bf16
// over the first half of their regions.  Query columns below `lo` precede the
// key and are masked out (kMasked only).
template <bool kMasked>
__device__ __forceinline__ void dkdv_half(uint32_t t_s, uint32_t t_dp, const float* nl,
                                          const float* nd, float2 sl2, int lo, int col0) {
#pragma unroll
  for (int c2 = 0; c2 < 2; ++c2) {
    uint32_t s[32], dp[32];
    tmem_ld32(t_s + 32 * c2, s);
    tmem_ld32(t_dp + 32 * c2, dp);
    tmem_wait_ld();
    uint32_t pk_p[16], pk_ds[16];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 nl4 = *reinterpret_cast<const float4*>(nl + 32 * c2 + i);
      const float4 nd4 = *reinterpret_cast<const float4*>(nd + 32 * c2 + i);
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        const float2 nlj = j == 0 ? make_float2(nl4.x, nl4.y) : make_float2(nl4.z, nl4.w);
        const float2 ndj = j == 0 ? make_float2(nd4.x, nd4.y) : make_float2(nd4.z, nd4.w);
        const float2 t2 = fma2(make_float2(__uint_as_float(s[i + j]),
                                           __uint_as_float(s[i + j + 1])), sl2, nlj);
        float p0 = ex2_approx(t2.x), p1 = ex2_approx(t2.y);
        if (kMasked) {
          const int qc = col0 + 32 * c2 + i + j;   // query column within the tile
          p0 = qc < lo ? 0.f : p0;
          p1 = qc + 1 < lo ? 0.f : p1;
        }
        const float2 dd = add2(make_float2(__uint_as_float(dp[i + j]),
                                           __uint_as_float(dp[i + j + 1])), ndj);
        const float2 ds = mul2(make_float2(p0, p1), dd);
        pk_p[(i + j) / 2] = pack_bf16x2(p0, p1);
        pk_ds[(i + j) / 2] = pack_bf16x2(ds.x, ds.y);
      }
    }
    tmem_st16(t_s + 16 * c2, pk_p);
    tmem_st16(t_dp + 16 * c2, pk_ds);
  }
}

// dQ pass, one half of a tile, one query row per thread: reads S and dP (64
// key columns starting at col0), writes dS as bf16 over the first half of the
// S region.  Key columns at or beyond `lim` are masked out (kMasked only).
template <bool kMasked>
__device__ __forceinline__ void dq_half(uint32_t t_s, uint32_t t_dp, float2 sl2, float2 nl2,
                                        float2 nd2, int lim, int col0) {
#pragma unroll
  for (int c2 = 0; c2 < 2; ++c2) {
    uint32_t s[32], dp[32];
    tmem_ld32(t_s + 32 * c2, s);
    tmem_ld32(t_dp + 32 * c2, dp);
    tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 t2 = fma2(make_float2(__uint_as_float(s[i]), __uint_as_float(s[i + 1])),
                             sl2, nl2);
      float p0 = ex2_approx(t2.x), p1 = ex2_approx(t2.y);
      if (kMasked) {
        const int kc = col0 + 32 * c2 + i;   // key column within the tile
        p0 = kc < lim ? p0 : 0.f;
        p1 = kc + 1 < lim ? p1 : 0.f;
      }
      const float2 dd = add2(make_float2(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])),
                             nd2);
      const float2 ds = mul2(make_float2(p0, p1), dd);
      pk[i / 2] = pack_bf16x2(ds.x, ds.y);
    }
    tmem_st16(t_s + 16 * c2, pk);
  }
}

// ---------------------------------------------------------------- dK / dV pass
template <int D, int kMode>
__global__ void __launch_bounds__(384, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  using Cfg = BwdCfg<D>;
  constexpr int kSt = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  DkdvSmem<D>& sm = *reinterpret_cast<DkdvSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  volatile int* abort_flag = &sm.abort_flag;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.kv_full), 1);
    mbar_init(smem_u32(&sm.kv_empty), 2);
    for (int i = 0; i < kSt; ++i) {
      mbar_init(smem_u32(&sm.st_full[i]), 1);
      mbar_init(smem_u32(&sm.st_empty[i]), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&sm.s_full[x]), 2);
      mbar_init(smem_u32(&sm.p_full[x]), 4);      // one arrival per elementwise warp
    }
    mbar_init(smem_u32(&sm.acc_full), 2);
    mbar_init(smem_u32(&sm.acc_empty), 8);
    mbar_init(smem_u32(&sm.drain[0]), 1);
    mbar_init(smem_u32(&sm.drain[1]), 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // The producer's positions: key/value tile loads issued (parity) and the
  // next streamed stage with its lap parity.  At function scope so that an
  // aborting CTA can wait for every load it issued.
  uint32_t tkv_ph = 0, tst = 0, tst_ph = 0;
  const CtaItems mine = cta_items(p.sched);
  auto item_at = [&](int64_t k) -> int64_t { return cta_item(mine, k, p.num_items); };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      for (int64_t k = 0;; ++k) {
        const int64_t item = item_at(k);
        if (item >= p.num_items) break;
        KUnit w;
        Geo gv;
        const Geo& g = kunit_get<kMode>(p, item, w, gv);
        const QTile kt = make_qtile(g, w.shard, w.seg, w.tile);
        QIter it;
        qiter_start<kMode>(p, g, it, w.hkv, w.shard, kt.qmin);
        if (!kt.valid || !qiter_next(g, it)) continue;
        if (!mbar_wait(smem_u32(&sm.kv_empty), tkv_ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag)) goto done;
        tkv_ph ^= 1;
        {
          const uint32_t bar = smem_u32(&sm.kv_full);
          mbar_arrive_expect_tx(bar, 2 * Cfg::kTileBytes);
          int phase, row;
          bwd_coords<kMode>(g, w.shard, kt.pos0, kt.local0, kt.off, w.row_base, phase, row);
#pragma unroll
          for (int s2 = 0; s2 < Cfg::kSubTiles; ++s2) {
            tma_load_4d(smem_u32(sm.k) + s2 * (kTile * 128), &tm_k, bar, 64 * s2, w.hkv, phase,
                        row, pol_kv);
            tma_load_4d(smem_u32(sm.v) + s2 * (kTile * 128), &tm_v, bar, 64 * s2, w.hkv, phase,
                        row, pol_kv);
          }
        }
        do {
          if (!mbar_wait(smem_u32(&sm.st_empty[tst]), tst_ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag))
            goto done;
          const uint32_t bar = smem_u32(&sm.st_full[tst]);
          mbar_arrive_expect_tx(bar, 2 * Cfg::kTileBytes + 2 * Cfg::kVecBytes);
          int phase, row;
          bwd_coords<kMode>(g, it.r, it.seg.pos0, it.seg.local0, it.a * kTile, w.row_base, phase, row);
#pragma unroll
          for (int s2 = 0; s2 < Cfg::kSubTiles; ++s2) {
            tma_load_4d(smem_u32(sm.q[tst]) + s2 * (kTile * 128), &tm_q, bar, 64 * s2, it.h, phase,
                        row, pol_q);
            tma_load_4d(smem_u32(sm.dO[tst]) + s2 * (kTile * 128), &tm_do, bar, 64 * s2, it.h,
                        phase, row, pol_q);
          }
          const int64_t vt = w.vbase + vec_slab<kMode>(g, w.b, it.h, it.r, it.sq, it.a) * kTile;
          bulk_load(smem_u32(sm.nlse2[tst]), p.nlse2 + vt, Cfg::kVecBytes, bar, pol_q);
          bulk_load(smem_u32(sm.ndelta[tst]), p.ndelta + vt, Cfg::kVecBytes, bar, pol_q);
          if (++tst == kSt) { tst = 0; tst_ph ^= 1; }
          ++it.a;
        } while (qiter_next(g, it));
      }
    }
  } else if (warp == 1 || warp == 3) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuers
      // Issuer 0 (warp 1): S^T_x = K Q_x^T and dV += P^T_x dO_x.
      // Issuer 1 (warp 3): dP^T_x = V dO_x^T and dK += dS^T_x Q_x.
      // Each accumulator has one issuer; s_full, st_empty, kv_empty and
      // acc_full complete when both have committed.
      const int w = warp == 1 ? 0 : 1;
      uint32_t kv_ph = 0, st = 0, st_ph = 0, p_ph0 = 0, p_ph1 = 0, acc_ph = 0;
      const uint32_t a_op = w == 0 ? smem_u32(sm.k) : smem_u32(sm.v);
      const uint32_t prod_col = w == 0 ? kColS : kColDP;    // product written, then its bf16 half read
      const uint32_t acc_col = w == 0 ? kColAcc0 : kColAcc1;
      for (int64_t k = 0;; ++k) {
        const int64_t item = item_at(k);
        if (item >= p.num_items) break;
        KUnit u;
        Geo gv;
        const Geo& g = kunit_get<kMode>(p, item, u, gv);
        const QTile kt = make_qtile(g, u.shard, u.seg, u.tile);
        QIter it;
        qiter_start<kMode>(p, g, it, u.hkv, u.shard, kt.qmin);
        if (!kt.valid || !qiter_next(g, it)) continue;
        if (!mbar_wait(smem_u32(&sm.kv_full), kv_ph, RA_DEV_TIMEOUT_MMA, abort_flag)) goto done;
        kv_ph ^= 1;
        if (!mbar_wait(smem_u32(&sm.st_full[st]), st_ph, RA_DEV_TIMEOUT_MMA, abort_flag)) goto done;
        tc_fence_after();
        // B operand of the product: Q (issuer 0) or dO (issuer 1); of the accumulation: the other
        auto prod_b = [&](uint32_t s_) { return w == 0 ? smem_u32(sm.q[s_]) : smem_u32(sm.dO[s_]); };
        auto acc_b = [&](uint32_t s_) { return w == 0 ? smem_u32(sm.dO[s_]) : smem_u32(sm.q[s_]); };
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          issue_half_product<D>(tmem + prod_col + 64 * x, a_op, prod_b(st), x);
          mma_commit(smem_u32(&sm.s_full[x]));
        }
        bool first = true;
        for (;;) {
          const uint32_t cur = st;
          ++it.a;
          const bool more = qiter_next(g, it);
          uint32_t nst = st + 1, nph = st_ph;
          if (nst == (uint32_t)kSt) { nst = 0; nph ^= 1; }
          // half 0
          if (!mbar_wait(smem_u32(&sm.p_full[0]), p_ph0, RA_DEV_TIMEOUT_MMA, abort_flag)) goto done;
          p_ph0 ^= 1;
          tc_fence_after();
          if (first) {
            if (!mbar_wait(smem_u32(&sm.acc_empty), acc_ph ^ 1, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            tc_fence_after();
          }
          issue_half_accumulate<D>(tmem + acc_col, tmem + prod_col, acc_b(cur), 0, first);
          if (more) {
            if (!mbar_wait(smem_u32(&sm.st_full[nst]), nph, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            tc_fence_after();
            issue_half_product<D>(tmem + prod_col, a_op, prod_b(nst), 0);
            mma_commit(smem_u32(&sm.s_full[0]));
          }
          // half 1
          if (!mbar_wait(smem_u32(&sm.p_full[1]), p_ph1, RA_DEV_TIMEOUT_MMA, abort_flag)) goto done;
          p_ph1 ^= 1;
          tc_fence_after();
          issue_half_accumulate<D>(tmem + acc_col, tmem + prod_col + 64, acc_b(cur), 1, false);
          mma_commit(smem_u32(&sm.st_empty[cur]));
          st = nst;
          st_ph = nph;
          first = false;
          if (!more) break;
          issue_half_product<D>(tmem + prod_col + 64, a_op, prod_b(st), 1);
          mma_commit(smem_u32(&sm.s_full[1]));
        }
        mma_commit(smem_u32(&sm.acc_full));
        mma_commit(smem_u32(&sm.kv_empty));
        acc_ph ^= 1;
      }
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- elementwise halves
    const int x = (warp - 4) / 4;                 // column half of S^T / dP^T
    const int quarter = warp % 4;                 // TMEM lanes [32*quarter, +32)
    const int row = quarter * 32 + lane;          // key row of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + kColS + 64 * x;
    const uint32_t t_dp = tmem + lane_addr + kColDP + 64 * x;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    uint32_t s_ph = 0, st = 0, st_ph = 0, acc_ph = 0;
    for (int64_t k = 0;; ++k) {
      const int64_t item = item_at(k);
      if (item >= p.num_items) break;
      KUnit w;
      Geo gv;
      const Geo& g = kunit_get<kMode>(p, item, w, gv);
      const QTile kt = make_qtile(g, w.shard, w.seg, w.tile);
      QIter it;
      qiter_start<kMode>(p, g, it, w.hkv, w.shard, kt.qmin);
      if (!kt.valid || !qiter_next(g, it)) {
        // A hop's key tile that no query of shard step_r sees: its rows of the
        // overwritten dv (half 0) / dk (half 1) are zero.  (In the ring modes
        // every key is seen at least by its own position.)
        if constexpr (kMode == BWD_STEP) {
          if (!p.accumulate && row < kt.valid) {
            float* dst = (x == 0 ? p.dv32 : p.dk32) +
                         (((int64_t)w.row_base + kt.local0 + kt.off + row) * g.Hkv + w.hkv) * D;
#pragma unroll
            for (int i = 0; i < D / 4; ++i)
              reinterpret_cast<float4*>(dst)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        continue;
      }
      const int kpos = kt.pos0 + kt.stride * (kt.off + row);
      do {
        // The tile's geometry does not depend on S: work it out while the
        // products are still running.
        const QTile qt = make_qtile(g, it.r, it.sq, it.a);
        int lo = 0;   // query columns below lo precede this key: masked out
        if (g.causal && qt.qmin < kt.qmax) {
          const int cnt = count_le(it.seg, kpos - 1) - qt.off;
          lo = cnt < 0 ? 0 : (cnt > kTile ? kTile : cnt);
        }
        const bool masked = __any_sync(0xffffffffu, lo > 64 * x);
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[x]), s_ph,
                                               RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
          goto done;
        s_ph ^= 1;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.st_full[st]), st_ph,
                                               RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
          goto done;
        tc_fence_after();
        const float* nl = sm.nlse2[st] + 64 * x;
        const float* nd = sm.ndelta[st] + 64 * x;
        if (masked)
          dkdv_half<true>(t_s, t_dp, nl, nd, sl2, lo, 64 * x);
        else
          dkdv_half<false>(t_s, t_dp, nl, nd, sl2, lo, 64 * x);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&sm.p_full[x]));
        if (++st == (uint32_t)kSt) { st = 0; st_ph ^= 1; }
        ++it.a;
      } while (qiter_next(g, it));
      // ---- epilogue: half 0 stores dV, half 1 stores scale * dK
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.acc_full), acc_ph,
                                             RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
        goto done;
      acc_ph ^= 1;
      tc_fence_after();
      {
        const float mul = x == 0 ? 1.f : p.scale;
        const uint32_t t_acc = tmem + lane_addr + (x == 0 ? kColAcc0 : kColAcc1);
        // natural order (ring modes) or this key's local slot (hop mode)
        const int64_t orow = kMode == BWD_STEP
            ? ((int64_t)w.row_base + kt.local0 + kt.off + row) * g.Hkv + w.hkv
            : ((int64_t)w.row_base + kpos) * g.Hkv + w.hkv;
#pragma unroll
        for (int cch = 0; cch < D / 32; ++cch) {
          uint32_t r[32];
          tmem_ld32(t_acc + 32 * cch, r);
          tmem_wait_ld();
          if (row < kt.valid) {
            if constexpr (kMode == BWD_STEP)
              store_row32_f32((x == 0 ? p.dv32 : p.dk32) + orow * D + 32 * cch, r, mul,
                              p.accumulate != 0);
            else
              store_row32_bf16((x == 0 ? p.dv : p.dk) + orow * D + 32 * cch, r, mul);
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(smem_u32(&sm.acc_empty));
    }
  }

done:
  tc_fence_before();
  __syncthreads();
  if (sm.abort_flag) {
    // Let whatever this CTA issued before the failure land before its tensor
    // memory and shared memory go away: each issuer's products (a commit
    // arrives once all of them are done), and every TMA load of the producer
    // (the last phase armed on each full barrier; a barrier never armed
    // reports parity 1 complete at once).
    if ((warp == 1 || warp == 3) && lane == 0) {
      const int w = warp == 1 ? 0 : 1;
      mma_commit(smem_u32(&sm.drain[w]));
      mbar_wait_for(smem_u32(&sm.drain[w]), 0, RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
    }
    if (warp == 0 && lane == 0) {
      mbar_wait_for(smem_u32(&sm.kv_full), tkv_ph ^ 1, RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
      for (uint32_t i = 0; i < (uint32_t)kSt; ++i)
        mbar_wait_for(smem_u32(&sm.st_full[i]), i < tst ? tst_ph : tst_ph ^ 1,
                      RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- dQ pass
template <int D, int kMode>
__global__ void __launch_bounds__(384, 1)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams p) {
  using Cfg = BwdCfg<D>;
  constexpr int kSt = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  DqSmem<D>& sm = *reinterpret_cast<DqSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  volatile int* abort_flag = &sm.abort_flag;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    mbar_init(smem_u32(&sm.q_empty), 8);
    mbar_init(smem_u32(&sm.qt_full), 8);
    for (int i = 0; i < kSt; ++i) {
      mbar_init(smem_u32(&sm.st_full[i]), 1);
      mbar_init(smem_u32(&sm.st_empty[i]), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&sm.s_full[x]), 2);
      mbar_init(smem_u32(&sm.p_full[x]), 4);      // one arrival per elementwise warp
    }
    mbar_init(smem_u32(&sm.acc_full), 1);
    mbar_init(smem_u32(&sm.acc_empty), 8);
    mbar_init(smem_u32(&sm.drain[0]), 1);
    mbar_init(smem_u32(&sm.drain[1]), 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // The producer's positions: query tile loads issued (parity) and the next
  // streamed stage with its lap parity.  At function scope so that an
  // aborting CTA can wait for every load it issued.
  uint32_t tq_ph = 0, tst = 0, tst_ph = 0;
  const CtaItems mine = cta_items(p.sched);
  auto item_at = [&](int64_t k) -> int64_t { return cta_item(mine, k, p.num_items); };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      for (int64_t k = 0;; ++k) {
        const int64_t item = item_at(k);
        if (item >= p.num_items) break;
        QUnit w;
        Geo gv;
        const Geo& g = qunit_get<kMode>(p, item, w, gv);
        const QTile qt = make_qtile(g, w.shard, w.seg, w.tile);
        if (!qt.valid) continue;
        KIterB it;
        kiterb_start<kMode>(p, g, it, w.shard, qt.qmax);
        if (!kiterb_next(g, it)) continue;
        if (!mbar_wait(smem_u32(&sm.q_empty), tq_ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag)) goto done;
        tq_ph ^= 1;
        {
          const uint32_t bar = smem_u32(&sm.q_full);
          mbar_arrive_expect_tx(bar, 2 * Cfg::kTileBytes);
          int phase, row;
          bwd_coords<kMode>(g, w.shard, qt.pos0, qt.local0, qt.off, w.row_base, phase, row);
#pragma unroll
          for (int s2 = 0; s2 < Cfg::kSubTiles; ++s2) {
            tma_load_4d(smem_u32(sm.q) + s2 * (kTile * 128), &tm_q, bar, 64 * s2, w.h, phase, row,
                        pol_q);
            tma_load_4d(smem_u32(sm.dO) + s2 * (kTile * 128), &tm_do, bar, 64 * s2, w.h, phase,
                        row, pol_q);
          }
        }
        const int hkv = w.h / (g.H / g.Hkv);
        do {
          if (!mbar_wait(smem_u32(&sm.st_empty[tst]), tst_ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag))
            goto done;
          const uint32_t bar = smem_u32(&sm.st_full[tst]);
          mbar_arrive_expect_tx(bar, 2 * Cfg::kTileBytes);
          int phase, row;
          bwd_coords<kMode>(g, it.s, it.seg.pos0, it.seg.local0, it.bt * kTile, w.row_base, phase, row);
#pragma unroll
          for (int s2 = 0; s2 < Cfg::kSubTiles; ++s2) {
            tma_load_4d(smem_u32(sm.k[tst]) + s2 * (kTile * 128), &tm_k, bar, 64 * s2, hkv, phase,
                        row, pol_kv);
            tma_load_4d(smem_u32(sm.v[tst]) + s2 * (kTile * 128), &tm_v, bar, 64 * s2, hkv, phase,
                        row, pol_kv);
          }
          if (++tst == kSt) { tst = 0; tst_ph ^= 1; }
          ++it.bt;
        } while (kiterb_next(g, it));
      }
    }
  } else if (warp == 1 || warp == 3) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuers
      // Issuer 0 (warp 1): S_x = Q K_x^T and dQ += dS_x K_x.
      // Issuer 1 (warp 3): dP_x = dO V_x^T.
      // s_full and st_empty complete when both have committed.  The A
      // operands (Q, dO) come from tensor memory, copied there per unit by the
      // elementwise warps (qt_full).
      const int w = warp == 1 ? 0 : 1;
      uint32_t q_ph = 0, st = 0, st_ph = 0, p_ph0 = 0, p_ph1 = 0, acc_ph = 0;
      const uint32_t a_op = tmem + (w == 0 ? kColQA : kColDOA);
      const uint32_t prod_col = w == 0 ? kColS : kColDP;
      auto prod_b = [&](uint32_t s_) { return w == 0 ? smem_u32(sm.k[s_]) : smem_u32(sm.v[s_]); };
      for (int64_t k = 0;; ++k) {
        const int64_t item = item_at(k);
        if (item >= p.num_items) break;
        QUnit u;
        Geo gv;
        const Geo& g = qunit_get<kMode>(p, item, u, gv);
        const QTile qt = make_qtile(g, u.shard, u.seg, u.tile);
        if (!qt.valid) continue;
        KIterB it;
        kiterb_start<kMode>(p, g, it, u.shard, qt.qmax);
        if (!kiterb_next(g, it)) continue;
        if (!mbar_wait(smem_u32(&sm.qt_full), q_ph, RA_DEV_TIMEOUT_MMA, abort_flag)) goto done;
        q_ph ^= 1;
        if (!mbar_wait(smem_u32(&sm.st_full[st]), st_ph, RA_DEV_TIMEOUT_MMA, abort_flag)) goto done;
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          issue_half_product_ta<D>(tmem + prod_col + 64 * x, a_op, prod_b(st), x);
          mma_commit(smem_u32(&sm.s_full[x]));
        }
        bool first = true;
        for (;;) {
          const uint32_t cur = st;
          ++it.bt;
          const bool more = kiterb_next(g, it);
          uint32_t nst = st + 1, nph = st_ph;
          if (nst == (uint32_t)kSt) { nst = 0; nph ^= 1; }
          // half 0: dS_0 is in TMEM, dP_0 has been read
          if (!mbar_wait(smem_u32(&sm.p_full[0]), p_ph0, RA_DEV_TIMEOUT_MMA, abort_flag)) goto done;
          p_ph0 ^= 1;
          tc_fence_after();
          if (w == 0) {
            if (first) {
              if (!mbar_wait(smem_u32(&sm.acc_empty), acc_ph ^ 1, RA_DEV_TIMEOUT_MMA, abort_flag))
                goto done;
              tc_fence_after();
            }
            issue_half_accumulate<D>(tmem + kColAcc0, tmem + kColS, smem_u32(sm.k[cur]), 0, first);
          }
          if (more) {
            if (!mbar_wait(smem_u32(&sm.st_full[nst]), nph, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            tc_fence_after();
            issue_half_product_ta<D>(tmem + prod_col, a_op, prod_b(nst), 0);
            mma_commit(smem_u32(&sm.s_full[0]));
          }
          // half 1
          if (!mbar_wait(smem_u32(&sm.p_full[1]), p_ph1, RA_DEV_TIMEOUT_MMA, abort_flag)) goto done;
          p_ph1 ^= 1;
          tc_fence_after();
          if (w == 0)
            issue_half_accumulate<D>(tmem + kColAcc0, tmem + kColS + 64, smem_u32(sm.k[cur]), 1,
                                     false);
          mma_commit(smem_u32(&sm.st_empty[cur]));
          st = nst;
          st_ph = nph;
          first = false;
          if (!more) break;
          issue_half_product_ta<D>(tmem + prod_col + 64, a_op, prod_b(st), 1);
          mma_commit(smem_u32(&sm.s_full[1]));
        }
        if (w == 0) mma_commit(smem_u32(&sm.acc_full));
        acc_ph ^= 1;
      }
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- elementwise halves
    const int x = (warp - 4) / 4;                 // key-column half of S / dP
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;          // query row of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + kColS + 64 * x;
    const uint32_t t_dp = tmem + lane_addr + kColDP + 64 * x;
    // the A operand these warps keep in tensor memory: Q (half 0) or dO (half 1)
    const uint32_t t_a = tmem + lane_addr + (x == 0 ? kColQA : kColDOA);
    const uint8_t* a_src = x == 0 ? sm.q : sm.dO;
    const float sl2 = p.scale_log2;
    uint32_t s_ph = 0, acc_ph = 0, q_ph = 0;
    // The previous unit's dQ rows are stored after this unit's A operands are
    // in place, so the issuers start the next unit during that store.
    bool owed = false, owed_ok = false;
    int64_t owed_orow = 0;
    auto store_dq = [&]() {
      const uint32_t t_acc = tmem + lane_addr + kColAcc0 + x * (D / 2);
#pragma unroll
      for (int cch = 0; cch < D / 64; ++cch) {
        uint32_t r[32];
        tmem_ld32(t_acc + 32 * cch, r);
        tmem_wait_ld();
        if (owed_ok) {
          if constexpr (kMode == BWD_STEP)
            store_row32_f32(p.dq32 + owed_orow * D + x * (D / 2) + 32 * cch, r, p.scale,
                            p.accumulate != 0);
          else
            store_row32_bf16(p.dq + owed_orow * D + x * (D / 2) + 32 * cch, r, p.scale);
        }
      }
      tc_fence_before();
      mbar_arrive_warp(smem_u32(&sm.acc_empty));
    };
    for (int64_t k = 0;; ++k) {
      const int64_t item = item_at(k);
      if (item >= p.num_items) break;
      QUnit w;
      Geo gv;
      const Geo& g = qunit_get<kMode>(p, item, w, gv);
      const QTile qt = make_qtile(g, w.shard, w.seg, w.tile);
      if (!qt.valid) continue;
      KIterB it;
      kiterb_start<kMode>(p, g, it, w.shard, qt.qmax);
      if (!kiterb_next(g, it)) {
        // A hop's query tile that sees no key of block step_s: its rows of an
        // overwritten dq are zero (half x writes columns [x*D/2, (x+1)*D/2)).
        if constexpr (kMode == BWD_STEP) {
          if (!p.accumulate && row < qt.valid) {
            float* dst = p.dq32 +
                         (((int64_t)w.row_base + qt.local0 + qt.off + row) * g.H + w.h) * D +
                         x * (D / 2);
#pragma unroll
            for (int i = 0; i < D / 8; ++i)
              reinterpret_cast<float4*>(dst)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        continue;
      }
      const int qpos = qt.pos0 + qt.stride * (qt.off + row);
      const int64_t vi = w.vbase + vec_slab<kMode>(g, w.b, w.h, w.shard, w.seg, w.tile) * kTile + row;
      const float nl = __ldg(p.nlse2 + vi);
      const float nd = __ldg(p.ndelta + vi);
      const float2 sl2_2 = make_float2(sl2, sl2), nl2 = make_float2(nl, nl), nd2 = make_float2(nd, nd);
      // Every product of the previous unit has completed once its dQ has:
      // only then may this unit's A operands overwrite that unit's.
      if (owed) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.acc_full), acc_ph,
                                               RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
          goto done;
        acc_ph ^= 1;
        tc_fence_after();
      }
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.q_full), q_ph, RA_DEV_TIMEOUT_SOFTMAX,
                                             abort_flag)))
        goto done;
      q_ph ^= 1;
      tile_row_to_tmem<D>(a_src, row, t_a);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(smem_u32(&sm.qt_full));
      mbar_arrive_warp(smem_u32(&sm.q_empty));
      if (owed) store_dq();
      do {
        const int k0 = it.bt * kTile;
        const int kleft = it.seg.len - k0;
        const int kvalid = kleft < kTile ? kleft : kTile;
        int lim = kvalid;   // key columns at or beyond `lim` are masked out
        if (g.causal && it.seg.pos0 + it.seg.stride * (k0 + kvalid - 1) > qt.qmin) {
          const int cl = count_le(it.seg, qpos) - k0;
          lim = cl < 0 ? 0 : (cl > kvalid ? kvalid : cl);
        }
        const bool masked = __any_sync(0xffffffffu, lim < 64 * x + 64);
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[x]), s_ph,
                                               RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
          goto done;
        s_ph ^= 1;
        tc_fence_after();
        if (masked)
          dq_half<true>(t_s, t_dp, sl2_2, nl2, nd2, lim, 64 * x);
        else
          dq_half<false>(t_s, t_dp, sl2_2, nl2, nd2, lim, 64 * x);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&sm.p_full[x]));
        ++it.bt;
      } while (kiterb_next(g, it));
      // ---- epilogue (deferred): half x stores dq columns [x*D/2, (x+1)*D/2), times scale
      owed = true;
      owed_ok = row < qt.valid;
      owed_orow = kMode == BWD_STEP
                      ? ((int64_t)w.row_base + qt.local0 + qt.off + row) * g.H + w.h
                      : ((int64_t)w.row_base + qpos) * g.H + w.h;
    }
    if (owed) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.acc_full), acc_ph,
                                             RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
        goto done;
      acc_ph ^= 1;
      tc_fence_after();
      store_dq();
    }
  }

done:
  tc_fence_before();
  __syncthreads();
  if (sm.abort_flag) {
    // Let whatever this CTA issued before the failure land before its tensor
    // memory and shared memory go away: each issuer's products (a commit
    // arrives once all of them are done), and every TMA load of the producer
    // (the last phase armed on each full barrier; a barrier never armed
    // reports parity 1 complete at once).
    if ((warp == 1 || warp == 3) && lane == 0) {
      const int w = warp == 1 ? 0 : 1;
      mma_commit(smem_u32(&sm.drain[w]));
      mbar_wait_for(smem_u32(&sm.drain[w]), 0, RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
    }
    if (warp == 0 && lane == 0) {
      mbar_wait_for(smem_u32(&sm.q_full), tq_ph ^ 1, RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
      for (uint32_t i = 0; i < (uint32_t)kSt; ++i)
        mbar_wait_for(smem_u32(&sm.st_full[i]), i < tst ? tst_ph : tst_ph ^ 1,
                      RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace ra
