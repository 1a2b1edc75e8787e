// geometry.cuh -- shard layouts, tiles and the ring block schedule, as integer
// arithmetic shared by the kernels (device) and the launcher / census (host).
//
// A shard's local slots split into "segments": runs whose global positions
// form an arithmetic progression pos0 + stride * o, o < len.
//   contiguous: one segment, pos0 = r*n, stride 1, len n
//     ("Sequenzparallelitaet und Ringaufmerksamkeit", "Tiefer Einblick":
//      every GPU owns a contiguous run of tokens);
//   striped:    one segment, pos0 = r, stride P, len n
//     ("Zig Zag Ring Attention": GPU 0 takes tokens 0, 4, 8, ..., GPU 1 takes
//      1, 5, 9, ...);
//   zig-zag:    two segments, chunks r and 2P-1-r of C = S/(2P) tokens.
// Tiles are 128 consecutive slots of one segment and never straddle two, so
// every tile is one TMA box in natural order and its positions are affine.
// Tiles of a segment are grouped in pairs (tile 2p and 2p+1): one CTA work
// unit, two 128-row query tiles sharing every key/value tile it loads.
#pragma once
#include <cstdint>

namespace ra {

constexpr int kTile = 128;
enum { LAYOUT_CONTIGUOUS = 0, LAYOUT_STRIPED = 1, LAYOUT_ZIGZAG = 2 };

// Positions, lengths and offsets are int32: the host rejects B*S >= 2^31.
struct Geo {
  int B, H, Hkv, P, layout, causal;
  int S, n, C;
  int nseg;          // segments per shard (1, or 2 for zig-zag)
  int seglen;        // slots per segment
  int ntile;         // tiles per segment = ceil(seglen / 128)
  int npair;         // tile pairs per segment = ceil(ntile / 2)
};

struct Seg {
  int pos0, stride, len, local0;
};

__host__ __device__ inline Geo make_geo(int B, int H, int Hkv, int64_t S, int P, int layout,
                                        int causal) {
  Geo g;
  g.B = B; g.H = H; g.Hkv = Hkv; g.P = P; g.layout = layout; g.causal = causal;
  g.S = (int)S; g.n = (int)(S / P); g.C = (int)(S / (2 * (int64_t)P));
  g.nseg = layout == LAYOUT_ZIGZAG ? 2 : 1;
  g.seglen = layout == LAYOUT_ZIGZAG ? g.C : g.n;
  g.ntile = (g.seglen + kTile - 1) / kTile;
  g.npair = (g.ntile + 1) / 2;
  return g;
}

__host__ __device__ inline Seg segment_of(const Geo& g, int shard, int seg) {
  Seg s;
  if (g.layout == LAYOUT_ZIGZAG) {
    int chunk = seg == 0 ? shard : 2 * g.P - 1 - shard;
    s.pos0 = chunk * g.C; s.stride = 1; s.len = g.C; s.local0 = seg * g.C;
  } else if (g.layout == LAYOUT_STRIPED) {
    s.pos0 = shard; s.stride = g.P; s.len = g.n; s.local0 = 0;
  } else {
    s.pos0 = shard * g.n; s.stride = 1; s.len = g.n; s.local0 = 0;
  }
  return s;
}

// Number of slots of segment k whose position is <= x (positions increase
// along the segment, so these are its first count_le slots).
__host__ __device__ inline int count_le(const Seg& k, int x) {
  if (x < k.pos0) return 0;
  int c = (x - k.pos0) / k.stride + 1;
  return c < k.len ? c : k.len;
}

// Global position of a shard's local slot j (host/test helper).
__host__ __device__ inline int64_t position_of(const Geo& g, int shard, int64_t j) {
  int seg = (g.layout == LAYOUT_ZIGZAG && j >= g.C) ? 1 : 0;
  Seg s = segment_of(g, shard, seg);
  return (int64_t)s.pos0 + (int64_t)s.stride * (j - s.local0);
}

// One 128-slot query tile.
struct QTile {
  int valid;        // 0 if the tile does not exist, else number of rows (1..128)
  int shard;
  int off;          // first slot offset within the segment
  int pos0, stride, local0;
  int qmin, qmax;
};

__host__ __device__ inline QTile make_qtile(const Geo& g, int shard, int seg, int tile) {
  QTile q;
  q.shard = shard;
  Seg s = segment_of(g, shard, seg);
  q.off = tile * kTile;
  q.pos0 = s.pos0; q.stride = s.stride; q.local0 = s.local0;
  if (tile >= g.ntile || q.off >= s.len) {
    q.valid = 0; q.qmin = 0; q.qmax = -1;
    return q;
  }
  int rows = s.len - q.off;
  q.valid = rows < kTile ? rows : kTile;
  q.qmin = s.pos0 + s.stride * q.off;
  q.qmax = s.pos0 + s.stride * (q.off + q.valid - 1);
  return q;
}

// Work unit u (a tile pair) in longest-first order.  Ring mode: all shards;
// the unit whose query tiles hold the largest positions (the most visible
// keys under a causal mask) comes first.  Step mode: only shard r.
struct Unit {
  int shard, seg, pair;
};

__host__ __device__ inline int64_t units_total(const Geo& g, bool step_mode) {
  return (int64_t)(step_mode ? 1 : g.P) * g.nseg * g.npair;
}

__host__ __device__ inline Unit unit_of(const Geo& g, int64_t u, bool step_mode, int step_r) {
  Unit w;
  const int64_t np = g.npair;
  if (step_mode) {
    // descending position within shard step_r: last segment, last pair first
    int64_t k = u;
    w.shard = step_r;
    w.seg = g.nseg - 1 - (int)(k / np);
    w.pair = (int)(np - 1 - k % np);
    return w;
  }
  if (g.layout == LAYOUT_STRIPED) {
    w.pair = (int)(np - 1 - u / g.P);
    w.shard = g.P - 1 - (int)(u % g.P);
    w.seg = 0;
  } else if (g.layout == LAYOUT_ZIGZAG) {
    int64_t chunk = 2 * (int64_t)g.P - 1 - u / np;
    w.pair = (int)(np - 1 - u % np);
    if (chunk < g.P) { w.shard = (int)chunk; w.seg = 0; }
    else { w.shard = (int)(2 * (int64_t)g.P - 1 - chunk); w.seg = 1; }
  } else {
    w.shard = g.P - 1 - (int)(u / np);
    w.pair = (int)(np - 1 - u % np);
    w.seg = 0;
  }
  return w;
}

// Key blocks of a unit in ring order: step t = 0..P-1 holds the block of
// shard s = (r - t) mod P ("Tiefer Einblick": each device keeps its queries
// while the key/value blocks hop around the ring).  For each (t, segment) the
// key tiles that a causal mask leaves visible to a query at position <= qmax
// are a prefix of the segment's tiles: nk = ceil(count_le / 128).
__host__ __device__ inline int ring_block(const Geo& g, int r, int t) {
  int s = (r - t) % g.P;
  return s < 0 ? s + g.P : s;
}

__host__ __device__ inline int visible_tiles(const Geo& g, const Seg& k, int qmax) {
  int c = g.causal ? count_le(k, qmax) : k.len;
  return (c + kTile - 1) / kTile;
}

// Number of key tiles a query tile multiplies over the whole schedule
// (ring mode) or against block s only (step mode, s >= 0).
__host__ __device__ inline int tile_work(const Geo& g, const QTile& q, int step_s) {
  if (!q.valid) return 0;
  int total = 0;
  const int t_end = step_s >= 0 ? 1 : g.P;
  for (int t = 0; t < t_end; ++t) {
    int s = step_s >= 0 ? step_s : ring_block(g, q.shard, t);
    for (int sk = 0; sk < g.nseg; ++sk) total += visible_tiles(g, segment_of(g, s, sk), q.qmax);
  }
  return total;
}

// The work items CTA c of a G-CTA persistent grid takes, in order: its list in
// a host-built schedule (int32 offsets[G + 1], then CTA 0's item ids, CTA 1's,
// ...), or without one a snake over the item order (round k gives item
// k*G + c for even k, k*G + G-1-c for odd k).
struct CtaItems {
  const int* list;
  int64_t count, G, c;
};

#ifdef __CUDACC__
__device__ __forceinline__ CtaItems cta_items(const int* sched) {
  CtaItems w;
  w.G = gridDim.x;
  w.c = blockIdx.x;
  w.list = nullptr;
  w.count = 0;
  if (sched != nullptr) {
    const int a0 = __ldg(sched + w.c);
    w.list = sched + w.G + 1 + a0;
    w.count = __ldg(sched + w.c + 1) - a0;
  }
  return w;
}

// Item k of the CTA's sequence, or `none` past its end.
__device__ __forceinline__ int64_t cta_item(const CtaItems& w, int64_t k, int64_t none) {
  if (w.list != nullptr) return k < w.count ? (int64_t)__ldg(w.list + k) : none;
  return k * w.G + ((k & 1) ? (w.G - 1 - w.c) : w.c);
}
#endif

}  // namespace ra
