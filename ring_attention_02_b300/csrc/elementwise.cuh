// elementwise.cuh -- the HBM-bound kernels: layout permutation and the merge
// of two partial results.
#pragma once
#include <cuda_runtime.h>
#include "geometry.cuh"
#include "sm103_ptx.cuh"

namespace ra {

// ---------------------------------------------------------------- permute
// dst[o][r*n + j] = src[o][pos_r(j)]  (gather, inverse = 0) or the scatter back.
// Each thread moves one VEC-byte piece of a row; consecutive threads move
// consecutive pieces, so reads and writes stay coalesced along a row.
template <typename VEC>
__global__ void permute_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                               int64_t outer, Geo g, int64_t row_bytes, int inverse) {
  const int64_t per_row = row_bytes / (int64_t)sizeof(VEC);
  const int64_t total = outer * g.S * per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t piece = idx % per_row;
    const int64_t slot_all = idx / per_row;       // o * S + slot
    const int64_t o = slot_all / g.S;
    const int64_t slot = slot_all % g.S;
    const int shard = (int)(slot / g.n);
    const int64_t pos = position_of(g, shard, slot % g.n);
    const int64_t from = inverse ? slot : pos;
    const int64_t to = inverse ? pos : slot;
    const VEC* s = reinterpret_cast<const VEC*>(src + (o * g.S + from) * row_bytes) + piece;
    VEC* d = reinterpret_cast<VEC*>(dst + (o * g.S + to) * row_bytes) + piece;
    *d = __ldg(s);
  }
}

// ---------------------------------------------------------------- shard-outer permute
// dst[r][o][j] = src[o][pos_r(j)]  (gather, inverse = 0) or the scatter back:
// the rows of every shard r gathered into one contiguous block per shard, with
// the `outer` slabs inside it.  This is the order an all-to-all exchanges
// (block r goes to, or came from, rank r).  Pieces are walked in shard-outer
// order, so the shard side is read or written contiguously.
template <typename VEC>
__global__ void permute_shards_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                      int64_t outer, Geo g, int64_t row_bytes, int inverse) {
  const int64_t per_row = row_bytes / (int64_t)sizeof(VEC);
  const int64_t total = outer * g.S * per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t piece = idx % per_row;
    int64_t t = idx / per_row;
    const int64_t j = t % g.n;
    t /= g.n;
    const int64_t o = t % outer;
    const int shard = (int)(t / outer);
    const int64_t pos = position_of(g, shard, j);
    const int64_t shard_row = ((int64_t)shard * outer + o) * g.n + j;
    const int64_t nat_row = o * g.S + pos;
    const int64_t from = inverse ? shard_row : nat_row;
    const int64_t to = inverse ? nat_row : shard_row;
    const VEC* s = reinterpret_cast<const VEC*>(src + from * row_bytes) + piece;
    VEC* d = reinterpret_cast<VEC*>(dst + to * row_bytes) + piece;
    *d = __ldg(s);
  }
}

// ---------------------------------------------------------------- head split
// dst[p][row] = src[row][p] (inverse = 0) or dst[row][p] = src[p][row], for
// `rows` rows of `parts` chunks of chunk_bytes each: a [B][n][H][D] tensor
// viewed as rows = B*n of H/parts-head chunks becomes one block per head
// group (the block sent to rank p), and back.
template <typename VEC>
__global__ void head_split_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                  int64_t rows, int parts, int64_t chunk_bytes, int inverse) {
  const int64_t per_chunk = chunk_bytes / (int64_t)sizeof(VEC);
  const int64_t total = rows * parts * per_chunk;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t piece = idx % per_chunk;
    const int64_t t = idx / per_chunk;
    const int64_t row = t % rows;
    const int64_t part = t / rows;
    const int64_t split = (part * rows + row) * per_chunk + piece;
    const int64_t merged = (row * parts + part) * per_chunk + piece;
    const VEC* s = reinterpret_cast<const VEC*>(src);
    VEC* d = reinterpret_cast<VEC*>(dst);
    if (inverse) d[merged] = __ldg(s + split);
    else d[split] = __ldg(s + merged);
  }
}

// ---------------------------------------------------------------- finalize
// out = bf16(acc): the ring's fp32 accumulator stored in the output type once
// the last block has been folded in.  Four values per thread step.
__global__ void finalize_bf16_kernel(const float4* __restrict__ acc, uint2* __restrict__ out,
                                     int64_t quads) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < quads; i += stride) {
    const float4 v = __ldg(acc + i);
    out[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

// ---------------------------------------------------------------- cache append
// cache[b][pos + t][:] = fresh[b][t][:] for the keys and the values of T new
// tokens (rows of `row` 16-byte vectors): the step that keeps the history's
// keys and values in the cache for the next decode.  blockIdx.y selects the
// tensor (0: keys, 1: values).
__global__ void cache_append_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                    const uint4* __restrict__ k_new,
                                    const uint4* __restrict__ v_new, int64_t B, int64_t S_cap,
                                    int64_t pos, int64_t T, int64_t row) {
  uint4* dst = blockIdx.y == 0 ? k_cache : v_cache;
  const uint4* src = blockIdx.y == 0 ? k_new : v_new;
  const int64_t total = B * T * row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t piece = idx % row;
    const int64_t bt = idx / row;
    const int64_t t = bt % T, b = bt / T;
    dst[(b * S_cap + pos + t) * row + piece] = __ldg(src + idx);
  }
}

// ---------------------------------------------------------------- merge
// (out_acc, lse_acc) <- fold of (out_part, lse_part) for rows (b, t, h):
//   lse = max + ln(e^(l1 - max) + e^(l2 - max)),
//   out = e^(l1 - lse) out_acc + e^(l2 - lse) out_part.
// A CTA takes a tile of kMergeTok consecutive tokens of one batch entry, all
// H heads.  It first folds the tile's lse values, head by head: kMergeTok
// consecutive floats of [B][H][n], one 32-byte sector per head, read and
// written once by this CTA, with the two weights of each row kept in shared
// memory.  Then it streams the tile's out rows, which are one contiguous run
// of kMergeTok * H * D floats in [B][n][H][D], four float4 of each tensor in
// flight per thread.  (A row-by-row order made every lse sector a read and a
// write from eight different CTAs: 69 % of the measured HBM rate on the
// 32-head shard against 90 % for this order.)
constexpr int kMergeTok = 8;
constexpr int kMergeThreads = 512;
constexpr int kMergeUnroll = 4;

template <int D>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(float* __restrict__ out_acc, float* __restrict__ lse_acc,
             const float* __restrict__ out_part, const float* __restrict__ lse_part, int B, int H,
             int n) {
  extern __shared__ float merge_w[];         // [2][H * kMergeTok]: the rows' two weights
  float* w1s = merge_w;
  float* w2s = merge_w + H * kMergeTok;
  constexpr int kQ = D / 4;                  // float4 per row
  const int tiles_per_b = (n + kMergeTok - 1) / kMergeTok;
  const int64_t tiles = (int64_t)B * tiles_per_b;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int b = (int)(tile / tiles_per_b);
    const int t0 = (int)(tile % tiles_per_b) * kMergeTok;
    const int nt = n - t0 < kMergeTok ? n - t0 : kMergeTok;
    for (int i = threadIdx.x; i < H * kMergeTok; i += kMergeThreads) {
      const int h = i / kMergeTok, t = i % kMergeTok;
      float w1 = 0.f, w2 = 0.f;
      if (t < nt) {
        const int64_t li = ((int64_t)b * H + h) * n + t0 + t;
        const float l1 = lse_acc[li], l2 = __ldg(lse_part + li);
        if (!(l1 == -INFINITY && l2 == -INFINITY)) {
          const float mx = fmaxf(l1, l2);
          const float lse = mx + logf(expf(l1 - mx) + expf(l2 - mx));
          w1 = expf(l1 - lse);
          w2 = expf(l2 - lse);
          lse_acc[li] = lse;
        }
      }
      w1s[i] = w1;
      w2s[i] = w2;
    }
    __syncthreads();
    const int64_t base = ((int64_t)b * n + t0) * H * kQ;
    const int q4n = nt * H * kQ;
    float4* oa = reinterpret_cast<float4*>(out_acc) + base;
    const float4* op = reinterpret_cast<const float4*>(out_part) + base;
    for (int j0 = threadIdx.x; j0 < q4n; j0 += kMergeThreads * kMergeUnroll) {
      float4 a[kMergeUnroll], c[kMergeUnroll];
#pragma unroll
      for (int u = 0; u < kMergeUnroll; ++u) {
        const int j = j0 + u * kMergeThreads;
        if (j < q4n) {
          a[u] = oa[j];
          c[u] = __ldg(op + j);
        }
      }
#pragma unroll
      for (int u = 0; u < kMergeUnroll; ++u) {
        const int j = j0 + u * kMergeThreads;
        if (j < q4n) {
          const int row = j / kQ;                 // t * H + h within the tile
          const int wi = (row % H) * kMergeTok + row / H;
          const float w1 = w1s[wi], w2 = w2s[wi];
          float4 o;
          o.x = w1 * a[u].x + w2 * c[u].x;
          o.y = w1 * a[u].y + w2 * c[u].y;
          o.z = w1 * a[u].z + w2 * c[u].z;
          o.w = w1 * a[u].w + w2 * c[u].w;
          oa[j] = o;
        }
      }
    }
    __syncthreads();   // the weights are rewritten for the next tile
  }
}

// ---------------------------------------------------------------- wait self-check
// One thread waits on an mbarrier that nothing ever arrives on, with the same
// bounded wait the kernels use but a caller-chosen limit: the wait gives up,
// records RA_DEV_TIMEOUT_SELFCHECK in the device status word and the kernel
// returns, leaving the context usable.  *waited_ns receives the time spent.
__global__ void wait_selfcheck_kernel(unsigned long long limit_ns, unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  const unsigned long long t0 = globaltimer();
  const bool ok = mbar_wait_for(b, 0, RA_DEV_TIMEOUT_SELFCHECK, limit_ns);
  *waited_ns = ok ? 0ull : globaltimer() - t0;
}

}  // namespace ra
