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
// (out_acc, lse_acc) <- fold of (out_part, lse_part), rows (b, j, h):
//   lse = max + ln(e^(l1 - max) + e^(l2 - max)),
//   out = e^(l1 - lse) out_acc + e^(l2 - lse) out_part.
// One row is handled by D/4 consecutive lanes of one warp (float4 each).  A
// warp takes kMergeUnroll groups of rows per step and issues every load of the
// step (both lse values and both float4 of each row) before it uses any, so a
// step costs one memory round trip instead of two per row.  The row's lse is
// read by all its lanes before lane 0 of the row writes it back (__syncwarp).
// Idx is uint32_t when B * n * H fits, uint64_t otherwise.
constexpr int kMergeUnroll = 4;
constexpr int kMergeThreads = 256;

template <int D, typename Idx>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(float* __restrict__ out_acc, float* __restrict__ lse_acc,
             const float* __restrict__ out_part, const float* __restrict__ lse_part, Idx H, Idx n,
             Idx rows) {
  constexpr int kLanesPerRow = D / 4;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  constexpr int kRowsPerStep = kRowsPerWarp * kMergeUnroll;
  const int lane = threadIdx.x % 32;
  const int sub = lane / kLanesPerRow;        // which row of the warp's group
  const int q4 = lane % kLanesPerRow;         // float4 index inside the row
  const Idx warps_total = (Idx)gridDim.x * (kMergeThreads / 32);
  const Idx warp0 = (Idx)blockIdx.x * (kMergeThreads / 32) + threadIdx.x / 32;
  for (Idx base = warp0 * kRowsPerStep; base < rows; base += warps_total * kRowsPerStep) {
    float l1[kMergeUnroll], l2[kMergeUnroll];
    float4 oa[kMergeUnroll], op[kMergeUnroll];
    Idx li[kMergeUnroll];
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const Idx r = base + (Idx)(u * kRowsPerWarp + sub);   // row index in [B][n][H] order
      l1[u] = -INFINITY;
      l2[u] = -INFINITY;
      li[u] = 0;
      if (r < rows) {
        const Idx h = r % H, t = r / H;
        li[u] = (t / n * H + h) * n + t % n;
        l1[u] = lse_acc[li[u]];
        l2[u] = __ldg(lse_part + li[u]);
        oa[u] = reinterpret_cast<const float4*>(out_acc + (uint64_t)r * D)[q4];
        op[u] = __ldg(reinterpret_cast<const float4*>(out_part + (uint64_t)r * D) + q4);
      }
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const Idx r = base + (Idx)(u * kRowsPerWarp + sub);
      if (r >= rows) continue;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      const bool empty = l1[u] == -INFINITY && l2[u] == -INFINITY;
      if (!empty) {
        const float mx = fmaxf(l1[u], l2[u]);
        const float lse = mx + logf(expf(l1[u] - mx) + expf(l2[u] - mx));
        const float w1 = expf(l1[u] - lse), w2 = expf(l2[u] - lse);
        o.x = w1 * oa[u].x + w2 * op[u].x;
        o.y = w1 * oa[u].y + w2 * op[u].y;
        o.z = w1 * oa[u].z + w2 * op[u].z;
        o.w = w1 * oa[u].w + w2 * op[u].w;
        if (q4 == 0) lse_acc[li[u]] = lse;
      }
      reinterpret_cast<float4*>(out_acc + (uint64_t)r * D)[q4] = o;
    }
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
