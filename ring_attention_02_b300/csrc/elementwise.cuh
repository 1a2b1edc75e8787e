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

// ---------------------------------------------------------------- merge
// (out_acc, lse_acc) <- fold of (out_part, lse_part), rows (b, j, h):
//   lse = max + ln(e^(l1 - max) + e^(l2 - max)),
//   out = e^(l1 - lse) out_acc + e^(l2 - lse) out_part.
// One row is handled by D/4 consecutive lanes of one warp (float4 each); the
// row's lse is read by all of them before lane 0 of the row writes it back.
template <int D>
__global__ void merge_kernel(float* __restrict__ out_acc, float* __restrict__ lse_acc,
                             const float* __restrict__ out_part,
                             const float* __restrict__ lse_part, int B, int H, int64_t n) {
  constexpr int kLanesPerRow = D / 4;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x % 32;
  const int sub = lane / kLanesPerRow;        // which row of the warp's group
  const int q4 = lane % kLanesPerRow;         // float4 index inside the row
  const int64_t rows = (int64_t)B * n * H;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  for (int64_t wr = warp0 * kRowsPerWarp; wr < rows; wr += warps_total * kRowsPerWarp) {
    const int64_t rrow = wr + sub;             // row index in [B][n][H] order
    const bool ok = rrow < rows;
    float l1 = -INFINITY, l2 = -INFINITY;
    int64_t li = 0;
    if (ok) {
      const int h = (int)(rrow % H);
      const int64_t j = (rrow / H) % n;
      const int b = (int)(rrow / ((int64_t)H * n));
      li = ((int64_t)b * H + h) * n + j;
      l1 = lse_acc[li];
      l2 = __ldg(lse_part + li);
    }
    __syncwarp();
    if (ok) {
      float4* oa = reinterpret_cast<float4*>(out_acc + rrow * D) + q4;
      const float4 op = __ldg(reinterpret_cast<const float4*>(out_part + rrow * D) + q4);
      if (l1 == -INFINITY && l2 == -INFINITY) {
        *oa = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        const float mx = fmaxf(l1, l2);
        const float lse = mx + logf(expf(l1 - mx) + expf(l2 - mx));
        const float w1 = expf(l1 - lse), w2 = expf(l2 - lse);
        float4 a = *oa;
        a.x = w1 * a.x + w2 * op.x;
        a.y = w1 * a.y + w2 * op.y;
        a.z = w1 * a.z + w2 * op.z;
        a.w = w1 * a.w + w2 * op.w;
        *oa = a;
        if (q4 == 0) lse_acc[li] = lse;
      }
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
