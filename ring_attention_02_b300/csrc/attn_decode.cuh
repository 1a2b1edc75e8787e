// attn_decode.cuh -- decode against a sharded key/value cache: T new query
// tokens (positions S-T .. S-1) attend to the S cached tokens, which the P
// virtual ring ranks hold under the shard layout.
//
// Method: the pages put ring attention to work for long-context inference
// ("Sequenzparallelitaet und Ringaufmerksamkeit", "Die Zukunft ..." and its
// use cases: ultra-long-context inference; the Chinese article on long-context
// inference: keep the history's keys and values in a cache and read them back
// instead of recomputing them).  Each rank computes the partial attention of
// the new queries against the cache block it holds, and the partials are
// combined with the online-softmax merge ("Tiefer Einblick").  Query t sees
// the keys at positions <= S - T + t.
//
// A decode step reads every cached key and value once and does only
// G * T multiply-adds per key element (G = H / Hkv query heads per key/value
// head), so it is bound by HBM bandwidth; the key/value tiles are staged into
// shared memory by TMA, three tiles in flight per CTA.
//
//   decode_partial_kernel  one CTA per (chunk of 128-slot tiles of one shard
//                          segment, b, kv head, group of 16 of the kv head's
//                          G*T query rows, the last padded); four
//                          warps, each with 32 keys of every tile and its own
//                          online softmax, merged at the end; writes a
//                          normalised partial and its lse.
//   decode_combine_kernel  LSE merge of a row's partials.
// The two small products per tile (16 rows x 32 keys x D, and back) use the
// warp-level mma.sync path with ldmatrix from the TMA-swizzled tiles: a few
// dozen instructions per warp where CUDA-core FMAs would need thousands.
#pragma once
#include "geometry.cuh"
#include "sm103_ptx.cuh"

namespace ra {

constexpr int kDecodeMaxRows = 16;   // query rows per CTA (one row group)
constexpr int kDecodeStages = 3;     // key/value tiles in flight per CTA

struct DecodeParams {
  Geo g;
  int T;               // new query tokens
  int rows;            // G * T
  int chunk_tiles;     // tiles per chunk
  int chunks_per_seg;  // ceil(ntile / chunk_tiles)
  float scale_log2;
  const __nv_bfloat16* q;   // [B][T][H][D]
  float* part_o;            // [B*Hkv][chunks][rows][D]
  float* part_lse;          // [B*Hkv][chunks][rows]
  int chunks;               // chunks per (b, kv head) = P * nseg * chunks_per_seg
  int row_groups;           // ceil(rows / kDecodeMaxRows): CTAs per chunk
};

template <int D>
struct __align__(1024) DecodeSmem {
  uint8_t k[kDecodeStages][kTile * D * 2];
  uint8_t v[kDecodeStages][kTile * D * 2];
  float q[kDecodeMaxRows][D];
  float sp[kDecodeMaxRows][kTile];      // scores, then probabilities, of one tile
  float m[kDecodeMaxRows], l[kDecodeMaxRows], corr[kDecodeMaxRows];
  uint64_t full[kDecodeStages];
};

// Byte offset of element d of row r in a 128 x D bf16 tile laid out by TMA
// with 128-byte swizzle: D/64 sub-tiles of 128 rows x 128 bytes; the 16-byte
// chunk c of row r sits at chunk position c ^ (r % 8).
template <int D>
__device__ __forceinline__ uint32_t sw128_offset(int r, int d) {
  const int sub = d / 64, dd = d % 64;
  const int c = dd / 8;
  return sub * (kTile * 128) + r * 128 + ((c ^ (r & 7)) << 4) + (dd % 8) * 2;
}

constexpr int kDecodeThreads = 128;   // 4 warps; warp w owns keys [32w, 32w+32) of each tile

// ---- legacy warp-level tensor-core pieces (m16n8k16, bf16 in, fp32 accumulate)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <int D>
__global__ void __launch_bounds__(kDecodeThreads)
decode_partial_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  DecodeSmem<D>& sm = *reinterpret_cast<DecodeSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Geo& g = p.g;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // the combine kernel that follows may be scheduled now: it waits for this
  // grid to complete before reading the partials
  griddep_launch_dependents();
  const int G = g.H / g.Hkv;
  const int bk = blockIdx.y;
  const int b = bk / g.Hkv, hkv = bk % g.Hkv;
  // the row groups of one chunk are adjacent in the grid, so they run side by
  // side and share the chunk's key/value tiles in L2
  const int chunk = blockIdx.x / p.row_groups;
  const int rg0 = (blockIdx.x % p.row_groups) * kDecodeMaxRows;   // first row of this group
  // chunk -> (shard, segment, tile range)
  const int rs = chunk / p.chunks_per_seg;
  const int shard = rs / g.nseg, seg = rs % g.nseg;
  const Seg sg = segment_of(g, shard, seg);
  const int a0 = (chunk % p.chunks_per_seg) * p.chunk_tiles;
  int a1 = a0 + p.chunk_tiles;
  if (a1 > g.ntile) a1 = g.ntile;
  const int ntiles = a1 > a0 ? a1 - a0 : 0;
  const int R = p.rows;

  if (tid == 0) {
    for (int s = 0; s < kDecodeStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
  }
  // query rows i = e * T + t (head hkv*G + e, token t) of this row group;
  // rows >= R are zero
  for (int idx = tid; idx < kDecodeMaxRows * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    float v = 0.f;
    if (rg0 + i < R) {
      const int e = (rg0 + i) / p.T, t = (rg0 + i) % p.T;
      v = __bfloat162float(p.q[(((int64_t)b * p.T + t) * g.H + hkv * G + e) * D + d]);
    }
    sm.q[i][d] = v;
  }
  __syncthreads();

  auto issue = [&](int it) {
    const int st = it % kDecodeStages;
    const uint32_t bar = smem_u32(&sm.full[st]);
    mbar_arrive_expect_tx(bar, 2 * kTile * D * 2);
    const int off = (a0 + it) * kTile;
    int phase, row;
    if (g.layout == LAYOUT_STRIPED) {
      phase = shard;
      row = b * g.n + off;
    } else {
      phase = 0;
      row = b * g.S + sg.pos0 + off;
    }
#pragma unroll
    for (int s2 = 0; s2 < D / 64; ++s2) {
      tma_load_4d(smem_u32(sm.k[st]) + s2 * (kTile * 128), &tm_k, bar, 64 * s2, hkv, phase, row,
                  policy_evict_first());
      tma_load_4d(smem_u32(sm.v[st]) + s2 * (kTile * 128), &tm_v, bar, 64 * s2, hkv, phase, row,
                  policy_evict_first());
    }
  };
  if (tid == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int it = 0; it < kDecodeStages - 1 && it < ntiles; ++it) issue(it);
  }

  // Q as A fragments (16 rows x D), once: a0/a1 rows r0 / r0+8, a2/a3 columns +8
  const int r0 = lane / 4, cq = (lane % 4) * 2;
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    qa[ks][0] = pack_bf16x2(sm.q[r0][16 * ks + cq], sm.q[r0][16 * ks + cq + 1]);
    qa[ks][1] = pack_bf16x2(sm.q[r0 + 8][16 * ks + cq], sm.q[r0 + 8][16 * ks + cq + 1]);
    qa[ks][2] = pack_bf16x2(sm.q[r0][16 * ks + 8 + cq], sm.q[r0][16 * ks + 8 + cq + 1]);
    qa[ks][3] = pack_bf16x2(sm.q[r0 + 8][16 * ks + 8 + cq], sm.q[r0 + 8][16 * ks + 8 + cq + 1]);
  }
  // the token each of this lane's two rows belongs to (rows >= R: none)
  const int qpos0 = g.S - p.T;
  const int lim0 = rg0 + r0 < R ? qpos0 + (rg0 + r0) % p.T : -1;   // last visible position
  const int lim1 = rg0 + r0 + 8 < R ? qpos0 + (rg0 + r0 + 8) % p.T : -1;
  float o[D / 8][4];                                       // O fragments: n-tile j = d [8j, 8j+8)
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // log2 units
  const float sl2 = p.scale_log2;

  bool ok = true;
  int failed_at = ntiles;   // the tile whose wait gave up, if one did
  for (int it = 0; it < ntiles; ++it) {
    const int st = it % kDecodeStages;
    if (tid == 0 && it + kDecodeStages - 1 < ntiles) issue(it + kDecodeStages - 1);
    ok = mbar_wait(smem_u32(&sm.full[st]), (it / kDecodeStages) & 1, RA_DEV_TIMEOUT_TMA, nullptr);
    if (!__syncthreads_and(ok)) {
      ok = false;
      failed_at = it;
      break;
    }
    const uint32_t kb = smem_u32(sm.k[st]), vb = smem_u32(sm.v[st]);
    const int kw = 32 * warp;                               // this warp's first key slot
    // ---- S = Q K^T for the warp's 32 keys: 4 n-tiles of 8 keys
    float sacc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        // matrices: (keys +0..7, d lo), (keys +0..7, d hi), (keys +8..15, d lo), (keys +8..15, d hi)
        const int key = kw + 16 * jj + (lane & 7) + ((lane >> 4) << 3);
        const int d = 16 * ks + ((lane >> 3) & 1) * 8;
        uint32_t bf[4];
        ldsm_x4(kb + sw128_offset<D>(key, d), bf);
        mma16816(sacc[2 * jj], qa[ks], bf[0], bf[1]);
        mma16816(sacc[2 * jj + 1], qa[ks], bf[2], bf[3]);
      }
    }
    // ---- mask, online softmax (log2 units) over the warp's keys
    const int off = (a0 + it) * kTile;
    float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int slot = off + kw + 8 * j + cq + c;
        const int kpos = sg.pos0 + sg.stride * slot;
        const bool valid = slot < sg.len;
        sacc[j][c] = (valid && kpos <= lim0) ? sacc[j][c] * sl2 : -INFINITY;
        sacc[j][2 + c] = (valid && kpos <= lim1) ? sacc[j][2 + c] * sl2 : -INFINITY;
        mt0 = fmaxf(mt0, sacc[j][c]);
        mt1 = fmaxf(mt1, sacc[j][2 + c]);
      }
    }
#pragma unroll
    for (int o2 = 1; o2 < 4; o2 *= 2) {
      mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, o2));
      mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, o2));
    }
    const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float c0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - base0);
    const float c1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    l0 *= c0;
    l1 *= c1;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      o[j][0] *= c0; o[j][1] *= c0;
      o[j][2] *= c1; o[j][3] *= c1;
    }
    uint32_t pa[2][4];                                      // P as A fragments, 2 k-steps of 16 keys
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float p0 = ex2_approx(sacc[j][0] - base0), p1 = ex2_approx(sacc[j][1] - base0);
      const float p2 = ex2_approx(sacc[j][2] - base1), p3 = ex2_approx(sacc[j][3] - base1);
      l0 += p0 + p1;
      l1 += p2 + p3;
      pa[j / 2][(j % 2) * 2 + 0] = pack_bf16x2(p0, p1);
      pa[j / 2][(j % 2) * 2 + 1] = pack_bf16x2(p2, p3);
    }
    // ---- O += P V over the warp's 32 keys: V fragments transposed from the swizzled tile
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int nd = 0; nd < D / 16; ++nd) {
        // matrices: (keys +0..7, d 16nd..+7), (keys +8..15, same d), (keys +0..7, d +8), (keys +8..15, d +8)
        const int key = kw + 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int d = 16 * nd + ((lane >> 4) << 3);
        uint32_t bf[4];
        ldsm_x4_t(vb + sw128_offset<D>(key, d), bf);
        mma16816(o[2 * nd], pa[ks], bf[0], bf[1]);
        mma16816(o[2 * nd + 1], pa[ks], bf[2], bf[3]);
      }
    }
    // every warp is done with stage st before it is refilled
    __syncthreads();
  }
  if (!ok) {
    // A wait gave up (status already recorded): the tiles issued from
    // failed_at on may still be landing.  Wait for each on its own barrier
    // before the shared memory is reused or given up, then report an empty
    // partial.
    if (tid == 0) {
      const int issued = failed_at + kDecodeStages < ntiles ? failed_at + kDecodeStages : ntiles;
      for (int j = failed_at; j < issued; ++j)
        mbar_wait_for(smem_u32(&sm.full[j % kDecodeStages]), (j / kDecodeStages) & 1,
                      RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
    }
    __syncthreads();
  }
  // ---- merge the four warps: rows' (m, l) and O through shared memory
#pragma unroll
  for (int o2 = 1; o2 < 4; o2 *= 2) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
  }
  __syncthreads();   // stage buffers are free: reuse them for the four warps' O
  float* ow = reinterpret_cast<float*>(sm.k[0]) + warp * (kDecodeMaxRows * D);
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    ow[r0 * D + 8 * j + cq] = o[j][0];
    ow[r0 * D + 8 * j + cq + 1] = o[j][1];
    ow[(r0 + 8) * D + 8 * j + cq] = o[j][2];
    ow[(r0 + 8) * D + 8 * j + cq + 1] = o[j][3];
  }
  if ((lane & 3) == 0) {
    sm.sp[r0][warp] = m0;
    sm.sp[r0][4 + warp] = l0;
    sm.sp[r0 + 8][warp] = m1;
    sm.sp[r0 + 8][4 + warp] = l1;
  }
  __syncthreads();
  const float* o_all = reinterpret_cast<const float*>(sm.k[0]);
  const int64_t cbase = (int64_t)bk * p.chunks + chunk;
  const int Rg = R - rg0 < kDecodeMaxRows ? R - rg0 : kDecodeMaxRows;   // rows of this group
  for (int idx = tid; idx < Rg * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < 4; ++w2) M = fmaxf(M, sm.sp[i][w2]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w2 = 0; w2 < 4; ++w2) {
        const float mw = sm.sp[i][w2];
        const float f = mw == -INFINITY ? 0.f : ex2_approx(mw - M);
        L += f * sm.sp[i][4 + w2];
        acc += f * o_all[(w2 * kDecodeMaxRows + i) * D + d];
      }
    }
    const bool has = ok && L > 0.f;
    p.part_o[(cbase * R + rg0 + i) * D + d] = has ? acc / L : 0.f;
    if (d == 0)
      p.part_lse[cbase * R + rg0 + i] = has ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
}

// out[b][t][h][:] and lse[b][h][t] from the partials of row i = e*T + t of
// (b, kv head), h = hkv*G + e: one CTA (16 warps) per row; the warps split the
// partials, first for the maximum lse, then for the weighted sum (unrolled so
// several partials' loads are in flight per warp).
constexpr int kCombineWarps = 16;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                      void* out, int out_f32, float* lse, Geo g, int T, int rows, int chunks) {
  constexpr int kPer = D / 32;
  __shared__ float red[kCombineWarps][D + 2];
  // launched to overlap the partial kernel's end: its partials are complete
  // and visible only after this
  griddep_wait();
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int item = blockIdx.x;                 // (bk, i)
  const int i = item % rows, bk = item / rows;
  const int64_t pbase = (int64_t)bk * chunks * rows + i;   // partial c at pbase + c * rows
  float m = -INFINITY;
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) m = fmaxf(m, __ldg(part_lse + pbase + (int64_t)c * rows));
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 /= 2) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o2));
  if (lane == 0) red[warp][D] = m;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w2 = 0; w2 < kCombineWarps; ++w2) M = fmaxf(M, red[w2][D]);
  float acc[kPer], s = 0.f;
#pragma unroll
  for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int c = warp; c < chunks; c += kCombineWarps) {
      const int64_t pi = pbase + (int64_t)c * rows;
      const float l = __ldg(part_lse + pi);
      const float w = l == -INFINITY ? 0.f : expf(l - M);
      const float* po = part_o + pi * D;
#pragma unroll
      for (int j = 0; j < kPer; ++j) acc[j] = fmaf(w, __ldg(po + lane + 32 * j), acc[j]);
      s += w;
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPer; ++j) red[warp][lane + 32 * j] = acc[j];
  if (lane == 0) red[warp][D + 1] = s;
  __syncthreads();
  if (warp == 0) {
    float S = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kCombineWarps; ++w2) S += red[w2][D + 1];
    const int b = bk / g.Hkv, hkv = bk % g.Hkv;
    const int G = g.H / g.Hkv;
    const int e = i / T, t = i % T;
    const int h = hkv * G + e;
    const float inv = S > 0.f ? 1.f / S : 0.f;
    const int64_t orow = ((int64_t)b * T + t) * g.H + h;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      float v = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kCombineWarps; ++w2) v += red[w2][lane + 32 * j];
      v *= inv;
      if (out_f32)
        static_cast<float*>(out)[orow * D + lane + 32 * j] = v;
      else
        static_cast<__nv_bfloat16*>(out)[orow * D + lane + 32 * j] = __float2bfloat16_rn(v);
    }
    if (lse != nullptr && lane == 0)
      lse[((int64_t)b * g.H + h) * T + t] = S > 0.f ? M + logf(S) : -INFINITY;
  }
}

}  // namespace ra
