// attn_fwd.cuh -- the forward kernel: blockwise attention over the ring block
// schedule with online softmax, on tcgen05 tensor cores (sm_103a).
//
// Method ("Sequenzparallelitaet und Ringaufmerksamkeit", "Tiefer Einblick";
// Thai edition, "technical insight"): each query shard stays put while the
// key/value blocks of the ring arrive one by one; for every block the partial
// attention is computed and folded into a running maximum m and normaliser l,
// the earlier partial sums rescaled when the maximum grows.  Causal masking
// compares global positions ("Zig Zag Ring Attention").
//
// One persistent CTA per SM.  A work unit is a pair of 128-row query tiles of
// one shard (plus batch b and head h); both tiles share every K/V tile loaded.
// Roles (384 threads):
//   warp 0       TMA producer: Q tiles once per unit, K and V tiles through a
//                ring of shared-memory stages (mbarrier full/empty pairs);
//   warp 1       MMA issuer: S_x = Q_x K^T (both operands in shared memory)
//                and O_x += P_x V (P read from tensor memory), tcgen05.mma
//                issued by one thread, completion signalled by tcgen05.commit;
//                the whole warp owns the TMEM allocation;
//   warps 4..7   softmax of query tile A, one row per thread;
//   warps 8..11  softmax of query tile B.
// The two softmax warpgroups ping-pong: while one turns S into P the tensor
// core runs the other tile's P V and next Q K^T.
//
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+D),
// O_B [384,384+D).  P (bf16, two per column) overwrites the first 64 columns
// of its S region after the softmax has read S into registers; the next
// Q K^T into that region is issued after the P V that reads it, and tcgen05
// MMAs of one thread execute in issue order.
//
// Lazy rescaling: a row keeps its running maximum until a tile raises it by
// more than 8 (log2 units); P entries then stay below 2^8, and the final O / l
// uses the same maximum in numerator and denominator, so the result is exact.
#pragma once
#include "geometry.cuh"
#include "sm103_ptx.cuh"

namespace ra {

enum { FWD_MODE_RING = 0, FWD_MODE_STEP = 1 };

struct FwdParams {
  Geo g;
  int mode;            // FWD_MODE_RING: natural-order tensors, all blocks in ring order
                       // FWD_MODE_STEP: shard-local tensors, one block step_s
  int step_r, step_s;
  float scale_log2;    // scale * log2(e)
  void* out;           // bf16 or fp32
  int out_f32;
  float* lse;          // may be null
  unsigned long long* shard_tiles;  // may be null: per-shard count of multiplied tile pairs
  int64_t num_items;
};

template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;       // one 128 x D bf16 tile
  static constexpr int kSubTiles = D / 64;                // 128-byte-wide TMA boxes per tile
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kThreads = 384;
};

// TMEM column of S_x and of O_x (x = 0: query tile A, 1: tile B).
__device__ __forceinline__ uint32_t col_s(int x) { return 128u * x; }
__device__ __forceinline__ uint32_t col_o(int x) { return 256u + 128u * x; }

template <int D>
struct __align__(1024) FwdSmem {
  uint8_t q[2][FwdCfg<D>::kTileBytes];
  uint8_t k[FwdCfg<D>::kKStages][FwdCfg<D>::kTileBytes];
  uint8_t v[FwdCfg<D>::kVStages][FwdCfg<D>::kTileBytes];
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[FwdCfg<D>::kKStages], k_empty[FwdCfg<D>::kKStages];
  uint64_t v_full[FwdCfg<D>::kVStages], v_empty[FwdCfg<D>::kVStages];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Per-unit schedule facts every role derives identically.
struct UnitInfo {
  int b, h, hkv;
  QTile qt[2];
  int64_t qmax;        // largest query position of the unit
  int ntiles[2];       // active key tiles per query tile
};

__device__ __forceinline__ UnitInfo unit_info(const FwdParams& p, int64_t item) {
  UnitInfo ui;
  const Geo& g = p.g;
  const int64_t bh = item % ((int64_t)g.B * g.H);
  const int64_t u = item / ((int64_t)g.B * g.H);
  ui.b = (int)(bh / g.H);
  ui.h = (int)(bh % g.H);
  ui.hkv = ui.h / (g.H / g.Hkv);
  const bool step = p.mode == FWD_MODE_STEP;
  Unit w = unit_of(g, u, step, p.step_r);
  ui.qt[0] = make_qtile(g, w.shard, w.seg, 2 * w.pair);
  ui.qt[1] = make_qtile(g, w.shard, w.seg, 2 * w.pair + 1);
  ui.qmax = ui.qt[1].valid ? ui.qt[1].qmax : ui.qt[0].qmax;
  if (ui.qt[0].valid && ui.qt[0].qmax > ui.qmax) ui.qmax = ui.qt[0].qmax;
  for (int x = 0; x < 2; ++x) ui.ntiles[x] = (int)tile_work(g, ui.qt[x], step ? p.step_s : -1);
  return ui;
}

// Iterator over the union of key tiles of a unit, in ring order.
struct KIter {
  int t, t_end, sk, bt, nk;
  int s;
  Seg seg;
};

__device__ __forceinline__ void kiter_setup(const FwdParams& p, const UnitInfo& ui, KIter& it) {
  it.t = 0;
  it.t_end = p.mode == FWD_MODE_STEP ? 1 : p.g.P;
  it.sk = 0;
  it.bt = 0;
  it.s = p.mode == FWD_MODE_STEP ? p.step_s : ring_block(p.g, ui.qt[0].shard, 0);
  it.seg = segment_of(p.g, it.s, 0);
  it.nk = visible_tiles(p.g, it.seg, ui.qmax);
}

// Advances to the next key tile; false when the schedule is exhausted.
__device__ __forceinline__ bool kiter_next(const FwdParams& p, const UnitInfo& ui, KIter& it) {
  while (it.bt >= it.nk) {
    it.bt = 0;
    if (++it.sk >= p.g.nseg) {
      it.sk = 0;
      if (++it.t >= it.t_end) return false;
      it.s = ring_block(p.g, ui.qt[0].shard, it.t);
    }
    it.seg = segment_of(p.g, it.s, it.sk);
    it.nk = visible_tiles(p.g, it.seg, ui.qmax);
  }
  return true;
}

// Is key tile (it.seg, it.bt) visible to query tile x?
__device__ __forceinline__ bool tile_active(const FwdParams& p, const UnitInfo& ui,
                                            const KIter& it, int x) {
  if (!ui.qt[x].valid) return false;
  if (!p.g.causal) return true;
  return it.seg.pos0 + it.seg.stride * ((int64_t)it.bt * kTile) <= ui.qt[x].qmax;
}

// TMA coordinates (phase, row) of a tile starting at offset `off` of segment
// (pos0, stride, local0) of shard `shard`, batch b.
__device__ __forceinline__ void tile_coords(const FwdParams& p, int shard, int64_t pos0,
                                            int64_t local0, int64_t off, int b, int& phase,
                                            int& row) {
  const Geo& g = p.g;
  if (p.mode == FWD_MODE_STEP) {
    phase = 0;
    row = (int)((int64_t)b * g.n + local0 + off);
  } else if (g.layout == LAYOUT_STRIPED) {
    phase = shard;
    row = (int)((int64_t)b * g.n + off);
  } else {
    phase = 0;
    row = (int)((int64_t)b * g.S + pos0 + off);
  }
}

template <int D>
__global__ void __launch_bounds__(384, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Cfg = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  volatile int* abort_flag = &sm.abort_flag;

  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&sm.q_full[x]), 1);
      mbar_init(smem_u32(&sm.q_empty[x]), 1);
      mbar_init(smem_u32(&sm.s_full[x]), 1);
      mbar_init(smem_u32(&sm.p_full[x]), 128);
      mbar_init(smem_u32(&sm.o_full[x]), 1);
    }
    for (int i = 0; i < Cfg::kKStages; ++i) {
      mbar_init(smem_u32(&sm.k_full[i]), 1);
      mbar_init(smem_u32(&sm.k_empty[i]), 1);
    }
    for (int i = 0; i < Cfg::kVStages; ++i) {
      mbar_init(smem_u32(&sm.v_full[i]), 1);
      mbar_init(smem_u32(&sm.v_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.drain), 1);
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

  // Static "snake" assignment of the longest-first item list: round k gives
  // CTA c item k*G + c (k even) or k*G + G-1-c (k odd).
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  auto item_at = [&](int64_t k) -> int64_t { return k * G + ((k & 1) ? (G - 1 - c) : c); };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t q_ph[2] = {0, 0};
      uint32_t kst = 0, k_ph = 0, vst = 0, v_ph = 0;
      for (int64_t k = 0;; ++k) {
        const int64_t item = item_at(k);
        if (item >= p.num_items) break;
        UnitInfo ui = unit_info(p, item);
        for (int x = 0; x < 2; ++x) {
          if (ui.ntiles[x] == 0) continue;
          if (!mbar_wait(smem_u32(&sm.q_empty[x]), q_ph[x] ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag))
            goto done;
          q_ph[x] ^= 1;
          const uint32_t bar = smem_u32(&sm.q_full[x]);
          mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
          int phase, row;
          const QTile& qt = ui.qt[x];
          tile_coords(p, qt.shard, qt.pos0, qt.local0, qt.off, ui.b, phase, row);
          for (int st = 0; st < Cfg::kSubTiles; ++st)
            tma_load_4d(smem_u32(sm.q[x]) + st * (kTile * 128), &tm_q, bar, 64 * st, ui.h, phase,
                        row, pol_q);
        }
        KIter it;
        kiter_setup(p, ui, it);
        while (kiter_next(p, ui, it)) {
          int phase, row;
          tile_coords(p, it.s, it.seg.pos0, it.seg.local0, (int64_t)it.bt * kTile, ui.b, phase,
                      row);
          if (!mbar_wait(smem_u32(&sm.k_empty[kst]), k_ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag))
            goto done;
          uint32_t bar = smem_u32(&sm.k_full[kst]);
          mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
          for (int st = 0; st < Cfg::kSubTiles; ++st)
            tma_load_4d(smem_u32(sm.k[kst]) + st * (kTile * 128), &tm_k, bar, 64 * st, ui.hkv,
                        phase, row, pol_kv);
          if (++kst == Cfg::kKStages) { kst = 0; k_ph ^= 1; }
          if (!mbar_wait(smem_u32(&sm.v_empty[vst]), v_ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag))
            goto done;
          bar = smem_u32(&sm.v_full[vst]);
          mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
          for (int st = 0; st < Cfg::kSubTiles; ++st)
            tma_load_4d(smem_u32(sm.v[vst]) + st * (kTile * 128), &tm_v, bar, 64 * st, ui.hkv,
                        phase, row, pol_kv);
          if (++vst == Cfg::kVStages) { vst = 0; v_ph ^= 1; }
          ++it.bt;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_pv = idesc_bf16(128, D, false, true);
      uint32_t q_ph[2] = {0, 0}, p_ph[2] = {0, 0};
      uint32_t kst = 0, k_ph = 0, vst = 0, v_ph = 0;
      for (int64_t k = 0;; ++k) {
        const int64_t item = item_at(k);
        if (item >= p.num_items) break;
        UnitInfo ui = unit_info(p, item);
        if (ui.ntiles[0] + ui.ntiles[1] == 0) continue;
        if (p.shard_tiles != nullptr)
          atomicAdd(p.shard_tiles + ui.qt[0].shard,
                    static_cast<unsigned long long>(ui.ntiles[0] + ui.ntiles[1]));
        int cnt_s[2] = {0, 0}, cnt_pv[2] = {0, 0};
        bool pend[2] = {false, false};   // a P V of the previous key tile is owed
        int prev_vst = -1;
        KIter it;
        kiter_setup(p, ui, it);
        bool more = kiter_next(p, ui, it);
        while (true) {
          bool act[2] = {false, false};
          if (more) {
            act[0] = tile_active(p, ui, it, 0);
            act[1] = tile_active(p, ui, it, 1);
            if (!mbar_wait(smem_u32(&sm.k_full[kst]), k_ph, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            tc_fence_after();
          }
          if (pend[0] || pend[1]) {
            if (!mbar_wait(smem_u32(&sm.v_full[prev_vst]), v_ph, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            tc_fence_after();
          }
          for (int x = 0; x < 2; ++x) {
            if (pend[x]) {
              // O_x += P_x V_prev
              if (!mbar_wait(smem_u32(&sm.p_full[x]), p_ph[x], RA_DEV_TIMEOUT_MMA, abort_flag))
                goto done;
              p_ph[x] ^= 1;
              tc_fence_after();
              const uint32_t vb = smem_u32(sm.v[prev_vst]);
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ts(tmem + col_o(x), tmem + col_s(x) + kk * 8,
                       sdesc_sw128(vb + kk * 2048, kTile * 128, 1024), id_pv,
                       (cnt_pv[x] > 0 || kk > 0) ? 1u : 0u);
              ++cnt_pv[x];
              pend[x] = false;
              if (cnt_pv[x] == ui.ntiles[x]) mma_commit(smem_u32(&sm.o_full[x]));
            }
            if (more && act[x]) {
              if (cnt_s[x] == 0) {
                if (!mbar_wait(smem_u32(&sm.q_full[x]), q_ph[x], RA_DEV_TIMEOUT_MMA, abort_flag))
                  goto done;
                q_ph[x] ^= 1;
                tc_fence_after();
              }
              // S_x = Q_x K^T
              const uint32_t qb = smem_u32(sm.q[x]);
              const uint32_t kb = smem_u32(sm.k[kst]);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk / 4) * (kTile * 128) + (kk % 4) * 32;
                mma_ss(tmem + col_s(x), sdesc_sw128(qb + off, 16, 1024),
                       sdesc_sw128(kb + off, 16, 1024), id_qk, kk > 0 ? 1u : 0u);
              }
              mma_commit(smem_u32(&sm.s_full[x]));
              ++cnt_s[x];
              if (cnt_s[x] == ui.ntiles[x]) mma_commit(smem_u32(&sm.q_empty[x]));
              pend[x] = true;
            }
          }
          if (prev_vst >= 0) {
            mma_commit(smem_u32(&sm.v_empty[prev_vst]));
            if (++vst == Cfg::kVStages) { vst = 0; v_ph ^= 1; }
            prev_vst = -1;
          }
          if (!more) break;
          mma_commit(smem_u32(&sm.k_empty[kst]));
          if (++kst == Cfg::kKStages) { kst = 0; k_ph ^= 1; }
          prev_vst = (int)vst;
          ++it.bt;
          more = kiter_next(p, ui, it);
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) / 4;                 // query tile A (0) or B (1)
    const int quarter = warp % 4;                 // TMEM lanes [32*quarter, +32)
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + col_s(x);
    const uint32_t t_o = tmem + lane_addr + col_o(x);
    const float sl2 = p.scale_log2;
    uint32_t s_ph = 0, o_ph = 0;
    for (int64_t k = 0;; ++k) {
      const int64_t item = item_at(k);
      if (item >= p.num_items) break;
      UnitInfo ui = unit_info(p, item);
      const QTile& qt = ui.qt[x];
      if (!qt.valid) continue;
      const bool row_ok = row < qt.valid;
      const int64_t qpos = qt.pos0 + qt.stride * (qt.off + row);
      float m_run = -INFINITY;   // running max, scaled log2 units
      float l_run = 0.f;         // running normaliser
      if (ui.ntiles[x] > 0) {
        KIter it;
        kiter_setup(p, ui, it);
        while (kiter_next(p, ui, it)) {
          if (!tile_active(p, ui, it, x)) { ++it.bt; continue; }
          const int64_t k0 = (int64_t)it.bt * kTile;
          const int64_t kleft = it.seg.len - k0;
          const int kvalid = kleft < kTile ? (int)kleft : kTile;
          int lim = kvalid;
          bool masked = kvalid < kTile;
          if (p.g.causal) {
            const int64_t kmax = it.seg.pos0 + it.seg.stride * (k0 + kvalid - 1);
            if (kmax > qt.qmin) masked = true;
            int64_t cl = count_le(it.seg, qpos) - k0;
            lim = cl < 0 ? 0 : (cl > kvalid ? kvalid : (int)cl);
          }
          if (!__all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&sm.s_full[x]), s_ph, RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
            goto done;
          s_ph ^= 1;
          tc_fence_after();
          float s[kTile];
#pragma unroll
          for (int cch = 0; cch < 4; ++cch) {
            uint32_t r[32];
            tmem_ld32(t_s + cch * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) s[cch * 32 + i] = __uint_as_float(r[i]);
          }
          tmem_wait_ld();
          // row extreme of the raw scores over the visible columns
          float mt;
          if (sl2 >= 0.f) {
            mt = -INFINITY;
            if (masked) {
#pragma unroll
              for (int i = 0; i < kTile; ++i) mt = fmaxf(mt, i < lim ? s[i] : -INFINITY);
            } else {
#pragma unroll
              for (int i = 0; i < kTile; ++i) mt = fmaxf(mt, s[i]);
            }
          } else {
            mt = INFINITY;
#pragma unroll
            for (int i = 0; i < kTile; ++i) mt = fminf(mt, i < lim ? s[i] : INFINITY);
          }
          const bool any = masked ? lim > 0 : true;
          const float m_tile = any ? mt * sl2 : -INFINITY;
          // lazy rescale: only when the max rises by more than 8 (log2 units)
          float corr = 1.f;
          bool need = false;
          if (m_run == -INFINITY) {
            m_run = m_tile;
          } else if (m_tile > m_run + 8.f) {
            corr = ex2_approx(m_run - m_tile);
            m_run = m_tile;
            need = true;
          }
          if (__any_sync(0xffffffffu, need)) {
            l_run *= corr;
#pragma unroll
            for (int cch = 0; cch < D / 32; ++cch) {
              uint32_t r[32];
              tmem_ld32(t_o + cch * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
              tmem_st32(t_o + cch * 32, r);
            }
          }
          const float m_use = m_run == -INFINITY ? 0.f : m_run;
          float lsum = 0.f;
#pragma unroll
          for (int cch = 0; cch < 4; ++cch) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int c0 = cch * 32 + 2 * i;
              float p0 = ex2_approx(fmaf(s[c0], sl2, -m_use));
              float p1 = ex2_approx(fmaf(s[c0 + 1], sl2, -m_use));
              if (masked) {
                p0 = c0 < lim ? p0 : 0.f;
                p1 = c0 + 1 < lim ? p1 : 0.f;
              }
              lsum += p0 + p1;
              pk[i] = pack_bf16x2(p0, p1);
            }
            tmem_st16(t_s + cch * 16, pk);
          }
          l_run += lsum;
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.p_full[x]));
          ++it.bt;
        }
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&sm.o_full[x]), o_ph, RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
          goto done;
        o_ph ^= 1;
        tc_fence_after();
      }
      // ---- epilogue: out = O / l, lse = (m + log2 l) * ln 2
      {
        const bool has = ui.ntiles[x] > 0 && l_run > 0.f;
        const float inv_l = has ? 1.f / l_run : 0.f;
        int64_t orow, lidx;
        const Geo& g = p.g;
        if (p.mode == FWD_MODE_STEP) {
          const int64_t j = qt.local0 + qt.off + row;
          orow = ((int64_t)ui.b * g.n + j) * g.H + ui.h;
          lidx = ((int64_t)ui.b * g.H + ui.h) * g.n + j;
        } else {
          orow = ((int64_t)ui.b * g.S + qpos) * g.H + ui.h;
          lidx = ((int64_t)ui.b * g.H + ui.h) * g.S + qpos;
        }
#pragma unroll
        for (int cch = 0; cch < D / 32; ++cch) {
          uint32_t r[32];
          if (ui.ntiles[x] > 0) {
            tmem_ld32(t_o + cch * 32, r);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          if (row_ok) {
            if (p.out_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * D + cch * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv_l,
                                     __uint_as_float(r[4 * i + 1]) * inv_l,
                                     __uint_as_float(r[4 * i + 2]) * inv_l,
                                     __uint_as_float(r[4 * i + 3]) * inv_l);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow * D + cch * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(
                    pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l),
                    pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l),
                    pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l),
                    pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l));
            }
          }
        }
        if (row_ok && p.lse != nullptr)
          p.lse[lidx] = has ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

done:
  tc_fence_before();
  __syncthreads();
  if (sm.abort_flag) {
    // Let whatever was issued before the failure land before TMEM goes away.
    if (warp == 1 && lane == 0) {
      mma_commit(smem_u32(&sm.drain));
      mbar_wait(smem_u32(&sm.drain), 0, RA_DEV_TIMEOUT_DRAIN, nullptr);
    }
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) {
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace ra
