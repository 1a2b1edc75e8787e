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
//   warps 1, 3   MMA issuers, one thread each: warp 1 for query tile A,
//                warp 3 for tile B.  Each issues S_x = Q_x K^T (both operands
//                in shared memory) and O_x += P_x V (P read from tensor
//                memory) with tcgen05.mma and signals completion with
//                tcgen05.commit; warp 1 owns the TMEM allocation;
//   warps 4..7   softmax of query tile A, one row per thread;
//   warps 8..11  softmax of query tile B.
// The two tiles run independent chains (S -> softmax -> P V -> next S).  The
// issuers pass a turn back and forth (two mbarriers): an issuer takes the turn
// before its P V and hands it on before its Q K^T, so the two chains stay half
// a batch apart: one tile's softmax runs while the other tile's products do,
// and the Q K^T of one overlaps the P V of the other at issue.  Measured on a
// B300 (32k causal forward): one issuing thread 1041 TFLOP/s (its own barrier
// waits serialise both chains), two free-running issuers 1111 (the chains fall
// into step, so both softmaxes leave the tensor core idle together), turn
// passed after each whole batch 1148, turn passed between P V and Q K^T 1250.
//
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+D),
// O_B [384,384+D).  P (bf16, two per column) overwrites the first 64 columns
// of its S region after the softmax has read S into registers; the next
// Q K^T into that region is issued after the P V that reads it, and tcgen05
// MMAs of one thread execute in issue order.
//
// Lazy rescaling: a row keeps its running maximum until a tile's exponentials
// against it sum above 2^12 (the exact pass then raises the maximum, with a
// slack of 8 in log2 units); P entries stay below 2^12, and the final O / l
// uses the same maximum in numerator and denominator, so the result is exact.
#pragma once
#include "geometry.cuh"
#include "sm103_ptx.cuh"

namespace ra {

enum { FWD_MODE_RING = 0, FWD_MODE_STEP = 1 };

// Register budget: 384 threads launched at kRegsLaunch registers each; the
// control warpgroup drops to kRegsControl and the two softmax warpgroups rise
// to kRegsSoftmax, using exactly the launched total.
constexpr int kRegsLaunch = 168;
constexpr uint32_t kRegsControl = 72;
constexpr uint32_t kRegsSoftmax = 216;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= 384 * kRegsLaunch,
              "register split exceeds the launch budget");

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
  // may be null: per work item, 4 words: the globaltimer when its CTA took it
  // up, when its last output row was stored (caller-zeroed, atomicMax), the
  // shard << 32 | CTA, and the number of key tiles its query tiles multiplied
  unsigned long long* trace;
  int64_t num_items;
  int kv_group;        // (b, kv head) pairs per scheduling group (see unit_head)
  const int* sched;    // may be null: per-CTA item lists (see cta_items)
  int early;           // launched with programmatic stream serialization
  // packed sequences (attn_fwd_kernel<D, true> only):
  const int4* units;          // (sequence, shard, segment, pair) per unit, longest first
  const int64_t* cu_seqlens;  // token offset of each sequence in the pack, and the total
  int total;                  // tokens in the pack
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
  uint64_t turn[2];      // issuer x may issue its next batch
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort_flag;
};

// Per-unit schedule facts every role derives identically.
struct UnitHead {
  int b, h, hkv, shard, seg, pair;
  int row_base;      // token row of position 0 of this (b or sequence) in q/k/v/out
  int64_t lse0;      // index of position 0 of this (b or sequence, h) in lse
};

// Work items are ordered group-major: the (b, kv head) pairs are cut into
// groups of p.kv_group, and a group's items all come before the next group's.
// Inside a group the units come longest first, each with all its heads side by
// side (the G query heads of one kv head adjacent).  With one group this is a
// global longest-first order; smaller groups keep the key/value tiles the
// running CTAs share inside L2 when all of them would not fit.
__device__ __forceinline__ UnitHead unit_head_dense(const FwdParams& p, int64_t item);

// Packed sequences: item = unit * H + h over the host's longest-first unit
// list; the geometry is the unit's sequence's (B = 1, S = its length).
template <bool kVarlen>
__device__ __forceinline__ const Geo& unit_head(const FwdParams& p, int64_t item, UnitHead& u,
                                                Geo& gv) {
  if constexpr (kVarlen) {
    const int H = p.g.H;
    const int64_t unit = item / H;
    u.h = (int)(item % H);
    u.hkv = u.h / (H / p.g.Hkv);
    u.b = 0;
    const int4 w = __ldg(p.units + unit);
    const int64_t t0 = __ldg(p.cu_seqlens + w.x), t1 = __ldg(p.cu_seqlens + w.x + 1);
    gv = make_geo(1, H, p.g.Hkv, t1 - t0, p.g.P, p.g.layout, p.g.causal);
    u.shard = w.y;
    u.seg = w.z;
    u.pair = w.w;
    u.row_base = (int)t0;
    u.lse0 = (int64_t)u.h * p.total + t0;
    return gv;
  } else {
    u = unit_head_dense(p, item);
    return p.g;
  }
}

// Item -> (unit, b * H + h) of the group-major order above (host and device).
__host__ __device__ __forceinline__ int64_t unit_index_dense(const FwdParams& p, int64_t item,
                                                            int* bh = nullptr) {
  const Geo& g = p.g;
  const int G = g.H / g.Hkv;
  const int BK = g.B * g.Hkv;
  const int64_t U = units_total(g, p.mode == FWD_MODE_STEP);
  const int64_t per_group = (int64_t)p.kv_group * G * U;
  const int grp = (int)(item / per_group);
  const int64_t rem = item % per_group;
  const int left = BK - grp * p.kv_group;
  const int hg = left < p.kv_group ? left : p.kv_group;   // pairs in this group
  const int r2 = (int)(rem % ((int64_t)hg * G));
  if (bh != nullptr) {
    const int bk = grp * p.kv_group + r2 / G;
    *bh = (bk / g.Hkv) * g.H + (bk % g.Hkv) * G + r2 % G;
  }
  return rem / ((int64_t)hg * G);
}

__device__ __forceinline__ UnitHead unit_head_dense(const FwdParams& p, int64_t item) {
  UnitHead u;
  const Geo& g = p.g;
  int bh = 0;
  const int64_t unit = unit_index_dense(p, item, &bh);
  u.b = bh / g.H;
  u.h = bh % g.H;
  u.hkv = u.h / (g.H / g.Hkv);
  Unit w = unit_of(g, unit, p.mode == FWD_MODE_STEP, p.step_r);
  u.shard = w.shard;
  u.seg = w.seg;
  u.pair = w.pair;
  u.row_base = u.b * g.S;
  u.lse0 = ((int64_t)u.b * g.H + u.h) * g.S;
  return u;
}

__device__ __forceinline__ int step_block(const FwdParams& p) {
  return p.mode == FWD_MODE_STEP ? p.step_s : -1;
}

// Iterator over the union of the key tiles a unit multiplies, in ring order.
struct KIter {
  int t, t_end, sk, bt, nk, s;
  int qmax, shard;
  Seg seg;
};

__device__ __forceinline__ void kiter_setup(const Geo& g, const FwdParams& p, int shard, int qmax,
                                            KIter& it) {
  it.t = 0;
  it.t_end = p.mode == FWD_MODE_STEP ? 1 : g.P;
  it.sk = 0;
  it.bt = 0;
  it.qmax = qmax;
  it.shard = shard;
  it.s = p.mode == FWD_MODE_STEP ? p.step_s : ring_block(g, shard, 0);
  it.seg = segment_of(g, it.s, 0);
  it.nk = visible_tiles(g, it.seg, qmax);
}

// Advances to the next key tile; false when the schedule is exhausted.
__device__ __forceinline__ bool kiter_next(const Geo& g, KIter& it) {
  while (it.bt >= it.nk) {
    it.bt = 0;
    if (++it.sk >= g.nseg) {
      it.sk = 0;
      if (++it.t >= it.t_end) return false;
      it.s = ring_block(g, it.shard, it.t);
    }
    it.seg = segment_of(g, it.s, it.sk);
    it.nk = visible_tiles(g, it.seg, it.qmax);
  }
  return true;
}

// Position of the first key of the iterator's current tile.
__device__ __forceinline__ int kiter_first_pos(const KIter& it) {
  return it.seg.pos0 + it.seg.stride * (it.bt * kTile);
}

// Is the current key tile visible to a query tile whose last position is qmax?
__device__ __forceinline__ bool visible_to(const Geo& g, const KIter& it, int valid, int qmax) {
  return valid && (!g.causal || kiter_first_pos(it) <= qmax);
}

// TMA coordinates (phase, row) of a tile starting at offset `off` of segment
// (pos0, local0) of shard `shard`, for the unit's batch entry or sequence
// whose position 0 sits at token row row_base (a multiple of P).
__device__ __forceinline__ void tile_coords(const Geo& g, const FwdParams& p, int shard, int pos0,
                                            int local0, int off, int row_base, int& phase,
                                            int& row) {
  if (p.mode == FWD_MODE_STEP) {
    phase = 0;
    row = row_base / g.P + local0 + off;     // shard-local tensors: n rows per batch entry
  } else if (g.layout == LAYOUT_STRIPED) {
    phase = shard;
    row = row_base / g.P + off;
  } else {
    phase = 0;
    row = row_base + pos0 + off;
  }
}

template <int D, bool kVarlen>
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
      mbar_init(smem_u32(&sm.p_full[x]), 4);      // one arrival per softmax warp
      mbar_init(smem_u32(&sm.o_full[x]), 1);
    }
    for (int i = 0; i < Cfg::kKStages; ++i) {
      mbar_init(smem_u32(&sm.k_full[i]), 1);
      mbar_init(smem_u32(&sm.k_empty[i]), 2);
    }
    for (int i = 0; i < Cfg::kVStages; ++i) {
      mbar_init(smem_u32(&sm.v_full[i]), 1);
      mbar_init(smem_u32(&sm.v_empty[i]), 2);
    }
    mbar_init(smem_u32(&sm.drain[0]), 1);
    mbar_init(smem_u32(&sm.drain[1]), 1);
    mbar_init(smem_u32(&sm.turn[0]), 1);
    mbar_init(smem_u32(&sm.turn[1]), 1);
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
  // Everything above touched only this CTA's shared and tensor memory; from
  // here on the kernel reads and writes global memory.
  if (p.early) {
    griddep_launch_dependents();
    griddep_wait();
  }
  const uint32_t tmem = sm.tmem_base;
  const int sblk = step_block(p);

  // The producer's positions in its rings: how many Q loads each query tile
  // slot received (parity) and the next K / V stage with its lap parity.  At
  // function scope so that an aborting CTA can wait for every load it issued.
  uint32_t q_ph0 = 0, q_ph1 = 0;
  uint32_t tk_st = 0, tk_ph = 0, tv_st = 0, tv_ph = 0;

  // This CTA's work items, in the order every role takes them.
  const CtaItems mine = cta_items(p.sched);
  auto item_at = [&](int64_t k) -> int64_t { return cta_item(mine, k, p.num_items); };

  if (warp < 4) {
    // Producer / MMA / idle warps give registers to the two softmax warpgroups.
    regs_dec<kRegsControl>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      for (int64_t k = 0;; ++k) {
        const int64_t item = item_at(k);
        if (item >= p.num_items) break;
        UnitHead u;
        Geo gv;
        const Geo& g = unit_head<kVarlen>(p, item, u, gv);
        const QTile qa = make_qtile(g, u.shard, u.seg, 2 * u.pair);
        const QTile qb = make_qtile(g, u.shard, u.seg, 2 * u.pair + 1);
        const int na = tile_work(g, qa, sblk), nb = tile_work(g, qb, sblk);
        if (p.trace != nullptr) {
          unsigned long long* rec = p.trace + 4 * item;
          rec[0] = globaltimer();
          rec[2] = (static_cast<unsigned long long>(u.shard) << 32) | blockIdx.x;
          rec[3] = static_cast<unsigned long long>(na + nb);
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const QTile& qt = x ? qb : qa;
          if ((x ? nb : na) == 0) continue;
          uint32_t& ph = x ? q_ph1 : q_ph0;
          if (!mbar_wait(smem_u32(&sm.q_empty[x]), ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag))
            goto done;
          ph ^= 1;
          const uint32_t bar = smem_u32(&sm.q_full[x]);
          mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
          int phase, row;
          tile_coords(g, p, qt.shard, qt.pos0, qt.local0, qt.off, u.row_base, phase, row);
#pragma unroll
          for (int st = 0; st < Cfg::kSubTiles; ++st)
            tma_load_4d(smem_u32(sm.q[x]) + st * (kTile * 128), &tm_q, bar, 64 * st, u.h, phase,
                        row, pol_q);
        }
        KIter it;
        kiter_setup(g, p, u.shard, qb.valid && qb.qmax > qa.qmax ? qb.qmax : qa.qmax, it);
        while (kiter_next(g, it)) {
          int phase, row;
          tile_coords(g, p, it.s, it.seg.pos0, it.seg.local0, it.bt * kTile, u.row_base, phase,
                      row);
          if (!mbar_wait(smem_u32(&sm.k_empty[tk_st]), tk_ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag))
            goto done;
          uint32_t bar = smem_u32(&sm.k_full[tk_st]);
          mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
#pragma unroll
          for (int st = 0; st < Cfg::kSubTiles; ++st)
            tma_load_4d(smem_u32(sm.k[tk_st]) + st * (kTile * 128), &tm_k, bar, 64 * st, u.hkv,
                        phase, row, pol_kv);
          if (++tk_st == Cfg::kKStages) { tk_st = 0; tk_ph ^= 1; }
          if (!mbar_wait(smem_u32(&sm.v_empty[tv_st]), tv_ph ^ 1, RA_DEV_TIMEOUT_TMA, abort_flag))
            goto done;
          bar = smem_u32(&sm.v_full[tv_st]);
          mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
#pragma unroll
          for (int st = 0; st < Cfg::kSubTiles; ++st)
            tma_load_4d(smem_u32(sm.v[tv_st]) + st * (kTile * 128), &tm_v, bar, 64 * st, u.hkv,
                        phase, row, pol_kv);
          if (++tv_st == Cfg::kVStages) { tv_st = 0; tv_ph ^= 1; }
          ++it.bt;
        }
      }
    } else if ((warp == 1 || warp == 3) && lane == 0) {
      // ---------------------------------------------------------- MMA issuers
      // One thread per query tile (warp 1: tile A, warp 3: tile B), each with
      // its own chain S_x = Q_x K^T -> softmax_x -> O_x += P_x V.  The tensor
      // core interleaves the two streams.  A key / value stage is released
      // when both issuers have committed it (barrier count 2), and each issuer
      // waits for every stage it passes, so neither can run a full ring ahead.
      const int x = warp == 1 ? 0 : 1;
      constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_pv = idesc_bf16(128, D, false, true);
      uint32_t q_ph = 0, p_ph = 0, turn_ph = 0;
      bool first_turn = x == 0;   // tile A's issuer opens the alternation
      uint32_t kst = 0, k_ph = 0, vst = 0, v_ph = 0;
      for (int64_t k = 0;; ++k) {
        const int64_t item = item_at(k);
        if (item >= p.num_items) break;
        UnitHead u;
        Geo gv;
        const Geo& g = unit_head<kVarlen>(p, item, u, gv);
        const QTile qa = make_qtile(g, u.shard, u.seg, 2 * u.pair);
        const QTile qb = make_qtile(g, u.shard, u.seg, 2 * u.pair + 1);
        const int na = tile_work(g, qa, sblk), nb = tile_work(g, qb, sblk);
        if (na + nb == 0) continue;
        if (x == 0 && p.shard_tiles != nullptr)
          atomicAdd(p.shard_tiles + u.shard, static_cast<unsigned long long>(na + nb));
        const QTile& qt = x ? qb : qa;
        const int nx = x ? nb : na;
        int cnt_s = 0, cnt_pv = 0;
        bool pend = false;   // a P V of the previous key tile is owed
        int prev_vst = -1;
        KIter it;
        kiter_setup(g, p, u.shard, qb.valid && qb.qmax > qa.qmax ? qb.qmax : qa.qmax, it);
        bool more = kiter_next(g, it);
        while (true) {
          bool act = false;
          if (more) {
            act = visible_to(g, it, qt.valid, qt.qmax);
            if (!mbar_wait(smem_u32(&sm.k_full[kst]), k_ph, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            tc_fence_after();
          }
          if (prev_vst >= 0) {
            if (!mbar_wait(smem_u32(&sm.v_full[prev_vst]), v_ph, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            tc_fence_after();
          }
          // The turn alternates between the two issuers (A, B, A, B, ...) and
          // is handed on between this issuer's P V and its Q K^T; left free,
          // the two chains fall into step and both softmaxes then leave the
          // tensor core idle at the same time.
          if (first_turn) {
            first_turn = false;
          } else {
            if (!mbar_wait(smem_u32(&sm.turn[x]), turn_ph, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            turn_ph ^= 1;
          }
          if (pend) {
            // O_x += P_x V_prev
            if (!mbar_wait(smem_u32(&sm.p_full[x]), p_ph, RA_DEV_TIMEOUT_MMA, abort_flag))
              goto done;
            p_ph ^= 1;
            tc_fence_after();
            const uint32_t vb = smem_u32(sm.v[prev_vst]);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts(tmem + col_o(x), tmem + col_s(x) + kk * 8,
                     sdesc_sw128(vb + kk * 2048, kTile * 128, 1024), id_pv,
                     (cnt_pv > 0 || kk > 0) ? 1u : 0u);
            ++cnt_pv;
            pend = false;
            if (cnt_pv == nx) mma_commit(smem_u32(&sm.o_full[x]));
          }
          mbar_arrive(smem_u32(&sm.turn[x ^ 1]));
          if (more && act) {
            if (cnt_s == 0) {
              if (!mbar_wait(smem_u32(&sm.q_full[x]), q_ph, RA_DEV_TIMEOUT_MMA, abort_flag))
                goto done;
              q_ph ^= 1;
              tc_fence_after();
            }
            // S_x = Q_x K^T
            const uint32_t qbase = smem_u32(sm.q[x]);
            const uint32_t kbase = smem_u32(sm.k[kst]);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk / 4) * (kTile * 128) + (kk % 4) * 32;
              mma_ss(tmem + col_s(x), sdesc_sw128(qbase + off, 16, 1024),
                     sdesc_sw128(kbase + off, 16, 1024), id_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&sm.s_full[x]));
            ++cnt_s;
            if (cnt_s == nx) mma_commit(smem_u32(&sm.q_empty[x]));
            pend = true;
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
          more = kiter_next(g, it);
        }
      }
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) / 4;                 // query tile A (0) or B (1)
    const int quarter = warp % 4;                 // TMEM lanes [32*quarter, +32)
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + col_s(x);
    const uint32_t t_o = tmem + lane_addr + col_o(x);
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 >= 0.f;
    uint32_t s_ph = 0, o_ph = 0;
    for (int64_t k = 0;; ++k) {
      const int64_t item = item_at(k);
      if (item >= p.num_items) break;
      UnitHead u;
      Geo gv;
      const Geo& g = unit_head<kVarlen>(p, item, u, gv);
      const QTile qt = make_qtile(g, u.shard, u.seg, 2 * u.pair + x);
      if (!qt.valid) continue;
      int qmax_u = qt.qmax;
      {
        const QTile other = make_qtile(g, u.shard, u.seg, 2 * u.pair + (x ^ 1));
        if (other.valid && other.qmax > qmax_u) qmax_u = other.qmax;
      }
      const int ntiles = tile_work(g, qt, sblk);
      const bool row_ok = row < qt.valid;
      const int qpos = qt.pos0 + qt.stride * (qt.off + row);
      float m_run = -INFINITY;   // running max, scaled log2 units
      float l_run = 0.f;         // running normaliser
      if (ntiles > 0) {
        KIter it;
        kiter_setup(g, p, u.shard, qmax_u, it);
        while (kiter_next(g, it)) {
          if (!visible_to(g, it, 1, qt.qmax)) { ++it.bt; continue; }
          const int k0 = it.bt * kTile;
          const int kleft = it.seg.len - k0;
          const int kvalid = kleft < kTile ? kleft : kTile;
          bool masked = kvalid < kTile;
          if (g.causal && it.seg.pos0 + it.seg.stride * (k0 + kvalid - 1) > qt.qmin) masked = true;
          int lim = kvalid;
          if (masked && g.causal) {
            const int cl = count_le(it.seg, qpos) - k0;
            lim = cl < 0 ? 0 : (cl > kvalid ? kvalid : cl);
          }
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[x]), s_ph,
                                                 RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
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
          float2 sum2 = make_float2(0.f, 0.f);
          bool done_p = false;
          if (!masked && pos_scale && m_run != -INFINITY) {
            // Speculative pass: exponentials against the running max, without
            // the tile max.  The tile's sum bounds its largest entry, so it is
            // kept when that sum stays <= 2^12 (entries <= 2^12: harmless in bf16
            // P and fp32 O, and O / l uses one max for both); otherwise the
            // exact pass below redoes the tile with the max updated.
            const float2 sl2_2 = make_float2(sl2, sl2);
            const float2 negm2 = make_float2(-m_run, -m_run);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int cch = 0; cch < 4; ++cch) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c0 = cch * 32 + 2 * i;
                const float2 t2 = fma2(make_float2(s[c0], s[c0 + 1]), sl2_2, negm2);
                const float p0 = ex2_approx(t2.x);
                const float p1 = ex2_approx(t2.y);
                acc[i % 4] = add2(acc[i % 4], make_float2(p0, p1));
                pk[i] = pack_bf16x2(p0, p1);
              }
              tmem_st16(t_s + cch * 16, pk);
            }
            const float2 sum_t = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
            const bool ok = sum_t.x + sum_t.y <= 4096.f;
            if (__all_sync(0xffffffffu, ok)) {
              sum2 = sum_t;
              done_p = true;
            }
          }
          if (!done_p) {
            // Exact pass: row extreme first.  Hidden columns take the value that
            // never wins it (-inf for a positive scale, +inf for a negative one).
            if (masked) {
              const float neutral = pos_scale ? -INFINITY : INFINITY;
#pragma unroll
              for (int i = 0; i < kTile; ++i) s[i] = i < lim ? s[i] : neutral;
            }
            float mq[4];
            if (pos_scale) {
#pragma unroll
              for (int j = 0; j < 4; ++j) mq[j] = -INFINITY;
#pragma unroll
              for (int i = 0; i < kTile; i += 2) mq[(i / 2) % 4] = max3f(mq[(i / 2) % 4], s[i], s[i + 1]);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) mq[j] = INFINITY;
#pragma unroll
              for (int i = 0; i < kTile; i += 2) mq[(i / 2) % 4] = min3f(mq[(i / 2) % 4], s[i], s[i + 1]);
            }
            const float mt = pos_scale ? max3f(mq[0], mq[1], fmaxf(mq[2], mq[3]))
                                       : min3f(mq[0], mq[1], fminf(mq[2], mq[3]));
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
              const float2 c2 = make_float2(corr, corr);
#pragma unroll
              for (int cch = 0; cch < D / 32; ++cch) {
                uint32_t r[32];
                tmem_ld32(t_o + cch * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                  float2 o2 = mul2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2);
                  r[i] = __float_as_uint(o2.x);
                  r[i + 1] = __float_as_uint(o2.y);
                }
                tmem_st32(t_o + cch * 32, r);
              }
            }
            const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
            const float2 sl2_2 = make_float2(sl2, sl2);
            const float2 negm2 = make_float2(neg_m, neg_m);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int cch = 0; cch < 4; ++cch) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c0 = cch * 32 + 2 * i;
                const float2 t2 = fma2(make_float2(s[c0], s[c0 + 1]), sl2_2, negm2);
                float p0 = ex2_approx(t2.x);
                float p1 = ex2_approx(t2.y);
                if (masked) {
                  p0 = c0 < lim ? p0 : 0.f;
                  p1 = c0 + 1 < lim ? p1 : 0.f;
                }
                acc[i % 4] = add2(acc[i % 4], make_float2(p0, p1));
                pk[i] = pack_bf16x2(p0, p1);
              }
              tmem_st16(t_s + cch * 16, pk);
            }
            sum2 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
          }
          l_run += sum2.x + sum2.y;
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive_warp(smem_u32(&sm.p_full[x]));
          ++it.bt;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.o_full[x]), o_ph,
                                               RA_DEV_TIMEOUT_SOFTMAX, abort_flag)))
          goto done;
        o_ph ^= 1;
        tc_fence_after();
      }
      // ---- epilogue: out = O / l, lse = (m + log2 l) * ln 2
      const bool has = ntiles > 0 && l_run > 0.f;
      const float inv_l = has ? 1.f / l_run : 0.f;
      int64_t orow, lidx;
      if (p.mode == FWD_MODE_STEP) {
        const int j = qt.local0 + qt.off + row;
        orow = ((int64_t)u.b * g.n + j) * g.H + u.h;
        lidx = ((int64_t)u.b * g.H + u.h) * g.n + j;
      } else {
        orow = ((int64_t)u.row_base + qpos) * g.H + u.h;
        lidx = u.lse0 + qpos;
      }
#pragma unroll
      for (int cch = 0; cch < D / 32; ++cch) {
        uint32_t r[32];
        if (ntiles > 0) {
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
      if (p.trace != nullptr) {
        __syncwarp();
        if (lane == 0) atomicMax(p.trace + 4 * item + 1, globaltimer());
      }
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
      const int x = warp == 1 ? 0 : 1;
      mma_commit(smem_u32(&sm.drain[x]));
      mbar_wait_for(smem_u32(&sm.drain[x]), 0, RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
    }
    if (warp == 0 && lane == 0) {
      mbar_wait_for(smem_u32(&sm.q_full[0]), q_ph0 ^ 1, RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
      mbar_wait_for(smem_u32(&sm.q_full[1]), q_ph1 ^ 1, RA_DEV_TIMEOUT_DRAIN, kDrainLimitNs);
      for (uint32_t i = 0; i < (uint32_t)Cfg::kKStages; ++i)
        mbar_wait_for(smem_u32(&sm.k_full[i]), i < tk_st ? tk_ph : tk_ph ^ 1, RA_DEV_TIMEOUT_DRAIN,
                      kDrainLimitNs);
      for (uint32_t i = 0; i < (uint32_t)Cfg::kVStages; ++i)
        mbar_wait_for(smem_u32(&sm.v_full[i]), i < tv_st ? tv_ph : tv_ph ^ 1, RA_DEV_TIMEOUT_DRAIN,
                      kDrainLimitNs);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace ra
