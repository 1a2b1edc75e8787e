// ring_attn.cu -- libringattn.so: the C ABI declared in include/ring_attn.h.
// Host side: argument checks, TMA tensor maps, launch shapes.  The library is
// one translation unit; the kernels live in the included headers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <queue>
#include <unordered_map>
#include <vector>

#include "../../include/ring_attn.h"
#include "attn_bwd.cuh"
#include "attn_decode.cuh"
#include "attn_fwd.cuh"
#include "elementwise.cuh"
#include "geometry.cuh"
#include "sm103_ptx.cuh"

namespace {

thread_local char g_last_error[512] = "";

ra_status fail(ra_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

ra_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- device facts
struct DeviceInfo {
  int sms = 0;
  int cc_major = 0;
  int l2_bytes = 0;
  bool fwd_attr_set[2] = {false, false};
  bool fwd_varlen_attr_set[2] = {false, false};
  bool bwd_attr_set[6] = {false, false, false, false, false, false};
  bool dec_attr_set[2] = {false, false};
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

ra_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(RA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.sms == 0) {
    int sms = 0, major = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(CC)");
    int l2 = 0;
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(L2 size)");
    d.sms = sms;
    d.cc_major = major;
    d.l2_bytes = l2;
  }
  if (d.cc_major != 10)
    return fail(RA_ERR_UNSUPPORTED, "needs a Blackwell sm_10x GPU (found compute capability %d.x)",
                d.cc_major);
  *out = &d;
  return RA_OK;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

ra_status encode_fn(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                           &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (cached == nullptr) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  *fn = cached;
  return RA_OK;
}

// 4-d bf16 view {D, heads, phases, rows} of a token tensor whose row `R` at
// phase `ph` starts at base + (R * phases + ph) * heads * D * 2 bytes.
// Box {64, 1, 1, 128}, 128-byte swizzle (the layout tcgen05 descriptors use).
ra_status encode_token_map(CUtensorMap* m, const void* base, int D, int heads, int64_t phases,
                           int64_t rows) {
  EncodeTiledFn fn = nullptr;
  ra_status st = encode_fn(&fn);
  if (st != RA_OK) return st;
  const cuuint64_t row_bytes = (cuuint64_t)heads * D * 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)phases, (cuuint64_t)rows};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, row_bytes, row_bytes * (cuuint64_t)phases};
  cuuint32_t box[4] = {64, 1, 1, (cuuint32_t)ra::kTile};
  cuuint32_t elem[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return RA_OK;
}

// The encoded map depends only on (base, D, heads, phases, rows), so each host
// thread keeps the last kMapCache maps it built: a caller that runs the same
// tensors again (a training or serving loop) skips the encode.
struct MapEntry {
  const void* base;
  int D, heads;
  int64_t phases, rows;
  CUtensorMap map;
};
constexpr int kMapCache = 32;
thread_local MapEntry t_maps[kMapCache];
thread_local int t_maps_used = 0, t_maps_next = 0;

ra_status make_token_map(CUtensorMap* m, const void* base, int D, int heads, int64_t phases,
                         int64_t rows) {
  for (int i = 0; i < t_maps_used; ++i) {
    const MapEntry& e = t_maps[i];
    if (e.base == base && e.D == D && e.heads == heads && e.phases == phases && e.rows == rows) {
      *m = e.map;
      return RA_OK;
    }
  }
  ra_status st = encode_token_map(m, base, D, heads, phases, rows);
  if (st != RA_OK) return st;
  MapEntry& e = t_maps[t_maps_next];
  e.base = base; e.D = D; e.heads = heads; e.phases = phases; e.rows = rows; e.map = *m;
  t_maps_next = (t_maps_next + 1) % kMapCache;
  if (t_maps_used < kMapCache) ++t_maps_used;
  return RA_OK;
}

// ---------------------------------------------------------------- work schedules
// A persistent kernel's work items come in a fixed order: grouped by (b, kv
// head) so that the CTAs running at one time share key/value (or query) tiles
// in L2, and longest first inside a group.  Without a schedule the kernels
// deal that list out as a snake (round k: CTA c takes item k*G + c, or
// k*G + G-1-c on odd rounds), which balances long against short only where a
// group's items happen to line up with the rounds.  Here the list is dealt out
// the way a queue would hand it to CTAs as they fall idle: each item, in
// order, goes to the CTA whose items so far add up to the least estimated work
// (the key or query tiles the item multiplies, plus a fixed cost per item).
// Every CTA still takes its items in list order, so the L2 grouping holds.
//
// Layout in device memory (int32): offsets[G + 1], then the item ids of CTA 0,
// CTA 1, ...; CTA c's are entries offsets[c] .. offsets[c+1]-1 after the
// offsets.  A schedule depends only on the launch's shape, so each is built
// once and kept for the life of the process (the kernels of a captured graph
// may read it at any later replay).
enum SchedKind { SCHED_FWD = 0, SCHED_DKDV = 1, SCHED_DQ = 2 };

struct SchedKey {
  int kind, dev, B, H, Hkv, P, layout, causal, mode, r, s, grid, kv_group;
  int64_t S;
  bool operator==(const SchedKey& o) const {
    return kind == o.kind && dev == o.dev && B == o.B && H == o.H && Hkv == o.Hkv && P == o.P &&
           layout == o.layout && causal == o.causal && mode == o.mode && r == o.r && s == o.s &&
           grid == o.grid && kv_group == o.kv_group && S == o.S;
  }
};
struct SchedKeyHash {
  size_t operator()(const SchedKey& k) const {
    const int64_t f[] = {k.kind,   k.dev,  k.B, k.H, k.Hkv,  k.P,        k.layout,
                         k.causal, k.mode, k.r, k.s, k.grid, k.kv_group, k.S};
    uint64_t h = 1469598103934665603ull;  // FNV-style: xor in a field, multiply
    for (int64_t v : f) {
      h ^= (uint64_t)v;
      h *= 1099511628211ull;
    }
    return (size_t)h;
  }
};
std::mutex g_sched_mu;
// The kept schedules; nullptr for a shape refused for lack of budget (it then
// runs unscheduled without being built again).
std::unordered_map<SchedKey, int*, SchedKeyHash> g_scheds;
// Device memory the kept schedules may take (a hop of a ring keys its own
// schedule by (r, s), so a P-rank ring keeps up to P^2 small ones); shapes
// past the budget run unscheduled.
constexpr size_t kSchedBytesMax = (size_t)64 << 20;
size_t g_sched_bytes = 0;
constexpr int64_t kSchedItemsMax = 1 << 22;  // larger lists run unscheduled
constexpr double kItemCost = 2.0;          // fixed cost of an item, in tile steps

// Deals items 0..n-1 (estimated cost cost_of(unit_of(item)), units 0..U-1) to
// G CTAs; returns offsets[G + 1] followed by the per-CTA item lists.
template <class UnitOf>
std::vector<int> deal_items(int64_t n, int G, const std::vector<double>& unit_cost, UnitOf unit_of) {
  std::vector<std::vector<int>> lists((size_t)G);
  typedef std::pair<double, int> Load;  // (work so far, CTA); ties go to the lower CTA
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> idle;
  for (int c = 0; c < G; ++c) idle.push(Load(0.0, c));
  for (int64_t i = 0; i < n; ++i) {
    Load l = idle.top();
    idle.pop();
    lists[(size_t)l.second].push_back((int)i);
    l.first += unit_cost[(size_t)unit_of(i)] + kItemCost;
    idle.push(l);
  }
  std::vector<int> out;
  out.reserve((size_t)(G + 1 + n));
  int off = 0;
  for (int c = 0; c < G; ++c) {
    out.push_back(off);
    off += (int)lists[(size_t)c].size();
  }
  out.push_back(off);
  for (int c = 0; c < G; ++c) out.insert(out.end(), lists[(size_t)c].begin(), lists[(size_t)c].end());
  return out;
}

// Query tiles (of shard r, or of every shard when r < 0) that see a key tile
// whose first position is kmin: under a causal mask, those whose last position
// is at or after kmin.  A segment's tiles past the one holding its first slot
// at or after kmin all qualify.
int64_t query_tiles_seeing(const ra::Geo& g, int kmin, int r) {
  int64_t n = 0;
  const int r0 = r < 0 ? 0 : r, r1 = r < 0 ? g.P : r + 1;
  for (int sh = r0; sh < r1; ++sh)
    for (int sg = 0; sg < g.nseg; ++sg) {
      const ra::Seg q = ra::segment_of(g, sh, sg);
      const int nt = (q.len + ra::kTile - 1) / ra::kTile;
      if (!g.causal) { n += nt; continue; }
      if (q.pos0 + q.stride * (q.len - 1) < kmin) continue;
      const int o = kmin <= q.pos0 ? 0 : (kmin - q.pos0 + q.stride - 1) / q.stride;
      n += nt - o / ra::kTile;
    }
  return n;
}

// The schedule for `key`, built on first use; nullptr (the kernels then use
// the snake) when the list is short or very long, when the schedules kept
// would exceed their memory budget, or when `stream` is being captured and the
// schedule does not exist yet.
bool schedule_worth(int64_t n_items, int grid) {
  return n_items > grid && n_items <= kSchedItemsMax;
}

template <class Build>
const int* work_schedule(const SchedKey& key, int64_t n_items, cudaStream_t stream, Build build) {
  if (!schedule_worth(n_items, key.grid)) return nullptr;
  std::lock_guard<std::mutex> lk(g_sched_mu);
  const auto hit = g_scheds.find(key);
  if (hit != g_scheds.end()) return hit->second;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return nullptr;
  // the list holds G + 1 offsets and n_items ids
  const size_t bytes = ((size_t)key.grid + 1 + (size_t)n_items) * sizeof(int);
  if (g_sched_bytes + bytes > kSchedBytesMax) {
    g_scheds.emplace(key, nullptr);
    return nullptr;
  }
  const std::vector<int> host = build();
  int* buf = nullptr;
  if (cudaMalloc(&buf, host.size() * sizeof(int)) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (cudaMemcpy(buf, host.data(), host.size() * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
    (void)cudaGetLastError();
    cudaFree(buf);
    return nullptr;
  }
  g_scheds.emplace(key, buf);
  g_sched_bytes += host.size() * sizeof(int);
  return buf;
}

int current_device() {
  int d = 0;
  return cudaGetDevice(&d) == cudaSuccess ? d : -1;
}

// Forward (ring or step mode): a unit is a pair of query tiles; it multiplies
// the union of the key tiles its two tiles see, i.e. those of its later tile.
std::vector<int> fwd_schedule_host(const ra::FwdParams& prm, int grid) {
  const ra::Geo& g = prm.g;
  const bool step = prm.mode == ra::FWD_MODE_STEP;
  const int64_t U = ra::units_total(g, step);
  std::vector<double> cost((size_t)U);
  for (int64_t u = 0; u < U; ++u) {
    const ra::Unit w = ra::unit_of(g, u, step, prm.step_r);
    ra::QTile q = ra::make_qtile(g, w.shard, w.seg, 2 * w.pair + 1);
    if (!q.valid) q = ra::make_qtile(g, w.shard, w.seg, 2 * w.pair);
    cost[(size_t)u] = ra::tile_work(g, q, step ? prm.step_s : -1);
  }
  return deal_items(prm.num_items, grid, cost,
                    [&](int64_t item) { return ra::unit_index_dense(prm, item); });
}

const int* fwd_schedule(const ra::FwdParams& prm, int grid, cudaStream_t stream) {
  const ra::Geo& g = prm.g;
  SchedKey key{SCHED_FWD, current_device(), g.B, g.H, g.Hkv, g.P, g.layout, g.causal, prm.mode,
               prm.step_r, prm.step_s, grid, prm.kv_group, (int64_t)g.S};
  return work_schedule(key, prm.num_items, stream, [&]() { return fwd_schedule_host(prm, grid); });
}

// Backward (ring or hop mode): a dK/dV unit is one key tile of a (b, kv head)
// and meets every query tile of the group's G heads that sees it; a dQ unit is
// one query tile and meets the key tiles it sees.
std::vector<int> bwd_schedule_host(const ra::BwdParams& prm, bool dkdv, bool step, int grid) {
  const ra::Geo& g = prm.g;
  const int64_t U = (int64_t)(step ? 1 : g.P) * g.nseg * g.ntile;
  std::vector<double> cost((size_t)U);
  const int G = g.H / g.Hkv;
  for (int64_t u = 0; u < U; ++u) {
    if (dkdv) {
      const ra::KUnit w = step ? ra::kunit_step(g, prm.step_s, u) : ra::kunit_of(g, u);
      const ra::Seg k = ra::segment_of(g, w.shard, w.seg);
      const int kmin = k.pos0 + k.stride * (w.tile * ra::kTile);
      cost[(size_t)u] = w.tile * ra::kTile < k.len
                            ? (double)G * query_tiles_seeing(g, kmin, step ? prm.step_r : -1)
                            : 0.0;
    } else {
      const ra::QUnit w = step ? ra::qunit_step(g, prm.step_r, u) : ra::qunit_of(g, u);
      const ra::QTile q = ra::make_qtile(g, w.shard, w.seg, w.tile);
      cost[(size_t)u] = ra::tile_work(g, q, step ? prm.step_s : -1);
    }
  }
  return deal_items(prm.num_items, grid, cost, [&](int64_t item) { return item % U; });
}

const int* bwd_schedule(const ra::BwdParams& prm, bool dkdv, bool step, int grid,
                        cudaStream_t stream) {
  const ra::Geo& g = prm.g;
  SchedKey key{dkdv ? SCHED_DKDV : SCHED_DQ, current_device(), g.B, g.H, g.Hkv, g.P, g.layout,
               g.causal, step ? 1 : 0, prm.step_r, prm.step_s, grid, 0, (int64_t)g.S};
  return work_schedule(key, prm.num_items, stream,
                       [&]() { return bwd_schedule_host(prm, dkdv, step, grid); });
}

// ---------------------------------------------------------------- checks
ra_status check_common(int B, int H, int Hkv, int64_t S, int D, int P, int layout, float scale) {
  if (B < 1 || H < 1 || Hkv < 1 || S < 1 || P < 1)
    return fail(RA_ERR_SHAPE, "sizes must be positive (B=%d H=%d Hkv=%d S=%lld P=%d)", B, H, Hkv,
                (long long)S, P);
  if (H % Hkv != 0) return fail(RA_ERR_SHAPE, "H=%d is not a multiple of Hkv=%d", H, Hkv);
  if (D != 64 && D != 128) return fail(RA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
  if (layout < 0 || layout > 2) return fail(RA_ERR_LAYOUT, "unknown layout %d", layout);
  if (S % P != 0) return fail(RA_ERR_LAYOUT, "S=%lld is not divisible by P=%d", (long long)S, P);
  if (layout == RA_LAYOUT_ZIGZAG && S % (2 * (int64_t)P) != 0)
    return fail(RA_ERR_LAYOUT, "zig-zag needs S=%lld divisible by 2P=%d", (long long)S, 2 * P);
  if (!std::isfinite(scale)) return fail(RA_ERR_UNSUPPORTED, "scale is not finite");
  if ((int64_t)B * S > 0x7fffffffLL)
    return fail(RA_ERR_SHAPE, "B*S=%lld exceeds the 2^31 rows a tensor map addresses",
                (long long)((int64_t)B * S));
  return RA_OK;
}

template <int D, bool kVarlen>
ra_status launch_fwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const ra::FwdParams& prm, DeviceInfo* dev, cudaStream_t stream) {
  const size_t smem = sizeof(ra::FwdSmem<D>) + 1024;
  const int di = D == 128 ? 1 : 0;
  bool& attr_set = kVarlen ? dev->fwd_varlen_attr_set[di] : dev->fwd_attr_set[di];
  if (!attr_set) {
    // The kernel moves registers between warpgroups (setmaxnreg); that only
    // completes if the launch holds exactly the budget the split assumes.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, ra::attn_fwd_kernel<D, kVarlen>);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(fwd)");
    if (fa.numRegs != ra::kRegsLaunch)
      return fail(RA_ERR_UNSUPPORTED, "forward kernel built with %d registers/thread, expected %d",
                  fa.numRegs, ra::kRegsLaunch);
    e = cudaFuncSetAttribute(ra::attn_fwd_kernel<D, kVarlen>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(fwd smem)");
    attr_set = true;
  }
  if (prm.num_items == 0) return RA_OK;
  const int64_t grid = prm.num_items < dev->sms ? prm.num_items : dev->sms;
  ra::FwdParams run = prm;
  if (!kVarlen) run.sched = fwd_schedule(prm, (int)grid, stream);
  // Programmatic stream serialization for a launch of fewer CTAs than SMs:
  // it may begin while the kernel before it in the stream finishes (its CTAs
  // land on SMs that are free and wait in griddep_wait() before touching
  // global memory), so back-to-back small calls overlap one kernel's start
  // with the previous one's end.  A full-width launch gains nothing from it
  // and measured slower with it.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(384);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // (a traced call follows its own memset: never early)
  run.early = prm.trace == nullptr && grid < dev->sms ? 1 : 0;
  cfg.numAttrs = run.early ? 1 : 0;
  cudaError_t le = cudaLaunchKernelEx(&cfg, ra::attn_fwd_kernel<D, kVarlen>, mq, mk, mv, run);
  if (le != cudaSuccess) return cuda_fail(le, "attn_fwd_kernel launch");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_kernel launch");
  return RA_OK;
}

// (b, kv head) pairs per scheduling group of the forward.  One group (a global
// longest-first order) unless the key/value tiles of all pairs would overflow
// L2: then groups whose keys and values fit in about 3/4 of L2, as long as a
// group still spans at least 8 rounds of the grid (fewer rounds would cost
// more in load balance than the L2 hits gain).
int fwd_kv_group(const ra::Geo& g, bool step, const DeviceInfo* dev, int D) {
  const int BK = g.B * g.Hkv;
  const int64_t kv_bytes_pair = (int64_t)(step ? g.n : g.S) * D * 2 * 2;
  const int64_t budget = (int64_t)dev->l2_bytes * 3 / 4;
  if (kv_bytes_pair * BK <= budget) return BK;
  int64_t hg = budget / kv_bytes_pair;
  if (hg < 1) hg = 1;
  const int G = g.H / g.Hkv;
  const int64_t items_per_group = hg * G * ra::units_total(g, step);
  if (items_per_group < 8 * (int64_t)dev->sms) return BK;
  return (int)(hg < BK ? hg : BK);
}

ra_status fwd_impl(int mode, const void* q, const void* k, const void* v, void* out, int out_f32,
                   float* lse, int B, int H, int Hkv, int64_t S, int D, int P, int layout,
                   int causal, float scale, int r, int s, unsigned long long* shard_tiles,
                   cudaStream_t stream, unsigned long long* trace = nullptr,
                   int64_t trace_capacity = 0) {
  if (!q || !k || !v || !out) return fail(RA_ERR_NULL, "q, k, v and out must be non-NULL");
  ra_status st = check_common(B, H, Hkv, S, D, P, layout, scale);
  if (st != RA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(RA_ERR_ALIGN, "q, k, v and out must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(RA_ERR_ALIGN, "lse must be 4-byte aligned");
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != RA_OK) return st;

  ra::FwdParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.g = ra::make_geo(B, H, Hkv, S, P, layout, causal ? 1 : 0);
  prm.mode = mode;
  prm.step_r = r;
  prm.step_s = s;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.out = out;
  prm.out_f32 = out_f32;
  prm.lse = lse;
  prm.shard_tiles = shard_tiles;
  const bool step = mode == ra::FWD_MODE_STEP;
  prm.num_items = ra::units_total(prm.g, step) * B * H;
  prm.kv_group = fwd_kv_group(prm.g, step, dev, D);
  if (trace != nullptr) {
    if (trace_capacity < prm.num_items)
      return fail(RA_ERR_SHAPE, "the trace holds %lld records; this call has %lld work items",
                  (long long)trace_capacity, (long long)prm.num_items);
    cudaError_t e = cudaMemsetAsync(trace, 0, (size_t)prm.num_items * 4 * sizeof(int64_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the trace");
    prm.trace = trace;
  }

  CUtensorMap mq, mk, mv;
  const int64_t n = S / P;
  if (step) {
    st = make_token_map(&mq, q, D, H, 1, (int64_t)B * n);
    if (st == RA_OK) st = make_token_map(&mk, k, D, Hkv, 1, (int64_t)B * n);
    if (st == RA_OK) st = make_token_map(&mv, v, D, Hkv, 1, (int64_t)B * n);
  } else if (layout == RA_LAYOUT_STRIPED) {
    st = make_token_map(&mq, q, D, H, P, (int64_t)B * n);
    if (st == RA_OK) st = make_token_map(&mk, k, D, Hkv, P, (int64_t)B * n);
    if (st == RA_OK) st = make_token_map(&mv, v, D, Hkv, P, (int64_t)B * n);
  } else {
    st = make_token_map(&mq, q, D, H, 1, (int64_t)B * S);
    if (st == RA_OK) st = make_token_map(&mk, k, D, Hkv, 1, (int64_t)B * S);
    if (st == RA_OK) st = make_token_map(&mv, v, D, Hkv, 1, (int64_t)B * S);
  }
  if (st != RA_OK) return st;
  return D == 128 ? launch_fwd_d<128, false>(mq, mk, mv, prm, dev, stream)
                  : launch_fwd_d<64, false>(mq, mk, mv, prm, dev, stream);
}

struct BwdArgs {
  const void *q, *k, *v, *out;
  const float* lse;
  const void* dout;
  void *dq, *dk, *dv;
  int B, H, Hkv;
  int64_t S;
  int D, P, layout, causal;
  float scale;
};

ra_status check_bwd(const BwdArgs& a) {
  if (!a.q || !a.k || !a.v || !a.out || !a.lse || !a.dout || !a.dq || !a.dk || !a.dv)
    return fail(RA_ERR_NULL, "q, k, v, out, lse, dout, dq, dk and dv must be non-NULL");
  ra_status st = check_common(a.B, a.H, a.Hkv, a.S, a.D, a.P, a.layout, a.scale);
  if (st != RA_OK) return st;
  const void* p16[] = {a.q, a.k, a.v, a.out, a.dout, a.dq, a.dk, a.dv};
  for (const void* ptr : p16)
    if (!aligned16(ptr)) return fail(RA_ERR_ALIGN, "q, k, v, out, dout, dq, dk, dv must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(a.lse) & 3u) return fail(RA_ERR_ALIGN, "lse must be 4-byte aligned");
  return RA_OK;
}

template <int D, int kMode>
ra_status bwd_attrs(DeviceInfo* dev) {
  const size_t smem_kv = sizeof(ra::DkdvSmem<D>) + 1024;
  const size_t smem_q = sizeof(ra::DqSmem<D>) + 1024;
  const int di = (D == 128 ? 1 : 0) + 2 * kMode;
  if (!dev->bwd_attr_set[di]) {
    cudaError_t e = cudaFuncSetAttribute(ra::attn_bwd_dkdv_kernel<D, kMode>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_kv);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dkdv smem)");
    e = cudaFuncSetAttribute(ra::attn_bwd_dq_kernel<D, kMode>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dq smem)");
    dev->bwd_attr_set[di] = true;
  }
  return RA_OK;
}

template <int D>
ra_status launch_bwd_d(const BwdArgs& a, float* nlse2, float* ndelta, DeviceInfo* dev,
                       cudaStream_t stream, bool scheduled) {
  const size_t smem_kv = sizeof(ra::DkdvSmem<D>) + 1024;
  const size_t smem_q = sizeof(ra::DqSmem<D>) + 1024;
  {
    ra_status st0 = bwd_attrs<D, ra::BWD_RING>(dev);
    if (st0 != RA_OK) return st0;
  }
  ra::BwdParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.g = ra::make_geo(a.B, a.H, a.Hkv, a.S, a.P, a.layout, a.causal ? 1 : 0);
  prm.scale = a.scale;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.nlse2 = nlse2;
  prm.ndelta = ndelta;
  prm.dq = static_cast<__nv_bfloat16*>(a.dq);
  prm.dk = static_cast<__nv_bfloat16*>(a.dk);
  prm.dv = static_cast<__nv_bfloat16*>(a.dv);
  const ra::Geo& g = prm.g;

  CUtensorMap mq, mk, mv, mdo;
  const int64_t n = a.S / a.P;
  const bool striped = a.layout == RA_LAYOUT_STRIPED;
  const int64_t phases = striped ? a.P : 1;
  const int64_t rows = striped ? (int64_t)a.B * n : (int64_t)a.B * a.S;
  ra_status st = make_token_map(&mq, a.q, D, a.H, phases, rows);
  if (st == RA_OK) st = make_token_map(&mk, a.k, D, a.Hkv, phases, rows);
  if (st == RA_OK) st = make_token_map(&mv, a.v, D, a.Hkv, phases, rows);
  if (st == RA_OK) st = make_token_map(&mdo, a.dout, D, a.H, phases, rows);
  if (st != RA_OK) return st;

  // delta and -lse*log2(e) in tile order
  const int64_t vrows = ra::vec_elems(g);
  const int rows_per_block = 8 * (32 / (D / 8));
  int64_t blocks = (vrows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = (int64_t)dev->sms * 8;
  if (blocks > cap) blocks = cap;
  ra::bwd_prep_kernel<D, ra::BWD_RING><<<(unsigned)blocks, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.out), static_cast<const __nv_bfloat16*>(a.dout), a.lse,
      nlse2, ndelta, g, nullptr, nullptr, 0, 0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bwd_prep_kernel launch");

  const int64_t units = (int64_t)g.P * g.nseg * g.ntile;
  prm.num_items = units * a.B * a.Hkv;
  int64_t grid = prm.num_items < dev->sms ? prm.num_items : dev->sms;
  prm.sched = scheduled ? bwd_schedule(prm, true, false, (int)grid, stream) : nullptr;
  ra::attn_bwd_dkdv_kernel<D, ra::BWD_RING><<<(unsigned)grid, 384, smem_kv, stream>>>(mq, mk, mv, mdo, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_dkdv_kernel launch");

  prm.num_items = units * a.B * a.H;
  grid = prm.num_items < dev->sms ? prm.num_items : dev->sms;
  prm.sched = scheduled ? bwd_schedule(prm, false, false, (int)grid, stream) : nullptr;
  ra::attn_bwd_dq_kernel<D, ra::BWD_RING><<<(unsigned)grid, 384, smem_q, stream>>>(mq, mk, mv, mdo, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_dq_kernel launch");
  return RA_OK;
}

// One ring hop of the backward: shard r's queries against block s, fp32
// gradient contributions written or added into dq32 / dk32 / dv32.
template <int D>
ra_status launch_bwd_step_d(const BwdArgs& a, int r, int s, int accumulate, float* dq32,
                            float* dk32, float* dv32, float* nlse2, float* ndelta, DeviceInfo* dev,
                            cudaStream_t stream) {
  const size_t smem_kv = sizeof(ra::DkdvSmem<D>) + 1024;
  const size_t smem_q = sizeof(ra::DqSmem<D>) + 1024;
  {
    ra_status st0 = bwd_attrs<D, ra::BWD_STEP>(dev);
    if (st0 != RA_OK) return st0;
  }
  ra::BwdParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.g = ra::make_geo(a.B, a.H, a.Hkv, a.S, a.P, a.layout, a.causal ? 1 : 0);
  prm.scale = a.scale;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.nlse2 = nlse2;
  prm.ndelta = ndelta;
  prm.step_r = r;
  prm.step_s = s;
  prm.accumulate = accumulate ? 1 : 0;
  prm.dq32 = dq32;
  prm.dk32 = dk32;
  prm.dv32 = dv32;
  const ra::Geo& g = prm.g;
  CUtensorMap mq, mk, mv, mdo;
  const int64_t rows = (int64_t)a.B * g.n;    // shard-local tensors
  ra_status st = make_token_map(&mq, a.q, D, a.H, 1, rows);
  if (st == RA_OK) st = make_token_map(&mk, a.k, D, a.Hkv, 1, rows);
  if (st == RA_OK) st = make_token_map(&mv, a.v, D, a.Hkv, 1, rows);
  if (st == RA_OK) st = make_token_map(&mdo, a.dout, D, a.H, 1, rows);
  if (st != RA_OK) return st;
  const int64_t vrows = ra::vec_elems_step(g);
  const int rows_per_block = 8 * (32 / (D / 8));
  int64_t blocks = (vrows + rows_per_block - 1) / rows_per_block;
  if (blocks > (int64_t)dev->sms * 8) blocks = (int64_t)dev->sms * 8;
  ra::bwd_prep_kernel<D, ra::BWD_STEP><<<(unsigned)blocks, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.out), static_cast<const __nv_bfloat16*>(a.dout), a.lse,
      nlse2, ndelta, g, nullptr, nullptr, 0, r);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bwd_prep_kernel launch");
  const int64_t tiles = (int64_t)g.nseg * g.ntile;
  prm.num_items = tiles * a.B * a.Hkv;
  int64_t grid = prm.num_items < dev->sms ? prm.num_items : dev->sms;
  prm.sched = bwd_schedule(prm, true, true, (int)grid, stream);
  ra::attn_bwd_dkdv_kernel<D, ra::BWD_STEP><<<(unsigned)grid, 384, smem_kv, stream>>>(mq, mk, mv, mdo, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_dkdv_kernel launch");
  prm.num_items = tiles * a.B * a.H;
  grid = prm.num_items < dev->sms ? prm.num_items : dev->sms;
  prm.sched = bwd_schedule(prm, false, true, (int)grid, stream);
  ra::attn_bwd_dq_kernel<D, ra::BWD_STEP><<<(unsigned)grid, 384, smem_q, stream>>>(mq, mk, mv, mdo, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_dq_kernel launch");
  return RA_OK;
}

// Launches the three backward kernels on `stream` with caller-provided
// workspace: nlse2 and ndelta each hold vec_elems(geometry) floats.
// `scheduled`: deal the work items by the cached host schedule (which is
// allocated on first use of a shape) rather than the snake.
ra_status bwd_launch(const BwdArgs& a, float* nlse2, float* ndelta, cudaStream_t stream,
                     bool scheduled) {
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  return a.D == 128 ? launch_bwd_d<128>(a, nlse2, ndelta, dev, stream, scheduled)
                    : launch_bwd_d<64>(a, nlse2, ndelta, dev, stream, scheduled);
}

// ---------------------------------------------------------------- fixed backward workspace
// ring_attn_bwd_noalloc runs the backward on this statically sized device
// array instead of a cudaMallocAsync workspace.  Every GPU that loads the
// library holds it (16 MiB) until the process exits.  Host code must never
// pass the array's name to a kernel: on the host it is only a stand-in
// symbol.  The device address comes from cudaGetSymbolAddress with the device
// current.  Outside stream capture it is looked up on every call, so a
// context that was reset and loaded the module again is followed; while
// `stream` is capturing, the address found by the last uncaptured call on this
// device is used (the first call on a device must therefore come before any
// capture).
constexpr int64_t kFixedVecMax = int64_t(1) << 21;  // floats per vector (-lse*log2e, -delta)
static __device__ __align__(256) float g_bwd_fixed_ws[2 * kFixedVecMax];

std::mutex g_fixed_mu;
float* g_fixed_ws_ptr[64] = {nullptr};

ra_status fixed_workspace(cudaStream_t stream, float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(RA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    (void)cudaGetLastError();
    cap = cudaStreamCaptureStatusActive;   // unknown: do not call into the runtime's module state
  }
  std::lock_guard<std::mutex> lk(g_fixed_mu);
  if (cap == cudaStreamCaptureStatusNone || g_fixed_ws_ptr[dev] == nullptr) {
    if (cap != cudaStreamCaptureStatusNone)
      return fail(RA_ERR_UNSUPPORTED,
                  "ring_attn_bwd_noalloc: the first call on device %d must come before stream "
                  "capture (it looks up the fixed workspace's address)", dev);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_fixed_ws);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(fixed backward workspace)");
    g_fixed_ws_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_fixed_ws_ptr[dev];
  return RA_OK;
}

// ---------------------------------------------------------------- decode
// Query rows (H/Hkv)*T per key/value head a decode call takes: groups of 16
// rows run as separate CTAs over the same key/value chunk.
constexpr int kDecodeRowsMax = 4096;

template <int D>
ra_status launch_decode_d(const CUtensorMap& mk, const CUtensorMap& mv, const ra::DecodeParams& prm,
                          void* out, int out_f32, float* lse, DeviceInfo* dev,
                          cudaStream_t stream) {
  const size_t smem = sizeof(ra::DecodeSmem<D>) + 1024;
  const int di = D == 128 ? 1 : 0;
  if (!dev->dec_attr_set[di]) {
    cudaError_t e = cudaFuncSetAttribute(ra::decode_partial_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode smem)");
    dev->dec_attr_set[di] = true;
  }
  const ra::Geo& g = prm.g;
  dim3 grid((unsigned)(prm.chunks * prm.row_groups), (unsigned)(g.B * g.Hkv));
  ra::decode_partial_kernel<D><<<grid, ra::kDecodeThreads, smem, stream>>>(mk, mv, prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_partial_kernel launch");
  const int64_t items = (int64_t)g.B * g.Hkv * prm.rows;
  // programmatic stream serialization: the combine is scheduled while the
  // partial kernel's last CTAs run and waits (griddep_wait) for its partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)items);
  cfg.blockDim = dim3(ra::kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, ra::decode_combine_kernel<D>, (const float*)prm.part_o,
                         (const float*)prm.part_lse, out, out_f32, lse, g, prm.T, prm.rows,
                         prm.chunks);
  if (e != cudaSuccess) return cuda_fail(e, "decode_combine_kernel launch");
  return RA_OK;
}

// ---------------------------------------------------------------- packed sequences
// Checks cu_seqlens (host) and builds the longest-first unit list of a pack:
// (sequence, shard, segment, tile pair), ordered by the key tiles the pair
// multiplies (ties in pack order).
ra_status varlen_units(const int64_t* cu, int nseq, int H, int Hkv, int P, int layout, int causal,
                       std::vector<int4>* units) {
  if (!cu) return fail(RA_ERR_NULL, "cu_seqlens must be non-NULL");
  if (nseq < 1) return fail(RA_ERR_SHAPE, "nseq=%d must be positive", nseq);
  if (cu[0] != 0) return fail(RA_ERR_SHAPE, "cu_seqlens[0]=%lld must be 0", (long long)cu[0]);
  if (cu[nseq] > 0x7fffffffLL)
    return fail(RA_ERR_SHAPE, "the pack holds %lld tokens; at most 2^31-1", (long long)cu[nseq]);
  const int64_t unit_mult = layout == RA_LAYOUT_ZIGZAG ? 2 * (int64_t)P : P;
  std::vector<std::pair<int, int4>> tmp;
  for (int i = 0; i < nseq; ++i) {
    const int64_t L = cu[i + 1] - cu[i];
    if (L < 1) return fail(RA_ERR_SHAPE, "sequence %d has length %lld", i, (long long)L);
    if (L % unit_mult != 0)
      return fail(RA_ERR_LAYOUT, "sequence %d: length %lld not divisible by %lld", i,
                  (long long)L, (long long)unit_mult);
    const ra::Geo g = ra::make_geo(1, H, Hkv, L, P, layout, causal ? 1 : 0);
    for (int r = 0; r < P; ++r)
      for (int sg = 0; sg < g.nseg; ++sg)
        for (int pr = 0; pr < g.npair; ++pr) {
          const ra::QTile qa = ra::make_qtile(g, r, sg, 2 * pr), qb = ra::make_qtile(g, r, sg, 2 * pr + 1);
          const int cost = ra::tile_work(g, qa, -1) + ra::tile_work(g, qb, -1);
          if (cost > 0) tmp.push_back({cost, make_int4(i, r, sg, pr)});
        }
  }
  std::stable_sort(tmp.begin(), tmp.end(),
                   [](const std::pair<int, int4>& a, const std::pair<int, int4>& b) {
                     return a.first > b.first;
                   });
  units->clear();
  for (auto& t : tmp) units->push_back(t.second);
  return RA_OK;
}

// Backward over packed sequences: unit lists, vector offsets and the launches.
template <int D>
ra_status launch_bwd_varlen_d(const BwdArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, const CUtensorMap& mdo, ra::BwdParams prm,
                              int nseq, int64_t max_vec, int nk, int nq, DeviceInfo* dev,
                              cudaStream_t stream) {
  ra_status st = bwd_attrs<D, ra::BWD_VARLEN>(dev);
  if (st != RA_OK) return st;
  const size_t smem_kv = sizeof(ra::DkdvSmem<D>) + 1024;
  const size_t smem_q = sizeof(ra::DqSmem<D>) + 1024;
  const int rows_per_block = 8 * (32 / (D / 8));
  int64_t bx = (max_vec + rows_per_block - 1) / rows_per_block;
  if (bx > (int64_t)dev->sms * 8) bx = (int64_t)dev->sms * 8;
  ra::bwd_prep_kernel<D, ra::BWD_VARLEN><<<dim3((unsigned)bx, (unsigned)nseq), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.out), static_cast<const __nv_bfloat16*>(a.dout), a.lse,
      const_cast<float*>(prm.nlse2), const_cast<float*>(prm.ndelta), prm.g, prm.cu_seqlens,
      prm.vbase, prm.total, 0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bwd_prep_kernel launch");
  const int4* qunits = prm.units + nk;
  prm.num_items = (int64_t)nk * a.Hkv;
  int64_t grid = prm.num_items < dev->sms ? prm.num_items : dev->sms;
  ra::attn_bwd_dkdv_kernel<D, ra::BWD_VARLEN><<<(unsigned)grid, 384, smem_kv, stream>>>(mq, mk, mv, mdo, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_dkdv_kernel launch");
  prm.units = qunits;
  prm.num_items = (int64_t)nq * a.H;
  grid = prm.num_items < dev->sms ? prm.num_items : dev->sms;
  ra::attn_bwd_dq_kernel<D, ra::BWD_VARLEN><<<(unsigned)grid, 384, smem_q, stream>>>(mq, mk, mv, mdo, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_dq_kernel launch");
  return RA_OK;
}

}  // namespace

extern "C" {

ra_status ring_attn_fwd(const void* q, const void* k, const void* v, void* out, ra_dtype out_dtype,
                        float* lse, int B, int H, int Hkv, int64_t S, int D, int P,
                        ra_layout layout, int causal, float scale, void* stream) {
  if (out_dtype != RA_BF16 && out_dtype != RA_F32)
    return fail(RA_ERR_UNSUPPORTED, "out_dtype %d", (int)out_dtype);
  return fwd_impl(ra::FWD_MODE_RING, q, k, v, out, out_dtype == RA_F32, lse, B, H, Hkv, S, D, P,
                  layout, causal, scale, 0, 0, nullptr, static_cast<cudaStream_t>(stream));
}

ra_status ring_attn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                               ra_dtype out_dtype, float* lse, const int64_t* cu_seqlens, int nseq,
                               int H, int Hkv, int D, int P, ra_layout layout, int causal,
                               float scale, void* stream) {
  if (!q || !k || !v || !out) return fail(RA_ERR_NULL, "q, k, v and out must be non-NULL");
  if (out_dtype != RA_BF16 && out_dtype != RA_F32)
    return fail(RA_ERR_UNSUPPORTED, "out_dtype %d", (int)out_dtype);
  if (!cu_seqlens || nseq < 1) return fail(RA_ERR_NULL, "cu_seqlens and nseq >= 1 are required");
  const int64_t total = cu_seqlens[nseq];
  ra_status st = check_common(1, H, Hkv, total > 0 ? total : 1, D, P, (int)layout, scale);
  if (st != RA_OK) return st;
  std::vector<int4> units;
  st = varlen_units(cu_seqlens, nseq, H, Hkv, P, (int)layout, causal, &units);
  if (st != RA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(RA_ERR_ALIGN, "q, k, v and out must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(RA_ERR_ALIGN, "lse must be 4-byte aligned");
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != RA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (units.empty()) return RA_OK;
  // the unit list and cu_seqlens go to the device with the call
  const size_t ub = units.size() * sizeof(int4), cb = (size_t)(nseq + 1) * sizeof(int64_t);
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, ub + cb, cs);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(RA_ERR_ALLOC, "cudaMallocAsync(%zu bytes) for the unit list: %s", ub + cb,
                cudaGetErrorString(e));
  }
  e = cudaMemcpyAsync(ws, units.data(), ub, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(static_cast<char*>(ws) + ub, cu_seqlens, cb, cudaMemcpyHostToDevice, cs);
  if (e != cudaSuccess) {
    cudaFreeAsync(ws, cs);
    return cuda_fail(e, "copying the unit list");
  }
  ra::FwdParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.g = ra::make_geo(1, H, Hkv, total, P, (int)layout, causal ? 1 : 0);
  prm.mode = ra::FWD_MODE_RING;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.out = out;
  prm.out_f32 = out_dtype == RA_F32;
  prm.lse = lse;
  prm.num_items = (int64_t)units.size() * H;
  prm.kv_group = Hkv;
  prm.units = static_cast<const int4*>(ws);
  prm.cu_seqlens = reinterpret_cast<const int64_t*>(static_cast<char*>(ws) + ub);
  prm.total = (int)total;
  CUtensorMap mq, mk, mv;
  const bool striped = layout == RA_LAYOUT_STRIPED;
  const int64_t phases = striped ? P : 1;
  const int64_t rows = striped ? total / P : total;
  st = make_token_map(&mq, q, D, H, phases, rows);
  if (st == RA_OK) st = make_token_map(&mk, k, D, Hkv, phases, rows);
  if (st == RA_OK) st = make_token_map(&mv, v, D, Hkv, phases, rows);
  if (st == RA_OK)
    st = D == 128 ? launch_fwd_d<128, true>(mq, mk, mv, prm, dev, cs)
                  : launch_fwd_d<64, true>(mq, mk, mv, prm, dev, cs);
  e = cudaFreeAsync(ws, cs);
  if (st != RA_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(unit list)");
  return RA_OK;
}

ra_status ring_attn_fwd_counted(const void* q, const void* k, const void* v, void* out,
                                ra_dtype out_dtype, float* lse, int B, int H, int Hkv, int64_t S,
                                int D, int P, ra_layout layout, int causal, float scale,
                                int64_t* shard_tiles, void* stream) {
  if (out_dtype != RA_BF16 && out_dtype != RA_F32)
    return fail(RA_ERR_UNSUPPORTED, "out_dtype %d", (int)out_dtype);
  if (!shard_tiles) return fail(RA_ERR_NULL, "shard_tiles must be non-NULL");
  if (reinterpret_cast<uintptr_t>(shard_tiles) & 7u)
    return fail(RA_ERR_ALIGN, "shard_tiles must be 8-byte aligned");
  return fwd_impl(ra::FWD_MODE_RING, q, k, v, out, out_dtype == RA_F32, lse, B, H, Hkv, S, D, P,
                  layout, causal, scale, 0, 0,
                  reinterpret_cast<unsigned long long*>(shard_tiles),
                  static_cast<cudaStream_t>(stream));
}

ra_status ring_attn_fwd_traced(const void* q, const void* k, const void* v, void* out,
                               ra_dtype out_dtype, float* lse, int B, int H, int Hkv, int64_t S,
                               int D, int P, ra_layout layout, int causal, float scale,
                               int64_t* records, int64_t capacity, int64_t* items, void* stream) {
  if (out_dtype != RA_BF16 && out_dtype != RA_F32)
    return fail(RA_ERR_UNSUPPORTED, "out_dtype %d", (int)out_dtype);
  if (!records || !items) return fail(RA_ERR_NULL, "records and items must be non-NULL");
  if (reinterpret_cast<uintptr_t>(records) & 7u)
    return fail(RA_ERR_ALIGN, "records must be 8-byte aligned");
  ra_status st = check_common(B, H, Hkv, S, D, P, (int)layout, scale);
  if (st != RA_OK) return st;
  *items = ra::units_total(ra::make_geo(B, H, Hkv, S, P, (int)layout, causal ? 1 : 0), false) *
           B * H;
  return fwd_impl(ra::FWD_MODE_RING, q, k, v, out, out_dtype == RA_F32, lse, B, H, Hkv, S, D, P,
                  layout, causal, scale, 0, 0, nullptr, static_cast<cudaStream_t>(stream),
                  reinterpret_cast<unsigned long long*>(records), capacity);
}

ra_status ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                        int H, int Hkv, int64_t S, int D, int P, ra_layout layout, int causal,
                        float scale, void* stream) {
  BwdArgs a{q, k, v, out, lse, dout, dq, dk, dv, B, H, Hkv, S, D, P, (int)layout, causal, scale};
  ra_status st = check_bwd(a);
  if (st != RA_OK) return st;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != RA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const ra::Geo g = ra::make_geo(B, H, Hkv, S, P, (int)layout, causal ? 1 : 0);
  const size_t vec_bytes = (size_t)ra::vec_elems(g) * sizeof(float);
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, 2 * vec_bytes, cs);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(RA_ERR_ALLOC, "cudaMallocAsync(%zu bytes) for the backward workspace: %s",
                2 * vec_bytes, cudaGetErrorString(e));
  }
  float* nlse2 = static_cast<float*>(ws);
  float* ndelta = reinterpret_cast<float*>(static_cast<char*>(ws) + vec_bytes);
  st = bwd_launch(a, nlse2, ndelta, cs, true);
  e = cudaFreeAsync(ws, cs);
  if (st != RA_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(backward workspace)");
  return RA_OK;
}

ra_status ring_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               const int64_t* cu_seqlens, int nseq, int H, int Hkv, int D, int P,
                               ra_layout layout, int causal, float scale, void* stream) {
  if (!cu_seqlens || nseq < 1) return fail(RA_ERR_NULL, "cu_seqlens and nseq >= 1 are required");
  const int64_t total = cu_seqlens[nseq];
  BwdArgs a{q, k, v, out, lse, dout, dq, dk, dv, 1, H, Hkv, total > 0 ? total : 1, D, P,
            (int)layout, causal, scale};
  ra_status st = check_bwd(a);
  if (st != RA_OK) return st;
  std::vector<int4> fwd_units;   // validates cu_seqlens against the layout
  st = varlen_units(cu_seqlens, nseq, H, Hkv, P, (int)layout, causal, &fwd_units);
  if (st != RA_OK) return st;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != RA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // key-tile and query-tile units, longest first; vector offsets per sequence
  std::vector<std::pair<int64_t, int4>> ku, qu;
  std::vector<int64_t> vbase(nseq);
  int64_t V = 0, max_vec = 0;
  for (int i = 0; i < nseq; ++i) {
    const ra::Geo g = ra::make_geo(1, H, Hkv, cu_seqlens[i + 1] - cu_seqlens[i], P, (int)layout,
                                   causal ? 1 : 0);
    vbase[i] = V;
    V += ra::vec_elems(g);
    if (ra::vec_elems(g) > max_vec) max_vec = ra::vec_elems(g);
    for (int r = 0; r < P; ++r)
      for (int sg = 0; sg < g.nseg; ++sg)
        for (int t = 0; t < g.ntile; ++t) {
          const ra::QTile tl = ra::make_qtile(g, r, sg, t);
          if (!tl.valid) continue;
          qu.push_back({ra::tile_work(g, tl, -1), make_int4(i, r, sg, t)});
          int64_t cost = 0;   // query tiles this key tile meets
          for (int rq = 0; rq < P; ++rq)
            for (int sq = 0; sq < g.nseg; ++sq) {
              const ra::Seg qs = ra::segment_of(g, rq, sq);
              const int first = g.causal ? ra::count_le(qs, tl.qmin - 1) : 0;
              if (first < qs.len) cost += g.ntile - first / ra::kTile;
            }
          ku.push_back({cost, make_int4(i, r, sg, t)});
        }
  }
  auto by_cost = [](const std::pair<int64_t, int4>& x, const std::pair<int64_t, int4>& y) {
    return x.first > y.first;
  };
  std::stable_sort(ku.begin(), ku.end(), by_cost);
  std::stable_sort(qu.begin(), qu.end(), by_cost);
  std::vector<int4> units;
  for (auto& x : ku) units.push_back(x.second);
  for (auto& x : qu) units.push_back(x.second);
  const int nk = (int)ku.size(), nq = (int)qu.size();
  // workspace: nlse2, ndelta [V] fp32 | units | cu_seqlens | vbase
  const size_t vb = (size_t)V * sizeof(float), ub = units.size() * sizeof(int4);
  const size_t cb = (size_t)(nseq + 1) * sizeof(int64_t), bb = (size_t)nseq * sizeof(int64_t);
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, 2 * vb + ub + cb + bb, cs);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(RA_ERR_ALLOC, "cudaMallocAsync(%zu bytes) for the backward workspace: %s",
                2 * vb + ub + cb + bb, cudaGetErrorString(e));
  }
  char* w8 = static_cast<char*>(ws);
  e = cudaMemcpyAsync(w8 + 2 * vb, units.data(), ub, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaMemcpyAsync(w8 + 2 * vb + ub, cu_seqlens, cb, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaMemcpyAsync(w8 + 2 * vb + ub + cb, vbase.data(), bb, cudaMemcpyHostToDevice, cs);
  if (e != cudaSuccess) {
    cudaFreeAsync(ws, cs);
    return cuda_fail(e, "copying the unit lists");
  }
  ra::BwdParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.g = ra::make_geo(1, H, Hkv, total, P, (int)layout, causal ? 1 : 0);
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.nlse2 = reinterpret_cast<float*>(w8);
  prm.ndelta = reinterpret_cast<float*>(w8 + vb);
  prm.dq = static_cast<__nv_bfloat16*>(dq);
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.units = reinterpret_cast<const int4*>(w8 + 2 * vb);
  prm.cu_seqlens = reinterpret_cast<const int64_t*>(w8 + 2 * vb + ub);
  prm.vbase = reinterpret_cast<const int64_t*>(w8 + 2 * vb + ub + cb);
  prm.total = (int)total;
  CUtensorMap mq, mk, mv, mdo;
  const bool striped = layout == RA_LAYOUT_STRIPED;
  const int64_t phases = striped ? P : 1;
  const int64_t rows = striped ? total / P : total;
  st = make_token_map(&mq, q, D, H, phases, rows);
  if (st == RA_OK) st = make_token_map(&mk, k, D, Hkv, phases, rows);
  if (st == RA_OK) st = make_token_map(&mv, v, D, Hkv, phases, rows);
  if (st == RA_OK) st = make_token_map(&mdo, dout, D, H, phases, rows);
  if (st == RA_OK)
    st = D == 128 ? launch_bwd_varlen_d<128>(a, mq, mk, mv, mdo, prm, nseq, max_vec, nk, nq, dev, cs)
                  : launch_bwd_varlen_d<64>(a, mq, mk, mv, mdo, prm, nseq, max_vec, nk, nq, dev, cs);
  e = cudaFreeAsync(ws, cs);
  if (st != RA_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(backward workspace)");
  return RA_OK;
}

ra_status ring_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                int B, int H, int Hkv, int64_t S, int D, int P, ra_layout layout,
                                int causal, float scale, void* stream) {
  BwdArgs a{q, k, v, out, lse, dout, dq, dk, dv, B, H, Hkv, S, D, P, (int)layout, causal, scale};
  ra_status st = check_bwd(a);
  if (st != RA_OK) return st;
  const ra::Geo g = ra::make_geo(B, H, Hkv, S, P, (int)layout, causal ? 1 : 0);
  const int64_t need = ra::vec_elems(g);
  if (need > kFixedVecMax)
    return fail(RA_ERR_SHAPE,
                "ring_attn_bwd_noalloc: this problem needs a workspace of 2 x %lld floats "
                "(B*H*P*T*128 with T 128-slot tiles per shard); the fixed workspace holds "
                "2 x %lld.  Use ring_attn_bwd instead",
                (long long)need, (long long)kFixedVecMax);
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != RA_OK) return st;
  float* ws = nullptr;
  st = fixed_workspace(static_cast<cudaStream_t>(stream), &ws);
  if (st != RA_OK) return st;
  return bwd_launch(a, ws, ws + kFixedVecMax, static_cast<cudaStream_t>(stream), false);
}

ra_status ring_attn_decode(const void* q, const void* k_cache, const void* v_cache, void* out,
                           ra_dtype out_dtype, float* lse, int B, int H, int Hkv, int T, int64_t S,
                           int D, int P, ra_layout layout, float scale, void* stream) {
  if (!q || !k_cache || !v_cache || !out)
    return fail(RA_ERR_NULL, "q, k_cache, v_cache and out must be non-NULL");
  if (out_dtype != RA_BF16 && out_dtype != RA_F32)
    return fail(RA_ERR_UNSUPPORTED, "out_dtype %d", (int)out_dtype);
  ra_status st = check_common(B, H, Hkv, S, D, P, (int)layout, scale);
  if (st != RA_OK) return st;
  if (T < 1 || T > S) return fail(RA_ERR_SHAPE, "T=%d new tokens must be in [1, S=%lld]", T, (long long)S);
  if ((int64_t)(H / Hkv) * T > kDecodeRowsMax)
    return fail(RA_ERR_UNSUPPORTED, "(H/Hkv)*T = %lld query rows per kv head; at most %d",
                (long long)(H / Hkv) * T, kDecodeRowsMax);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(RA_ERR_ALIGN, "q, k_cache, v_cache and out must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(RA_ERR_ALIGN, "lse must be 4-byte aligned");
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != RA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  ra::DecodeParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.g = ra::make_geo(B, H, Hkv, S, P, (int)layout, 1);
  const ra::Geo& g = prm.g;
  prm.T = T;
  prm.rows = (H / Hkv) * T;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.row_groups = (prm.rows + ra::kDecodeMaxRows - 1) / ra::kDecodeMaxRows;
  // Chunks of a shard segment's 128-slot tiles: about two CTAs per SM in all
  // (each chunk runs one CTA per row group).
  const int64_t tiles = (int64_t)B * Hkv * P * g.nseg * g.ntile * prm.row_groups;
  int64_t ct = (tiles + 2 * dev->sms - 1) / (2 * (int64_t)dev->sms);
  if (ct < 1) ct = 1;
  if (ct > g.ntile) ct = g.ntile;
  const int64_t per_seg = (g.ntile + ct - 1) / ct;
  ct = (g.ntile + per_seg - 1) / per_seg;        // even out the chunks of a segment
  prm.chunk_tiles = (int)ct;
  prm.chunks_per_seg = (g.ntile + prm.chunk_tiles - 1) / prm.chunk_tiles;
  prm.chunks = P * g.nseg * prm.chunks_per_seg;

  const size_t n_lse = (size_t)B * Hkv * prm.chunks * prm.rows;
  const size_t bytes = n_lse * sizeof(float) * (size_t)(D + 1);
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, bytes, cs);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(RA_ERR_ALLOC, "cudaMallocAsync(%zu bytes) for decode partials: %s", bytes,
                cudaGetErrorString(e));
  }
  prm.part_o = static_cast<float*>(ws);
  prm.part_lse = prm.part_o + n_lse * D;

  CUtensorMap mk, mv;
  const int64_t n = S / P;
  const bool striped = layout == RA_LAYOUT_STRIPED;
  const int64_t phases = striped ? P : 1;
  const int64_t rows = striped ? (int64_t)B * n : (int64_t)B * S;
  st = make_token_map(&mk, k_cache, D, Hkv, phases, rows);
  if (st == RA_OK) st = make_token_map(&mv, v_cache, D, Hkv, phases, rows);
  if (st == RA_OK)
    st = D == 128 ? launch_decode_d<128>(mk, mv, prm, out, out_dtype == RA_F32, lse, dev, cs)
                  : launch_decode_d<64>(mk, mv, prm, out, out_dtype == RA_F32, lse, dev, cs);
  e = cudaFreeAsync(ws, cs);
  if (st != RA_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(decode partials)");
  return RA_OK;
}

ra_status ring_attn_cache_append(void* k_cache, void* v_cache, const void* k_new,
                                 const void* v_new, int B, int Hkv, int64_t S_cap, int64_t pos,
                                 int T, int D, void* stream) {
  if (!k_cache || !v_cache || !k_new || !v_new)
    return fail(RA_ERR_NULL, "k_cache, v_cache, k_new and v_new must be non-NULL");
  if (B < 1 || Hkv < 1 || T < 1 || S_cap < 1 || pos < 0)
    return fail(RA_ERR_SHAPE, "sizes must be positive (B=%d Hkv=%d T=%d S_cap=%lld pos=%lld)", B,
                Hkv, T, (long long)S_cap, (long long)pos);
  if (pos + T > S_cap)
    return fail(RA_ERR_SHAPE, "pos=%lld + T=%d exceeds the cache's %lld rows", (long long)pos, T,
                (long long)S_cap);
  if (D != 64 && D != 128) return fail(RA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
    return fail(RA_ERR_ALIGN, "cache and new-token pointers must be 16-byte aligned");
  const int64_t row = (int64_t)Hkv * D * 2 / 16;   // 16-byte vectors per token row
  const int64_t nb = (int64_t)B * T * row * 16;
  const char* ranges[4] = {static_cast<const char*>(k_cache), static_cast<const char*>(v_cache),
                           static_cast<const char*>(k_new), static_cast<const char*>(v_new)};
  const int64_t lens[4] = {(int64_t)B * S_cap * row * 16, (int64_t)B * S_cap * row * 16, nb, nb};
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (ranges[i] < ranges[j] + lens[j] && ranges[j] < ranges[i] + lens[i])
        return fail(RA_ERR_SHAPE, "cache and new-token buffers overlap");
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  const int64_t total = (int64_t)B * T * row;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)dev->sms * 8) blocks = (int64_t)dev->sms * 8;
  ra::cache_append_kernel<<<dim3((unsigned)blocks, 2), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), B, S_cap, pos, T, row);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "cache_append_kernel launch");
  return RA_OK;
}

ra_status ring_attn_step(const void* q_shard, const void* k_shard, const void* v_shard,
                         float* out_part, float* lse_part, int B, int H, int Hkv, int64_t S, int D,
                         int P, ra_layout layout, int r, int s, int causal, float scale,
                         void* stream) {
  if (!lse_part) return fail(RA_ERR_NULL, "lse_part must be non-NULL");
  if (P >= 1 && (r < 0 || r >= P || s < 0 || s >= P))
    return fail(RA_ERR_SHAPE, "shard indices r=%d s=%d outside [0, %d)", r, s, P);
  return fwd_impl(ra::FWD_MODE_STEP, q_shard, k_shard, v_shard, out_part, 1, lse_part, B, H, Hkv,
                  S, D, P, layout, causal, scale, r, s, nullptr, static_cast<cudaStream_t>(stream));
}

ra_status ring_attn_step_bwd(const void* q_shard, const void* k_shard, const void* v_shard,
                             const void* out_shard, const float* lse_shard, const void* dout_shard,
                             float* dq_part, float* dk_part, float* dv_part, int B, int H, int Hkv,
                             int64_t S, int D, int P, ra_layout layout, int r, int s, int causal,
                             float scale, int accumulate, void* stream) {
  if (!dq_part || !dk_part || !dv_part) return fail(RA_ERR_NULL, "dq_part, dk_part and dv_part must be non-NULL");
  BwdArgs a{q_shard, k_shard, v_shard, out_shard, lse_shard, dout_shard, dq_part, dk_part, dv_part,
            B, H, Hkv, S, D, P, (int)layout, causal, scale};
  ra_status st = check_bwd(a);
  if (st != RA_OK) return st;
  if (r < 0 || r >= P || s < 0 || s >= P)
    return fail(RA_ERR_SHAPE, "shard indices r=%d s=%d outside [0, %d)", r, s, P);
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != RA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const ra::Geo g = ra::make_geo(B, H, Hkv, S, P, (int)layout, causal ? 1 : 0);
  const size_t vec_bytes = (size_t)ra::vec_elems_step(g) * sizeof(float);
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, 2 * vec_bytes, cs);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(RA_ERR_ALLOC, "cudaMallocAsync(%zu bytes) for the hop workspace: %s",
                2 * vec_bytes, cudaGetErrorString(e));
  }
  float* nlse2 = static_cast<float*>(ws);
  float* ndelta = reinterpret_cast<float*>(static_cast<char*>(ws) + vec_bytes);
  st = D == 128 ? launch_bwd_step_d<128>(a, r, s, accumulate, dq_part, dk_part, dv_part, nlse2,
                                         ndelta, dev, cs)
                : launch_bwd_step_d<64>(a, r, s, accumulate, dq_part, dk_part, dv_part, nlse2,
                                        ndelta, dev, cs);
  e = cudaFreeAsync(ws, cs);
  if (st != RA_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(hop workspace)");
  return RA_OK;
}

ra_status ring_attn_merge(float* out_acc, float* lse_acc, const float* out_part,
                          const float* lse_part, int B, int H, int64_t n, int D, void* stream) {
  if (!out_acc || !lse_acc || !out_part || !lse_part)
    return fail(RA_ERR_NULL, "merge pointers must be non-NULL");
  if (B < 1 || H < 1 || n < 1) return fail(RA_ERR_SHAPE, "sizes must be positive");
  if (D != 64 && D != 128) return fail(RA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
  if (!aligned16(out_acc) || !aligned16(out_part))
    return fail(RA_ERR_ALIGN, "out_acc and out_part must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse_acc) | reinterpret_cast<uintptr_t>(lse_part)) & 3u)
    return fail(RA_ERR_ALIGN, "lse pointers must be 4-byte aligned");
  if (H > 2048) return fail(RA_ERR_UNSUPPORTED, "H=%d heads; the merge takes at most 2048", H);
  if (n > 0x7fffffffLL) return fail(RA_ERR_SHAPE, "n=%lld exceeds 2^31-1", (long long)n);
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  const size_t smem = 2 * (size_t)H * ra::kMergeTok * sizeof(float);
  const void* fn = D == 128 ? (const void*)ra::merge_kernel<128> : (const void*)ra::merge_kernel<64>;
  if (smem > 48 * 1024) {
    cudaError_t ae = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem);
    if (ae != cudaSuccess) return cuda_fail(ae, "cudaFuncSetAttribute(merge smem)");
  }
  // one wave of resident blocks; each strides over the token tiles
  int per_sm = 0;
  cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, ra::kMergeThreads,
                                                                 smem);
  if (oe != cudaSuccess) return cuda_fail(oe, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(merge)");
  const int64_t tiles = (int64_t)B * ((n + ra::kMergeTok - 1) / ra::kMergeTok);
  const int64_t cap = (int64_t)dev->sms * (per_sm > 0 ? per_sm : 1);
  const int64_t blocks = tiles < cap ? tiles : cap;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (D == 128)
    ra::merge_kernel<128><<<(unsigned)blocks, ra::kMergeThreads, smem, cs>>>(
        out_acc, lse_acc, out_part, lse_part, B, H, (int)n);
  else
    ra::merge_kernel<64><<<(unsigned)blocks, ra::kMergeThreads, smem, cs>>>(
        out_acc, lse_acc, out_part, lse_part, B, H, (int)n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "merge_kernel launch");
  return RA_OK;
}

ra_status ring_attn_permute(const void* src, void* dst, int64_t outer, int64_t S, int64_t row_bytes,
                            int P, ra_layout layout, int inverse, void* stream) {
  if (!src || !dst) return fail(RA_ERR_NULL, "src and dst must be non-NULL");
  if (outer < 1 || S < 1 || P < 1 || row_bytes < 4 || row_bytes % 4 != 0)
    return fail(RA_ERR_SHAPE, "bad permute sizes (outer=%lld S=%lld row_bytes=%lld P=%d)",
                (long long)outer, (long long)S, (long long)row_bytes, P);
  if ((int)layout < 0 || (int)layout > 2) return fail(RA_ERR_LAYOUT, "unknown layout %d", (int)layout);
  if (S % P != 0) return fail(RA_ERR_LAYOUT, "S=%lld is not divisible by P=%d", (long long)S, P);
  if (layout == RA_LAYOUT_ZIGZAG && S % (2 * (int64_t)P) != 0)
    return fail(RA_ERR_LAYOUT, "zig-zag needs S divisible by 2P");
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (a & 3u) return fail(RA_ERR_ALIGN, "src and dst must be 4-byte aligned");
  const char* s8 = static_cast<const char*>(src);
  const char* d8 = static_cast<const char*>(dst);
  const int64_t bytes = outer * S * row_bytes;
  if (s8 < d8 + bytes && d8 < s8 + bytes) return fail(RA_ERR_SHAPE, "src and dst overlap");
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  ra::Geo g = ra::make_geo(1, 1, 1, S, P, layout, 0);
  const bool v16 = (a & 15u) == 0 && row_bytes % 16 == 0;
  const int64_t pieces = outer * S * (row_bytes / (v16 ? 16 : 4));
  int64_t blocks = (pieces + 255) / 256;
  const int64_t cap = (int64_t)dev->sms * 16;
  if (blocks > cap) blocks = cap;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (v16)
    ra::permute_kernel<uint4><<<(unsigned)blocks, 256, 0, cs>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), outer, g, row_bytes, inverse);
  else
    ra::permute_kernel<uint32_t><<<(unsigned)blocks, 256, 0, cs>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), outer, g, row_bytes, inverse);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "permute_kernel launch");
  return RA_OK;
}

ra_status ring_attn_permute_shards(const void* src, void* dst, int64_t outer, int64_t S,
                                   int64_t row_bytes, int P, ra_layout layout, int inverse,
                                   void* stream) {
  if (!src || !dst) return fail(RA_ERR_NULL, "src and dst must be non-NULL");
  if (outer < 1 || S < 1 || P < 1 || row_bytes < 4 || row_bytes % 4 != 0)
    return fail(RA_ERR_SHAPE, "bad permute sizes (outer=%lld S=%lld row_bytes=%lld P=%d)",
                (long long)outer, (long long)S, (long long)row_bytes, P);
  if ((int)layout < 0 || (int)layout > 2) return fail(RA_ERR_LAYOUT, "unknown layout %d", (int)layout);
  if (S % P != 0) return fail(RA_ERR_LAYOUT, "S=%lld is not divisible by P=%d", (long long)S, P);
  if (layout == RA_LAYOUT_ZIGZAG && S % (2 * (int64_t)P) != 0)
    return fail(RA_ERR_LAYOUT, "zig-zag needs S divisible by 2P");
  if (S > 0x7fffffffLL) return fail(RA_ERR_SHAPE, "S=%lld exceeds 2^31-1", (long long)S);
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (a & 3u) return fail(RA_ERR_ALIGN, "src and dst must be 4-byte aligned");
  const char* s8 = static_cast<const char*>(src);
  const char* d8 = static_cast<const char*>(dst);
  const int64_t bytes = outer * S * row_bytes;
  if (s8 < d8 + bytes && d8 < s8 + bytes) return fail(RA_ERR_SHAPE, "src and dst overlap");
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  ra::Geo g = ra::make_geo(1, 1, 1, S, P, layout, 0);
  const bool v16 = (a & 15u) == 0 && row_bytes % 16 == 0;
  const int64_t pieces = outer * S * (row_bytes / (v16 ? 16 : 4));
  int64_t blocks = (pieces + 255) / 256;
  if (blocks > (int64_t)dev->sms * 16) blocks = (int64_t)dev->sms * 16;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (v16)
    ra::permute_shards_kernel<uint4><<<(unsigned)blocks, 256, 0, cs>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), outer, g, row_bytes, inverse);
  else
    ra::permute_shards_kernel<uint32_t><<<(unsigned)blocks, 256, 0, cs>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), outer, g, row_bytes, inverse);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "permute_shards_kernel launch");
  return RA_OK;
}

ra_status ring_attn_head_split(const void* src, void* dst, int64_t rows, int parts,
                               int64_t chunk_bytes, int inverse, void* stream) {
  if (!src || !dst) return fail(RA_ERR_NULL, "src and dst must be non-NULL");
  if (rows < 1 || parts < 1 || chunk_bytes < 4 || chunk_bytes % 4 != 0)
    return fail(RA_ERR_SHAPE, "bad head-split sizes (rows=%lld parts=%d chunk_bytes=%lld)",
                (long long)rows, parts, (long long)chunk_bytes);
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (a & 3u) return fail(RA_ERR_ALIGN, "src and dst must be 4-byte aligned");
  const char* s8 = static_cast<const char*>(src);
  const char* d8 = static_cast<const char*>(dst);
  const int64_t bytes = rows * parts * chunk_bytes;
  if (s8 < d8 + bytes && d8 < s8 + bytes) return fail(RA_ERR_SHAPE, "src and dst overlap");
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  const bool v16 = (a & 15u) == 0 && chunk_bytes % 16 == 0;
  const int64_t pieces = rows * parts * (chunk_bytes / (v16 ? 16 : 4));
  int64_t blocks = (pieces + 255) / 256;
  if (blocks > (int64_t)dev->sms * 16) blocks = (int64_t)dev->sms * 16;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (v16)
    ra::head_split_kernel<uint4><<<(unsigned)blocks, 256, 0, cs>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), rows, parts, chunk_bytes,
        inverse);
  else
    ra::head_split_kernel<uint32_t><<<(unsigned)blocks, 256, 0, cs>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), rows, parts, chunk_bytes,
        inverse);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "head_split_kernel launch");
  return RA_OK;
}

ra_status ring_attn_finalize(const float* acc, void* out, int64_t count, void* stream) {
  if (!acc || !out) return fail(RA_ERR_NULL, "acc and out must be non-NULL");
  if (count < 1 || count % 4 != 0)
    return fail(RA_ERR_SHAPE, "count=%lld must be a positive multiple of 4", (long long)count);
  if (!aligned16(acc) || (reinterpret_cast<uintptr_t>(out) & 7u))
    return fail(RA_ERR_ALIGN, "acc must be 16-byte and out 8-byte aligned");
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  const int64_t quads = count / 4;
  int64_t blocks = (quads + 255) / 256;
  if (blocks > (int64_t)dev->sms * 16) blocks = (int64_t)dev->sms * 16;
  ra::finalize_bf16_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const float4*>(acc), static_cast<uint2*>(out), quads);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "finalize_bf16_kernel launch");
  return RA_OK;
}

ra_status ring_attn_index_map(int64_t S, int P, ra_layout layout, int64_t* pos) {
  if (!pos) return fail(RA_ERR_NULL, "pos must be non-NULL");
  if (S < 1 || P < 1) return fail(RA_ERR_SHAPE, "S and P must be positive");
  if ((int)layout < 0 || (int)layout > 2) return fail(RA_ERR_LAYOUT, "unknown layout %d", (int)layout);
  if (S % P != 0) return fail(RA_ERR_LAYOUT, "S is not divisible by P");
  if (layout == RA_LAYOUT_ZIGZAG && S % (2 * (int64_t)P) != 0)
    return fail(RA_ERR_LAYOUT, "zig-zag needs S divisible by 2P");
  ra::Geo g = ra::make_geo(1, 1, 1, S, P, layout, 0);
  for (int r = 0; r < P; ++r)
    for (int64_t j = 0; j < g.n; ++j) pos[r * g.n + j] = ra::position_of(g, r, j);
  return RA_OK;
}

ra_status ring_attn_census(int64_t S, int P, ra_layout layout, int causal, int64_t* visible_pairs,
                           int64_t* computed_tiles) {
  if (S < 1 || P < 1) return fail(RA_ERR_SHAPE, "S and P must be positive");
  if ((int)layout < 0 || (int)layout > 2) return fail(RA_ERR_LAYOUT, "unknown layout %d", (int)layout);
  if (S % P != 0) return fail(RA_ERR_LAYOUT, "S is not divisible by P");
  if (layout == RA_LAYOUT_ZIGZAG && S % (2 * (int64_t)P) != 0)
    return fail(RA_ERR_LAYOUT, "zig-zag needs S divisible by 2P");
  ra::Geo g = ra::make_geo(1, 1, 1, S, P, layout, causal ? 1 : 0);
  for (int r = 0; r < P; ++r) {
    int64_t pairs = 0, tiles = 0;
    for (int sq = 0; sq < g.nseg; ++sq) {
      ra::Seg qs = ra::segment_of(g, r, sq);
      for (int a = 0; a < g.ntile; ++a) {
        ra::QTile qt = ra::make_qtile(g, r, sq, a);
        if (!qt.valid) continue;
        tiles += ra::tile_work(g, qt, -1);
        // a query at position x sees keys 0..x (causal) or all S keys
        for (int i = 0; i < qt.valid; ++i)
          pairs += causal ? qs.pos0 + qs.stride * (qt.off + i) + 1 : S;
      }
    }
    if (visible_pairs) visible_pairs[r] = pairs;
    if (computed_tiles) computed_tiles[r] = tiles;
  }
  return RA_OK;
}

ra_status ring_attn_work_schedule(int kind, int B, int H, int Hkv, int64_t S, int D, int P,
                                  ra_layout layout, int causal, int sms, int64_t l2_bytes,
                                  int* out, int64_t capacity, int64_t* n_out) {
  if (n_out == nullptr) return fail(RA_ERR_NULL, "n_out must be non-NULL");
  *n_out = 0;
  if (kind < 0 || kind > 2)
    return fail(RA_ERR_SHAPE, "kind %d: 0 (forward), 1 (dK/dV pass) or 2 (dQ pass)", kind);
  if (sms < 1 || l2_bytes < 0 || l2_bytes > 0x7fffffffLL)
    return fail(RA_ERR_SHAPE, "sms=%d and l2_bytes=%lld must be positive", sms, (long long)l2_bytes);
  ra_status st = check_common(B, H, Hkv, S, D, P, (int)layout, 1.0f);
  if (st != RA_OK) return st;
  DeviceInfo dev;
  dev.sms = sms;
  dev.l2_bytes = (int)l2_bytes;
  std::vector<int> v;
  if (kind == 0) {
    ra::FwdParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.g = ra::make_geo(B, H, Hkv, S, P, (int)layout, causal ? 1 : 0);
    prm.mode = ra::FWD_MODE_RING;
    prm.num_items = ra::units_total(prm.g, false) * B * H;
    prm.kv_group = fwd_kv_group(prm.g, false, &dev, D);
    const int grid = (int)(prm.num_items < sms ? prm.num_items : sms);
    if (schedule_worth(prm.num_items, grid)) v = fwd_schedule_host(prm, grid);
  } else {
    ra::BwdParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.g = ra::make_geo(B, H, Hkv, S, P, (int)layout, causal ? 1 : 0);
    const int64_t units = (int64_t)prm.g.P * prm.g.nseg * prm.g.ntile;
    prm.num_items = units * B * (kind == 1 ? Hkv : H);
    const int grid = (int)(prm.num_items < sms ? prm.num_items : sms);
    if (schedule_worth(prm.num_items, grid)) v = bwd_schedule_host(prm, kind == 1, false, grid);
  }
  *n_out = (int64_t)v.size();
  if (out == nullptr) return RA_OK;
  if ((int64_t)v.size() > capacity)
    return fail(RA_ERR_SHAPE, "the schedule holds %lld ints; the buffer %lld", (long long)v.size(),
                (long long)capacity);
  if (!v.empty()) memcpy(out, v.data(), v.size() * sizeof(int));
  return RA_OK;
}

ra_status ring_attn_check_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&word, ra::g_dev_status, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "reading device status");
  if (word != 0) {
    e = cudaMemcpyToSymbol(ra::g_dev_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clearing device status");
    return fail(RA_ERR_DEVICE_TIMEOUT, "a kernel gave up on a bounded wait (status 0x%x)", word);
  }
  return RA_OK;
}

ra_status ring_attn_set_wait_limit(int64_t limit_ns) {
  if (limit_ns < 0 || limit_ns > 60000000000LL)
    return fail(RA_ERR_SHAPE, "limit_ns=%lld outside [0, 6e10]", (long long)limit_ns);
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  const unsigned long long v = limit_ns == 0 ? ra::kWaitLimitNs : (unsigned long long)limit_ns;
  cudaError_t e = cudaMemcpyToSymbol(ra::g_wait_limit_ns, &v, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "setting the wait limit");
  return RA_OK;
}

ra_status ring_attn_wait_selfcheck(int limit_ms, int64_t* waited_ns, void* stream) {
  if (!waited_ns) return fail(RA_ERR_NULL, "waited_ns must be non-NULL");
  if (limit_ms < 1 || limit_ms > 1000)
    return fail(RA_ERR_SHAPE, "limit_ms=%d outside [1, 1000]", limit_ms);
  if (reinterpret_cast<uintptr_t>(waited_ns) & 7u) return fail(RA_ERR_ALIGN, "waited_ns must be 8-byte aligned");
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  ra::wait_selfcheck_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      (unsigned long long)limit_ms * 1000000ull, reinterpret_cast<unsigned long long*>(waited_ns));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "wait_selfcheck_kernel launch");
  return RA_OK;
}

const char* ring_attn_last_error(void) { return g_last_error; }

const char* ring_attn_version(void) { return "ring_attn 0.1.0 (sm_103a)"; }

}  // extern "C"
