// gemm_tcgen05.cu -- host side of the FP8 GEMM: tensor maps, the choice of
// kernel and tile shape per GEMM, the K-split schedule, launches, and the
// description of a GEMM's kernel and schedule.  The kernels themselves are in
// gemm_kernels.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "gemm_kernels.cuh"

namespace fp8lin {
namespace {

// ------------------------------------------------------------------ host side

thread_local CUresult g_last_encode_result = CUDA_SUCCESS;
thread_local char g_map_site[128];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Every 2-D tiled map of the library goes through here.  Encoding is a pure
// function of its arguments, and a training loop encodes the same few maps
// over and over (its buffers do not move), so each host thread keeps the
// last kMapCache encodings and reuses one whose arguments all match.
struct MapKey {
  const void* base;
  uint64_t inner, rows, stride;
  uint32_t box_inner, box_rows;
  int dtype, swizzle, promo;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && rows == o.rows && stride == o.stride &&
           box_inner == o.box_inner && box_rows == o.box_rows && dtype == o.dtype &&
           swizzle == o.swizzle && promo == o.promo;
  }
};

constexpr int kMapCache = 64;
struct MapCache {
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int used = 0, next = 0;
};
thread_local MapCache g_map_cache;

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
               uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
  const MapKey k = {base, inner, rows, row_stride_bytes, box_inner, box_rows,
                    static_cast<int>(dtype), static_cast<int>(swizzle), static_cast<int>(promo)};
  MapCache& c = g_map_cache;
  for (int i = 0; i < c.used; ++i) {
    if (c.key[i] == k) {
      *map = c.map[i];
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_bytes)};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  g_last_encode_result = r;
  if (r != CUDA_SUCCESS) return false;
  const int slot = c.used < kMapCache ? c.used++ : c.next;
  if (slot == c.next) c.next = (c.next + 1) % kMapCache;
  c.key[slot] = k;
  c.map[slot] = *map;
  return true;
}

// 2-D map over an 8-bit [rows, k] matrix (row stride ld bytes), box
// [box_rows, 128 bytes], 128-byte swizzle, zero fill outside the matrix.
bool make_map_k_major(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t k, int64_t ld,
                      int box_rows) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, static_cast<uint64_t>(k),
                   static_cast<uint64_t>(rows), static_cast<uint64_t>(ld), kBK,
                   static_cast<uint32_t>(box_rows), CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// 2-D map over the bf16 output [rows, cols] (row stride ldd elements), box
// 32 rows x 64 columns (128-byte rows), 128-byte swizzle, for the
// epilogue's TMA stores.
bool make_map_out(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ldd) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, static_cast<uint64_t>(cols),
                   static_cast<uint64_t>(rows), static_cast<uint64_t>(ldd) * 2, kBoxCols, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// How the `tiles` tiles of rows_per_tile x bn, with `num_kb` K blocks each,
// are dealt to `slots` persistent units (CTAs or pairs), given `split_bytes`
// of workspace for fp32 partials: tiles [0, t_full) run whole, round-robin;
// each tile after them runs as `ways` K slices that the slices reduce
// together (see epilogue_unit).
//   Few tiles (fewer than slots) with a K loop of at least 16 blocks: every
//   tile is split, ways = slots / tiles, so the work runs on all slots.
//   Several waves with a long K loop (at least kTailSplitMinKb blocks) and a
//   last wave at most half full: the whole waves run whole and only the r
//   tiles of the last wave are split, ways = slots / r, so the last round
//   takes a fraction of a tile instead of a whole one (e.g. the dW product
//   of a 65536-token step: 256 tiles on 76 pairs, r = 28, ways = 2).  With a
//   short K loop the partials' traffic and the extra reductions cost more
//   than the idle tail, as measured on 4096 x 4096 x 4096 products.
struct SplitPlan {
  int t_full, ways;
};

constexpr int kTailSplitMinKb = 96;

SplitPlan plan_split(int tiles, int slots, int num_kb, int rows_per_tile, int bn,
                     size_t split_bytes) {
  const SplitPlan whole = {tiles, 1};
  if (split_bytes == 0 || slots < 2 || tiles < 1) return whole;
  int r, t_full;
  if (tiles < slots) {
    if (num_kb < 16) return whole;
    r = tiles;
    t_full = 0;
  } else {
    r = tiles % slots;
    if (r == 0 || 2 * r > slots || num_kb < kTailSplitMinKb) return whole;
    t_full = tiles - r;
  }
  const size_t groups = static_cast<size_t>(rows_per_tile) / 32 * (bn >= 64 ? 2 : 1);
  const size_t tile_bytes = static_cast<size_t>(rows_per_tile) * bn * sizeof(float);
  int s = slots / r;
  if (s > kMaxSplit) s = kMaxSplit;
  if (s > num_kb) s = num_kb;
  if (s < 2) return whole;
  const int per = (num_kb + s - 1) / s;
  s = (num_kb + per - 1) / per;  // no empty slice
  if (s < 2) return whole;
  const size_t need_tickets = 2 * static_cast<size_t>(r) * groups;
  if (static_cast<size_t>(r) * s * tile_bytes > split_bytes || need_tickets > kWsTickets)
    return whole;
  return {t_full, s};
}

void plan_schedule(GemmParams& p, int tiles, int slots, int num_kb, int rows_per_tile, int bn,
                   const GemmArgs& g) {
  const bool can_split = g.ws_split != nullptr && g.ws_tickets != nullptr;
  const SplitPlan sp =
      plan_split(tiles, slots, num_kb, rows_per_tile, bn, can_split ? g.ws_split_bytes : 0);
  p.t_full = sp.t_full;
  p.s_tail = sp.ways;
  p.partials = sp.ways > 1 ? g.ws_split : nullptr;
  p.tickets = sp.ways > 1 ? g.ws_tickets : nullptr;
}

// One-time per-device set-up of a kernel's shared-memory limit (and, for the
// pair kernel, the number of co-resident clusters of 2 it gets), kept per
// device and guarded, so concurrent first calls from several host threads or
// alternating devices are safe.
constexpr int kMaxDevices = 64;

template <int BN, int STAGES, bool kTransStore>
cudaError_t one_cta_setup(const DeviceInfo& dev) {
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  if (dev.device < 0 || dev.device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev.device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_fp8_kernel<BN, STAGES, kTransStore>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg<BN, STAGES>::kSmemBytes));
  if (e == cudaSuccess) done[dev.device] = true;
  return e;
}

// Epilogue warps of a pair-kernel launch: 4 when at least one whole round of
// tiles runs whole and each tile's main loop has at least kLeanMinKb K
// blocks, so that a tile's epilogue hides under the next tile's main loop;
// else 8.  Measured on GB300: 4 warps took 0.5-3 % off products of 13 or
// more K blocks a tile; with 8 or fewer (K = 1024: 4 % slower; K = 256:
// 14 % slower) and under one round the epilogue is on the critical path.
constexpr int kLeanMinKb = 12;

int pair_epi(int t_full, int slots, int num_kb) {
  return t_full >= slots && num_kb >= kLeanMinKb ? 4 : 8;
}

// The same for a grouped launch of two GEMMs of kb0 and kb1 K blocks a tile.
int group_epi(int units, int slots, int kb0, int kb1) {
  return pair_epi(units, slots, kb0 < kb1 ? kb0 : kb1);
}

template <int BN, int STAGES, int EPI>
cudaError_t pair_setup(const DeviceInfo& dev, int* slots) {
  using C = PairCfg<BN, STAGES>;
  auto kernel = gemm_fp8_pair_kernel<BN, STAGES, EPI>;
  static std::mutex mu;
  static int max_pairs[kMaxDevices] = {};
  if (dev.device < 0 || dev.device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (max_pairs[dev.device] == 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t probe = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    probe.gridDim = dim3(2 * (dev.num_sms / 2));
    probe.blockDim = dim3(pair_threads<EPI>());
    probe.dynamicSmemBytes = C::kSmemBytes;
    probe.attrs = attr;
    probe.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &probe) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = dev.num_sms / 2;
    }
    max_pairs[dev.device] = n;
  }
  *slots = max_pairs[dev.device];
  return cudaSuccess;
}

template <int BN, int STAGES, bool kTransStore>
cudaError_t run(const uint8_t* a, int64_t lda, const uint8_t* b, int64_t ldb, GemmParams p,
                const GemmArgs& g, const DeviceInfo& dev, cudaStream_t stream) {
  using C = Cfg<BN, STAGES>;
  auto kernel = gemm_fp8_kernel<BN, STAGES, kTransStore>;
  cudaError_t e = one_cta_setup<BN, STAGES, kTransStore>(dev);
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb, md;
  if (!make_map_k_major(&ma, a, p.M, p.K, lda, kBM)) return map_failed("GEMM operand A map");
  if (!make_map_k_major(&mb, b, p.N, p.K, ldb, BN)) return map_failed("GEMM operand B map");
  if (kTransStore)
    md = mb;  // unused: the transposed store writes D directly
  else if (!make_map_out(&md, p.d, p.M, p.N, p.ldd))
    return map_failed("GEMM output map");
  const int tiles = ((p.M + kBM - 1) / kBM) * ((p.N + BN - 1) / BN);
  plan_schedule(p, tiles, dev.num_sms, (p.K + kBK - 1) / kBK, kBM, BN, g);
  set_error_site("one-CTA GEMM launch");
  const int units = p.t_full + (tiles - p.t_full) * p.s_tail;
  const int grid = units < dev.num_sms ? units : dev.num_sms;
  return launch_kernel(kernel, dim3(grid), dim3(kGemmThreads), C::kSmemBytes, stream, 1, false, ma,
                       mb, md, p);
}

template <int BN, int STAGES>
cudaError_t run_pair(const uint8_t* a, int64_t lda, const uint8_t* b, int64_t ldb, GemmParams p,
                     const GemmArgs& g, const DeviceInfo& dev, cudaStream_t stream) {
  using C = PairCfg<BN, STAGES>;
  int max_pairs = 0;
  cudaError_t e = pair_setup<BN, STAGES, 8>(dev, &max_pairs);
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb, md;
  if (!make_map_k_major(&ma, a, p.M, p.K, lda, kBM)) return map_failed("pair GEMM operand A map");
  if (!make_map_k_major(&mb, b, p.N, p.K, ldb, BN / 2))
    return map_failed("pair GEMM operand B map");
  if (!make_map_out(&md, p.d, p.M, p.N, p.ldd)) return map_failed("pair GEMM output map");
  const int tiles = ((p.M + 2 * kBM - 1) / (2 * kBM)) * ((p.N + BN - 1) / BN);
  plan_schedule(p, tiles, max_pairs, (p.K + kBK - 1) / kBK, 2 * kBM, BN, g);
  set_error_site("pair GEMM launch");
  const int units = p.t_full + (tiles - p.t_full) * p.s_tail;
  const int pairs = units < max_pairs ? units : max_pairs;
  if constexpr (BN == 256) {  // (the 128-wide tiles, for N <= 128, keep 8 warps)
    if (pair_epi(p.t_full, max_pairs, (p.K + kBK - 1) / kBK) == 4) {
      int slots4 = 0;
      if ((e = pair_setup<BN, STAGES, 4>(dev, &slots4)) != cudaSuccess) return e;
      if (slots4 >= pairs)  // (the same shared memory: as many pairs fit)
          return launch_kernel(gemm_fp8_pair_kernel<BN, STAGES, 4>, dim3(2 * pairs),
                             dim3(pair_threads<4>()), C::kSmemBytes, stream, 2, false, ma, mb,
                             md, p);
    }
  }
  return launch_kernel(gemm_fp8_pair_kernel<BN, STAGES, 8>, dim3(2 * pairs),
                       dim3(pair_threads<8>()), C::kSmemBytes, stream, 2, false, ma, mb, md, p);
}

template <int BN, int STAGES, int EPI>
cudaError_t pair2_setup(const DeviceInfo& dev) {
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  if (dev.device < 0 || dev.device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev.device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_fp8_pair2_kernel<BN, STAGES, EPI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(PairCfg<BN, STAGES>::kSmemBytes));
  if (e == cudaSuccess) done[dev.device] = true;
  return e;
}

// Estimated time of a pair-kernel GEMM alone, in K blocks of its busiest
// pair (a split tail tile's slices add kSplitExtraKb for their partials,
// measured at about 4 us beyond a whole tile's epilogue).
constexpr int kSplitExtraKb = 13;
constexpr int kLaunchExtraKb = 9;  // a launch boundary, about 3 us
// Grouping is chosen only when the estimate gains at least this share.  In a
// graphed step the second of two launches overlaps its prologue with the
// first's drain, so small estimated gains were measured as none (a 4096-token
// Linear of 4096 x 4096, 0.976 of the separate estimate: no faster) or as a
// loss (the 8192 x 4096 x 14336 FFN projections, 0.994: 1% slower), while
// 0.88 and below gained 3 to 11% of the whole step.
constexpr int kGroupMinGainPct = 8;

int alone_kb(int tiles, int num_kb, int slots, size_t split_bytes) {
  const SplitPlan sp = plan_split(tiles, slots, num_kb, 2 * kBM, 256, split_bytes);
  if (sp.ways == 1) return (tiles + slots - 1) / slots * num_kb;
  const int per = (num_kb + sp.ways - 1) / sp.ways;
  return sp.t_full / slots * num_kb + per + kSplitExtraKb;
}

// K blocks of the busiest pair under unit_at_grouped's deal with this d
// (the counts unit_at_grouped deals to each pair, in closed form).
int grouped_kb(const GroupSched& gs, int kb0, int kb1, int slots) {
  const int ll = gs.tiles0 / slots, heavy = gs.tiles0 % slots, light = slots - heavy;
  const int e = gs.tiles1 < light * gs.d ? gs.tiles1 : light * gs.d;
  const int r = gs.tiles1 - e;
  int worst = 0;
  for (int p = 0; p < slots; ++p) {
    const int q = p - heavy;
    const int ep = p >= heavy && e > q ? (e - q + light - 1) / light : 0;
    const int pos = p >= heavy ? q : light + p;
    const int rp = r > pos ? (r - pos + slots - 1) / slots : 0;
    const int load = (ll + (p < heavy ? 1 : 0)) * kb0 + (ep + rp) * kb1;
    if (load > worst) worst = load;
  }
  return worst;
}

// The grouped plan for two pair-kernel GEMMs (problem 0: the longer K loop):
// the d with the least busiest pair, and whether it beats two launches.
struct GroupPlan {
  bool use;
  GroupSched gs;
  int grouped, alone;  // estimated K blocks of the busiest pair
};

GroupPlan plan_group(int tiles0, int kb0, int tiles1, int kb1, int slots, size_t split_bytes) {
  GroupPlan g = {false, {tiles0, tiles1, 0}, 0, 0};
  g.alone = alone_kb(tiles0, kb0, slots, split_bytes) + alone_kb(tiles1, kb1, slots, split_bytes) +
            kLaunchExtraKb;
  const int dmax = kb1 > 0 ? kb0 / kb1 + 2 : 0;
  g.grouped = 1 << 30;
  for (int d = 0; d <= dmax; ++d) {
    const GroupSched gs = {tiles0, tiles1, d};
    const int kb = grouped_kb(gs, kb0, kb1, slots);
    if (kb < g.grouped) {
      g.grouped = kb;
      g.gs = gs;
    }
  }
  g.use = static_cast<int64_t>(g.grouped) * 100 <
          static_cast<int64_t>(g.alone) * (100 - kGroupMinGainPct);
  return g;
}

// FP8LIN_GROUP: 0 never runs two GEMMs in one launch, 2 always when they
// qualify, anything else when the plan expects it to be faster.
int group_mode() {
  static const int mode = [] {
    const char* v = std::getenv("FP8LIN_GROUP");
    if (v != nullptr && v[0] == '0') return 0;
    if (v != nullptr && v[0] == '2') return 2;
    return 1;
  }();
  return mode;
}

}  // namespace

cudaError_t map_failed(const char* what) {
  std::snprintf(g_map_site, sizeof(g_map_site), "%s (cuTensorMapEncodeTiled CUresult %d)", what,
                static_cast<int>(g_last_encode_result));
  set_error_site(g_map_site);
  return cudaErrorInvalidValue;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle) {
  return encode_2d(map, dtype, base, inner, rows, row_stride_bytes, box_inner, box_rows, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

size_t gemm_split_workspace_bytes(int num_sms) {
  // At most `num_sms` one-CTA slices of 128 x 256 fp32 (or num_sms / 2 pair
  // slices of 256 x 256): the tail split never has more slices than slots.
  return static_cast<size_t>(num_sms) * kBM * 256 * sizeof(float);
}

namespace {

// The kernel and tile shape for a Linear GEMM of M rows and N columns:
// swap-AB (D^T = B . A^T, the weight-side operand fills the 128-row MMA and
// the few rows of A become N = 16 / 32 / 64) for M <= 64; one-CTA 128-row
// tiles up to M = 128; CTA pairs with 256-row tiles above.  BN = 256 except
// for N <= 128: a 128-wide tile costs about 1.7x more per FLOP (each CTA
// reads the same A block per K step for half the columns), which outweighs
// the padding it saves everywhere else -- e.g. the N = 1600 products of a
// 1600-wide model run 1.5-1.8x faster on 256-wide tiles, padding included.
enum class Variant { kSwap16, kSwap32, kSwap64, kOne128, kOne256, kPair128, kPair256 };

Variant choose_variant(int64_t M, int64_t N) {
  if (M <= 16) return Variant::kSwap16;
  if (M <= 32) return Variant::kSwap32;
  if (M <= 64) return Variant::kSwap64;
  const bool narrow = N <= 128;
  if (M > kBM) return narrow ? Variant::kPair128 : Variant::kPair256;
  return narrow ? Variant::kOne128 : Variant::kOne256;
}

bool is_swap(Variant v) {
  return v == Variant::kSwap16 || v == Variant::kSwap32 || v == Variant::kSwap64;
}

}  // namespace

namespace {

GemmParams base_params(const GemmArgs& g) {
  GemmParams p;
  p.inv_a = g.inv_a;
  p.inv_b = g.inv_b;
  p.d = static_cast<uint16_t*>(g.d);
  p.ldd = g.ldd;
  p.err = g.ws_error;
  p.K = static_cast<int>(g.K);
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  p.amax_out = g.d_amax;
  p.amax_acc = g.ws_amax_acc;
  p.amax_ticket = g.ws_amax_ticket;
  p.t_full = 0;
  p.s_tail = 1;
  p.partials = nullptr;
  p.tickets = nullptr;
  return p;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& g, const DeviceInfo& dev, cudaStream_t stream) {
  GemmParams p;
  p.inv_a = g.inv_a;
  p.inv_b = g.inv_b;
  p.d = static_cast<uint16_t*>(g.d);
  p.ldd = g.ldd;
  p.err = g.ws_error;
  p.K = static_cast<int>(g.K);
  p.amax_out = g.d_amax;
  p.amax_acc = g.ws_amax_acc;
  p.amax_ticket = g.ws_amax_ticket;
  const Variant v = choose_variant(g.M, g.N);
  if (is_swap(v)) {
    p.M = static_cast<int>(g.N);
    p.N = static_cast<int>(g.M);
    if (v == Variant::kSwap16) {
      p.idesc = make_idesc_f8(g.fmt_b, g.fmt_a, kBM, 16);
      return run<16, 8, true>(g.b, g.ldb, g.a, g.lda, p, g, dev, stream);
    }
    if (v == Variant::kSwap32) {
      p.idesc = make_idesc_f8(g.fmt_b, g.fmt_a, kBM, 32);
      return run<32, 8, true>(g.b, g.ldb, g.a, g.lda, p, g, dev, stream);
    }
    p.idesc = make_idesc_f8(g.fmt_b, g.fmt_a, kBM, 64);
    return run<64, 8, true>(g.b, g.ldb, g.a, g.lda, p, g, dev, stream);
  }
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  switch (v) {
    case Variant::kPair128:
      p.idesc = make_idesc_f8(g.fmt_a, g.fmt_b, 2 * kBM, 128);
      return run_pair<128, 8>(g.a, g.lda, g.b, g.ldb, p, g, dev, stream);
    case Variant::kPair256:
      p.idesc = make_idesc_f8(g.fmt_a, g.fmt_b, 2 * kBM, 256);
      return run_pair<256, 6>(g.a, g.lda, g.b, g.ldb, p, g, dev, stream);
    case Variant::kOne128:
      p.idesc = make_idesc_f8(g.fmt_a, g.fmt_b, kBM, 128);
      return run<128, 6, false>(g.a, g.lda, g.b, g.ldb, p, g, dev, stream);
    default:
      p.idesc = make_idesc_f8(g.fmt_a, g.fmt_b, kBM, 256);
      return run<256, 4, false>(g.a, g.lda, g.b, g.ldb, p, g, dev, stream);
  }
}

void describe_plan(int64_t M, int64_t N, int64_t K, int num_sms, int pair_slots, char* buf,
                   size_t len) {
  const Variant v = choose_variant(M, N);
  const char* name = "";
  int rows = kBM, bn = 256, slots = num_sms;
  switch (v) {
    case Variant::kSwap16: name = "gemm_fp8_kernel<16, 8, 1>"; bn = 16; break;
    case Variant::kSwap32: name = "gemm_fp8_kernel<32, 8, 1>"; bn = 32; break;
    case Variant::kSwap64: name = "gemm_fp8_kernel<64, 8, 1>"; bn = 64; break;
    case Variant::kOne128: name = "gemm_fp8_kernel<128, 6, 0>"; bn = 128; break;
    case Variant::kOne256: name = "gemm_fp8_kernel<256, 4, 0>"; break;
    case Variant::kPair128:
      name = "gemm_fp8_pair_kernel<128, 8, 8>";
      bn = 128;
      rows = 2 * kBM;
      slots = pair_slots;
      break;
    case Variant::kPair256:
      name = "gemm_fp8_pair_kernel<256, 6, 8>";
      rows = 2 * kBM;
      slots = pair_slots;
      break;
  }
  const int64_t tm = is_swap(v) ? N : M, tn = is_swap(v) ? M : N;  // as the kernel sees it
  const int64_t tiles64 = ((tm + rows - 1) / rows) * ((tn + bn - 1) / bn);
  const int tiles = tiles64 > (1 << 30) ? (1 << 30) : static_cast<int>(tiles64);
  const int num_kb = static_cast<int>((K + kBK - 1) / kBK);
  const SplitPlan sp =
      plan_split(tiles, slots, num_kb, rows, bn, gemm_split_workspace_bytes(num_sms));
  if (v == Variant::kPair256 && pair_epi(sp.t_full, slots, num_kb) == 4)
    name = "gemm_fp8_pair_kernel<256, 6, 4>";
  const int units = sp.t_full + (tiles - sp.t_full) * sp.ways;
  const int used = units < slots ? units : slots;
  char sched[64] = "whole tiles";
  if (sp.ways > 1 && sp.t_full == 0)
    std::snprintf(sched, sizeof(sched), "K split %d ways", sp.ways);
  else if (sp.ways > 1)
    std::snprintf(sched, sizeof(sched), "last %d tiles K split %d ways", tiles - sp.t_full,
                  sp.ways);
  std::snprintf(buf, len, "%s: %s%dx%d tiles, %d tiles on %d of %d %s, %s", name,
                is_swap(v) ? "swap-AB (D^T = B.A^T), " : "", rows, bn, tiles, used, slots,
                rows == 2 * kBM ? "CTA pairs" : "CTAs", sched);
}

cudaError_t describe_gemm(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev, char* buf,
                          size_t len) {
  // The pair kernel's slots are the clusters of 2 the device holds at once.
  int pair_slots = dev.num_sms / 2;
  cudaError_t e = cudaSuccess;
  switch (choose_variant(M, N)) {
    case Variant::kPair128: e = pair_setup<128, 8, 8>(dev, &pair_slots); break;
    case Variant::kPair256: e = pair_setup<256, 6, 8>(dev, &pair_slots); break;
    default: break;
  }
  if (e != cudaSuccess) return e;
  describe_plan(M, N, K, dev.num_sms, pair_slots, buf, len);
  return cudaSuccess;
}

static bool group_qualifies(const GemmArgs& g0, const GemmArgs& g1) {
  return choose_variant(g0.M, g0.N) == Variant::kPair256 &&
         choose_variant(g1.M, g1.N) == Variant::kPair256 &&
         (g0.d_amax == nullptr || g1.d_amax == nullptr) && g0.K > 0 && g1.K > 0;
}

namespace {

// The grouped plan for two qualifying GEMMs: problem 0 the one with the
// longer K loop (*swap: b), its tiles and the deal.
struct Pair2 {
  bool use, swap;
  int tiles0, tiles1, max_pairs;
  GroupSched gs;
};

cudaError_t pair2_plan(const GemmArgs& ga, const GemmArgs& gb, const DeviceInfo& dev, Pair2* out) {
  out->use = false;
  if (group_mode() == 0 || !group_qualifies(ga, gb)) return cudaSuccess;
  int max_pairs = 0;
  cudaError_t e = pair_setup<256, 6, 8>(dev, &max_pairs);
  if (e != cudaSuccess) return e;
  out->swap = (gb.K + kBK - 1) / kBK > (ga.K + kBK - 1) / kBK;
  const GemmArgs& g0 = out->swap ? gb : ga;
  const GemmArgs& g1 = out->swap ? ga : gb;
  out->tiles0 = static_cast<int>(((g0.M + 2 * kBM - 1) / (2 * kBM)) * ((g0.N + 255) / 256));
  out->tiles1 = static_cast<int>(((g1.M + 2 * kBM - 1) / (2 * kBM)) * ((g1.N + 255) / 256));
  out->max_pairs = max_pairs;
  const int kb0 = static_cast<int>((g0.K + kBK - 1) / kBK);
  const int kb1 = static_cast<int>((g1.K + kBK - 1) / kBK);
  const size_t split = g0.ws_split != nullptr && g0.ws_tickets != nullptr ? g0.ws_split_bytes : 0;
  const GroupPlan plan = plan_group(out->tiles0, kb0, out->tiles1, kb1, max_pairs, split);
  out->gs = plan.gs;
  out->use = plan.use || group_mode() == 2;
  return cudaSuccess;
}

}  // namespace

cudaError_t plan_gemm_pair2(const GemmArgs& a, const GemmArgs& b, const DeviceInfo& dev,
                            bool* use) {
  Pair2 pl;
  cudaError_t e = pair2_plan(a, b, dev, &pl);
  *use = pl.use;
  return e;
}

cudaError_t launch_gemm_pair2(const GemmArgs& ga, const GemmArgs& gb, const DeviceInfo& dev,
                              cudaStream_t stream) {
  Pair2 pl;
  cudaError_t e = pair2_plan(ga, gb, dev, &pl);
  if (e != cudaSuccess) return e;
  if (!pl.use) return cudaErrorInvalidValue;
  const GemmArgs& g0 = pl.swap ? gb : ga;
  const GemmArgs& g1 = pl.swap ? ga : gb;
  GemmParams p0 = base_params(g0), p1 = base_params(g1);
  p0.t_full = pl.tiles0;
  p1.t_full = pl.tiles1;
  p0.idesc = make_idesc_f8(g0.fmt_a, g0.fmt_b, 2 * kBM, 256);
  p1.idesc = make_idesc_f8(g1.fmt_a, g1.fmt_b, 2 * kBM, 256);
  CUtensorMap ma0, mb0, md0, ma1, mb1, md1;
  if (!make_map_k_major(&ma0, g0.a, p0.M, p0.K, g0.lda, kBM) ||
      !make_map_k_major(&ma1, g1.a, p1.M, p1.K, g1.lda, kBM))
    return map_failed("grouped pair GEMM operand A map");
  if (!make_map_k_major(&mb0, g0.b, p0.N, p0.K, g0.ldb, 128) ||
      !make_map_k_major(&mb1, g1.b, p1.N, p1.K, g1.ldb, 128))
    return map_failed("grouped pair GEMM operand B map");
  if (!make_map_out(&md0, p0.d, p0.M, p0.N, p0.ldd) || !make_map_out(&md1, p1.d, p1.M, p1.N, p1.ldd))
    return map_failed("grouped pair GEMM output map");
  set_error_site("grouped pair GEMM launch");
  const int units = pl.tiles0 + pl.tiles1;
  const int pairs = units < pl.max_pairs ? units : pl.max_pairs;
  GroupSched gs = pl.gs;
  if (pairs < pl.max_pairs) gs = {pl.tiles0, pl.tiles1, 0};  // one round: a pair per unit
  const int kb0 = (p0.K + kBK - 1) / kBK, kb1 = (p1.K + kBK - 1) / kBK;
  if (group_epi(units, pl.max_pairs, kb0, kb1) == 4) {
    if ((e = pair2_setup<256, 6, 4>(dev)) != cudaSuccess) return e;
    return launch_kernel(gemm_fp8_pair2_kernel<256, 6, 4>, dim3(2 * pairs),
                         dim3(pair_threads<4>()), PairCfg<256, 6>::kSmemBytes, stream, 2, false,
                         ma0, mb0, md0, p0, ma1, mb1, md1, p1, gs);
  }
  if ((e = pair2_setup<256, 6, 8>(dev)) != cudaSuccess) return e;
  return launch_kernel(gemm_fp8_pair2_kernel<256, 6, 8>, dim3(2 * pairs), dim3(pair_threads<8>()),
                       PairCfg<256, 6>::kSmemBytes, stream, 2, false, ma0, mb0, md0, p0, ma1, mb1,
                       md1, p1, gs);
}

void describe_group_plan(int64_t Ma, int64_t Na, int64_t Ka, int64_t Mb, int64_t Nb, int64_t Kb,
                         int num_sms, int pair_slots, char* buf, size_t len) {
  if (choose_variant(Ma, Na) != Variant::kPair256 || choose_variant(Mb, Nb) != Variant::kPair256) {
    std::snprintf(buf, len, "separate: not both on 256-wide pair tiles");
    return;
  }
  const int kba = static_cast<int>((Ka + kBK - 1) / kBK), kbb = static_cast<int>((Kb + kBK - 1) / kBK);
  const bool swap = kbb > kba;
  const int64_t M0 = swap ? Mb : Ma, N0 = swap ? Nb : Na, M1 = swap ? Ma : Mb, N1 = swap ? Na : Nb;
  const int kb0 = swap ? kbb : kba, kb1 = swap ? kba : kbb;
  const int tiles0 = static_cast<int>(((M0 + 2 * kBM - 1) / (2 * kBM)) * ((N0 + 255) / 256));
  const int tiles1 = static_cast<int>(((M1 + 2 * kBM - 1) / (2 * kBM)) * ((N1 + 255) / 256));
  const GroupPlan plan =
      plan_group(tiles0, kb0, tiles1, kb1, pair_slots, gemm_split_workspace_bytes(num_sms));
  // Every unit dealt exactly once, with the pairs and the deal the launch
  // uses (the device deals with the same function; under one round, one unit
  // a pair).
  const int units = tiles0 + tiles1;
  const int pairs = units < pair_slots ? units : pair_slots;
  const GroupSched gs = pairs < pair_slots ? GroupSched{tiles0, tiles1, 0} : plan.gs;
  std::vector<int> seen(static_cast<size_t>(units), 0);
  bool ok = true;
  for (int p = 0; p < pairs; ++p) {
    Unit u;
    for (int n = 0; unit_at_grouped(p, pairs, n, gs, kb0, kb1, u); ++n) {
      const int i = u.prob == 0 ? u.tile : tiles0 + u.tile;
      if (u.tile < 0 || u.tile >= (u.prob == 0 ? tiles0 : tiles1)) ok = false;
      else ++seen[static_cast<size_t>(i)];
    }
  }
  for (int c : seen) ok = ok && c == 1;
  std::snprintf(buf, len, "%s: %d + %d tiles (K blocks %d, %d), d = %d; busiest pair %d K blocks "
                "grouped, %d alone; %d epilogue warps%s",
                plan.use ? "grouped" : "separate", tiles0, tiles1, kb0, kb1, plan.gs.d,
                plan.grouped, plan.alone, group_epi(units, pair_slots, kb0, kb1),
                ok ? "" : "; DEAL BROKEN");
}

}  // namespace fp8lin
