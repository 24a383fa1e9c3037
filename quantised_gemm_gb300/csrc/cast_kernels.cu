// cast_kernels.cu -- host side of the amax, scale and cast kernels: grid
// sizes, launches, the choice between the cluster, cooperative and two-pass
// paths, and the file-scope scratch of the allocation-free amax.  The
// kernels themselves are in cast_kernels.cuh.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "cast_kernels.cuh"

namespace fp8lin {

// ------------------------------------------------------------------ launchers

int amax_grid(const DeviceInfo& dev, int64_t rows, int64_t cols) {
  const int64_t cvec = cols >> 3;
  const int64_t ntiles = ((rows + kAmaxRows - 1) / kAmaxRows) * ((cvec + 31) >> 5);
  int64_t g = static_cast<int64_t>(dev.num_sms) * 8;
  if (g > kMaxPartials) g = kMaxPartials;
  if (ntiles < g) g = ntiles;
  return g < 1 ? 1 : static_cast<int>(g);
}

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint32_t* out,
                        bool atomic, int grid, cudaStream_t stream, uint32_t* ws_acc,
                        uint32_t* ws_ticket) {
  uint32_t* none = nullptr;
  if (!atomic)
    return launch_kernel(amax_kernel<0>, dim3(grid), dim3(kThreads), 0, stream, 1, false, x, rows,
                         cols, ld, out, none, none);
  if (ws_ticket == nullptr)
    return launch_kernel(amax_kernel<1>, dim3(grid), dim3(kThreads), 0, stream, 1, false, x, rows,
                         cols, ld, out, none, none);
  return launch_kernel(amax_kernel<2>, dim3(grid), dim3(kThreads), 0, stream, 1, false, x, rows,
                       cols, ld, out, ws_acc, ws_ticket);
}

cudaError_t launch_amax_final(const uint32_t* partials, int n, uint32_t* amax_bits,
                              cudaStream_t stream) {
  return launch_kernel(amax_final_kernel, dim3(1), dim3(kThreads), 0, stream, 1, false, partials, n,
                       amax_bits);
}

// ------------------------------------------------------------------ amax without a workspace
//
// The two-kernel REDUCTION amax needs somewhere to keep one partial maximum
// per CTA.  For callers that cannot allocate device memory and have no
// workspace to hand over, that scratch lives in this file-scope array instead:
// kStaticAmaxPartials words (16 KiB), resident on every GPU that loads the
// library until the process exits.  Host code must not pass the array's name
// to a kernel (on the host it only stands in for the symbol); the device
// address is looked up with cudaGetSymbolAddress on every call (no
// allocation), so it stays right after a device reset reloads the module.
static __device__ __align__(256) uint32_t g_static_amax_partials[kStaticAmaxPartials];

namespace {

// Device address of g_static_amax_partials in the current context.
cudaError_t static_partials(uint32_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_amax_partials);
  if (e != cudaSuccess) return e;
  *out = static_cast<uint32_t*>(p);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_amax_static_scratch(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                       float* amax_out, int grid, cudaStream_t stream) {
  if (grid < 1 || grid > kStaticAmaxPartials) return cudaErrorInvalidValue;
  uint32_t* part = nullptr;
  cudaError_t e = static_partials(&part);
  if (e != cudaSuccess) return e;
  // Every CTA of the first kernel writes its own slot before the second
  // kernel reads slots [0, grid): nothing in the array has to start at zero.
  amax_kernel<0><<<grid, kThreads, 0, stream>>>(x, rows, cols, ld, part, nullptr, nullptr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  amax_final_kernel<<<1, kThreads, 0, stream>>>(part, grid, reinterpret_cast<uint32_t*>(amax_out));
  return cudaGetLastError();
}

cudaError_t launch_scale(const float* amax, float* scale, float* inv, float* ring, int32_t* head,
                         int32_t history_len, bool delayed, int fmt, float eps,
                         cudaStream_t stream) {
  const float F = fmt == 0 ? 448.0f : 57344.0f;
  return launch_kernel(scale_kernel, dim3(1), dim3(1), 0, stream, 1, false, amax, scale, inv, ring,
                       head, history_len, delayed ? 1 : 0, F, eps);
}

cudaError_t launch_scale_batch(const ScaleArgs* a, int n, cudaStream_t stream) {
  if (n < 1 || n > kScaleBatch) return cudaErrorInvalidValue;
  ScaleBatch b = {};
  b.n = n;
  for (int i = 0; i < n; ++i) {
    b.amax[i] = a[i].amax;
    b.scale[i] = a[i].scale;
    b.inv[i] = a[i].inv;
    b.ring[i] = a[i].ring;
    b.head[i] = a[i].head;
    b.H[i] = a[i].history_len;
    b.delayed[i] = a[i].delayed ? 1 : 0;
    b.F[i] = a[i].fmt == 0 ? 448.0f : 57344.0f;
    b.eps[i] = a[i].eps;
  }
  return launch_kernel(scale_batch_kernel, dim3(1), dim3(32), 0, stream, 1, false, b);
}

namespace {

template <int kFmt, bool kTrans>
cudaError_t stream_prepare(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(cast_stream_kernel<kFmt, kTrans>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kStreamSmem));
  if (e == cudaSuccess) done[device] = true;
  return e;
}

// The TMA streaming cast: one persistent CTA per SM over the tiles.
cudaError_t launch_cast_stream(const CastParams& p, const CastArgs& a, const DeviceInfo& dev,
                               cudaStream_t stream) {
  const bool trans = a.out_t != nullptr;
  CUtensorMap tx, tq, tqt;
  if (!make_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, static_cast<uint64_t>(a.cols),
                   static_cast<uint64_t>(a.rows), static_cast<uint64_t>(a.ld) * 2, kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return map_failed("streaming cast input map");
  // q [rows, cols] and q^T [cols, rows]; the map of an absent output is a
  // valid copy of the other and is never used.
  const bool has_q = a.out != nullptr;
  if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, has_q ? static_cast<const void*>(a.out)
                                                             : a.out_t,
                   static_cast<uint64_t>(has_q ? a.cols : a.rows),
                   static_cast<uint64_t>(has_q ? a.rows : a.cols),
                   static_cast<uint64_t>(has_q ? a.cols : a.rows), kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return map_failed("streaming cast output map");
  if (trans) {
    if (!make_map_2d(&tqt, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.out_t, static_cast<uint64_t>(a.rows),
                     static_cast<uint64_t>(a.cols), static_cast<uint64_t>(a.rows), kTile, kTile,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return map_failed("streaming cast transposed output map");
  } else {
    tqt = tq;
  }
  const int64_t ntiles = ((a.rows + kTile - 1) / kTile) * ((a.cols + kTile - 1) / kTile);
  const unsigned grid =
      static_cast<unsigned>(ntiles < dev.num_sms ? ntiles : static_cast<int64_t>(dev.num_sms));
  void (*fn)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CastParams);
  cudaError_t e;
  if (a.fmt == 0) {
    e = trans ? stream_prepare<0, true>(dev.device) : stream_prepare<0, false>(dev.device);
    fn = trans ? cast_stream_kernel<0, true> : cast_stream_kernel<0, false>;
  } else {
    e = trans ? stream_prepare<1, true>(dev.device) : stream_prepare<1, false>(dev.device);
    fn = trans ? cast_stream_kernel<1, true> : cast_stream_kernel<1, false>;
  }
  if (e != cudaSuccess) return e;
  set_error_site("streaming cast launch");
  return launch_kernel(fn, dim3(grid), dim3(kStreamThreads), kStreamSmem, stream, 1, false, tx,
                       tq, tqt, p);
}

}  // namespace

cudaError_t launch_cast(const CastArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  CastParams p;
  p.x = a.x;
  p.rows = a.rows;
  p.cols = a.cols;
  p.ld = a.ld;
  p.scale_in = a.scale_in;
  p.amax_in = a.amax_in;
  p.derive_scale = a.derive_scale ? 1 : 0;
  p.eps = a.eps;
  p.scale_out = a.scale_out;
  p.inv_out = a.inv_out;
  p.out = a.out;
  p.out_t = a.out_t;
  p.amax_rec = a.amax_rec;
  p.rec_acc = a.rec_acc;
  p.rec_ticket = a.rec_ticket;
  p.err = a.err;
  // With a workspace error word (forward, backward, cast_dynamic) the TMA
  // streaming kernel runs; the bare fp8lin_cast keeps the per-thread kernel.
  if (a.err != nullptr) return launch_cast_stream(p, a, dev, stream);
  const int64_t ntiles = ((a.rows + kTile - 1) / kTile) * ((a.cols + kTile - 1) / kTile);
  int64_t grid = static_cast<int64_t>(dev.num_sms) * 4;
  if (ntiles < grid) grid = ntiles;
  if (grid < 1) grid = 1;
  const bool trans = a.out_t != nullptr;
  const dim3 g(static_cast<unsigned>(grid)), b(kThreads);
  if (a.fmt == 0)
    return trans ? launch_kernel(cast_kernel<0, true>, g, b, 0, stream, 1, false, p)
                 : launch_kernel(cast_kernel<0, false>, g, b, 0, stream, 1, false, p);
  return trans ? launch_kernel(cast_kernel<1, true>, g, b, 0, stream, 1, false, p)
               : launch_kernel(cast_kernel<1, false>, g, b, 0, stream, 1, false, p);
}

namespace {
constexpr size_t kSinglePassSmem =
    static_cast<size_t>(kSinglePassTilesPerCta) * kTile * kTile * 2 + 1024;  // + alignment slack

// Opt the kernel into its shared memory and count its resident CTAs per SM,
// once per device (the answers do not change; the calls cost host time).
template <int kFmt, bool kTrans>
cudaError_t single_pass_prepare(int* ctas_per_sm) {
  static std::mutex mu;
  static int per_sm[64] = {};  // 0: not prepared yet on that device
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (per_sm[d] == 0) {
    auto k = cast_single_pass_kernel<kFmt, kTrans>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSinglePassSmem));
    if (e != cudaSuccess) return e;
    const int n = resident_ctas(k, kSpThreads, kSinglePassSmem);
    if (n < 1) {
      *ctas_per_sm = 0;  // cannot run here; not cached, the caller falls back
      return cudaSuccess;
    }
    per_sm[d] = n;
  }
  *ctas_per_sm = per_sm[d];
  return cudaSuccess;
}
}  // namespace

int64_t single_pass_capacity_elems(const DeviceInfo& dev) {
  if (static_cast<size_t>(dev.max_smem_optin) < kSinglePassSmem + 1024) return 0;
  int per_sm = 0;
  if (single_pass_prepare<0, true>(&per_sm) != cudaSuccess || per_sm < 1) return 0;
  return static_cast<int64_t>(dev.num_sms) * per_sm * kSinglePassTilesPerCta * kTile * kTile;
}

bool single_pass_fits(const DeviceInfo& dev, int64_t rows, int64_t cols) {
  const int64_t ntiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
  return ntiles * kTile * kTile <= single_pass_capacity_elems(dev);
}

namespace {
int cluster_tile_rows(int64_t rows) {
  return rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
}

int64_t cluster_tiles(int64_t rows, int64_t cols) {
  const int tr = cluster_tile_rows(rows);
  const int64_t tc = kClusterTileElems / tr;
  return ((rows + tr - 1) / tr) * ((cols + tc - 1) / tc);
}

template <int kFmt, bool kTrans>
void (*cluster_kernel_for(int tr))(const ClusterCastParams) {
  switch (tr) {
    case 16: return cast_cluster_kernel<kFmt, kTrans, 16>;
    case 32: return cast_cluster_kernel<kFmt, kTrans, 32>;
    case 64: return cast_cluster_kernel<kFmt, kTrans, 64>;
    default: return cast_cluster_kernel<kFmt, kTrans, 128>;
  }
}
}  // namespace

bool cluster_cast_fits(int64_t rows, int64_t cols) {
  return rows > 0 && cols > 0 && cluster_tiles(rows, cols) <= kClusterCtas * kClusterTilesPerCta;
}

cudaError_t launch_cast_cluster(const SinglePassArgs& a, cudaStream_t stream) {
  if (!cluster_cast_fits(a.rows, a.cols)) return cudaErrorInvalidValue;
  ClusterCastParams p;
  p.x = a.x;
  p.rows = a.rows;
  p.cols = a.cols;
  p.ld = a.ld;
  p.eps = a.eps;
  p.amax_out = a.amax_out;
  p.scale_out = a.scale_out;
  p.inv_out = a.inv_out;
  p.out = a.out;
  p.out_t = a.out_t;
  const int tr = cluster_tile_rows(a.rows);
  const int64_t ntiles = cluster_tiles(a.rows, a.cols);
  const int ctas = static_cast<int>(ntiles < kClusterCtas ? ntiles : kClusterCtas);
  const bool trans = a.out_t != nullptr;
  void (*fn)(const ClusterCastParams);
  if (a.fmt == 0)
    fn = trans ? cluster_kernel_for<0, true>(tr) : cluster_kernel_for<0, false>(tr);
  else
    fn = trans ? cluster_kernel_for<1, true>(tr) : cluster_kernel_for<1, false>(tr);
  set_error_site("cluster single-pass launch");
  return launch_kernel(fn, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), 0, stream, ctas,
                       false, p);
}

cudaError_t launch_cast_single_pass(const SinglePassArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream) {
  SinglePassParams p;
  p.rows = a.rows;
  p.cols = a.cols;
  p.eps = a.eps;
  p.amax_out = a.amax_out;
  p.scale_out = a.scale_out;
  p.inv_out = a.inv_out;
  p.out = a.out;
  p.out_t = a.out_t;
  p.ws_barrier = a.ws_barrier;
  p.ws_exits = a.ws_exits;
  p.ws_amax = a.ws_amax;
  p.ws_error = a.ws_error;
  const bool trans = a.out_t != nullptr;
  int per_sm = 0;
  cudaError_t e;
  void (*fn)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const SinglePassParams);
  if (a.fmt == 0) {
    e = trans ? single_pass_prepare<0, true>(&per_sm) : single_pass_prepare<0, false>(&per_sm);
    fn = trans ? cast_single_pass_kernel<0, true> : cast_single_pass_kernel<0, false>;
  } else {
    e = trans ? single_pass_prepare<1, true>(&per_sm) : single_pass_prepare<1, false>(&per_sm);
    fn = trans ? cast_single_pass_kernel<1, true> : cast_single_pass_kernel<1, false>;
  }
  if (e != cudaSuccess) {
    set_error_site("single-pass kernel set-up");
    return e;
  }
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  const int64_t ntiles = ((a.rows + kTile - 1) / kTile) * ((a.cols + kTile - 1) / kTile);
  int64_t grid = (ntiles + kSinglePassTilesPerCta - 1) / kSinglePassTilesPerCta;
  const int64_t max_grid = static_cast<int64_t>(dev.num_sms) * per_sm;
  if (grid > max_grid) return cudaErrorCooperativeLaunchTooLarge;
  // Spread the tiles over as many SMs as possible (fewer tiles per CTA).
  grid = ntiles < max_grid ? ntiles : max_grid;
  if (grid < 1) grid = 1;
  CUtensorMap tm, tq, tqt;
  if (!make_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, static_cast<uint64_t>(a.cols),
                   static_cast<uint64_t>(a.rows), static_cast<uint64_t>(a.ld) * 2, kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_NONE)) {
    return map_failed("single-pass input map");
  }
  // fp8 outputs: q [rows, cols] and q^T [cols, rows], dense, 128 x 128 boxes
  // (maps of absent outputs are never used; they describe a valid dummy).
  const void* qbase = a.out != nullptr ? static_cast<const void*>(a.out) : a.out_t;
  if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qbase,
                   static_cast<uint64_t>(a.out != nullptr ? a.cols : a.rows),
                   static_cast<uint64_t>(a.out != nullptr ? a.rows : a.cols),
                   static_cast<uint64_t>(a.out != nullptr ? a.cols : a.rows), kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_128B)) {
    return map_failed("single-pass output map");
  }
  if (trans) {
    if (!make_map_2d(&tqt, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.out_t, static_cast<uint64_t>(a.rows),
                     static_cast<uint64_t>(a.cols), static_cast<uint64_t>(a.rows), kTile, kTile,
                     CU_TENSOR_MAP_SWIZZLE_128B)) {
      return map_failed("single-pass transposed output map");
    }
  } else {
    tqt = tq;
  }
  set_error_site("single-pass cooperative launch");
  return launch_kernel(fn, dim3(static_cast<unsigned>(grid)), dim3(kSpThreads), kSinglePassSmem,
                       stream, 1, true, tm, tq, tqt, p);
}

namespace {

// The paired kernel's shared memory and resident CTAs per SM (once per device).
cudaError_t pair_prepare(int* ctas_per_sm) {
  static std::mutex mu;
  static int per_sm[64] = {};
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (per_sm[d] == 0) {
    auto k = cast_pair_single_pass_kernel<0, true>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSinglePassSmem));
    if (e != cudaSuccess) return e;
    const int n = resident_ctas(k, kSpThreads, kSinglePassSmem);
    if (n < 1) {
      *ctas_per_sm = 0;
      return cudaSuccess;
    }
    per_sm[d] = n;
  }
  *ctas_per_sm = per_sm[d];
  return cudaSuccess;
}

int64_t tiles_of(int64_t rows, int64_t cols) {
  return ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
}

}  // namespace

bool single_pass_pair_fits(const DeviceInfo& dev, int64_t w_rows, int64_t w_cols, int64_t x_rows,
                           int64_t x_cols) {
  if (w_rows <= 0 || w_cols <= 0 || x_rows <= 0 || x_cols <= 0) return false;
  if (cluster_cast_fits(w_rows, w_cols) || !single_pass_fits(dev, w_rows, w_cols)) return false;
  int per_sm = 0;
  if (pair_prepare(&per_sm) != cudaSuccess || per_sm < 1) return false;
  const int64_t max_grid = static_cast<int64_t>(dev.num_sms) * per_sm;
  const int64_t wt = tiles_of(w_rows, w_cols);
  const int64_t grid = wt < max_grid ? wt : max_grid;
  return wt <= max_grid * kSinglePassTilesPerCta && tiles_of(x_rows, x_cols) <= grid;
}

cudaError_t launch_cast_single_pass_pair(const SinglePassArgs& a, const SinglePassArgs& x,
                                         const DeviceInfo& dev, cudaStream_t stream) {
  if (a.fmt != 0 || x.fmt != 0 || a.out_t == nullptr || x.out_t == nullptr)
    return cudaErrorInvalidValue;
  if (!single_pass_pair_fits(dev, a.rows, a.cols, x.rows, x.cols)) return cudaErrorInvalidValue;
  int per_sm = 0;
  cudaError_t e = pair_prepare(&per_sm);
  if (e != cudaSuccess) return e;
  SinglePassParams p;
  p.rows = a.rows;
  p.cols = a.cols;
  p.eps = a.eps;
  p.amax_out = a.amax_out;
  p.scale_out = a.scale_out;
  p.inv_out = a.inv_out;
  p.out = a.out;
  p.out_t = a.out_t;
  p.ws_barrier = a.ws_barrier;
  p.ws_exits = a.ws_exits;
  p.ws_amax = a.ws_amax;
  p.ws_error = a.ws_error;
  p.x2 = x.x;
  p.rows2 = x.rows;
  p.cols2 = x.cols;
  p.ld2 = x.ld;
  p.eps2 = x.eps;
  p.amax2_out = x.amax_out;
  p.scale2_out = x.scale_out;
  p.inv2_out = x.inv_out;
  p.out2 = x.out;
  p.out2_t = x.out_t;
  p.ws_amax2 = x.ws_amax;
  const int64_t wt = tiles_of(a.rows, a.cols);
  const int64_t max_grid = static_cast<int64_t>(dev.num_sms) * per_sm;
  const int64_t grid = wt < max_grid ? wt : max_grid;
  CUtensorMap tm, tq, tqt, tq2, tqt2;
  if (!make_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, static_cast<uint64_t>(a.cols),
                   static_cast<uint64_t>(a.rows), static_cast<uint64_t>(a.ld) * 2, kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return map_failed("paired single-pass input map");
  const void* qw = a.out != nullptr ? static_cast<const void*>(a.out) : a.out_t;
  const void* qx = x.out != nullptr ? static_cast<const void*>(x.out) : x.out_t;
  if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw,
                   static_cast<uint64_t>(a.out != nullptr ? a.cols : a.rows),
                   static_cast<uint64_t>(a.out != nullptr ? a.rows : a.cols),
                   static_cast<uint64_t>(a.out != nullptr ? a.cols : a.rows), kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&tqt, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.out_t, static_cast<uint64_t>(a.rows),
                   static_cast<uint64_t>(a.cols), static_cast<uint64_t>(a.rows), kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&tq2, CU_TENSOR_MAP_DATA_TYPE_UINT8, qx,
                   static_cast<uint64_t>(x.out != nullptr ? x.cols : x.rows),
                   static_cast<uint64_t>(x.out != nullptr ? x.rows : x.cols),
                   static_cast<uint64_t>(x.out != nullptr ? x.cols : x.rows), kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&tqt2, CU_TENSOR_MAP_DATA_TYPE_UINT8, x.out_t, static_cast<uint64_t>(x.rows),
                   static_cast<uint64_t>(x.cols), static_cast<uint64_t>(x.rows), kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return map_failed("paired single-pass output map");
  set_error_site("paired single-pass cooperative launch");
  return launch_kernel(cast_pair_single_pass_kernel<0, true>, dim3(static_cast<unsigned>(grid)),
                       dim3(kSpThreads), kSinglePassSmem, stream, 1, true, tm, tq, tqt, p, tq2,
                       tqt2);
}

}  // namespace fp8lin
