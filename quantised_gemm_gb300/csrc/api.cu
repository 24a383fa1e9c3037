// api.cu -- the C ABI of libfp8lin: argument checks, orchestration of the
// forward and backward of the fp8 Linear on the caller's stream, workspace
// layout, error reporting and the measurement hooks.  No device memory is
// allocated here; every buffer comes from the caller.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "../../include/fp8lin.h"
#include "internal.h"

namespace fp8lin {
namespace {

thread_local int g_last_cuda_error = 0;
thread_local const char* g_error_site = nullptr;
thread_local char g_error_detail[256];
std::atomic<uint64_t> g_launches{0};

// Record a failed CUDA call: its error, and where (the site a launcher named
// with set_error_site, else the line of this file that saw the failure).
fp8lin_status cuda_fail(cudaError_t e, int line = __builtin_LINE()) {
  g_last_cuda_error = static_cast<int>(e);
  if (g_error_site != nullptr)
    std::snprintf(g_error_detail, sizeof(g_error_detail), "%s in %s", cudaGetErrorName(e),
                  g_error_site);
  else
    std::snprintf(g_error_detail, sizeof(g_error_detail), "%s at api.cu:%d", cudaGetErrorName(e),
                  line);
  g_error_site = nullptr;
  return FP8LIN_ECUDA;
}

// ---------------------------------------------------------------- profiling

constexpr int kProfPairs = 8192;
struct ProfRecord {
  cudaEvent_t start, stop;
  int kind;
};
bool g_prof_on = false;
int g_prof_used = 0;
ProfRecord g_prof[kProfPairs];
bool g_prof_created[kProfPairs];

struct ProfScope {
  ProfRecord* rec = nullptr;
  cudaStream_t stream;
  ProfScope(int kind, cudaStream_t s) : stream(s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_prof_on || g_prof_used >= kProfPairs) return;
    const int i = g_prof_used;
    if (!g_prof_created[i]) {
      if (cudaEventCreate(&g_prof[i].start) != cudaSuccess) return;
      if (cudaEventCreate(&g_prof[i].stop) != cudaSuccess) return;
      g_prof_created[i] = true;
    }
    rec = &g_prof[i];
    rec->kind = kind;
    ++g_prof_used;
    cudaEventRecord(rec->start, stream);
  }
  ~ProfScope() {
    if (rec) cudaEventRecord(rec->stop, stream);
  }
};

// ---------------------------------------------------------------- helpers

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int* ws_error(void* ws) {
  return reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + kWsErrorOffset);
}
uint32_t* ws_u32(void* ws, size_t off) {
  return reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + off);
}

bool valid_fmt(int32_t f) { return f == FP8LIN_E4M3 || f == FP8LIN_E5M2; }

// Checks shared by amax and cast: bf16 [rows, cols] with row stride ld.
fp8lin_status check_bf16(const void* x, int64_t rows, int64_t cols, int64_t ld) {
  if (rows < 0 || cols < 0) return FP8LIN_EINVAL;
  if (rows == 0 || cols == 0) return FP8LIN_OK;
  if (x == nullptr || !aligned16(x)) return FP8LIN_EINVAL;
  if (ld < cols) return FP8LIN_EINVAL;
  if (cols % 16 != 0 || ld % 8 != 0) return FP8LIN_EUNSUPPORTED;
  if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31)) return FP8LIN_EUNSUPPORTED;
  return FP8LIN_OK;
}

fp8lin_status check_state(const fp8lin_scaling_state* st, bool need_delayed_buffers) {
  if (st == nullptr) return FP8LIN_EINVAL;
  if (!valid_fmt(st->fmt)) return FP8LIN_EUNSUPPORTED;
  if (st->kind != FP8LIN_DYNAMIC && st->kind != FP8LIN_DELAYED) return FP8LIN_EUNSUPPORTED;
  if (st->amax == nullptr || st->scale == nullptr || st->inv_scale == nullptr)
    return FP8LIN_EINVAL;
  if (!(st->eps > 0.0f)) return FP8LIN_EINVAL;
  if (st->kind == FP8LIN_DELAYED && need_delayed_buffers) {
    if (st->history_len < 1) return FP8LIN_EINVAL;
    if (st->amax_history == nullptr || st->head == nullptr) return FP8LIN_EINVAL;
  }
  if (st->amax_algo < FP8LIN_AMAX_ATOMIC || st->amax_algo > FP8LIN_AMAX_PRECOMPUTED)
    return FP8LIN_EUNSUPPORTED;
  if (st->amax_algo == FP8LIN_AMAX_PRECOMPUTED && st->kind != FP8LIN_DYNAMIC)
    return FP8LIN_EUNSUPPORTED;  // delayed scaling records the amax in its own cast pass
  return FP8LIN_OK;
}

// amax into a device fp32 (ATOMIC or REDUCTION).
fp8lin_status do_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, float* amax_out,
                      int32_t algo, void* ws, const DeviceInfo& dev, cudaStream_t stream) {
  uint32_t* out_bits = reinterpret_cast<uint32_t*>(amax_out);
  if (rows == 0 || cols == 0) {
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), stream);
    return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
  }
  const int grid = amax_grid(dev, rows, cols);
  if (algo == FP8LIN_AMAX_REDUCTION) {
    uint32_t* part = ws_u32(ws, kWsPartialOffset);
    {
      ProfScope ps(FP8LIN_PROF_AMAX, stream);
      cudaError_t e = launch_amax(static_cast<const uint16_t*>(x), rows, cols, ld, part, false,
                                  grid, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    ProfScope ps(FP8LIN_PROF_AMAX, stream);
    cudaError_t e = launch_amax_final(part, grid, out_bits, stream);
    return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
  }
  if (ws != nullptr) {
    // One atomic max per CTA through the workspace's self-cleaning words.
    ProfScope ps(FP8LIN_PROF_AMAX, stream);
    cudaError_t e = launch_amax(static_cast<const uint16_t*>(x), rows, cols, ld, out_bits, true,
                                grid, stream, ws_u32(ws, kWsAtomicAccOffset),
                                ws_u32(ws, kWsAtomicTicketOffset));
    return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
  }
  cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), stream);
  if (e != cudaSuccess) return cuda_fail(e);
  ProfScope ps(FP8LIN_PROF_AMAX, stream);
  e = launch_amax(static_cast<const uint16_t*>(x), rows, cols, ld, out_bits, true, grid, stream);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

fp8lin_status do_cast(const CastArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (a.rows == 0 || a.cols == 0) return FP8LIN_OK;
  ProfScope ps(FP8LIN_PROF_CAST, stream);
  cudaError_t e = launch_cast(a, dev, stream);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

// Dynamic scaling of one tensor: amax -> scale -> cast (+T) per st->amax_algo.
// FP8LIN_PAIR_CAST=0 casts x and W of the forward in separate launches even
// where one paired single pass would take both.
bool pair_cast_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("FP8LIN_PAIR_CAST");
    return !(v != nullptr && v[0] == '0');
  }();
  return on;
}

bool single_pass_algo(int32_t algo) {
  return algo == FP8LIN_AMAX_AUTO || algo == FP8LIN_AMAX_SINGLE_PASS;
}

SinglePassArgs single_pass_args(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                const fp8lin_scaling_state* st, uint8_t* out, uint8_t* out_t,
                                void* ws) {
  SinglePassArgs sp;
  sp.x = static_cast<const uint16_t*>(x);
  sp.rows = rows;
  sp.cols = cols;
  sp.ld = ld;
  sp.fmt = st->fmt;
  sp.eps = st->eps;
  sp.amax_out = st->amax;
  sp.scale_out = st->scale;
  sp.inv_out = st->inv_scale;
  sp.out = out;
  sp.out_t = out_t;
  sp.ws_barrier = ws_u32(ws, kWsBarrierOffset);
  sp.ws_exits = ws_u32(ws, kWsExitsOffset);
  sp.ws_amax = ws_u32(ws, kWsAmaxOffset);
  sp.ws_error = ws_error(ws);
  return sp;
}

// SINGLE_PASS falls back to ATOMIC when the tensor does not fit on chip and
// `allow_fallback` is set.  PRECOMPUTED takes *st->amax as given (written by
// the producer of x, e.g. a GEMM epilogue) and runs scale + cast only.
fp8lin_status cast_dynamic_scaled(const void* x, int64_t rows, int64_t cols, int64_t ld,
                           const fp8lin_scaling_state* st, uint8_t* out, uint8_t* out_t, void* ws,
                           const DeviceInfo& dev, cudaStream_t stream, bool allow_fallback) {
  int32_t algo = st->amax_algo;
  if ((algo == FP8LIN_AMAX_SINGLE_PASS || algo == FP8LIN_AMAX_AUTO) && rows > 0 && cols > 0) {
    const bool cluster = cluster_cast_fits(rows, cols);
    if (cluster || single_pass_fits(dev, rows, cols)) {
      SinglePassArgs sp;
      sp.x = static_cast<const uint16_t*>(x);
      sp.rows = rows;
      sp.cols = cols;
      sp.ld = ld;
      sp.fmt = st->fmt;
      sp.eps = st->eps;
      sp.amax_out = st->amax;
      sp.scale_out = st->scale;
      sp.inv_out = st->inv_scale;
      sp.out = out;
      sp.out_t = out_t;
      sp.ws_barrier = ws_u32(ws, kWsBarrierOffset);
      sp.ws_exits = ws_u32(ws, kWsExitsOffset);
      sp.ws_amax = ws_u32(ws, kWsAmaxOffset);
      sp.ws_error = ws_error(ws);
      ProfScope ps(FP8LIN_PROF_CAST_FUSED, stream);
      cudaError_t e =
          cluster ? launch_cast_cluster(sp, stream) : launch_cast_single_pass(sp, dev, stream);
      return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
    }
    if (!allow_fallback && algo == FP8LIN_AMAX_SINGLE_PASS) return FP8LIN_EUNSUPPORTED;
    algo = FP8LIN_AMAX_ATOMIC;
  }
  if (algo != FP8LIN_AMAX_PRECOMPUTED) {
    fp8lin_status s = do_amax(x, rows, cols, ld, st->amax, algo, ws, dev, stream);
    if (s != FP8LIN_OK) return s;
  }
  if (rows == 0 || cols == 0) {
    ProfScope ps(FP8LIN_PROF_SCALE, stream);
    cudaError_t e = launch_scale(st->amax, st->scale, st->inv_scale, nullptr, nullptr, 1, false,
                                 st->fmt, st->eps, stream);
    return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
  }
  CastArgs c;
  c.x = static_cast<const uint16_t*>(x);
  c.rows = rows;
  c.cols = cols;
  c.ld = ld;
  c.fmt = st->fmt;
  c.scale_in = nullptr;
  c.amax_in = st->amax;
  c.derive_scale = true;
  c.eps = st->eps;
  c.scale_out = st->scale;
  c.inv_out = st->inv_scale;
  c.out = out;
  c.out_t = out_t;
  c.amax_rec = nullptr;
  c.err = ws_error(ws);
  return do_cast(c, dev, stream);
}

// Delayed scaling of one tensor inside forward/backward: cast with the stored
// scale and record this tensor's amax in the same pass; on the first step
// (needs_init) take the scale from the tensor's own amax first.
fp8lin_status delayed_cast(const void* x, int64_t rows, int64_t cols, int64_t ld,
                           fp8lin_scaling_state* st, uint8_t* out, uint8_t* out_t, void* ws,
                           const DeviceInfo& dev, cudaStream_t stream) {
  if (st->needs_init) {
    fp8lin_status s = do_amax(x, rows, cols, ld, st->amax, FP8LIN_AMAX_ATOMIC, ws, dev, stream);
    if (s != FP8LIN_OK) return s;
    ProfScope ps(FP8LIN_PROF_SCALE, stream);
    cudaError_t e = launch_scale(st->amax, st->scale, st->inv_scale, nullptr, nullptr, 1, false,
                                 st->fmt, st->eps, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    st->needs_init = 0;
  }
  if (rows == 0 || cols == 0) {
    cudaError_t e = cudaMemsetAsync(st->amax, 0, sizeof(float), stream);
    return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
  }
  CastArgs c;
  c.x = static_cast<const uint16_t*>(x);
  c.rows = rows;
  c.cols = cols;
  c.ld = ld;
  c.fmt = st->fmt;
  c.scale_in = st->scale;
  c.amax_in = nullptr;
  c.derive_scale = false;
  c.eps = st->eps;
  c.scale_out = nullptr;
  c.inv_out = nullptr;
  c.out = out;
  c.out_t = out_t;
  c.amax_rec = reinterpret_cast<uint32_t*>(st->amax);
  c.rec_acc = ws_u32(ws, kWsAtomicAccOffset);
  c.rec_ticket = ws_u32(ws, kWsAtomicTicketOffset);
  c.err = ws_error(ws);
  return do_cast(c, dev, stream);
}

GemmArgs gemm_args(const uint8_t* a, const uint8_t* b, int64_t M, int64_t N, int64_t K,
                   int64_t lda, int64_t ldb, int32_t fa, int32_t fb, const float* inv_a,
                   const float* inv_b, void* d, int64_t ldd, float* d_amax, void* ws,
                   size_t ws_bytes) {
  GemmArgs g;
  g.a = a;
  g.b = b;
  g.M = M;
  g.N = N;
  g.K = K;
  g.lda = lda;
  g.ldb = ldb;
  g.fmt_a = fa;
  g.fmt_b = fb;
  g.inv_a = inv_a;
  g.inv_b = inv_b;
  g.d = d;
  g.ldd = ldd;
  g.d_amax = reinterpret_cast<uint32_t*>(d_amax);
  g.ws_amax_acc = ws_u32(ws, kWsGemmAmaxAccOffset);
  g.ws_amax_ticket = ws_u32(ws, kWsGemmAmaxTicketOffset);
  g.ws_error = ws_error(ws);
  if (ws_bytes > kWsSplitOffset) {
    g.ws_tickets = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + kWsTicketOffset);
    g.ws_split = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsSplitOffset);
    g.ws_split_bytes = ws_bytes - kWsSplitOffset;
  } else {
    g.ws_tickets = nullptr;
    g.ws_split = nullptr;
    g.ws_split_bytes = 0;
  }
  return g;
}

fp8lin_status do_gemm(const uint8_t* a, const uint8_t* b, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int32_t fa, int32_t fb, const float* inv_a,
                      const float* inv_b, void* d, int64_t ldd, float* d_amax, void* ws,
                      size_t ws_bytes, const DeviceInfo& dev, cudaStream_t stream) {
  if (M == 0 || N == 0 || K == 0) {
    // Nothing to multiply: D (if any) is zeros, and so is its amax.
    cudaError_t e = cudaSuccess;
    if (M > 0 && N > 0)
      e = cudaMemset2DAsync(d, static_cast<size_t>(ldd) * 2, 0, static_cast<size_t>(N) * 2,
                            static_cast<size_t>(M), stream);
    if (e == cudaSuccess && d_amax != nullptr)
      e = cudaMemsetAsync(d_amax, 0, sizeof(float), stream);
    return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
  }
  const GemmArgs g = gemm_args(a, b, M, N, K, lda, ldb, fa, fb, inv_a, inv_b, d, ldd, d_amax, ws,
                               ws_bytes);
  ProfScope ps(FP8LIN_PROF_GEMM, stream);
  cudaError_t e = launch_gemm(g, dev, stream);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

fp8lin_status get_dev(DeviceInfo* dev) {
  cudaError_t e = current_device_info(dev);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

bool ws_ok(const void* ws) {
  return ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0;
}

fp8lin_status run_scale(const fp8lin_scaling_state* st, cudaStream_t stream) {
  const bool delayed = st->kind == FP8LIN_DELAYED;
  ProfScope ps(FP8LIN_PROF_SCALE, stream);
  cudaError_t e = launch_scale(st->amax, st->scale, st->inv_scale, st->amax_history, st->head,
                               delayed ? st->history_len : 1, delayed, st->fmt, st->eps, stream);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

}  // namespace

void set_error_site(const char* site) { g_error_site = site; }

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("FP8LIN_PDL");
    return !(v != nullptr && v[0] == '0');
  }();
  return on;
}

cudaError_t current_device_info(DeviceInfo* info) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  // Bind the device's primary context to this thread: a thread that never
  // called cudaSetDevice (e.g. an autograd worker) may have none current, and
  // the driver-level tensor-map encoding needs one.
  e = cudaSetDevice(d);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[d]) {
    DeviceInfo x;
    x.device = d;
    e = cudaDeviceGetAttribute(&x.num_sms, cudaDevAttrMultiProcessorCount, d);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&x.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    if (e != cudaSuccess) return e;
    cache[d] = x;
    have[d] = true;
  }
  *info = cache[d];
  return cudaSuccess;
}

}  // namespace fp8lin

using namespace fp8lin;

extern "C" {

const char* fp8lin_status_string(int status) {
  switch (status) {
    case FP8LIN_OK: return "FP8LIN_OK";
    case FP8LIN_EINVAL: return "FP8LIN_EINVAL: invalid argument";
    case FP8LIN_EUNSUPPORTED: return "FP8LIN_EUNSUPPORTED: shape, format or size not supported";
    case FP8LIN_ECUDA: return "FP8LIN_ECUDA: a CUDA call failed";
    case FP8LIN_ETIMEOUT: return "FP8LIN_ETIMEOUT: a bounded device wait ran out";
    default: return "unknown fp8lin status";
  }
}

int fp8lin_last_cuda_error(void) { return g_last_cuda_error; }

const char* fp8lin_last_error_detail(void) {
  return g_last_cuda_error == 0 ? "" : g_error_detail;
}

int fp8lin_version(void) { return 101; }

size_t fp8lin_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  (void)M;
  (void)K;
  (void)N;
  // Fixed part (error word, grid barrier, amax partials), the K-split tickets
  // and room for the K-split partials of the GEMMs' tail wave.
  int num_sms = 152;
  DeviceInfo dev;
  if (current_device_info(&dev) == cudaSuccess) num_sms = dev.num_sms;
  else cudaGetLastError();
  return kWsSplitOffset + gemm_split_workspace_bytes(num_sms);
}

int64_t fp8lin_single_pass_max_elems(void) {
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return 0;
  return single_pass_capacity_elems(dev);
}

fp8lin_status fp8lin_check(void* ws, cudaStream_t stream) {
  if (!ws_ok(ws)) return FP8LIN_EINVAL;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int code = 0;
  e = cudaMemcpy(&code, ws_error(ws), sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (code == 0) return FP8LIN_OK;
  // A wait that ran out can leave counters of the workspace mid-count: clear
  // the error word and the GEMM split tickets so the workspace is usable again.
  e = cudaMemset(ws_error(ws), 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemset(static_cast<uint8_t*>(ws) + kWsTicketOffset, 0, sizeof(int) * kWsTickets);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemset(static_cast<uint8_t*>(ws) + kWsScratchBegin, 0,
                 kWsPartialOffset - kWsScratchBegin);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8LIN_ETIMEOUT;
}

fp8lin_status fp8lin_amax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                          float* amax_out, int32_t algo, void* ws, cudaStream_t stream) {
  fp8lin_status s = check_bf16(x, rows, cols, ld);
  if (s != FP8LIN_OK) return s;
  if (amax_out == nullptr || (reinterpret_cast<uintptr_t>(amax_out) & 3u)) return FP8LIN_EINVAL;
  if (algo != FP8LIN_AMAX_ATOMIC && algo != FP8LIN_AMAX_REDUCTION) return FP8LIN_EUNSUPPORTED;
  if (algo == FP8LIN_AMAX_REDUCTION && !ws_ok(ws)) return FP8LIN_EINVAL;
  DeviceInfo dev;
  if ((s = get_dev(&dev)) != FP8LIN_OK) return s;
  return do_amax(x, rows, cols, ld, amax_out, algo, ws, dev, stream);
}

fp8lin_status fp8lin_amax_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                  float* amax_out, cudaStream_t stream) {
  fp8lin_status s = check_bf16(x, rows, cols, ld);
  if (s != FP8LIN_OK) return s;
  if (amax_out == nullptr || (reinterpret_cast<uintptr_t>(amax_out) & 3u)) return FP8LIN_EINVAL;
  DeviceInfo dev;
  if ((s = get_dev(&dev)) != FP8LIN_OK) return s;
  if (rows == 0 || cols == 0) {
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), stream);
    return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
  }
  const int grid = amax_grid(dev, rows, cols);
  if (grid > kStaticAmaxPartials) return FP8LIN_EUNSUPPORTED;  // more CTAs than scratch slots
  g_launches.fetch_add(2, std::memory_order_relaxed);
  cudaError_t e = launch_amax_static_scratch(static_cast<const uint16_t*>(x), rows, cols, ld,
                                             amax_out, grid, stream);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

fp8lin_status fp8lin_scale(const fp8lin_scaling_state* st, cudaStream_t stream) {
  fp8lin_status s = check_state(st, true);
  if (s != FP8LIN_OK) return s;
  return run_scale(st, stream);
}

// The device byte ranges the scale update of one state writes (scale, inverse
// and, delayed, the ring and its head); it reads only these and *amax.
struct ByteRange {
  uintptr_t lo, hi;
};

int scale_written_ranges(const fp8lin_scaling_state* st, ByteRange* r) {
  auto at = [](const void* p, size_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return ByteRange{lo, lo + bytes};
  };
  int n = 0;
  r[n++] = at(st->scale, sizeof(float));
  r[n++] = at(st->inv_scale, sizeof(float));
  if (st->kind == FP8LIN_DELAYED) {
    r[n++] = at(st->amax_history, sizeof(float) * static_cast<size_t>(st->history_len));
    r[n++] = at(st->head, sizeof(int32_t));
  }
  return n;
}

bool ranges_overlap(const ByteRange& a, const ByteRange& b) { return a.lo < b.hi && b.lo < a.hi; }

// True if a buffer that one of the n states' updates writes overlaps any
// buffer of another state (one thread per state would race on it).  States
// may share an amax, which the update only reads.
bool scale_states_overlap(const fp8lin_scaling_state* states, int n) {
  for (int i = 0; i < n; ++i) {
    ByteRange wi[4];
    const int ni = scale_written_ranges(&states[i], wi);
    for (int j = 0; j < n; ++j) {
      if (j == i) continue;
      ByteRange bj[5];
      int nj = scale_written_ranges(&states[j], bj);
      const uintptr_t amax = reinterpret_cast<uintptr_t>(states[j].amax);
      bj[nj++] = {amax, amax + sizeof(float)};
      for (int x = 0; x < ni; ++x)
        for (int y = 0; y < nj; ++y)
          if (ranges_overlap(wi[x], bj[y])) return true;
    }
  }
  return false;
}

fp8lin_status fp8lin_scale_many(const fp8lin_scaling_state* states, int32_t n,
                                cudaStream_t stream) {
  if (n < 0 || n > 8 || (n > 0 && states == nullptr)) return FP8LIN_EINVAL;
  ScaleArgs a[8];
  for (int i = 0; i < n; ++i) {
    const fp8lin_scaling_state* st = &states[i];
    fp8lin_status s = check_state(st, true);
    if (s != FP8LIN_OK) return s;
    const bool delayed = st->kind == FP8LIN_DELAYED;
    a[i] = {st->amax, st->scale, st->inv_scale, st->amax_history, st->head,
            delayed ? st->history_len : 1, delayed, st->fmt, st->eps};
  }
  if (n == 0) return FP8LIN_OK;
  if (scale_states_overlap(states, n)) return FP8LIN_EINVAL;
  ProfScope ps(FP8LIN_PROF_SCALE, stream);
  cudaError_t e = launch_scale_batch(a, n, stream);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

fp8lin_status fp8lin_cast(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t fmt,
                          const float* scale, uint8_t* out, uint8_t* out_t, float* amax_out,
                          cudaStream_t stream) {
  fp8lin_status s = check_bf16(x, rows, cols, ld);
  if (s != FP8LIN_OK) return s;
  if (!valid_fmt(fmt)) return FP8LIN_EUNSUPPORTED;
  if (scale == nullptr) return FP8LIN_EINVAL;
  if (out == nullptr && out_t == nullptr) return FP8LIN_EINVAL;
  if (out != nullptr && !aligned16(out)) return FP8LIN_EINVAL;
  if (out_t != nullptr) {
    if (!aligned16(out_t)) return FP8LIN_EINVAL;
    if (rows % 16 != 0) return FP8LIN_EUNSUPPORTED;
  }
  DeviceInfo dev;
  if ((s = get_dev(&dev)) != FP8LIN_OK) return s;
  if (amax_out != nullptr) {
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  CastArgs c;
  c.x = static_cast<const uint16_t*>(x);
  c.rows = rows;
  c.cols = cols;
  c.ld = ld;
  c.fmt = fmt;
  c.scale_in = scale;
  c.amax_in = nullptr;
  c.derive_scale = false;
  c.eps = 1e-12f;
  c.scale_out = nullptr;
  c.inv_out = nullptr;
  c.out = out;
  c.out_t = out_t;
  c.amax_rec = reinterpret_cast<uint32_t*>(amax_out);
  return do_cast(c, dev, stream);
}

fp8lin_status fp8lin_cast_dynamic(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                  const fp8lin_scaling_state* st, uint8_t* out, uint8_t* out_t,
                                  void* ws, cudaStream_t stream) {
  fp8lin_status s = check_bf16(x, rows, cols, ld);
  if (s != FP8LIN_OK) return s;
  if ((s = check_state(st, false)) != FP8LIN_OK) return s;
  if (st->kind != FP8LIN_DYNAMIC) return FP8LIN_EINVAL;
  if (!ws_ok(ws)) return FP8LIN_EINVAL;
  if (out == nullptr && out_t == nullptr) return FP8LIN_EINVAL;
  if (out != nullptr && !aligned16(out)) return FP8LIN_EINVAL;
  if (out_t != nullptr) {
    if (!aligned16(out_t)) return FP8LIN_EINVAL;
    if (rows % 16 != 0) return FP8LIN_EUNSUPPORTED;
  }
  DeviceInfo dev;
  if ((s = get_dev(&dev)) != FP8LIN_OK) return s;
  return cast_dynamic_scaled(x, rows, cols, ld, st, out, out_t, ws, dev, stream, false);
}

fp8lin_status fp8lin_cast_delayed(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                  fp8lin_scaling_state* st, uint8_t* out, uint8_t* out_t,
                                  void* ws, cudaStream_t stream) {
  fp8lin_status s = check_bf16(x, rows, cols, ld);
  if (s != FP8LIN_OK) return s;
  if ((s = check_state(st, false)) != FP8LIN_OK) return s;
  if (st->kind != FP8LIN_DELAYED) return FP8LIN_EINVAL;
  if (!ws_ok(ws)) return FP8LIN_EINVAL;
  if (out == nullptr && out_t == nullptr) return FP8LIN_EINVAL;
  if (out != nullptr && !aligned16(out)) return FP8LIN_EINVAL;
  if (out_t != nullptr) {
    if (!aligned16(out_t)) return FP8LIN_EINVAL;
    if (rows % 16 != 0) return FP8LIN_EUNSUPPORTED;
  }
  DeviceInfo dev;
  if ((s = get_dev(&dev)) != FP8LIN_OK) return s;
  return delayed_cast(x, rows, cols, ld, st, out, out_t, ws, dev, stream);
}

fp8lin_status fp8lin_gemm(const uint8_t* a, const uint8_t* b, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int32_t fmt_a, int32_t fmt_b,
                          const float* inv_a, const float* inv_b, void* d, int64_t ldd,
                          float* d_amax, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0) return FP8LIN_EINVAL;
  if (!valid_fmt(fmt_a) || !valid_fmt(fmt_b)) return FP8LIN_EUNSUPPORTED;
  if (!ws_ok(ws) || ws_bytes < kWsFixedBytes) return FP8LIN_EINVAL;
  if (d_amax != nullptr && (reinterpret_cast<uintptr_t>(d_amax) & 3u) != 0) return FP8LIN_EINVAL;
  if (M == 0 || N == 0) {
    if (d_amax == nullptr) return FP8LIN_OK;
    DeviceInfo dev;
    fp8lin_status s = get_dev(&dev);
    if (s != FP8LIN_OK) return s;
    return do_gemm(a, b, M, N, K, lda, ldb, fmt_a, fmt_b, inv_a, inv_b, d, ldd, d_amax, ws,
                   ws_bytes, dev, stream);
  }
  if (d == nullptr || !aligned16(d) || ldd < N) return FP8LIN_EINVAL;
  if (inv_a == nullptr || inv_b == nullptr) return FP8LIN_EINVAL;
  if (K > 0) {
    if (a == nullptr || b == nullptr || !aligned16(a) || !aligned16(b)) return FP8LIN_EINVAL;
    if (lda < K || ldb < K) return FP8LIN_EINVAL;
    if (lda % 16 != 0 || ldb % 16 != 0 || K % 16 != 0) return FP8LIN_EUNSUPPORTED;
  }
  if (N % 16 != 0 || ldd % 8 != 0) return FP8LIN_EUNSUPPORTED;
  if (M > (int64_t(1) << 31) - 256 || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - 256)
    return FP8LIN_EUNSUPPORTED;
  DeviceInfo dev;
  fp8lin_status s = get_dev(&dev);
  if (s != FP8LIN_OK) return s;
  return do_gemm(a, b, M, N, K, lda, ldb, fmt_a, fmt_b, inv_a, inv_b, d, ldd, d_amax, ws, ws_bytes,
                 dev, stream);
}

fp8lin_status fp8lin_gemm_describe(int64_t M, int64_t N, int64_t K, char* buf, size_t buf_len) {
  if (M < 0 || N < 0 || K < 0 || buf == nullptr || buf_len == 0) return FP8LIN_EINVAL;
  buf[0] = '\0';
  DeviceInfo dev;
  fp8lin_status s = get_dev(&dev);
  if (s != FP8LIN_OK) return s;
  cudaError_t e = describe_gemm(M, N, K, dev, buf, buf_len);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

fp8lin_status fp8lin_gemm_describe_for(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                                       char* buf, size_t buf_len) {
  if (M < 0 || N < 0 || K < 0 || num_sms < 2 || buf == nullptr || buf_len == 0)
    return FP8LIN_EINVAL;
  describe_plan(M, N, K, num_sms, num_sms / 2, buf, buf_len);
  return FP8LIN_OK;
}

fp8lin_status fp8lin_gemm_group_describe_for(int64_t Ma, int64_t Na, int64_t Ka, int64_t Mb,
                                             int64_t Nb, int64_t Kb, int32_t num_sms, char* buf,
                                             size_t buf_len) {
  if (Ma < 1 || Na < 1 || Ka < 1 || Mb < 1 || Nb < 1 || Kb < 1 || num_sms < 2 || buf == nullptr ||
      buf_len == 0)
    return FP8LIN_EINVAL;
  describe_group_plan(Ma, Na, Ka, Mb, Nb, Kb, num_sms, num_sms / 2, buf, buf_len);
  return FP8LIN_OK;
}

static fp8lin_status check_linear_sizes(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || K < 0 || N < 0) return FP8LIN_EINVAL;
  if (M % 16 != 0 || K % 16 != 0 || N % 16 != 0) return FP8LIN_EUNSUPPORTED;
  if (M > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - 256 ||
      N > (int64_t(1) << 31) - 256)
    return FP8LIN_EUNSUPPORTED;
  return FP8LIN_OK;
}

static bool dev_ptrs_ok(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr || !aligned16(p)) return false;
  return true;
}

}  // extern "C"

namespace {

fp8lin_status check_forward(const void* x, const void* w, int64_t M, int64_t K, int64_t N,
                            const fp8lin_scaling_state* sx, const fp8lin_scaling_state* sw,
                            const void* y, const float* y_amax, const uint8_t* x8,
                            const uint8_t* x8t, const uint8_t* w8, const uint8_t* w8t,
                            const void* ws, size_t ws_bytes) {
  fp8lin_status s = check_linear_sizes(M, K, N);
  if (s != FP8LIN_OK) return s;
  if ((s = check_state(sx, true)) != FP8LIN_OK) return s;
  if ((s = check_state(sw, true)) != FP8LIN_OK) return s;
  if (sx->fmt != FP8LIN_E4M3 || sw->fmt != FP8LIN_E4M3) return FP8LIN_EUNSUPPORTED;
  if (!ws_ok(ws) || ws_bytes < kWsFixedBytes) return FP8LIN_EINVAL;
  if (M * K > 0 && !dev_ptrs_ok({x, x8, x8t})) return FP8LIN_EINVAL;
  if (N * K > 0 && !dev_ptrs_ok({w8, w8t})) return FP8LIN_EINVAL;
  if (w != nullptr && N * K > 0 && !dev_ptrs_ok({w})) return FP8LIN_EINVAL;
  // w == NULL reuses w8 / w8t / sw from an earlier call: there must have been one.
  if (w == nullptr && sw->kind == FP8LIN_DELAYED && sw->needs_init) return FP8LIN_EINVAL;
  if (M * N > 0 && !dev_ptrs_ok({y})) return FP8LIN_EINVAL;
  if (y_amax != nullptr && (reinterpret_cast<uintptr_t>(y_amax) & 3u) != 0) return FP8LIN_EINVAL;
  return FP8LIN_OK;
}

// Few-token products run as one fused launch each (small_m.cu) when the
// token side has dynamic scaling; FP8LIN_SMALL_M=0 turns this off.
bool small_m_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("FP8LIN_SMALL_M");
    return !(v != nullptr && v[0] == '0');
  }();
  return on;
}

// The backward's few-token product also computes dW unless FP8LIN_SMALL_M_DW=0.
bool small_m_dw_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("FP8LIN_SMALL_M_DW");
    return !(v != nullptr && v[0] == '0');
  }();
  return on;
}

bool few_token_state(const fp8lin_scaling_state* st, int64_t M) {
  return small_m_enabled() && M >= 1 && M <= kSmallMaxRows && st->kind == FP8LIN_DYNAMIC &&
         (st->amax_algo == FP8LIN_AMAX_AUTO || st->amax_algo == FP8LIN_AMAX_SINGLE_PASS ||
          st->amax_algo == FP8LIN_AMAX_PRECOMPUTED);
}

size_t split_bytes(size_t ws_bytes) {
  return ws_bytes > kWsSplitOffset ? ws_bytes - kWsSplitOffset : 0;
}

// The fused few-token product D = B8 . A8^T (token side B cast in the launch).
SmallMArgs small_m_args(const fp8lin_scaling_state* sb, const void* b, int64_t M, uint8_t* b8,
                        uint8_t* b8t, void* d, int64_t ldd, float* d_amax, void* ws,
                        size_t ws_bytes) {
  SmallMArgs a = {};
  a.MB = M;
  a.b = static_cast<const uint16_t*>(b);
  a.eps = sb->eps;
  a.fmt_b = sb->fmt;
  a.b_amax_in = sb->amax_algo == FP8LIN_AMAX_PRECOMPUTED ? sb->amax : nullptr;
  a.b_amax = sb->amax;
  a.b_scale = sb->scale;
  a.b_inv = sb->inv_scale;
  a.b8 = b8;
  a.b8t = b8t;
  a.d = d;
  a.ldd = ldd;
  a.d_amax = reinterpret_cast<uint32_t*>(d_amax);
  a.ws_amax_acc = ws_u32(ws, kWsGemmAmaxAccOffset);
  a.ws_amax_ticket = ws_u32(ws, kWsGemmAmaxTicketOffset);
  a.ws_partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsSplitOffset);
  a.ws_partial_bytes = split_bytes(ws_bytes);
  a.ws_tickets = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + kWsTicketOffset);
  a.ws_barrier = ws_u32(ws, kWsBarrierOffset);
  a.ws_exits = ws_u32(ws, kWsExitsOffset);
  a.ws_amax = ws_u32(ws, kWsAmaxOffset);
  a.ws_b_amax = ws_u32(ws, kWsSmallBAmaxOffset);
  a.ws_error = ws_error(ws);
  return a;
}

fp8lin_status run_small_m(const SmallMArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  ProfScope ps(FP8LIN_PROF_SMALL_M, stream);
  cudaError_t e = launch_small_m(a, dev, stream);
  return e == cudaSuccess ? FP8LIN_OK : cuda_fail(e);
}

fp8lin_status run_forward(const void* x, const void* w, int64_t M, int64_t K, int64_t N,
                          fp8lin_scaling_state* sx, fp8lin_scaling_state* sw, void* y,
                          float* y_amax, uint8_t* x8, uint8_t* x8t, uint8_t* w8, uint8_t* w8t,
                          void* ws, size_t ws_bytes, const DeviceInfo& dev, cudaStream_t stream) {
  // A few tokens: x's cast, W's cast (unless W8 is reused) and y in one launch.
  if (K > 0 && N > 0 && few_token_state(sx, M)) {
    const bool cast_w = w != nullptr;
    const bool w_ok = !cast_w || (sw->kind == FP8LIN_DYNAMIC &&
                                  (sw->amax_algo == FP8LIN_AMAX_AUTO ||
                                   sw->amax_algo == FP8LIN_AMAX_SINGLE_PASS));
    if (w_ok && small_m_fits(dev, cast_w, 0, M, N, K, split_bytes(ws_bytes))) {
      SmallMArgs a = small_m_args(sx, x, M, x8, x8t, y, N, y_amax, ws, ws_bytes);
      a.cast_a = cast_w;
      a.NA = N;
      a.KA = K;
      a.ldb = K;
      if (cast_w) {
        a.a = w;
        a.a8 = w8;
        a.a8t = w8t;
        a.a_amax = sw->amax;
        a.a_scale = sw->scale;
        a.a_inv = sw->inv_scale;
      } else {
        a.a = w8;
        a.a_inv_in = sw->inv_scale;
      }
      return run_small_m(a, dev, stream);
    }
  }
  // W's single pass with x's cast in the same launch, where x has at most one
  // tile for each of its CTAs (a few hundred tokens): one launch and one grid
  // barrier fewer.
  if (w != nullptr && pair_cast_enabled() && sx->kind == FP8LIN_DYNAMIC &&
      sw->kind == FP8LIN_DYNAMIC && single_pass_algo(sx->amax_algo) &&
      single_pass_algo(sw->amax_algo) && x8t != nullptr && w8t != nullptr &&
      single_pass_pair_fits(dev, N, K, M, K)) {
    SinglePassArgs wa = single_pass_args(w, N, K, K, sw, w8, w8t, ws);
    SinglePassArgs xa = single_pass_args(x, M, K, K, sx, x8, x8t, ws);
    xa.ws_amax = ws_u32(ws, kWsAmax2Offset);
    {
      ProfScope ps(FP8LIN_PROF_CAST_FUSED, stream);
      cudaError_t e = launch_cast_single_pass_pair(wa, xa, dev, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return do_gemm(x8, w8, M, N, K, K, K, FP8LIN_E4M3, FP8LIN_E4M3, sx->inv_scale, sw->inv_scale,
                   y, N, y_amax, ws, ws_bytes, dev, stream);
  }
  fp8lin_status s;
  if (sx->kind == FP8LIN_DYNAMIC)
    s = cast_dynamic_scaled(x, M, K, K, sx, x8, x8t, ws, dev, stream, true);
  else
    s = delayed_cast(x, M, K, K, sx, x8, x8t, ws, dev, stream);
  if (s != FP8LIN_OK) return s;
  if (w != nullptr) {
    if (sw->kind == FP8LIN_DYNAMIC)
      s = cast_dynamic_scaled(w, N, K, K, sw, w8, w8t, ws, dev, stream, true);
    else
      s = delayed_cast(w, N, K, K, sw, w8, w8t, ws, dev, stream);
    if (s != FP8LIN_OK) return s;
  }
  // y = x8 . W8^T : A = x8 [M, K], B = W8 [N, K]
  return do_gemm(x8, w8, M, N, K, K, K, FP8LIN_E4M3, FP8LIN_E4M3, sx->inv_scale, sw->inv_scale, y,
                 N, y_amax, ws, ws_bytes, dev, stream);
}

fp8lin_status check_backward(const void* dy, int64_t M, int64_t K, int64_t N, const uint8_t* x8t,
                             const uint8_t* w8t, const fp8lin_scaling_state* sx,
                             const fp8lin_scaling_state* sw, const fp8lin_scaling_state* sdy,
                             const uint8_t* dy8, const uint8_t* dy8t, const void* dx,
                             const void* dw, const float* dx_amax, const float* dw_amax,
                             const void* ws, size_t ws_bytes) {
  fp8lin_status s = check_linear_sizes(M, K, N);
  if (s != FP8LIN_OK) return s;
  if ((s = check_state(sx, false)) != FP8LIN_OK) return s;
  if ((s = check_state(sw, false)) != FP8LIN_OK) return s;
  if ((s = check_state(sdy, true)) != FP8LIN_OK) return s;
  if (sdy->fmt != FP8LIN_E5M2) return FP8LIN_EUNSUPPORTED;
  if (!ws_ok(ws) || ws_bytes < kWsFixedBytes) return FP8LIN_EINVAL;
  if (M * N > 0 && !dev_ptrs_ok({dy, dy8, dy8t})) return FP8LIN_EINVAL;
  if (dx != nullptr && M * K > 0 && !dev_ptrs_ok({dx})) return FP8LIN_EINVAL;
  if (dx != nullptr && N * K > 0 && !dev_ptrs_ok({w8t})) return FP8LIN_EINVAL;
  if (dw != nullptr && N * K > 0 && !dev_ptrs_ok({dw})) return FP8LIN_EINVAL;
  if (dw != nullptr && M * K > 0 && !dev_ptrs_ok({x8t})) return FP8LIN_EINVAL;
  if ((dx_amax != nullptr && (dx == nullptr || (reinterpret_cast<uintptr_t>(dx_amax) & 3u))) ||
      (dw_amax != nullptr && (dw == nullptr || (reinterpret_cast<uintptr_t>(dw_amax) & 3u))))
    return FP8LIN_EINVAL;
  return FP8LIN_OK;
}

fp8lin_status run_backward(const void* dy, int64_t M, int64_t K, int64_t N, const uint8_t* x8t,
                           const uint8_t* w8t, const fp8lin_scaling_state* sx,
                           const fp8lin_scaling_state* sw, fp8lin_scaling_state* sdy,
                           uint8_t* dy8, uint8_t* dy8t, void* dx, void* dw, float* dx_amax,
                           float* dw_amax, void* ws, size_t ws_bytes, const DeviceInfo& dev,
                           cudaStream_t stream) {
  fp8lin_status s;
  bool dx_done = false, dw_done = false;
  if (dx != nullptr && K > 0 && N > 0 && few_token_state(sdy, M) &&
      small_m_fits(dev, false, FP8LIN_E5M2, M, K, N, split_bytes(ws_bytes))) {
    // A few tokens: dY's cast and dX = dY8 . W8 (A = W8^T [K, N]) in one launch,
    // and dW = dY8^T . x8 in the same launch when its amax is not wanted.
    SmallMArgs a = small_m_args(sdy, dy, M, dy8, dy8t, dx, K, dx_amax, ws, ws_bytes);
    a.cast_a = false;
    a.NA = K;
    a.KA = N;
    a.ldb = N;
    a.a = w8t;
    a.a_inv_in = sw->inv_scale;
    if (dw != nullptr && dw_amax == nullptr && small_m_dw_enabled() &&
        small_m_fits(dev, false, FP8LIN_E5M2, M, K, N, split_bytes(ws_bytes), true)) {
      a.fuse_dw = true;
      a.x8t = x8t;
      a.x_inv = sx->inv_scale;
      a.dw = dw;
      dw_done = true;
    }
    if ((s = run_small_m(a, dev, stream)) != FP8LIN_OK) return s;
    dx_done = true;
  } else if (sdy->kind == FP8LIN_DYNAMIC) {
    s = cast_dynamic_scaled(dy, M, N, N, sdy, dy8, dy8t, ws, dev, stream, true);
  } else {
    s = delayed_cast(dy, M, N, N, sdy, dy8, dy8t, ws, dev, stream);
  }
  if (!dx_done && s != FP8LIN_OK) return s;
  if (dx != nullptr && !dx_done && dw != nullptr && !dw_done && M > 0 && N > 0 && K > 0) {
    // dX and dW in one launch when the grouped plan expects it to be faster
    const GemmArgs gx = gemm_args(dy8, w8t, M, K, N, N, N, FP8LIN_E5M2, FP8LIN_E4M3,
                                  sdy->inv_scale, sw->inv_scale, dx, K, dx_amax, ws, ws_bytes);
    const GemmArgs gw = gemm_args(dy8t, x8t, N, K, M, M, M, FP8LIN_E5M2, FP8LIN_E4M3,
                                  sdy->inv_scale, sx->inv_scale, dw, K, dw_amax, ws, ws_bytes);
    bool grouped = false;
    cudaError_t e = plan_gemm_pair2(gx, gw, dev, &grouped);
    if (e != cudaSuccess) return cuda_fail(e);
    if (grouped) {
      ProfScope ps(FP8LIN_PROF_GEMM, stream);
      e = launch_gemm_pair2(gx, gw, dev, stream);
      if (e != cudaSuccess) return cuda_fail(e);
      dx_done = dw_done = true;
    }
  }
  if (dx != nullptr && !dx_done) {
    // dX = dY8 . W8 : A = dY8 [M, N], B = W8^T [K, N], contract over N
    s = do_gemm(dy8, w8t, M, K, N, N, N, FP8LIN_E5M2, FP8LIN_E4M3, sdy->inv_scale, sw->inv_scale,
                dx, K, dx_amax, ws, ws_bytes, dev, stream);
    if (s != FP8LIN_OK) return s;
  }
  if (dw != nullptr && !dw_done) {
    // dW = dY8^T . x8 : A = dY8^T [N, M], B = x8^T [K, M], contract over M
    s = do_gemm(dy8t, x8t, N, K, M, M, M, FP8LIN_E5M2, FP8LIN_E4M3, sdy->inv_scale, sx->inv_scale,
                dw, K, dw_amax, ws, ws_bytes, dev, stream);
    if (s != FP8LIN_OK) return s;
  }
  return FP8LIN_OK;
}

}  // namespace

extern "C" {

fp8lin_status fp8lin_forward(const void* x, const void* w, int64_t M, int64_t K, int64_t N,
                             fp8lin_scaling_state* sx, fp8lin_scaling_state* sw, void* y,
                             float* y_amax, uint8_t* x8, uint8_t* x8t, uint8_t* w8, uint8_t* w8t,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
  fp8lin_status s =
      check_forward(x, w, M, K, N, sx, sw, y, y_amax, x8, x8t, w8, w8t, ws, ws_bytes);
  if (s != FP8LIN_OK) return s;
  DeviceInfo dev;
  if ((s = get_dev(&dev)) != FP8LIN_OK) return s;
  return run_forward(x, w, M, K, N, sx, sw, y, y_amax, x8, x8t, w8, w8t, ws, ws_bytes, dev,
                     stream);
}

fp8lin_status fp8lin_backward(const void* dy, int64_t M, int64_t K, int64_t N,
                              const uint8_t* x8t, const uint8_t* w8t,
                              const fp8lin_scaling_state* sx, const fp8lin_scaling_state* sw,
                              fp8lin_scaling_state* sdy, uint8_t* dy8, uint8_t* dy8t, void* dx,
                              void* dw, float* dx_amax, float* dw_amax, void* ws, size_t ws_bytes,
                              cudaStream_t stream) {
  fp8lin_status s = check_backward(dy, M, K, N, x8t, w8t, sx, sw, sdy, dy8, dy8t, dx, dw, dx_amax,
                                   dw_amax, ws, ws_bytes);
  if (s != FP8LIN_OK) return s;
  DeviceInfo dev;
  if ((s = get_dev(&dev)) != FP8LIN_OK) return s;
  return run_backward(dy, M, K, N, x8t, w8t, sx, sw, sdy, dy8, dy8t, dx, dw, dx_amax, dw_amax, ws,
                      ws_bytes, dev, stream);
}

fp8lin_status fp8lin_step_host(const void* x_h, const void* w_h, const void* dy_h, void* y_h,
                               void* dx_h, void* dw_h, int64_t M, int64_t K, int64_t N,
                               fp8lin_scaling_state* sx, fp8lin_scaling_state* sw,
                               fp8lin_scaling_state* sdy, const fp8lin_step_slot* slot,
                               cudaStream_t compute, cudaStream_t h2d, cudaStream_t d2h,
                               int wait) {
  if (slot == nullptr) return FP8LIN_EINVAL;
  const fp8lin_step_slot& d = *slot;
  fp8lin_status s = check_forward(d.x, d.w, M, K, N, sx, sw, d.y, nullptr, d.x8, d.x8t, d.w8,
                                  d.w8t, d.ws, d.ws_bytes);
  if (s != FP8LIN_OK) return s;
  if ((s = check_backward(d.dy, M, K, N, d.x8t, d.w8t, sx, sw, sdy, d.dy8, d.dy8t, d.dx, d.dw,
                          nullptr, nullptr, d.ws, d.ws_bytes)) != FP8LIN_OK)
    return s;
  if (M * K > 0 && (x_h == nullptr || dx_h == nullptr || d.dx == nullptr)) return FP8LIN_EINVAL;
  if (N * K > 0 && (w_h == nullptr || dw_h == nullptr || d.w == nullptr || d.dw == nullptr))
    return FP8LIN_EINVAL;
  if (M * N > 0 && (dy_h == nullptr || y_h == nullptr)) return FP8LIN_EINVAL;
  for (cudaEvent_t e : d.ev)
    if (e == nullptr) return FP8LIN_EINVAL;
  DeviceInfo dev;
  if ((s = get_dev(&dev)) != FP8LIN_OK) return s;

  enum { kXwIn = 0, kDyIn = 1, kFwdDone = 2, kBwdDone = 3, kOutDone = 4 };
  const size_t bx = static_cast<size_t>(M) * K * 2, bw = static_cast<size_t>(N) * K * 2,
               by = static_cast<size_t>(M) * N * 2;
  cudaError_t e;
  // Uploads: x and W once this slot's previous forward has read them; dY once
  // its previous backward has.
  if ((e = cudaStreamWaitEvent(h2d, d.ev[kFwdDone], 0)) != cudaSuccess) return cuda_fail(e);
  if (bx > 0 && (e = cudaMemcpyAsync(d.x, x_h, bx, cudaMemcpyHostToDevice, h2d)) != cudaSuccess)
    return cuda_fail(e);
  if (bw > 0 && (e = cudaMemcpyAsync(d.w, w_h, bw, cudaMemcpyHostToDevice, h2d)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaEventRecord(d.ev[kXwIn], h2d)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaStreamWaitEvent(h2d, d.ev[kBwdDone], 0)) != cudaSuccess) return cuda_fail(e);
  if (by > 0 && (e = cudaMemcpyAsync(d.dy, dy_h, by, cudaMemcpyHostToDevice, h2d)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaEventRecord(d.ev[kDyIn], h2d)) != cudaSuccess) return cuda_fail(e);
  // Forward once x and W are in and this slot's outputs have gone out.
  if ((e = cudaStreamWaitEvent(compute, d.ev[kXwIn], 0)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaStreamWaitEvent(compute, d.ev[kOutDone], 0)) != cudaSuccess) return cuda_fail(e);
  s = run_forward(d.x, d.w, M, K, N, sx, sw, d.y, nullptr, d.x8, d.x8t, d.w8, d.w8t, d.ws,
                  d.ws_bytes, dev, compute);
  if (s != FP8LIN_OK) return s;
  if ((e = cudaEventRecord(d.ev[kFwdDone], compute)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaStreamWaitEvent(d2h, d.ev[kFwdDone], 0)) != cudaSuccess) return cuda_fail(e);
  if (by > 0 && (e = cudaMemcpyAsync(y_h, d.y, by, cudaMemcpyDeviceToHost, d2h)) != cudaSuccess)
    return cuda_fail(e);
  // Backward once dY is in, then the delayed states' history sync.
  if ((e = cudaStreamWaitEvent(compute, d.ev[kDyIn], 0)) != cudaSuccess) return cuda_fail(e);
  s = run_backward(d.dy, M, K, N, d.x8t, d.w8t, sx, sw, sdy, d.dy8, d.dy8t, d.dx, d.dw, nullptr,
                   nullptr, d.ws, d.ws_bytes, dev, compute);
  if (s != FP8LIN_OK) return s;
  for (const fp8lin_scaling_state* st : {static_cast<const fp8lin_scaling_state*>(sx),
                                         static_cast<const fp8lin_scaling_state*>(sw),
                                         static_cast<const fp8lin_scaling_state*>(sdy)}) {
    if (st->kind != FP8LIN_DELAYED) continue;
    if ((s = run_scale(st, compute)) != FP8LIN_OK) return s;
  }
  if ((e = cudaEventRecord(d.ev[kBwdDone], compute)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaStreamWaitEvent(d2h, d.ev[kBwdDone], 0)) != cudaSuccess) return cuda_fail(e);
  if (bx > 0 && (e = cudaMemcpyAsync(dx_h, d.dx, bx, cudaMemcpyDeviceToHost, d2h)) != cudaSuccess)
    return cuda_fail(e);
  if (bw > 0 && (e = cudaMemcpyAsync(dw_h, d.dw, bw, cudaMemcpyDeviceToHost, d2h)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaEventRecord(d.ev[kOutDone], d2h)) != cudaSuccess) return cuda_fail(e);
  if (wait && (e = cudaStreamWaitEvent(compute, d.ev[kOutDone], 0)) != cudaSuccess)
    return cuda_fail(e);
  return FP8LIN_OK;
}

uint64_t fp8lin_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void fp8lin_profile_enable(int on) {
  g_prof_on = on != 0;
  if (g_prof_on) g_prof_used = 0;
}

int64_t fp8lin_profile_launches(double* ms, int32_t* kind, int64_t capacity) {
  if (ms == nullptr || kind == nullptr || capacity < 0) return -static_cast<int64_t>(FP8LIN_EINVAL);
  const int64_t n = g_prof_used < capacity ? g_prof_used : capacity;
  for (int64_t i = 0; i < n; ++i) {
    cudaError_t e = cudaEventSynchronize(g_prof[i].stop);
    if (e != cudaSuccess) return -static_cast<int64_t>(cuda_fail(e));
    float t = 0.0f;
    e = cudaEventElapsedTime(&t, g_prof[i].start, g_prof[i].stop);
    if (e != cudaSuccess) return -static_cast<int64_t>(cuda_fail(e));
    ms[i] = t;
    kind[i] = g_prof[i].kind;
  }
  g_prof_used = 0;
  return n;
}

fp8lin_status fp8lin_profile_collect(double* ms, int64_t* count) {
  if (ms == nullptr || count == nullptr) return FP8LIN_EINVAL;
  for (int k = 0; k < FP8LIN_PROF_KINDS; ++k) {
    ms[k] = 0.0;
    count[k] = 0;
  }
  for (int i = 0; i < g_prof_used; ++i) {
    cudaError_t e = cudaEventSynchronize(g_prof[i].stop);
    if (e != cudaSuccess) return cuda_fail(e);
    float t = 0.0f;
    e = cudaEventElapsedTime(&t, g_prof[i].start, g_prof[i].stop);
    if (e != cudaSuccess) return cuda_fail(e);
    ms[g_prof[i].kind] += t;
    count[g_prof[i].kind] += 1;
  }
  g_prof_used = 0;
  return FP8LIN_OK;
}

}  // extern "C"
