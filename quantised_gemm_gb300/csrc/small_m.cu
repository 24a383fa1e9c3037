// small_m.cu -- host side of the few-token fused products: the fit test,
// tensor maps, one-time set-up per device, and the launch.  The kernel is in
// small_m_kernels.cuh.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "small_m_kernels.cuh"

namespace fp8lin {
namespace {

template <bool kCastA, int kFmtB, int kMN, bool kDW>
cudaError_t small_m_prepare(const DeviceInfo& dev, bool* resident) {
  static std::mutex mu;
  static int state[64] = {};  // 0: not yet; 1: ready, fits; 2: ready, does not fit
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (state[dev.device] == 0) {
    auto k = small_m_kernel<kCastA, kFmtB, kMN, kDW>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmSmem));
    if (e != cudaSuccess) return e;
    state[dev.device] = resident_ctas(k, kSmThreads, kSmSmem) >= 1 ? 1 : 2;
  }
  *resident = state[dev.device] == 1;
  return cudaSuccess;
}

int64_t small_m_tiles(int64_t NA, int64_t KA) {
  return ((NA + kTile - 1) / kTile) * ((KA + kTile - 1) / kTile);
}

template <bool kCastA, int kFmtB, int kMN, bool kDW>
cudaError_t run_small_m(const SmallMArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  bool resident = false;
  cudaError_t e = small_m_prepare<kCastA, kFmtB, kMN, kDW>(dev, &resident);
  if (e != cudaSuccess) return e;
  if (!resident) return cudaErrorCooperativeLaunchTooLarge;
  SmallParams p;
  p.NA = static_cast<int>(a.NA);
  p.KA = static_cast<int>(a.KA);
  p.MB = static_cast<int>(a.MB);
  p.b = a.b;
  p.ldb = a.ldb;
  p.eps = a.eps;
  p.b_amax_in = a.b_amax_in;
  p.b_amax = a.b_amax;
  p.b_scale = a.b_scale;
  p.b_inv = a.b_inv;
  p.b8 = a.b8;
  p.b8t = a.b8t;
  p.a_amax = a.a_amax;
  p.a_scale = a.a_scale;
  p.a_inv = a.a_inv;
  p.a_inv_in = a.a_inv_in;
  p.d = static_cast<uint16_t*>(a.d);
  p.ldd = a.ldd;
  p.d_amax = a.d_amax;
  p.d_amax_acc = a.ws_amax_acc;
  p.d_amax_ticket = a.ws_amax_ticket;
  p.partials = a.ws_partials;
  p.tickets = a.ws_tickets;
  p.ws_barrier = a.ws_barrier;
  p.ws_exits = a.ws_exits;
  p.ws_amax = a.ws_amax;
  p.ws_b_amax = a.ws_b_amax;
  p.err = a.ws_error;
  p.x8t = a.x8t;
  p.x_inv = a.x_inv;
  // A's maps: bf16 input (kCastA) and the fp8 matrix, 128 x 128 boxes; the
  // fp8 one is the W8 output of kCastA (TMA stores) or the fp8 input.
  CUtensorMap ma, ma8;
  const void* a8base = kCastA ? static_cast<const void*>(a.a8) : a.a;
  if (!make_map_2d(&ma8, CU_TENSOR_MAP_DATA_TYPE_UINT8, a8base, static_cast<uint64_t>(a.KA),
                   static_cast<uint64_t>(a.NA), static_cast<uint64_t>(a.KA), kTile, kTile,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return map_failed("few-token product fp8 weight map");
  if (kCastA) {
    if (!make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.a, static_cast<uint64_t>(a.KA),
                     static_cast<uint64_t>(a.NA), static_cast<uint64_t>(a.KA) * 2, kTile, kTile,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return map_failed("few-token product bf16 weight map");
  } else {
    ma = ma8;
  }
  // The third map: dW [KA, NA] bf16 (kDW; 32-row x 64-column boxes, 128-byte
  // rows, 128-byte swizzle) or W8^T [KA, NA] fp8 (kCastA; 128 x 128 boxes).
  CUtensorMap mc = ma8;
  if (kDW && !make_map_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.dw, static_cast<uint64_t>(a.NA),
                          static_cast<uint64_t>(a.KA), static_cast<uint64_t>(a.NA) * 2, 64, 32,
                          CU_TENSOR_MAP_SWIZZLE_128B))
    return map_failed("few-token product weight-gradient map");
  if (kCastA && !make_map_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a8t, static_cast<uint64_t>(a.NA),
                             static_cast<uint64_t>(a.KA), static_cast<uint64_t>(a.NA), kTile, kTile,
                             CU_TENSOR_MAP_SWIZZLE_128B))
    return map_failed("few-token product fp8 weight transpose map");
  const int64_t tiles = small_m_tiles(a.NA, a.KA);
  const int64_t grid = tiles < dev.num_sms ? tiles : dev.num_sms;
  set_error_site(kCastA ? "few-token fused product (weight cast) cooperative launch"
                 : kDW  ? "few-token fused product (with dW) cooperative launch"
                        : "few-token fused product cooperative launch");
  // Cooperative: the CTAs wait for one another (the amaxes), so all must be resident.
  return launch_kernel(small_m_kernel<kCastA, kFmtB, kMN, kDW>, dim3(static_cast<unsigned>(grid)),
                       dim3(kSmThreads), kSmSmem, stream, 1, true, ma, ma8, mc, p);
}

}  // namespace

bool small_m_fits(const DeviceInfo& dev, bool cast_a, int fmt_b, int64_t MB, int64_t NA,
                  int64_t KA, size_t partial_bytes, bool fuse_dw) {
  if (MB < 1 || MB > kSmallMaxRows || NA < 1 || KA < 1) return false;
  // dW's K is the tokens: 16 or 32 of them, the rows of x8^T exactly 16 or 32 bytes.
  if (fuse_dw && (cast_a || fmt_b != 1 || MB % 16 != 0 || NA % 16 != 0)) return false;
  if (NA > (int64_t(1) << 30) || KA > (int64_t(1) << 30)) return false;
  if (static_cast<size_t>(dev.max_smem_optin) < kSmSmem) return false;
  const int64_t tiles = small_m_tiles(NA, KA);
  const int kmn = MB <= 16 ? 16 : 32;
  if (tiles > static_cast<int64_t>(dev.num_sms) * kSmTilesPerCta) return false;
  if (static_cast<size_t>(tiles) * kmn * kTile * sizeof(float) > partial_bytes) return false;
  if ((NA + kTile - 1) / kTile > kWsTickets) return false;
  if (cast_a && fmt_b != 0) return false;  // the forward casts x and W, both e4m3
  // One CTA of 512 threads and ~225 KB of shared memory per SM must fit
  // (once per device and kernel; the cooperative launch needs every CTA resident).
  bool resident = false;
  cudaError_t e;
  if (cast_a)
    e = kmn == 16 ? small_m_prepare<true, 0, 16, false>(dev, &resident)
                  : small_m_prepare<true, 0, 32, false>(dev, &resident);
  else if (fmt_b == 0)
    e = kmn == 16 ? small_m_prepare<false, 0, 16, false>(dev, &resident)
                  : small_m_prepare<false, 0, 32, false>(dev, &resident);
  else if (fuse_dw)
    e = kmn == 16 ? small_m_prepare<false, 1, 16, true>(dev, &resident)
                  : small_m_prepare<false, 1, 32, true>(dev, &resident);
  else
    e = kmn == 16 ? small_m_prepare<false, 1, 16, false>(dev, &resident)
                  : small_m_prepare<false, 1, 32, false>(dev, &resident);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return resident;
}

cudaError_t launch_small_m(const SmallMArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (!small_m_fits(dev, a.cast_a, a.fmt_b, a.MB, a.NA, a.KA, a.ws_partial_bytes, a.fuse_dw))
    return cudaErrorInvalidValue;
  if (a.fuse_dw && (a.dw == nullptr || a.x8t == nullptr || a.x_inv == nullptr))
    return cudaErrorInvalidValue;
  const bool m16 = a.MB <= 16;
  if (a.cast_a) {  // the forward: the weight and x, both e4m3
    return m16 ? run_small_m<true, 0, 16, false>(a, dev, stream)
               : run_small_m<true, 0, 32, false>(a, dev, stream);
  }
  if (a.fmt_b == 0)
    return m16 ? run_small_m<false, 0, 16, false>(a, dev, stream)
               : run_small_m<false, 0, 32, false>(a, dev, stream);
  if (a.fuse_dw)  // the backward with dW
    return m16 ? run_small_m<false, 1, 16, true>(a, dev, stream)
               : run_small_m<false, 1, 32, true>(a, dev, stream);
  return m16 ? run_small_m<false, 1, 16, false>(a, dev, stream)
             : run_small_m<false, 1, 32, false>(a, dev, stream);
}

}  // namespace fp8lin
