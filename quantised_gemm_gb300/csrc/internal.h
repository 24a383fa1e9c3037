// internal.h -- launchers shared between the C ABI layer and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fp8lin {

// Workspace layout (bytes from the 256-byte aligned base).
constexpr size_t kWsErrorOffset = 0;      // int32: first device error code (0 = none)
constexpr size_t kWsBarrierOffset = 64;   // uint32: grid barrier arrivals (single pass)
constexpr size_t kWsExitsOffset = 68;     // uint32: CTAs past the barrier (single pass)
constexpr size_t kWsAmaxOffset = 128;     // uint32: amax bits (single pass)
constexpr size_t kWsAtomicAccOffset = 192;     // uint32: ticketed amax accumulator
constexpr size_t kWsAtomicTicketOffset = 196;  // uint32: ticketed amax arrivals
constexpr size_t kWsGemmAmaxAccOffset = 200;     // uint32: GEMM output amax accumulator
constexpr size_t kWsGemmAmaxTicketOffset = 204;  // uint32: GEMM epilogue warps arrived
constexpr size_t kWsSmallBAmaxOffset = 208;      // uint32: few-token product, token-side amax
constexpr size_t kWsAmax2Offset = 212;           // uint32: paired single pass, x's amax bits
constexpr size_t kWsScratchBegin = 64;    // [64, 256): self-cleaning counters
constexpr size_t kWsPartialOffset = 256;  // uint32[kMaxPartials]: REDUCTION partial maxima
constexpr int kMaxPartials = 4096;
constexpr size_t kWsFixedBytes = kWsPartialOffset + sizeof(uint32_t) * kMaxPartials;
constexpr size_t kWsTicketOffset = (kWsFixedBytes + 255) / 256 * 256;  // int32[kWsTickets]
constexpr int kWsTickets = 4096;
constexpr size_t kWsSplitOffset = kWsTicketOffset + sizeof(int) * kWsTickets;  // fp32 partials

// Device error codes written at kWsErrorOffset.
enum DeviceError : int {
  kErrNone = 0,
  kErrGemmProducerWait = 1,
  kErrGemmMmaWait = 2,
  kErrGemmEpilogueWait = 3,
  kErrGridBarrier = 4,
  kErrCastWait = 5,          // a streaming cast's load ring wait ran out
};

// Name the operation a launcher failed in (reported by
// fp8lin_last_error_detail together with the cudaError_t).
void set_error_site(const char* site);

// Whether launches use programmatic dependent launch (default on; the
// environment variable FP8LIN_PDL=0 turns it off).
bool pdl_enabled();

// Launch `kernel` on `stream` with cudaLaunchKernelEx: programmatic
// dependent launch when enabled, a cluster of `cluster_x` CTAs when > 1, and
// a cooperative launch when `cooperative`.  A cooperative grid launched
// early waits in griddepcontrol.wait, before its grid barrier, until the
// grid ahead of it has finished and freed its SMs; it lets the next grid
// launch only after its barrier, when all of its own CTAs are resident.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, int cluster_x, bool cooperative, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[3];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct DeviceInfo {
  int device;
  int num_sms;
  int max_smem_optin;
};
// Properties of the current device (cached per device).
cudaError_t current_device_info(DeviceInfo* info);

// ---- amax / scale / cast (cast_kernels.cu)

// Grid size the amax kernel uses for this tensor.
int amax_grid(const DeviceInfo& dev, int64_t rows, int64_t cols);

// Block maxima of |x| as fp32 bits.  atomic: one atomicMax per CTA, either
// into out[0] (which must hold 0 beforehand; ws_ticket == nullptr) or through
// the self-cleaning workspace words ws_acc / ws_ticket (the last CTA writes
// out[0]); otherwise out[blockIdx.x] = partial.
cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint32_t* out,
                        bool atomic, int grid, cudaStream_t stream, uint32_t* ws_acc = nullptr,
                        uint32_t* ws_ticket = nullptr);

// amax = max(partials[0..n)) written as fp32 bits into *amax_bits.
cudaError_t launch_amax_final(const uint32_t* partials, int n, uint32_t* amax_bits,
                              cudaStream_t stream);

// REDUCTION amax with its partial maxima in a static device array instead of
// a workspace (at most kStaticAmaxPartials CTAs); two launches.
constexpr int kStaticAmaxPartials = 4096;
cudaError_t launch_amax_static_scratch(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                       float* amax_out, int grid, cudaStream_t stream);

// One-thread scale update (dynamic or delayed ring).
// One state of a batched scale update (launch_scale's arguments).
struct ScaleArgs {
  const float* amax;
  float* scale;
  float* inv;
  float* ring;
  int32_t* head;
  int32_t history_len;
  bool delayed;
  int fmt;
  float eps;
};
// Up to 8 states in one launch, one thread each.
cudaError_t launch_scale_batch(const ScaleArgs* a, int n, cudaStream_t stream);
cudaError_t launch_scale(const float* amax, float* scale, float* inv, float* ring, int32_t* head,
                         int32_t history_len, bool delayed, int fmt, float eps,
                         cudaStream_t stream);

// Cast (+ transpose) of a bf16 tensor.
//   derive_scale == false: scale read from scale_in[0];
//   derive_scale == true:  scale = F / max(amax_in[0], eps), and CTA 0 writes
//                          scale_out[0] / inv_out[0].
//   amax_rec != nullptr: atomicMax of the tensor's amax bits (pre-zeroed).
struct CastArgs {
  const uint16_t* x;
  int64_t rows, cols, ld;
  int fmt;
  const float* scale_in;
  const float* amax_in;
  bool derive_scale;
  float eps;
  float* scale_out;
  float* inv_out;
  uint8_t* out;
  uint8_t* out_t;
  uint32_t* amax_rec;
  uint32_t* rec_acc = nullptr;     // non-null: record through the self-cleaning
  uint32_t* rec_ticket = nullptr;  // workspace words instead of a pre-zeroed amax_rec
  int* err = nullptr;              // workspace error word: use the TMA streaming kernel
};
cudaError_t launch_cast(const CastArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// Cooperative single pass: amax -> scale -> cast (+T) with the tensor held in
// shared memory.  Writes amax/scale/inv.  Requires tiles <= capacity.
struct SinglePassArgs {
  const uint16_t* x;
  int64_t rows, cols, ld;
  int fmt;
  float eps;
  float* amax_out;
  float* scale_out;
  float* inv_out;
  uint8_t* out;
  uint8_t* out_t;
  uint32_t* ws_barrier;   // self-cleaning workspace counters (zero between launches)
  uint32_t* ws_exits;
  uint32_t* ws_amax;
  int* ws_error;
};
int64_t single_pass_capacity_elems(const DeviceInfo& dev);
// W's single pass with x's cast in the same launch (the forward, both e4m3
// with transposed copies): W must take the cooperative single pass and x have
// at most one 128 x 128 tile for each of its CTAs.  x's amax goes through the
// workspace word of x_args.ws_amax.
bool single_pass_pair_fits(const DeviceInfo& dev, int64_t w_rows, int64_t w_cols,
                           int64_t x_rows, int64_t x_cols);
cudaError_t launch_cast_single_pass_pair(const SinglePassArgs& w, const SinglePassArgs& x,
                                         const DeviceInfo& dev, cudaStream_t stream);
bool single_pass_fits(const DeviceInfo& dev, int64_t rows, int64_t cols);
// Small tensors: the same single pass in one thread-block cluster (no grid
// barrier, no workspace).  Results are identical to the cooperative kernel's.
bool cluster_cast_fits(int64_t rows, int64_t cols);
cudaError_t launch_cast_cluster(const SinglePassArgs& a, cudaStream_t stream);
cudaError_t launch_cast_single_pass(const SinglePassArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream);

// 2-D tiled TMA map over a row-major [rows, inner] tensor (row stride in
// bytes), box [box_rows, box_inner], zero fill outside (gemm_tcgen05.cu).
bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle);

// Record a failed tensor-map encoding (with its CUresult) as the error site;
// returns cudaErrorInvalidValue.
cudaError_t map_failed(const char* what);

// ---- few-token products fused with their casts (small_m.cu)
//
// D [MB, NA] = B8 [MB, KA] . A8 [NA, KA]^T * inv_b * inv_a in one launch, for
// MB <= kSmallMaxRows tokens: B (bf16) is cast with a dynamic tensorwise
// scale in the same launch (its amax computed, or given by b_amax_in), and
// with cast_a the bf16 A (the weight) too (cooperative launch: its amax is a
// grid-wide reduction).  Writes B's fp8 copies and state, A's with cast_a,
// and D (+ its amax).
constexpr int kSmallMaxRows = 32;
struct SmallMArgs {
  bool cast_a;
  int fmt_b;
  int64_t MB, NA, KA;
  const void* a;            // cast_a: bf16 A [NA, KA]; else fp8 A8 [NA, KA] (dense)
  uint8_t* a8;              // cast_a: fp8 outputs A8 [NA, KA] and A8^T [KA, NA]
  uint8_t* a8t;
  float* a_amax;            // cast_a: A's state outputs
  float* a_scale;
  float* a_inv;
  const float* a_inv_in;    // !cast_a: A's inverse scale
  const uint16_t* b;        // bf16 B [MB, KA], row stride ldb
  int64_t ldb;
  float eps;
  const float* b_amax_in;   // nullptr: computed in the launch
  float* b_amax;
  float* b_scale;
  float* b_inv;
  uint8_t* b8;              // fp8 B [MB, KA] and B^T [KA, MB]
  uint8_t* b8t;
  void* d;                  // bf16 D [MB, NA], row stride ldd
  int64_t ldd;
  uint32_t* d_amax;
  uint32_t* ws_amax_acc;
  uint32_t* ws_amax_ticket;
  float* ws_partials;
  size_t ws_partial_bytes;
  int* ws_tickets;
  uint32_t* ws_barrier;
  uint32_t* ws_exits;
  uint32_t* ws_amax;
  uint32_t* ws_b_amax;
  int* ws_error;
  bool fuse_dw;             // the backward also computes dW [KA, NA] = dY8^T . x8
  const uint8_t* x8t;       // fuse_dw: fp8 x^T [NA, MB]
  const float* x_inv;       // fuse_dw: x's inverse scale
  void* dw;                 // fuse_dw: bf16 dW [KA, NA], dense
};
// Whether launch_small_m takes these sizes on this device with this much
// workspace for partials (fuse_dw: with the weight gradient in the launch).
bool small_m_fits(const DeviceInfo& dev, bool cast_a, int fmt_b, int64_t MB, int64_t NA,
                  int64_t KA, size_t partial_bytes, bool fuse_dw = false);
cudaError_t launch_small_m(const SmallMArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// ---- GEMM (gemm_tcgen05.cu)

struct GemmArgs {
  const uint8_t* a;   // [M, K] K fastest, row stride lda bytes
  const uint8_t* b;   // [N, K] K fastest, row stride ldb bytes
  int64_t M, N, K, lda, ldb;
  int fmt_a, fmt_b;
  const float* inv_a;
  const float* inv_b;
  void* d;            // bf16 [M, N], row stride ldd elements
  int64_t ldd;
  uint32_t* d_amax;   // fp32 bits of max |d| over the stored bf16 values (nullptr: not wanted)
  uint32_t* ws_amax_acc;     // self-cleaning words of the ticketed d_amax
  uint32_t* ws_amax_ticket;
  int* ws_error;
  int* ws_tickets;     // kWsTickets zero-initialised counters (nullptr: no K split)
  float* ws_split;     // fp32 partials of K-split tail tiles (nullptr: no K split)
  size_t ws_split_bytes;
};
cudaError_t launch_gemm(const GemmArgs& g, const DeviceInfo& dev, cudaStream_t stream);

// One line naming the kernel, tile shape and schedule launch_gemm uses for
// an M x N x K GEMM (given a workspace of fp8lin_workspace_bytes).
cudaError_t describe_gemm(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev, char* buf,
                          size_t len);
// The same line for a device of num_sms SMs holding pair_slots clusters of
// the pair kernel at once; pure host logic, no CUDA call.
void describe_plan(int64_t M, int64_t N, int64_t K, int num_sms, int pair_slots, char* buf,
                   size_t len);

// Two GEMMs of the pair kernel (256-wide tiles) in one launch, whole tiles
// dealt by cost.  plan_gemm_pair2 tells whether the plan expects that to beat
// two launches (always with FP8LIN_GROUP=2, never with FP8LIN_GROUP=0; both
// must qualify, and at most one may ask for its output amax);
// launch_gemm_pair2 runs them so, cudaErrorInvalidValue if the plan says no.
cudaError_t plan_gemm_pair2(const GemmArgs& a, const GemmArgs& b, const DeviceInfo& dev,
                            bool* use);
cudaError_t launch_gemm_pair2(const GemmArgs& a, const GemmArgs& b, const DeviceInfo& dev,
                              cudaStream_t stream);
// The grouped plan for two GEMMs (M x N x K each) on a device of num_sms SMs
// holding pair_slots clusters: grouped or separate, the deal's d, the
// estimated K blocks of the busiest pair both ways, and a check that the deal
// hands out every tile once.  Pure host logic.
void describe_group_plan(int64_t Ma, int64_t Na, int64_t Ka, int64_t Mb, int64_t Nb, int64_t Kb,
                         int num_sms, int pair_slots, char* buf, size_t len);

// Workspace bytes the tail K split can use at most on a device with num_sms SMs.
size_t gemm_split_workspace_bytes(int num_sms);

}  // namespace fp8lin
