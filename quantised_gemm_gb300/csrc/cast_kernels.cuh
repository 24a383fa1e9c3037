// cast_kernels.cuh -- device code of the HBM-bound kernels of the fp8 Linear:
// amax (one-pass
// atomic and two-kernel reduction), scale (dynamic and delayed ring), cast
// to e4m3/e5m2 with an optional transposed copy, and a cooperative single
// pass amax -> scale -> cast that keeps the tensor in shared memory.
//
// Numerics (the plain reading of tensorwise scaling in "Integrate
// float8nocompile, an experimental feature for high performance",
// pytorch/torchtitan PR 778, Summary):
//   amax  = max |x|, computed on the bf16 bit patterns (|x| is bits & 0x7FFF,
//           whose unsigned order is the order of magnitudes), so it is exact;
//   scale = __fdiv_rn(F, max(amax, eps)), inv = __fdiv_rn(1, scale);
//   q     = cvt.rn.satfinite(x * scale) -- one RN fp32 product, then one
//           saturating RNE rounding to the 8-bit format.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace fp8lin {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;          // cast tile: 128 rows x 128 columns
constexpr int kSqWords = 33;        // shared fp8 tile row pitch: 132 bytes
constexpr int kAmaxRows = 64;       // amax tile: 64 rows x 256 columns
constexpr int kSinglePassTilesPerCta = 7;

template <int kFmt>
__device__ __forceinline__ float fp8_max() {
  return kFmt == 0 ? 448.0f : 57344.0f;
}

__device__ __forceinline__ float scale_from_amax(float amax, float eps, float F) {
  const float d = amax > eps ? amax : eps;
  return __fdiv_rn(F, d);
}

// Max of the 16-bit magnitudes held in a 16-byte vector of 8 bf16 values.
__device__ __forceinline__ uint32_t vec_absmax(uint32_t acc, const uint4& v) {
  acc = __vmaxu2(acc, v.x & 0x7FFF7FFFu);
  acc = __vmaxu2(acc, v.y & 0x7FFF7FFFu);
  acc = __vmaxu2(acc, v.z & 0x7FFF7FFFu);
  acc = __vmaxu2(acc, v.w & 0x7FFF7FFFu);
  return acc;
}

// The same maximum with the low and the high bf16 of each 32-bit word kept
// apart (bits & 0x7FFF, bits & 0x7FFF0000): each step is an AND and a native
// 32-bit max.  It issues twice as many instructions as vec_absmax, which
// costs the streaming kernels, but its steps are short: the kernels whose
// amax is a latency chain (data already on chip) run faster with it.
struct AbsMax {
  uint32_t lo = 0, hi = 0;
  __device__ __forceinline__ void add(const uint4& v) {
    lo = max(lo, max(max(v.x & 0x7FFFu, v.y & 0x7FFFu), max(v.z & 0x7FFFu, v.w & 0x7FFFu)));
    hi = max(hi, max(max(v.x & 0x7FFF0000u, v.y & 0x7FFF0000u),
                     max(v.z & 0x7FFF0000u, v.w & 0x7FFF0000u)));
  }
  __device__ __forceinline__ void merge(const AbsMax& o) {
    lo = max(lo, o.lo);
    hi = max(hi, o.hi);
  }
  // As vec_absmax's packed pair: the maximum in the low 16 bits.
  __device__ __forceinline__ uint32_t packed() const { return max(lo, hi >> 16); }
};

// Block-wide max of per-thread 2x16-bit magnitudes; result (as fp32 bits)
// valid in thread 0.
__device__ __forceinline__ uint32_t block_absmax_bits(uint32_t acc) {
  __shared__ uint32_t red[kThreads / 32];
  uint32_t m = max(acc & 0xFFFFu, acc >> 16);
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kThreads / 32 ? red[lane] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
  }
  return m << 16;
}

// 8 bf16 -> 8 fp8 codes (two words, element order preserved).
template <int kFmt>
__device__ __forceinline__ uint2 cast8(const uint4& v, float s) {
  uint2 q;
  q.x = static_cast<uint32_t>(cvt_fp8x2<kFmt>(__fmul_rn(bf16lo_to_f32(v.x), s),
                                              __fmul_rn(bf16hi_to_f32(v.x), s))) |
        (static_cast<uint32_t>(cvt_fp8x2<kFmt>(__fmul_rn(bf16lo_to_f32(v.y), s),
                                               __fmul_rn(bf16hi_to_f32(v.y), s)))
         << 16);
  q.y = static_cast<uint32_t>(cvt_fp8x2<kFmt>(__fmul_rn(bf16lo_to_f32(v.z), s),
                                              __fmul_rn(bf16hi_to_f32(v.z), s))) |
        (static_cast<uint32_t>(cvt_fp8x2<kFmt>(__fmul_rn(bf16lo_to_f32(v.w), s),
                                               __fmul_rn(bf16hi_to_f32(v.w), s)))
         << 16);
  return q;
}

// Transposed write of one 128x128 fp8 tile held in shared memory (rows of
// kSqWords words).  Each thread moves a 16-row x 4-column block: 16 word
// reads, a 4x4 byte transpose per 4 rows (prmt), four 16-byte stores.  Lane
// pairs cover 32 contiguous output bytes; the pitch of 33 words makes the
// reads of a warp hit 32 distinct banks.
__device__ __forceinline__ void store_transposed_tile(const uint32_t* sq, uint8_t* out_t,
                                                      int64_t rows, int64_t cols, int64_t r0,
                                                      int64_t c0, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int jg = (warp & 1) * 16 + (lane >> 1);  // 4-column group 0..31
  const int ig = (warp >> 1) * 2 + (lane & 1);   // 16-row group 0..7
  const int i0 = ig * 16, j0 = jg * 4;
  if (c0 + j0 >= cols || r0 + i0 >= rows) return;
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k] = sq[(i0 + k) * kSqWords + jg];
  uint32_t o[4][4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t t0 = __byte_perm(w[4 * g + 0], w[4 * g + 1], 0x5140);
    const uint32_t t1 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x5140);
    const uint32_t t2 = __byte_perm(w[4 * g + 0], w[4 * g + 1], 0x7362);
    const uint32_t t3 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x7362);
    o[0][g] = __byte_perm(t0, t1, 0x5410);
    o[1][g] = __byte_perm(t0, t1, 0x7632);
    o[2][g] = __byte_perm(t2, t3, 0x5410);
    o[3][g] = __byte_perm(t2, t3, 0x7632);
  }
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    uint8_t* dst = out_t + (c0 + j0 + jj) * rows + r0 + i0;
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[jj][0], o[jj][1], o[jj][2], o[jj][3]);
  }
}

// ------------------------------------------------------------------ amax

// Ticketed atomic maximum: fold `bits` into *acc, and let the last of `n`
// arrivals publish the result to *out and clear *acc and *ticket, so the
// scratch words are zero again for the next launch (no memset needed).
__device__ __forceinline__ void ticketed_max(uint32_t bits, uint32_t* acc, uint32_t* ticket,
                                             uint32_t* out, unsigned n) {
  atomicMax(acc, bits);
  __threadfence();
  if (atomicAdd(ticket, 1u) == n - 1) {
    __threadfence();
    *out = atomicExch(acc, 0u);
    atomicExch(ticket, 0u);
  }
}

// kMode: 0 = write this CTA's partial maximum to out[blockIdx.x];
//        1 = atomicMax into out[0] (zero beforehand);
//        2 = ticketed maximum through the workspace words acc / ticket.
template <int kMode>
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t* __restrict__ x,
                                                        int64_t rows, int64_t cols, int64_t ld,
                                                        uint32_t* __restrict__ out,
                                                        uint32_t* acc_word, uint32_t* ticket) {
  griddep_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t cvec = cols >> 3;                 // 8-element vectors per row
  const int64_t ntc = (cvec + 31) >> 5;           // 32 vectors per tile row
  const int64_t ntr = (rows + kAmaxRows - 1) / kAmaxRows;
  const int64_t ntiles = ntr * ntc;
  uint32_t acc = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t tr = t / ntc, tc = t - tr * ntc;
    const int64_t c = (tc << 5) + lane;
    if (c < cvec) {
      uint4 v[8];  // eight 16-byte loads in flight per thread
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t r = tr * kAmaxRows + warp + u * 8;
        v[u] = r < rows ? ld_stream_v4(x + r * ld + c * 8) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) acc = vec_absmax(acc, v[u]);
    }
  }
  griddep_launch_dependents();
  const uint32_t bits = block_absmax_bits(acc);
  if (threadIdx.x == 0) {
    if (kMode == 0)
      out[blockIdx.x] = bits;
    else if (kMode == 1)
      atomicMax(out, bits);
    else
      ticketed_max(bits, acc_word, ticket, out, gridDim.x);
  }
}

__global__ void __launch_bounds__(kThreads) amax_final_kernel(const uint32_t* __restrict__ part,
                                                              int n, uint32_t* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  uint32_t m = 0;
  for (int i = threadIdx.x; i < n; i += kThreads) m = max(m, part[i]);
  // part[] already holds fp32 bits of non-negative values: order-preserving.
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t red[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int w = 0; w < kThreads / 32; ++w) r = max(r, red[w]);
    *out = r;
  }
}

// ------------------------------------------------------------------ scale

// One state's scale update: delayed, the ring takes the amax at its head and
// the scale comes from the ring's maximum; dynamic, from the amax itself.
__device__ __forceinline__ void scale_update(const float* amax, float* scale, float* inv,
                                             float* ring, int32_t* head, int32_t H, int delayed,
                                             float F, float eps) {
  float a = *amax;
  if (delayed) {
    int32_t h = *head;
    h = ((h % H) + H) % H;  // a corrupted head still indexes inside the ring
    ring[h] = a;
    *head = (h + 1 == H) ? 0 : h + 1;
    float m = 0.0f;
    for (int32_t i = 0; i < H; ++i) m = ring[i] > m ? ring[i] : m;
    a = m;
  }
  const float s = scale_from_amax(a, eps, F);
  *scale = s;
  *inv = __fdiv_rn(1.0f, s);
}

__global__ void scale_kernel(const float* __restrict__ amax, float* __restrict__ scale,
                             float* __restrict__ inv, float* __restrict__ ring,
                             int32_t* __restrict__ head, int32_t H, int delayed, float F,
                             float eps) {
  griddep_wait();
  griddep_launch_dependents();
  scale_update(amax, scale, inv, ring, head, H, delayed, F, eps);
}

// Up to kScaleBatch states updated by one launch, one thread each.
constexpr int kScaleBatch = 8;
struct ScaleBatch {
  const float* amax[kScaleBatch];
  float* scale[kScaleBatch];
  float* inv[kScaleBatch];
  float* ring[kScaleBatch];
  int32_t* head[kScaleBatch];
  int32_t H[kScaleBatch];
  int32_t delayed[kScaleBatch];
  float F[kScaleBatch];
  float eps[kScaleBatch];
  int32_t n;
};

__global__ void scale_batch_kernel(const __grid_constant__ ScaleBatch b) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = static_cast<int>(threadIdx.x);
  if (i < b.n)
    scale_update(b.amax[i], b.scale[i], b.inv[i], b.ring[i], b.head[i], b.H[i], b.delayed[i],
                 b.F[i], b.eps[i]);
}

// ------------------------------------------------------------------ cast

struct CastParams {
  const uint16_t* x;
  int64_t rows, cols, ld;
  const float* scale_in;
  const float* amax_in;
  int derive_scale;
  float eps;
  float* scale_out;
  float* inv_out;
  uint8_t* out;
  uint8_t* out_t;
  uint32_t* amax_rec;
  uint32_t* rec_acc;     // non-null: ticketed recording through the workspace
  uint32_t* rec_ticket;
  int* err;              // workspace error word (streaming kernel; may be null)
};

template <int kFmt, bool kTrans>
__global__ void __launch_bounds__(kThreads, 4) cast_kernel(const CastParams p) {
  __shared__ __align__(16) uint32_t sq[kTrans ? kTile * kSqWords : 1];
  griddep_wait();
  float s;
  if (p.derive_scale) {
    s = scale_from_amax(*p.amax_in, p.eps, fp8_max<kFmt>());
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      *p.scale_out = s;
      *p.inv_out = __fdiv_rn(1.0f, s);
    }
  } else {
    s = *p.scale_in;
  }
  const int64_t ntc = (p.cols + kTile - 1) / kTile;
  const int64_t ntiles = ((p.rows + kTile - 1) / kTile) * ntc;
  uint32_t acc = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t r0 = (t / ntc) * kTile, c0 = (t % ntc) * kTile;
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int vi = threadIdx.x + kThreads * u;
      const int64_t row = r0 + (vi >> 4), col = c0 + (vi & 15) * 8;
      v[u] = (row < p.rows && col < p.cols) ? ld_stream_v4(p.x + row * p.ld + col)
                                             : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int vi = threadIdx.x + kThreads * u;
      const int rl = vi >> 4, cv = vi & 15;
      const int64_t row = r0 + rl, col = c0 + cv * 8;
      acc = vec_absmax(acc, v[u]);
      const uint2 q = cast8<kFmt>(v[u], s);
      if (p.out != nullptr && row < p.rows && col < p.cols)
        *reinterpret_cast<uint2*>(p.out + row * p.cols + col) = q;
      if (kTrans) {
        sq[rl * kSqWords + cv * 2] = q.x;
        sq[rl * kSqWords + cv * 2 + 1] = q.y;
      }
    }
    if (kTrans) {
      __syncthreads();
      store_transposed_tile(sq, p.out_t, p.rows, p.cols, r0, c0, threadIdx.x);
      __syncthreads();
    }
  }
  griddep_launch_dependents();
  if (p.amax_rec != nullptr) {
    const uint32_t bits = block_absmax_bits(acc);
    if (threadIdx.x == 0) {
      if (p.rec_ticket != nullptr)
        ticketed_max(bits, p.rec_acc, p.rec_ticket, p.amax_rec, gridDim.x);
      else
        atomicMax(p.amax_rec, bits);
    }
  }
}

// ------------------------------------------------------------------ streaming cast (TMA)
//
// The same cast (+ transpose, optional amax record) as cast_kernel, with the
// data moved by TMA: one persistent CTA per SM, a producer lane that loads
// 128 x 128 bf16 tiles into a kStreamStages-deep ring, and eight consumer
// warps that cast a tile from shared memory, stage the fp8 tile and its
// transpose in the 128-byte TMA swizzle (double-buffered across tiles) and
// write both with TMA bulk stores.  No thread issues a global load or store
// of its own.
constexpr int kStreamStages = 3;
constexpr int kStreamBlockRows = 8;  // tile rows per block of the walk order

// Tile t of the streaming walk as (tile row, tile column): blocks of
// kStreamBlockRows tile rows, column by column inside a block, so that the
// tiles in flight at once cover a few rows and columns and both outputs, q
// and its transpose, are written in runs of several tiles.
__device__ __forceinline__ void stream_tile(int64_t t, int64_t ntr, int64_t ntc, int64_t& tr,
                                            int64_t& tc) {
  const int64_t per_block = static_cast<int64_t>(kStreamBlockRows) * ntc;
  const int64_t b = t / per_block, i = t - b * per_block;
  const int64_t rows = min(static_cast<int64_t>(kStreamBlockRows), ntr - b * kStreamBlockRows);
  tr = b * kStreamBlockRows + i % rows;
  tc = i / rows;
}
constexpr int kStreamConsumers = 256;
constexpr int kStreamThreads = 32 + kStreamConsumers;
constexpr int kTileBytesBf16 = kTile * kTile * 2;
constexpr size_t kStreamSmem = 1024 + static_cast<size_t>(kStreamStages) * kTileBytesBf16 +
                               2 * static_cast<size_t>(kTileBytesBf16) + 256;

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kStreamConsumers) : "memory");
}

// Barrier of the consumer warps that also returns, to every one of them, the
// OR of `bad` over all of them: one decision for the whole group.
__device__ __forceinline__ bool consumer_sync_or(bool bad) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(bad ? 1u : 0u), "r"(kStreamConsumers)
      : "memory");
  return r != 0;
}

// Offset of byte `col` (0..127) of row `row` in a 128 x 128-byte fp8 tile
// laid out as the 128-byte TMA swizzle expects: 16-byte chunk c of row r is
// stored at chunk c ^ (r & 7).
__device__ __forceinline__ int sw128(int row, int col) {
  return row * 128 + ((((col >> 4) ^ (row & 7))) << 4) + (col & 15);
}

// Cast 8 vectors per thread (this thread's share of a 128 x 128 bf16 tile in
// shared memory, 256 threads) into the swizzled fp8 tile `sqt` and, with
// kTrans, its transpose `stt`.  `sync` separates the writes of `sqt` from
// the reads of it for the transpose.
template <int kTrans, typename Sync>
__device__ __forceinline__ void stage_tile_fp8(const uint2 (&q)[8], uint8_t* sqt, uint8_t* stt,
                                               int tid, Sync sync) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int vi = tid + 256 * u;
    *reinterpret_cast<uint2*>(sqt + sw128(vi >> 4, (vi & 15) * 8)) = q[u];
  }
  if (kTrans) {
    sync();
    // Each thread moves a 16-row x 4-column block: 16 words down a column
    // group of the tile, 4x4 byte transposes, four 16-byte rows of the
    // transpose.
    const int lane = tid & 31, warp = tid >> 5;
    const int jg = (warp & 1) * 16 + (lane >> 1);  // 4-column group 0..31
    const int ig = (warp >> 1) * 2 + (lane & 1);   // 16-row group 0..7
    uint32_t w[16];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk)
      w[kk] = *reinterpret_cast<const uint32_t*>(sqt + sw128(ig * 16 + kk, jg * 4));
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t t0 = __byte_perm(w[4 * g + 0], w[4 * g + 1], 0x5140);
      const uint32_t t1 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x5140);
      const uint32_t t2 = __byte_perm(w[4 * g + 0], w[4 * g + 1], 0x7362);
      const uint32_t t3 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x7362);
      w[4 * g + 0] = __byte_perm(t0, t1, 0x5410);
      w[4 * g + 1] = __byte_perm(t0, t1, 0x7632);
      w[4 * g + 2] = __byte_perm(t2, t3, 0x5410);
      w[4 * g + 3] = __byte_perm(t2, t3, 0x7632);
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      *reinterpret_cast<uint4*>(stt + sw128(jg * 4 + jj, ig * 16)) =
          make_uint4(w[jj], w[4 + jj], w[8 + jj], w[12 + jj]);
  }
}

template <int kFmt, bool kTrans>
__global__ void __launch_bounds__(kStreamThreads, 1)
    cast_stream_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmQT, const CastParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* in = base;                                      // kStreamStages bf16 tiles
  uint8_t* outb = base + kStreamStages * kTileBytesBf16;   // 2 x (fp8 tile | transpose)
  uint64_t* full = reinterpret_cast<uint64_t*>(outb + 2 * kTileBytesBf16);
  uint64_t* empty = full + kStreamStages;
  __shared__ int s_abort;
  __shared__ uint32_t s_red[kStreamConsumers / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ntc = (p.cols + kTile - 1) / kTile;
  const int64_t ntr = (p.rows + kTile - 1) / kTile;
  const int64_t ntiles = ntr * ntc;
  const int64_t mine = blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStreamStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    s_abort = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmX);
    if (p.out != nullptr) tma_prefetch_map(&tmQ);
    if (kTrans) tma_prefetch_map(&tmQT);
  }
  __syncthreads();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t fills[kStreamStages] = {};
      bool ok = true;
      for (int64_t i = 0; i < mine; ++i) {
        const int st = static_cast<int>(i % kStreamStages);
        const uint32_t ph = static_cast<uint32_t>((i / kStreamStages) & 1);
        if (!mbar_wait_bounded(&empty[st], ph ^ 1u, &s_abort)) {
          ok = false;
          break;
        }
        int64_t tr, tc;
        stream_tile(blockIdx.x + i * gridDim.x, ntr, ntc, tr, tc);
        mbar_arrive_expect_tx(&full[st], kTileBytesBf16);
        tma_load_2d(in + st * kTileBytesBf16, &tmX, &full[st], static_cast<int32_t>(tc * kTile),
                    static_cast<int32_t>(tr * kTile));
        ++fills[st];
      }
      if (!ok) {
        if (p.err != nullptr) atomicCAS(p.err, 0, kErrCastWait);
        s_abort = 1;
      }
      // Stay until every copy this lane issued has landed, whatever the
      // consumers do: the CTA (and its shared memory) lives as long as this
      // lane does, so no copy can land in a CTA that has left.  Only the last
      // phase of each stage can still be open; without a failure the
      // consumers have waited for all of them already, or are about to.
      volatile int never = 0;
      for (int st = 0; st < kStreamStages; ++st)
        if (fills[st] > 0) mbar_wait_bounded(&full[st], (fills[st] - 1) & 1u, &never);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = threadIdx.x - 32;
  const bool issuer = ctid == 0;
  float s;
  if (p.derive_scale) {
    s = scale_from_amax(*p.amax_in, p.eps, fp8_max<kFmt>());
    if (blockIdx.x == 0 && issuer) {
      *p.scale_out = s;
      *p.inv_out = __fdiv_rn(1.0f, s);
    }
  } else {
    s = *p.scale_in;
  }
  uint32_t acc = 0;
  for (int64_t i = 0; i < mine; ++i) {
    const int st = static_cast<int>(i % kStreamStages);
    const uint32_t ph = static_cast<uint32_t>((i / kStreamStages) & 1);
    const int o = static_cast<int>(i & 1);
    int64_t tr, tc;
    stream_tile(blockIdx.x + i * gridDim.x, ntr, ntc, tr, tc);
    const int64_t r0 = tr * kTile, c0 = tc * kTile;
    const bool ready = mbar_wait_bounded(&full[st], ph, &s_abort);
    // One decision for all consumers, whatever each one's wait returned.
    if (consumer_sync_or(!ready)) {
      if (issuer && p.err != nullptr) atomicCAS(p.err, 0, kErrCastWait);
      s_abort = 1;  // the producer stops refilling and drains its copies
      break;
    }
    if (issuer && i >= 2) bulk_wait_group_read<1>();  // output buffer o has been read
    uint2 q[8];
    const uint8_t* buf = in + st * kTileBytesBf16;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int vi = ctid + 256 * u;
      const uint4 v = *reinterpret_cast<const uint4*>(buf + (vi >> 4) * (kTile * 2) +
                                                      (vi & 15) * 16);
      if (p.amax_rec != nullptr) acc = vec_absmax(acc, v);
      q[u] = cast8<kFmt>(v, s);
    }
    consumer_sync();  // the stage is read; output buffer o is free
    if (issuer) mbar_arrive(&empty[st]);
    uint8_t* sqt = outb + o * kTileBytesBf16;
    stage_tile_fp8<kTrans>(q, sqt, sqt + kTile * kTile, ctid, consumer_sync);
    fence_proxy_async_shared();
    consumer_sync();
    if (issuer) {
      if (p.out != nullptr)
        tma_store_2d(&tmQ, sqt, static_cast<int32_t>(c0), static_cast<int32_t>(r0));
      if (kTrans)
        tma_store_2d(&tmQT, sqt + kTile * kTile, static_cast<int32_t>(r0),
                     static_cast<int32_t>(c0));
      bulk_commit_group();
    }
  }
  griddep_launch_dependents();
  if (issuer) bulk_wait_group<0>();  // stores done before the shared memory goes away
  if (p.amax_rec != nullptr) {
    uint32_t m = max(acc & 0xFFFFu, acc >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) s_red[ctid >> 5] = m;
    consumer_sync();
    if (issuer) {
      for (int w = 1; w < kStreamConsumers / 32; ++w) m = max(m, s_red[w]);
      if (p.rec_ticket != nullptr)
        ticketed_max(m << 16, p.rec_acc, p.rec_ticket, p.amax_rec, gridDim.x);
      else
        atomicMax(p.amax_rec, m << 16);
    }
  }
}

// ------------------------------------------------------------------ single pass

struct SinglePassParams {
  int64_t rows, cols;
  float eps;
  float* amax_out;
  float* scale_out;
  float* inv_out;
  uint8_t* out;
  uint8_t* out_t;
  uint32_t* ws_barrier;   // arrivals  } zero between launches: the last CTA
  uint32_t* ws_exits;     // leavers   } past the barrier clears all three
  uint32_t* ws_amax;      // amax bits }
  int* ws_error;
  // The paired launch only: a second tensor of at most one 128 x 128 tile a
  // CTA (x of the forward, cast with W), loaded into registers by group 0 of
  // CTA b < its tile count, its amax taken at the same grid barrier (its own
  // word ws_amax2, cleared with the others), cast after the CTA's own tiles.
  const uint16_t* x2;
  int64_t rows2, cols2, ld2;
  float eps2;
  float* amax2_out;
  float* scale2_out;
  float* inv2_out;
  uint8_t* out2;
  uint8_t* out2_t;
  uint32_t* ws_amax2;
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Phase 1: one TMA load per 128 x 128 bf16 tile brings this CTA's tiles
// (tile t = blockIdx.x + k * gridDim.x) into shared memory; the CTA folds
// their amax into ws_amax and arrives on a grid barrier.  Phase 2 derives the
// scale from the global amax and casts the tiles from shared memory, the two
// 256-thread groups of the CTA working on alternate tiles (each group
// synchronises on its own named barrier).  Launched cooperatively, so all
// CTAs are co-resident and the grid barrier completes; its time limit only
// guards against a launch that broke that promise.  The counters clean
// themselves: the last CTA past the barrier resets them, so consecutive
// launches need no memset.
constexpr int kSpGroups = 2;
constexpr int kSpThreads = kSpGroups * kThreads;

__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(kThreads) : "memory");
}

template <int kFmt, bool kTrans, bool kPair>
__device__ __forceinline__ void single_pass_body(const CUtensorMap* tmX, const CUtensorMap* tmQ,
                                                 const CUtensorMap* tmQT,
                                                 const SinglePassParams& p,
                                                 const CUtensorMap* tmQ2,
                                                 const CUtensorMap* tmQT2) {
  extern __shared__ __align__(1024) uint8_t tiles_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tiles_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t loaded[kSinglePassTilesPerCta];  // one per tile
  __shared__ uint32_t s_amax_bits, s_amax2_bits;
  __shared__ uint32_t s_red[kSpThreads / 32];
  __shared__ int s_abort;
  const int group = threadIdx.x / kThreads, tid = threadIdx.x % kThreads;
  const int64_t ntc = (p.cols + kTile - 1) / kTile;
  const int64_t ntiles = ((p.rows + kTile - 1) / kTile) * ntc;
  int mine = 0;
  while (mine < kSinglePassTilesPerCta &&
         blockIdx.x + static_cast<int64_t>(mine) * gridDim.x < ntiles)
    ++mine;

  griddep_wait();
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int k = 0; k < mine; ++k) mbar_init(&loaded[k], 1);
    fence_barrier_init();
    for (int k = 0; k < mine; ++k) {
      const int64_t t = blockIdx.x + static_cast<int64_t>(k) * gridDim.x;
      mbar_arrive_expect_tx(&loaded[k], kTile * kTile * 2);
      tma_load_2d(tiles + k * (kTile * kTile * 2), tmX, &loaded[k],
                  static_cast<int32_t>((t % ntc) * kTile), static_cast<int32_t>((t / ntc) * kTile));
    }
  }
  __syncthreads();
  // kPair: group 0 of CTA b < ntiles2 loads tile b of the second tensor into
  // registers (8 vectors a thread, as the casts below read a tile), in flight
  // with the TMA loads.
  uint4 v2[kPair ? 8 : 1];
  AbsMax x0;
  int64_t ntc2 = 1, ntiles2 = 0;
  if constexpr (kPair) {
    ntc2 = (p.cols2 + kTile - 1) / kTile;
    ntiles2 = ((p.rows2 + kTile - 1) / kTile) * ntc2;
    if (static_cast<int64_t>(blockIdx.x) < ntiles2 && group == 0) {
      const int64_t r0 = (blockIdx.x / ntc2) * kTile, c0 = (blockIdx.x % ntc2) * kTile;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int vi = tid + kThreads * u;
        const int64_t row = r0 + (vi >> 4), col = c0 + (vi & 15) * 8;
        v2[u] = row < p.rows2 && col < p.cols2 ? ld_stream_v4(p.x2 + row * p.ld2 + col)
                                               : make_uint4(0u, 0u, 0u, 0u);
        x0.add(v2[u]);
      }
    }
  }
  const bool has2 = kPair && static_cast<int64_t>(blockIdx.x) < ntiles2;  // CTA-uniform
  // The amax of each tile as soon as it lands.  Two independent accumulators
  // of the short-step kind: the tile is on chip, so this loop is a latency
  // chain, not a bandwidth stream.
  AbsMax a0, a1;
  bool landed = true;
  for (int k = group; k < mine; k += kSpGroups) {
    volatile int never = 0;
    if (!mbar_wait_bounded(&loaded[k], 0, &never)) {
      landed = false;
      break;
    }
    const uint8_t* buf = tiles + k * (kTile * kTile * 2);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int vi = tid + kThreads * u;
      (u & 1 ? a1 : a0).add(*reinterpret_cast<const uint4*>(buf + (vi >> 4) * (kTile * 2) +
                                                             (vi & 15) * 16));
    }
  }
  {
    a0.merge(a1);
    const uint32_t acc = a0.packed();
    uint32_t m = max(acc & 0xFFFFu, acc >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
  }
  __shared__ uint32_t s_red2[kThreads / 32];
  if constexpr (kPair) {  // group 0's maximum of the second tensor's tile
    const uint32_t acc = x0.packed();
    uint32_t m = max(acc & 0xFFFFu, acc >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (group == 0 && (tid & 31) == 0) s_red2[tid >> 5] = m;
  }
  if (__syncthreads_and(landed ? 1 : 0) == 0) {  // one decision for the CTA
    if (threadIdx.x == 0) {
      atomicCAS(p.ws_error, 0, kErrGridBarrier);
      volatile int never = 0;  // copies in flight land before the shared memory goes away
      for (int k = 0; k < mine; ++k) mbar_wait_bounded(&loaded[k], 0, &never);
    }
    return;
  }
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int w = 0; w < kSpThreads / 32; ++w) m = max(m, s_red[w]);
    atomicMax(p.ws_amax, m << 16);
    if (has2) {
      uint32_t m2 = 0;
      for (int w = 0; w < kThreads / 32; ++w) m2 = max(m2, s_red2[w]);
      atomicMax(p.ws_amax2, m2 << 16);
    }
    red_release_add(p.ws_barrier, 1u);  // the maxima above are visible to whoever sees this
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_u32(p.ws_barrier) < gridDim.x) {
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicCAS(p.ws_error, 0, kErrGridBarrier);
        s_abort = 1;
        break;
      }
    }
    // Ordered after every arrival by the acquiring poll above.
    if (!s_abort) {
      s_amax_bits = *reinterpret_cast<volatile uint32_t*>(p.ws_amax);
      if (kPair) s_amax2_bits = *reinterpret_cast<volatile uint32_t*>(p.ws_amax2);
    }
  }
  __syncthreads();
  if (s_abort) return;
  griddep_launch_dependents();

  const float amax = __uint_as_float(s_amax_bits);
  const float s = scale_from_amax(amax, p.eps, fp8_max<kFmt>());
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *p.amax_out = amax;
    *p.scale_out = s;
    *p.inv_out = __fdiv_rn(1.0f, s);
  }
  float s2 = 1.0f;
  if constexpr (kPair) {
    const float amax2 = __uint_as_float(s_amax2_bits);
    s2 = scale_from_amax(amax2, p.eps2, fp8_max<kFmt>());
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      *p.amax2_out = amax2;
      *p.scale2_out = s2;
      *p.inv2_out = __fdiv_rn(1.0f, s2);
    }
  }
  // Phase 2, per tile: cast from shared memory into registers, then stage the
  // fp8 tile (first 16 KB of the tile's own 32 KB buffer, free once read)
  // and its transpose (second 16 KB) in the 128-byte TMA swizzle, and write
  // both with TMA bulk stores, which clip ragged edges.  One thread of each
  // group issues its group's stores and waits for them before the CTA ends.
  const bool issuer = tid == 0;
  for (int k = group; k < mine; k += kSpGroups) {
    const int64_t t = blockIdx.x + static_cast<int64_t>(k) * gridDim.x;
    uint8_t* buf = tiles + k * (kTile * kTile * 2);
    const int64_t r0 = (t / ntc) * kTile, c0 = (t % ntc) * kTile;
    uint2 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int vi = tid + kThreads * u;
      const uint4 v = *reinterpret_cast<const uint4*>(buf + (vi >> 4) * (kTile * 2) +
                                                      (vi & 15) * 16);
      q[u] = cast8<kFmt>(v, s);
    }
    group_sync(group);  // the group has read the whole bf16 tile
    uint8_t* sqt = buf;                       // fp8 tile [128 rows][128 bytes]
    uint8_t* stt = buf + kTile * kTile;       // its transpose
    stage_tile_fp8<kTrans>(q, sqt, stt, tid, [&] { group_sync(group); });
    fence_proxy_async_shared();
    group_sync(group);
    if (issuer) {
      if (p.out != nullptr)
        tma_store_2d(tmQ, sqt, static_cast<int32_t>(c0), static_cast<int32_t>(r0));
      if (kTrans)
        tma_store_2d(tmQT, stt, static_cast<int32_t>(r0), static_cast<int32_t>(c0));
      bulk_commit_group();
    }
  }
  if constexpr (kPair) {
    // The second tensor's tile, by group 0, staged in slot 0 (group 0's
    // first tile) once that tile's stores have read it.
    if (has2 && group == 0) {
      if (issuer) bulk_wait_group_read<0>();
      group_sync(0);
      const int64_t r0 = (blockIdx.x / ntc2) * kTile, c0 = (blockIdx.x % ntc2) * kTile;
      uint2 q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) q[u] = cast8<kFmt>(v2[u], s2);
      uint8_t* sqt = tiles;
      uint8_t* stt = tiles + kTile * kTile;
      stage_tile_fp8<kTrans>(q, sqt, stt, tid, [&] { group_sync(0); });
      fence_proxy_async_shared();
      group_sync(0);
      if (issuer) {
        if (p.out2 != nullptr)
          tma_store_2d(tmQ2, sqt, static_cast<int32_t>(c0), static_cast<int32_t>(r0));
        if (kTrans)
          tma_store_2d(tmQT2, stt, static_cast<int32_t>(r0), static_cast<int32_t>(c0));
        bulk_commit_group();
      }
    }
  }
  // Count this CTA out (it has read the amax; after its casts, so that the
  // atomic's round trip delays no group); the last one clears the three words
  // for the next launch.
  if (threadIdx.x == 0 && atomicAdd(p.ws_exits, 1u) == gridDim.x - 1) {
    atomicExch(p.ws_barrier, 0u);
    atomicExch(p.ws_exits, 0u);
    atomicExch(p.ws_amax, 0u);
    if (kPair) atomicExch(p.ws_amax2, 0u);
  }
  if (issuer) bulk_wait_group<0>();  // stores done before the shared memory goes away
}

template <int kFmt, bool kTrans>
__global__ void __launch_bounds__(kSpThreads, 1)
    cast_single_pass_kernel(const __grid_constant__ CUtensorMap tmX,
                            const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmQT,
                            const __grid_constant__ SinglePassParams p) {
  single_pass_body<kFmt, kTrans, false>(&tmX, &tmQ, &tmQT, p, &tmQ, &tmQT);
}

// The single pass of W with x's cast in the same launch (x: at most one tile
// a CTA); one grid barrier for both maxima.
template <int kFmt, bool kTrans>
__global__ void __launch_bounds__(kSpThreads, 1)
    cast_pair_single_pass_kernel(const __grid_constant__ CUtensorMap tmX,
                                 const __grid_constant__ CUtensorMap tmQ,
                                 const __grid_constant__ CUtensorMap tmQT,
                                 const __grid_constant__ SinglePassParams p,
                                 const __grid_constant__ CUtensorMap tmQ2,
                                 const __grid_constant__ CUtensorMap tmQT2) {
  single_pass_body<kFmt, kTrans, true>(&tmX, &tmQ, &tmQT, p, &tmQ2, &tmQT2);
}

// ------------------------------------------------------------------ cluster single pass
//
// Dynamic amax -> scale -> cast (+ transpose) of a small tensor in ONE
// thread-block cluster of at most kClusterCtas CTAs.  Each CTA loads its
// tiles into registers and takes their maximum; the CTAs exchange their
// maxima through distributed shared memory between two cluster barriers; each
// then casts from registers.  No grid barrier, no global atomics and no
// workspace words, so the latency of a few-token tensor is one load, one
// cluster exchange and one store.  Tiles are kTR rows x (16384 / kTR) columns,
// kTR the smallest of 16, 32, 64, 128 covering the rows, so that a short,
// wide tensor (a few tokens x 4096) is not padded to 128-row tiles.
constexpr int kClusterCtas = 8;
constexpr int kClusterTilesPerCta = 2;
constexpr int kClusterTileElems = kThreads * 8 * 8;  // 8 vectors of 8 values per thread

struct ClusterCastParams {
  const uint16_t* x;
  int64_t rows, cols, ld;
  float eps;
  float* amax_out;
  float* scale_out;
  float* inv_out;
  uint8_t* out;
  uint8_t* out_t;
};

// Transposed write of one kTR x kTC fp8 tile held in shared memory (rows of
// kTC / 4 + 1 words): each thread moves one 16-row x 4-column block with the
// same 4x4 byte transposes as store_transposed_tile.  A warp reads 32
// consecutive words of a row: conflict-free.
template <int kTR, int kTC>
__device__ __forceinline__ void store_transposed_block(const uint32_t* sq, uint8_t* out_t,
                                                       int64_t rows, int64_t cols, int64_t r0,
                                                       int64_t c0, int tid) {
  constexpr int kPitch = kTC / 4 + 1;
  const int jg = tid % (kTC / 4), ig = tid / (kTC / 4);
  const int i0 = ig * 16, j0 = jg * 4;
  if (c0 + j0 >= cols || r0 + i0 >= rows) return;
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k] = sq[(i0 + k) * kPitch + jg];
  uint32_t o[4][4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t t0 = __byte_perm(w[4 * g + 0], w[4 * g + 1], 0x5140);
    const uint32_t t1 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x5140);
    const uint32_t t2 = __byte_perm(w[4 * g + 0], w[4 * g + 1], 0x7362);
    const uint32_t t3 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x7362);
    o[0][g] = __byte_perm(t0, t1, 0x5410);
    o[1][g] = __byte_perm(t0, t1, 0x7632);
    o[2][g] = __byte_perm(t2, t3, 0x5410);
    o[3][g] = __byte_perm(t2, t3, 0x7632);
  }
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    uint8_t* dst = out_t + (c0 + j0 + jj) * rows + r0 + i0;
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[jj][0], o[jj][1], o[jj][2], o[jj][3]);
  }
}

template <int kFmt, bool kTrans, int kTR>
__global__ void __launch_bounds__(kThreads, 1) cast_cluster_kernel(const ClusterCastParams p) {
  constexpr int kTC = kClusterTileElems / kTR;
  constexpr int kVR = kTC / 8;  // 8-value vectors per tile row
  constexpr int kPitch = kTC / 4 + 1;
  static_assert(kTR % 16 == 0 && kTC % 128 == 0, "tile shape");
  __shared__ __align__(16) uint32_t sq[kTrans ? kTR * kPitch : 1];
  __shared__ uint32_t s_max;  // this CTA's maximum, read by every CTA of the cluster
  __shared__ uint32_t s_all;
  const uint32_t rank = cluster_ctarank();
  const int nctas = static_cast<int>(gridDim.x);  // the grid is one cluster
  const int64_t ntc = (p.cols + kTC - 1) / kTC;
  const int64_t ntiles = ((p.rows + kTR - 1) / kTR) * ntc;
  griddep_wait();
  uint4 v[kClusterTilesPerCta][8];
  AbsMax a0, a1;
#pragma unroll
  for (int k = 0; k < kClusterTilesPerCta; ++k) {
    const int64_t t = rank + static_cast<int64_t>(k) * nctas;
    const int64_t r0 = (t / ntc) * kTR, c0 = (t % ntc) * kTC;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int vi = threadIdx.x + kThreads * u;
      const int64_t row = r0 + vi / kVR, col = c0 + (vi % kVR) * 8;
      v[k][u] = (t < ntiles && row < p.rows && col < p.cols)
                    ? ld_stream_v4(p.x + row * p.ld + col)
                    : make_uint4(0, 0, 0, 0);
      (u & 1 ? a1 : a0).add(v[k][u]);
    }
  }
  a0.merge(a1);
  const uint32_t bits = block_absmax_bits(a0.packed());
  if (threadIdx.x == 0) s_max = bits;
  // A lone CTA (launched without a cluster) keeps to CTA-scope barriers.
  if (nctas > 1)
    cluster_sync_all();  // every CTA's s_max is written
  else
    __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t m = 0;
    if (static_cast<int>(threadIdx.x) < nctas)
      m = nctas > 1 ? ld_shared_cluster_u32(map_to_cta(smem_addr(&s_max), threadIdx.x)) : s_max;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (threadIdx.x == 0) s_all = m;
  }
  if (nctas > 1)
    cluster_sync_all();  // no CTA leaves or moves on while a peer may read its s_max
  else
    __syncthreads();
  griddep_launch_dependents();

  const float amax = __uint_as_float(s_all);
  const float s = scale_from_amax(amax, p.eps, fp8_max<kFmt>());
  if (rank == 0 && threadIdx.x == 0) {
    *p.amax_out = amax;
    *p.scale_out = s;
    *p.inv_out = __fdiv_rn(1.0f, s);
  }
#pragma unroll
  for (int k = 0; k < kClusterTilesPerCta; ++k) {
    const int64_t t = rank + static_cast<int64_t>(k) * nctas;
    if (t < ntiles) {  // uniform in the CTA
      const int64_t r0 = (t / ntc) * kTR, c0 = (t % ntc) * kTC;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int vi = threadIdx.x + kThreads * u;
        const int rl = vi / kVR, cv = vi % kVR;
        const int64_t row = r0 + rl, col = c0 + cv * 8;
        const uint2 q = cast8<kFmt>(v[k][u], s);
        if (p.out != nullptr && row < p.rows && col < p.cols)
          *reinterpret_cast<uint2*>(p.out + row * p.cols + col) = q;
        if (kTrans) {
          sq[rl * kPitch + cv * 2] = q.x;
          sq[rl * kPitch + cv * 2 + 1] = q.y;
        }
      }
      if (kTrans) {
        __syncthreads();
        store_transposed_block<kTR, kTC>(sq, p.out_t, p.rows, p.cols, r0, c0, threadIdx.x);
        __syncthreads();
      }
    }
  }
}

template <typename Kernel>
int resident_ctas(Kernel k, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess) return 0;
  return n;
}

}  // namespace

}  // namespace fp8lin
