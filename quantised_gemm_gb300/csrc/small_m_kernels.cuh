// small_m_kernels.cuh -- device code of the few-token Linear products: a
// GEMM with few rows (M <= 32 tokens) against a large weight, fused with the
// casts around it, in ONE launch per product.
//
//   D [M, NA] = (B8 [M, KA] . A8 [NA, KA]^T) * inv_b * inv_a      (bf16)
//
// A is the weight side (W8 for y, W8^T for dX), B the few-token side (x for
// y, dY for dX).  With few tokens the products are short of work and long on
// fixed costs: the step of a 16-token 4096 x 4096 Linear ran as six kernels
// whose boundaries cost more than their bytes.  Here one kernel
//   1. loads its A tiles (128 x 128) by TMA, each on its own mbarrier --
//      bf16 W when kCastA (the weight is cast in the same launch), else the
//      fp8 copy, which is loaded after the grid barrier when B's amax is
//      taken here (ahead of the barrier, those loads held up the few bytes of
//      B the barrier waits for); the CTA owning each 128-column slice of B
//      takes that slice's amax (unless the amax is given) and keeps the
//      slice in registers;
//   2. kCastA: folds the amax of its W tiles, each as it lands; every CTA
//      then passes a bounded grid barrier (cooperative launch: all CTAs are
//      resident) that makes both amaxes complete -- for !kCastA the barrier
//      counts only the slices of B -- and the slice owners write B's fp8 copy
//      and its transpose (x8 / x8^T, dY8 / dY8^T) from those registers;
//   3. per tile: casts the W tile (kCastA) into the 128-byte-swizzled K-major
//      layout the tensor cores read and stores W8 by TMA; casts B's slice of
//      the tile's K range into the same layout beside it, and its group's
//      thread issues the tile's tcgen05 MMAs (M = 128 rows of A, N = kMN
//      tokens, K = 128) into the tile's own TMEM columns at once.  Tiles are
//      numbered band-major (128 rows of A, then K), so the few consecutive
//      tiles of a CTA fall in one or two bands;
//   4. once the MMAs are done, sums the accumulators of its tiles of each
//      band in tile order and writes that fp32 partial of D^T to the
//      workspace; one lane per band adds the CTA's tile count to the band's
//      ticket with a release atomic.  While those are in flight, kCastA
//      stages each tile's transpose in the second half of its slot and
//      stores W8^T by TMA (kDW computes dW, below).  The CTA that completes a
//      band (all its K tiles counted) sums the band's partials in K order
//      (deterministic), scales by alpha = fl32(inv_a * inv_b) and stores
//      bf16 D, plus the amax of D when asked for.
//
// kDW (the backward): the same launch also computes the weight gradient
//   dW [KA, NA] = (dY8^T . x8) * inv_dy * inv_x          (bf16)
// with K = MB tokens, once the MMAs of dX are done.  dW has as many 128 x 128
// tiles as dX's product, row-band-major, and each CTA takes the same tile
// numbers t0 .. t0 + mine - 1, split between the two groups.  Per tile the
// group writes dY8^T's 128 rows (dY re-cast from bf16 with the scale just
// found: the same bytes the slice owners store) and x8^T's 128 rows (the
// forward's transposed x8) into 128-byte-swizzled K-major operands, zero
// beyond the tokens; one MMA of K = 32 puts the tile into the group's 128
// TMEM columns; each of the group's 8 warps stores its 32 x 64 block as one
// TMA box.  The next tile's operand loads are in flight meanwhile.
//
// Numerics are those of the separate kernels: amax of the bf16 bit patterns,
// scale = __fdiv_rn(F, max(amax, eps)), q = cvt.rn.satfinite(x * scale), fp32
// accumulation on the tensor cores; only the order in which the fp32 partial
// sums of D are added differs from the split-K GEMM's.
#pragma once

#include "cast_kernels.cuh"

namespace fp8lin {
namespace {

constexpr int kSmThreads = 512;                        // two 256-thread tile groups
constexpr int kSmMmaK = 32;                            // K of one kind::f8f6f4 MMA
constexpr int kSmTilesPerCta = 7;
constexpr int kSmTileBytes = kTile * kTile * 2;        // one bf16 tile; fp8 uses the first half
constexpr int kSmBSliceOffset = kTile * kTile;         // B's slice sits in the second half
constexpr size_t kSmSmem = static_cast<size_t>(kSmTilesPerCta) * kSmTileBytes + 1024;

constexpr int kSmDwTmemCol = 256;                      // kDW: dW accumulators, 128 columns per group
constexpr int kSmDwStageOffset = 4 * kTile * kTile;    // kDW: operands (2 x 2 x 16 KB), then boxes
constexpr int kSmDwBoxBytes = 32 * 64 * 2;             // one 32-row x 64-column bf16 box
static_assert(kSmDwStageOffset + 16 * 2 * kSmDwBoxBytes <= kSmTilesPerCta * kSmTileBytes,
              "dW operands and staging boxes fit in the tile slots");

struct SmallParams {
  int NA, KA, MB;               // D^T [NA, MB] = A [NA, KA] . B [MB, KA]^T
  const uint16_t* b;            // bf16 B [MB, KA], row stride ldb elements
  int64_t ldb;
  float eps;
  const float* b_amax_in;       // amax of B given by its producer (nullptr: computed here)
  float* b_amax;                // B's state: amax, scale, inverse (written by CTA 0)
  float* b_scale;
  float* b_inv;
  uint8_t* b8;                  // fp8 B [MB, KA] and B^T [KA, MB]
  uint8_t* b8t;
  float* a_amax;                // kCastA: A's state outputs
  float* a_scale;
  float* a_inv;
  const float* a_inv_in;        // !kCastA: A's inverse scale
  uint16_t* d;                  // bf16 D [MB, NA], row stride ldd elements
  int64_t ldd;
  uint32_t* d_amax;             // max |D| as fp32 bits (nullptr: not wanted)
  uint32_t* d_amax_acc;         // self-cleaning workspace words of that maximum
  uint32_t* d_amax_ticket;
  float* partials;              // fp32 partials, [first tile of the CTA in the band][kMN][128]
  int* tickets;                 // per 128-row band of A (zero between launches)
  uint32_t* ws_barrier;         // grid barrier words (zero between launches)
  uint32_t* ws_exits;
  uint32_t* ws_amax;            // amax of A (kCastA)
  uint32_t* ws_b_amax;          // amax of B (unless given)
  int* err;
  const uint8_t* x8t;           // kDW: fp8 x^T [NA, MB] (e4m3, from the forward)
  const float* x_inv;           // kDW: x's inverse scale
};

__device__ __forceinline__ void sm_group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(256) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Atomic add with release semantics at GPU scope (this thread's earlier
// writes, and those ordered before it by a CTA barrier, are visible to a
// thread that acquires the new value); returns the old value.
__device__ __forceinline__ int atom_add_release(int* p, int v) {
  int old;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// AND of `pred` over the 256 threads of `group` (also a barrier of the group).
__device__ __forceinline__ bool sm_group_and(int group, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %2, 0;\n\t"
      "bar.red.and.pred p, %1, 256, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(1 + group), "r"(pred ? 1u : 0u)
      : "memory");
  return r != 0;
}

// Max over the 512 threads of a 16-bit magnitude pattern; result in s_out
// (as fp32 bits) after the call, visible to every thread.
__device__ __forceinline__ void sm_block_max(uint32_t m16, uint32_t* s_red, uint32_t* s_out) {
  m16 = __reduce_max_sync(0xFFFFFFFFu, m16);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m16;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t m = threadIdx.x < kSmThreads / 32 ? s_red[threadIdx.x] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (threadIdx.x == 0) *s_out = m << 16;
  }
  __syncthreads();
}

template <int kMN>
__device__ __forceinline__ void sm_tmem_load(uint32_t taddr, uint32_t (&r)[kMN]) {
  if constexpr (kMN == 32)
    tmem_load_32cols(taddr, r);
  else
    tmem_load_16cols(taddr, r);
  tmem_load_wait();
}

// kCastA: the transpose of a cast 128 x 128 fp8 tile (128-byte swizzled, as
// the tensor cores read it) into `dst` in the same layout, for one TMA store
// of W8^T.  Each thread of the group takes a 16-row x 4-column block: four
// 16-byte rows of the transpose.
__device__ __forceinline__ void stage_transpose(const uint8_t* src, uint8_t* dst, int gtid) {
  const int lw = gtid & 31, gw = gtid >> 5;
  const int jg = (gw & 1) * 16 + (lw >> 1);  // 4-column group 0..31
  const int ig = (gw >> 1) * 2 + (lw & 1);   // 16-row group 0..7
  uint32_t w[16];
#pragma unroll
  for (int kk = 0; kk < 16; ++kk)
    w[kk] = *reinterpret_cast<const uint32_t*>(src + sw128(ig * 16 + kk, jg * 4));
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t x0 = __byte_perm(w[4 * g + 0], w[4 * g + 1], 0x5140);
    const uint32_t x1 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x5140);
    const uint32_t x2 = __byte_perm(w[4 * g + 0], w[4 * g + 1], 0x7362);
    const uint32_t x3 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x7362);
    w[4 * g + 0] = __byte_perm(x0, x1, 0x5410);
    w[4 * g + 1] = __byte_perm(x0, x1, 0x7632);
    w[4 * g + 2] = __byte_perm(x2, x3, 0x5410);
    w[4 * g + 3] = __byte_perm(x2, x3, 0x7632);
  }
#pragma unroll
  for (int jj = 0; jj < 4; ++jj)
    *reinterpret_cast<uint4*>(dst + sw128(jg * 4 + jj, ig * 16)) =
        make_uint4(w[jj], w[4 + jj], w[8 + jj], w[12 + jj]);
}

// kDW: the global operand bytes of one dW tile for this thread of its group
// -- dY vectors of the tile's 128 rows of dW (kMN / 16 per thread) and one
// 16-byte piece of x8^T's 128 rows.
template <int kMN>
struct DwLoads {
  uint4 y[kMN / 16];
  uint4 x;
};

template <int kMN>
__device__ __forceinline__ void dw_load(const SmallParams& p, int t, int nbands, int gtid,
                                        DwLoads<kMN>& l) {
  const int n0 = (t / nbands) * kTile, k0 = (t % nbands) * kTile;
#pragma unroll
  for (int u = 0; u < kMN / 16; ++u) {
    const int i = gtid + 256 * u, m = i >> 4, n = n0 + (i & 15) * 8;
    l.y[u] = n < p.KA ? ld_stream_v4(p.b + static_cast<int64_t>(m) * p.ldb + n)
                      : make_uint4(0u, 0u, 0u, 0u);
  }
  // x8^T rows are kMN bytes: one 16-byte piece per thread (16 tokens: the first 128 threads).
  const int row = kMN == 16 ? gtid : gtid >> 1, piece = kMN == 16 ? 0 : gtid & 1;
  const int k = k0 + row;
  l.x = (row < kTile && k < p.NA)
            ? *reinterpret_cast<const uint4*>(p.x8t + static_cast<int64_t>(k) * kMN + 16 * piece)
            : make_uint4(0u, 0u, 0u, 0u);
}

// kDW: the group's dW tiles (its share of t0 .. t0 + mine - 1), after the
// MMAs of dX are done: operands into the group's two 16 KB buffers, one MMA
// (K = 32, the tokens zero-padded), the group's 8 warps each take a 32-row x
// 64-column block out of TMEM and store it as one TMA box (two boxes per
// warp, used in turn).  `l` holds the group's first tile's loads on entry.
// Returns false (group-uniform) when the wait for an MMA ran out.
template <int kFmtB, int kMN>
__device__ __forceinline__ bool dw_tiles(const SmallParams& p, const CUtensorMap* tmDW,
                                         uint8_t* tiles, uint32_t tmem, uint64_t* done, int t0,
                                         int mine, int nbands, float s_dy, float alpha,
                                         DwLoads<kMN>& l) {
  constexpr uint32_t kIdesc = make_idesc_f8(static_cast<uint32_t>(kFmtB), 0u, 128u, 128u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = tid >> 8, gtid = tid & 255;
  uint8_t* opA = tiles + group * (2 * kTile * kTile);  // dY8^T rows, 128 B each (swizzled)
  uint8_t* opB = opA + kTile * kTile;                   // x8^T rows
  const uint32_t d_tmem = tmem + static_cast<uint32_t>(kSmDwTmemCol + 128 * group);
  if constexpr (kMN == 16) {  // tokens 16..31 of every row stay zero
    uint8_t* buf = gtid < kTile ? opA : opB;
    *reinterpret_cast<uint4*>(buf + sw128(gtid & (kTile - 1), 16)) = make_uint4(0u, 0u, 0u, 0u);
  }
  const int quarter = warp & 3, half = (warp >> 2) & 1;
  bool prev_stored = false, ok = true;
  uint32_t phase = 0;
  int band = -1;
  for (int k = group, kq = 0; k < mine; k += 2, ++kq) {
    const int t = t0 + k, nb = t / nbands;
    if (nb != band) {  // dY8^T of this band of dW rows: byte m of row n (8 rows per vector)
      band = nb;
#pragma unroll
      for (int u = 0; u < kMN / 16; ++u) {
        const int i = gtid + 256 * u, m = i >> 4, j = i & 15;
        const uint2 q = cast8<kFmtB>(l.y[u], s_dy);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = (e + j) & 7;  // rotated: the warp's rows fall in different chunks
          opA[sw128(8 * j + r, m)] = static_cast<uint8_t>(((r < 4 ? q.x : q.y) >> (8 * (r & 3))));
        }
      }
    }
    if (kMN == 32 || gtid < kTile) {
      const int row = kMN == 16 ? gtid : gtid >> 1, piece = kMN == 16 ? 0 : gtid & 1;
      *reinterpret_cast<uint4*>(opB + sw128(row, 16 * piece)) = l.x;
    }
    if (k + 2 < mine) dw_load<kMN>(p, t + 2, nbands, gtid, l);  // lands during this tile
    fence_proxy_async_shared();
    sm_group_sync(group);
    if (gtid == 0) {
      tc_fence_after_sync();
      mma_f8f6f4(d_tmem, smem_desc_k_sw128(smem_addr(opA)), smem_desc_k_sw128(smem_addr(opB)),
                 kIdesc, 0u);
      mma_commit(&done[group]);
    }
    volatile int never = 0;
    const bool landed = mbar_wait_bounded(&done[group], phase, &never);
    phase ^= 1u;
    if (!sm_group_and(group, landed)) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    uint32_t ra[32], rb[32];
    const uint32_t taddr = d_tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                           static_cast<uint32_t>(half * 64);
    tmem_load_32cols(taddr, ra);
    tmem_load_32cols(taddr + 32, rb);
    tmem_load_wait();
    tc_fence_before_sync();  // the reads are done before the group's next MMA
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float v0, v1;
      mul2_rn(ra[2 * j], ra[2 * j + 1], alpha, v0, v1);
      w[j] = cvt_bf16x2(v0, v1);
      mul2_rn(rb[2 * j], rb[2 * j + 1], alpha, v0, v1);
      w[16 + j] = cvt_bf16x2(v0, v1);
    }
    uint8_t* box = tiles + kSmDwStageOffset + (warp * 2 + (kq & 1)) * kSmDwBoxBytes;
    if (lane == 0) {  // the box's last store has read it
      if (prev_stored)
        bulk_wait_group_read<1>();
      else
        bulk_wait_group_read<0>();
    }
    __syncwarp();
    uint8_t* rowp = box + lane * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(rowp + ((c ^ (lane & 7)) << 4)) =
          make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    fence_proxy_async_shared();
    __syncwarp();
    const int row0 = nb * kTile + quarter * 32, col0 = (t % nbands) * kTile + half * 64;
    prev_stored = row0 < p.KA && col0 < p.NA;  // boxes are clipped at dW's edges
    if (lane == 0 && prev_stored) {
      tma_store_2d(tmDW, box, col0, row0);
      bulk_commit_group();
    }
  }
  return ok;
}

template <bool kCastA, int kFmtB, int kMN, bool kDW>
__global__ void __launch_bounds__(kSmThreads, 1)
    small_m_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA8,
                   const __grid_constant__ CUtensorMap tmC, const SmallParams p) {
  static_assert(kMN == 16 || kMN == 32, "tokens per MMA");
  static_assert(!(kDW && kCastA), "dW is fused into the backward product only");
  constexpr int kTmemCols = kDW ? 512 : (kSmTilesPerCta * kMN <= 128 ? 128 : 256);
  constexpr int kBVec = kMN * 16 / 256;  // B slice vectors per thread of a group, per tile
  constexpr int kGroupTiles = (kSmTilesPerCta + 1) / 2;
  constexpr uint32_t kIdesc = make_idesc_f8(0u, static_cast<uint32_t>(kFmtB), 128u, kMN);
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t loaded[kSmTilesPerCta];
  __shared__ __align__(8) uint64_t mma_done[2];
  __shared__ __align__(8) uint64_t dw_done[2];
  __shared__ uint32_t s_tmem;
  __shared__ uint32_t s_red[kSmThreads / 32];
  __shared__ uint32_t s_b_bits, s_a_bits, s_d_bits;
  __shared__ int s_abort;
  __shared__ int s_nbands;
  __shared__ int s_bands[kSmTilesPerCta];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = tid >> 8, gtid = tid & 255;
  const int nbands = (p.NA + kTile - 1) / kTile, nks = (p.KA + kTile - 1) / kTile;
  const int ntiles = nbands * nks;
  const int G = static_cast<int>(gridDim.x);
  const int per = ntiles / G, extra = ntiles % G;
  const int t0 = static_cast<int>(blockIdx.x) * per + min(static_cast<int>(blockIdx.x), extra);
  const int mine = per + (static_cast<int>(blockIdx.x) < extra ? 1 : 0);  // <= kSmTilesPerCta
  const int band0 = t0 / nks;  // tile t: band t / nks, K slice t % nks
  const bool b_given = p.b_amax_in != nullptr;

  if (tid == 0) {
    s_abort = 0;
    for (int k = 0; k < kSmTilesPerCta; ++k) mbar_init(&loaded[k], 1);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    if (kDW) {
      mbar_init(&dw_done[0], 1);
      mbar_init(&dw_done[1], 1);
    }
    if (kDW || kCastA) tma_prefetch_map(&tmC);
    fence_barrier_init();
    if (kCastA) tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmA8);
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;
  griddep_wait();  // B, A and the states are ready; D and the outputs are free

  // ---- phase 1: A tiles in flight (one barrier each); this thread's B
  // vectors for its group's tiles in one batch; the amax of B's slices.
  // The fp8 variant whose token side needs the grid barrier loads its tiles
  // after the barrier instead: the barrier waits on the few bytes of B's
  // slices, which would otherwise queue behind every CTA's tile loads.
  const bool late_a = !kCastA && !b_given;  // grid-uniform
  auto issue_a = [&] {
    constexpr uint32_t kTileIn = kCastA ? kTile * kTile * 2 : kTile * kTile;
    for (int k = 0; k < mine; ++k) {
      const int t = t0 + k;
      mbar_arrive_expect_tx(&loaded[k], kTileIn);
      tma_load_2d(tiles + k * kSmTileBytes, kCastA ? &tmA : &tmA8, &loaded[k], (t % nks) * kTile,
                  (t / nks) * kTile);
    }
  };
  if (tid == 0 && !late_a) issue_a();
  uint4 bv[kGroupTiles][kBVec];
#pragma unroll
  for (int kq = 0; kq < kGroupTiles; ++kq) {
    const int k = group + 2 * kq;
    const int c0 = ((t0 + k) % nks) * kTile;
#pragma unroll
    for (int u = 0; u < kBVec; ++u) {
      const int i = gtid + 256 * u, m = i >> 4, j = c0 + (i & 15) * 8;
      bv[kq][u] = (k < mine && m < p.MB && j < p.KA)
                      ? ld_stream_v4(p.b + static_cast<int64_t>(m) * p.ldb + j)
                      : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  int my_slices = 0;  // B slices this CTA owns: blockIdx.x, blockIdx.x + G, ...
  uint4 b_own = make_uint4(0u, 0u, 0u, 0u);  // this thread's vector of slice blockIdx.x, kept
  if (!b_given) {                            // for B's fp8 copies (MB * 16 <= threads)
    AbsMax am;
    for (int c = blockIdx.x; c < nks; c += G, ++my_slices) {
      for (int i = tid; i < p.MB * 16; i += kSmThreads) {
        const int m = i >> 4, j = c * kTile + (i & 15) * 8;
        if (j < p.KA) {
          const uint4 v = ld_stream_v4(p.b + static_cast<int64_t>(m) * p.ldb + j);
          am.add(v);
          if (c == static_cast<int>(blockIdx.x)) b_own = v;
        }
      }
    }
    if (my_slices > 0) {  // CTA-uniform
      const uint32_t pk = am.packed();
      sm_block_max(max(pk & 0xFFFFu, pk >> 16), s_red, &s_b_bits);
    }
  } else {
    if (tid == 0) s_b_bits = __float_as_uint(*p.b_amax_in);
    if (static_cast<int>(blockIdx.x) < nks && tid < p.MB * 16) {
      const int j = static_cast<int>(blockIdx.x) * kTile + (tid & 15) * 8;
      if (j < p.KA) b_own = ld_stream_v4(p.b + static_cast<int64_t>(tid >> 4) * p.ldb + j);
    }
  }

  bool ok = true;
  if constexpr (kCastA) {
    // The amax of each W tile as soon as it lands.
    volatile int never = 0;
    AbsMax a0, a1;
    for (int k = group; k < mine; k += 2) {
      if (!mbar_wait_bounded(&loaded[k], 0, &never)) {
        ok = false;
        break;
      }
      const uint8_t* buf = tiles + k * kSmTileBytes;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int vi = gtid + 256 * u;
        (u & 1 ? a1 : a0).add(*reinterpret_cast<const uint4*>(buf + (vi >> 4) * (kTile * 2) +
                                                               (vi & 15) * 16));
      }
    }
    a0.merge(a1);
    const uint32_t pk = a0.packed();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (ok) sm_block_max(max(pk & 0xFFFFu, pk >> 16), s_red, &s_a_bits);
  }
  if (!ok && tid == 0) atomicCAS(p.err, 0, kErrCastWait);

  // ---- the grid barrier: A's amax (kCastA) and B's slices complete
  const bool need_barrier = kCastA || !b_given;  // grid-uniform
  if (ok && need_barrier) {
    if (tid == 0) {
      if (kCastA) atomicMax(p.ws_amax, s_a_bits);
      if (!b_given && my_slices > 0) atomicMax(p.ws_b_amax, s_b_bits);
      // kCastA: every CTA arrives once; else each slice of B arrives once.
      const uint32_t arrive = kCastA ? 1u : static_cast<uint32_t>(my_slices);
      const uint32_t target = kCastA ? gridDim.x : static_cast<uint32_t>(nks);
      if (arrive > 0) red_release_add(p.ws_barrier, arrive);
      const uint64_t start = global_timer_ns();
      while (ld_acquire_u32(p.ws_barrier) < target) {
        if (global_timer_ns() - start > kWaitLimitNs) {
          atomicCAS(p.err, 0, kErrGridBarrier);
          s_abort = 1;
          break;
        }
      }
      if (!s_abort) {  // ordered after every arrival by the acquiring poll; both in flight at once
        const uint32_t a_bits = kCastA ? ld_relaxed_u32(p.ws_amax) : 0u;
        const uint32_t b_bits = b_given ? 0u : ld_relaxed_u32(p.ws_b_amax);
        if (kCastA) s_a_bits = a_bits;
        if (!b_given) s_b_bits = b_bits;
      }
    }
    __syncthreads();
    ok = s_abort == 0;
  } else {
    __syncthreads();
  }
  const bool passed = need_barrier && ok;  // counts out once its MMAs are issued
  const bool a_issued = !late_a || ok;      // CTA-uniform
  if (late_a && ok && tid == 0) issue_a();

  const float amax_b = __uint_as_float(s_b_bits);
  const float s_b = scale_from_amax(amax_b, p.eps, fp8_max<kFmtB>());
  const float inv_b = __fdiv_rn(1.0f, s_b);
  float s_a = 1.0f, inv_a;
  if constexpr (kCastA) {
    s_a = scale_from_amax(__uint_as_float(s_a_bits), p.eps, fp8_max<0>());
    inv_a = __fdiv_rn(1.0f, s_a);
  } else {
    inv_a = *p.a_inv_in;
  }
  if (ok && blockIdx.x == 0 && tid == 0) {
    *p.b_amax = amax_b;
    *p.b_scale = s_b;
    *p.b_inv = inv_b;
    if constexpr (kCastA) {
      *p.a_amax = __uint_as_float(s_a_bits);
      *p.a_scale = s_a;
      *p.a_inv = inv_a;
    }
  }

  // ---- B's fp8 copies (for the later kernels): the CTA of each K slice
  // writes it (q [MB, KA], q^T [KA, MB]), the first slice from the registers
  // its amax was taken from.  Before the tiles' casts: behind their stores
  // these few bytes waited about a microsecond.
  if (ok) {
    for (int c = blockIdx.x; c < nks; c += G) {
      for (int i = tid; i < kMN * 16; i += kSmThreads) {
        const int m = i >> 4, j = (c * kTile) + (i & 15) * 8;
        if (m < p.MB && j < p.KA) {
          const uint4 v = c == static_cast<int>(blockIdx.x)
                              ? b_own
                              : ld_stream_v4(p.b + static_cast<int64_t>(m) * p.ldb + j);
          const uint2 q = cast8<kFmtB>(v, s_b);
          *reinterpret_cast<uint2*>(p.b8 + static_cast<int64_t>(m) * p.KA + j) = q;
#pragma unroll
          for (int e = 0; e < 8; ++e)
            p.b8t[static_cast<int64_t>(j + e) * p.MB + m] =
                static_cast<uint8_t>(((e < 4 ? q.x : q.y) >> (8 * (e & 3))) & 0xFFu);
        }
      }
    }
  }

  // ---- phase 2: per tile, the casts into the MMA layout, then its MMAs
  bool issued = false;
  if (ok) {
    volatile int never = 0;
#pragma unroll
    for (int kq = 0; kq < kGroupTiles; ++kq) {
      const int k = group + 2 * kq;
      if (k >= mine) break;
      const int t = t0 + k, c0 = (t % nks) * kTile, r0 = (t / nks) * kTile;
      uint8_t* buf = tiles + k * kSmTileBytes;
      uint8_t* bsl = buf + kSmBSliceOffset;
      if constexpr (kCastA) {
        uint2 q[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int vi = gtid + 256 * u;
          q[u] = cast8<0>(*reinterpret_cast<const uint4*>(buf + (vi >> 4) * (kTile * 2) +
                                                          (vi & 15) * 16),
                          s_a);
        }
        sm_group_sync(group);  // the group has read the bf16 tile: the buffer is free
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int vi = gtid + 256 * u;
          *reinterpret_cast<uint2*>(buf + sw128(vi >> 4, (vi & 15) * 8)) = q[u];
        }
      } else {
        mbar_wait_bounded(&loaded[k], 0, &never);  // the fp8 tile has landed (bounded)
      }
      // B's slice of this tile's K range, [kMN rows][128 bytes], same swizzle.
#pragma unroll
      for (int u = 0; u < kBVec; ++u) {
        const int i = gtid + 256 * u;
        *reinterpret_cast<uint2*>(bsl + sw128(i >> 4, (i & 15) * 8)) = cast8<kFmtB>(bv[kq][u], s_b);
      }
      fence_proxy_async_shared();
      sm_group_sync(group);
      if (gtid == 0) {
        const bool landed = kCastA || mbar_try_wait(&loaded[k], 0);
        if (landed) {
          tc_fence_after_sync();
          const uint64_t a_desc = smem_desc_k_sw128(smem_addr(buf));
          const uint64_t b_desc = smem_desc_k_sw128(smem_addr(bsl));
#pragma unroll
          for (int kk = 0; kk < kTile / kSmMmaK; ++kk)  // K offset kk * 32 bytes (encoded >> 4)
            mma_f8f6f4(tmem + static_cast<uint32_t>(k * kMN),
                       a_desc + static_cast<uint64_t>(kk * (kSmMmaK >> 4)),
                       b_desc + static_cast<uint64_t>(kk * (kSmMmaK >> 4)), kIdesc,
                       kk > 0 ? 1u : 0u);
          issued = true;
        } else {
          atomicCAS(p.err, 0, kErrCastWait);
          s_abort = 1;
        }
      }
      if constexpr (kCastA) {
        if (gtid == 0) {
          tma_store_2d(&tmA8, buf, c0, r0);  // W8 tile (clipped at the edges)
          bulk_commit_group();
        }
      }
    }
  }
  if (gtid == 0) {
    if (issued)
      mma_commit(&mma_done[group]);  // arrives once this thread's MMAs are complete
    else
      mbar_arrive(&mma_done[group]);
  }
  DwLoads<kMN> dwl;
  if (kDW && ok && group < mine) dw_load<kMN>(p, t0 + group, nbands, gtid, dwl);

  griddep_launch_dependents();
  // Count this CTA out of the grid barrier (it has read its words); the last
  // one clears them for the next launch.  Off the path: the MMAs are running.
  if (passed && tid == 0 && atomicAdd(p.ws_exits, 1u) == gridDim.x - 1) {
    atomicExch(p.ws_barrier, 0u);
    atomicExch(p.ws_exits, 0u);
    atomicExch(p.ws_amax, 0u);
    atomicExch(p.ws_b_amax, 0u);
  }
  {
    volatile int never = 0;
    bool done = mbar_wait_bounded(&mma_done[0], 0, &never);
    done = mbar_wait_bounded(&mma_done[1], 0, &never) && done;
    if (!done && tid == 0) atomicCAS(p.err, 0, kErrGemmMmaWait);
    ok = __syncthreads_and(ok && done && s_abort == 0 ? 1 : 0) != 0;
  }
  tc_fence_after_sync();

  // ---- phase 3: one partial per band of this CTA (its tiles summed in tile
  // order), tickets, the last one reduces
  const int nacc = mine > 0 ? (t0 + mine - 1) / nks - band0 + 1 : 0;
  if (ok) {
    const int quarter = warp & 3;
    for (int a = warp >> 2; a < nacc; a += kSmThreads / 128) {
      const int band = band0 + a;
      const int lo = max(t0, band * nks), hi = min(t0 + mine, (band + 1) * nks);
      float acc[kMN];
#pragma unroll
      for (int m = 0; m < kMN; ++m) acc[m] = 0.0f;
      for (int t = lo; t < hi; ++t) {
        uint32_t r[kMN];
        sm_tmem_load<kMN>(tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>((t - t0) * kMN),
                          r);
#pragma unroll
        for (int m = 0; m < kMN; ++m) acc[m] += __uint_as_float(r[m]);
      }
      float* dst = p.partials + static_cast<size_t>(lo) * kMN * kTile + quarter * 32 + lane;
#pragma unroll
      for (int m = 0; m < kMN; ++m)
        if (m < p.MB) __stcg(dst + m * kTile, acc[m]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  // Tickets: one lane of the last warp per band of this CTA adds the CTA's
  // tile count, releasing its partials (ordered before the lane by the
  // barrier).  The old values are looked at only after dW (kDW), so the
  // warp does not wait for them.
  int old_ticket = 0, my_band = -1, my_count = 0;
  if (warp == kSmThreads / 32 - 1 && ok && lane < nacc) {
    my_band = band0 + lane;
    const int lo = max(t0, my_band * nks), hi = min(t0 + mine, (my_band + 1) * nks);
    my_count = hi - lo;
    old_ticket = atom_add_release(&p.tickets[my_band], my_count);
  }
  if constexpr (kCastA) {
    // W8^T: each tile's transpose staged in the second half of its slot (the
    // bf16 data and B's slice there are used up: the MMAs are done) and
    // stored by TMA, while the tickets' atomics are in flight.  Stored from
    // registers during the casts, these 16-byte rows took 3.7 us of them;
    // staged before the partials, they held the partials back by 2.5 us.
    if (ok) {
      for (int k = group; k < mine; k += 2) {  // each tile's store leaves as it is staged
        stage_transpose(tiles + k * kSmTileBytes, tiles + k * kSmTileBytes + kSmBSliceOffset,
                        gtid);
        fence_proxy_async_shared();
        sm_group_sync(group);
        if (gtid == 0) {
          const int t = t0 + k;
          tma_store_2d(&tmC, tiles + k * kSmTileBytes + kSmBSliceOffset, (t / nks) * kTile,
                       (t % nks) * kTile);  // W8^T [KA, NA] at (K slice, band)
          bulk_commit_group();
        }
      }
    }
  }
  if constexpr (kDW) {
    // dW (the tile slots are free: the MMAs that read them are done)
    if (ok) {
      const float alpha_dw = __fmul_rn(inv_b, *p.x_inv);
      const bool dw_ok = dw_tiles<kFmtB, kMN>(p, &tmC, tiles, tmem, dw_done, t0, mine, nbands,
                                              s_b, alpha_dw, dwl);
      if (!dw_ok && gtid == 0) atomicCAS(p.err, 0, kErrGemmMmaWait);
    }
  }
  if (warp == kSmThreads / 32 - 1) {
    const bool completes = my_band >= 0 && old_ticket + my_count == nks;
    if (completes) {
      p.tickets[my_band] = 0;  // every K tile has arrived: clear for the next launch
      fence_acq_rel_gpu();     // ...and every partial of the band is visible to this CTA
    }
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, completes);
    if (completes) s_bands[__popc(m & ((1u << lane) - 1u))] = my_band;
    if (lane == 0) s_nbands = __popc(m);
  }
  __syncthreads();
  const float alpha = __fmul_rn(inv_a, inv_b);
  float vmax = 0.0f;
  const int nb = s_nbands;
  for (int bi = 0; bi < nb; ++bi) {
    const int band = s_bands[bi];
    // The band's partials: one per CTA holding some of its K tiles, at that
    // CTA's first tile in the band, in K order.  The CTA holding the band's
    // first tile (CTAs below `extra` hold per + 1 tiles) is one division
    // away; the next slots are the starts of the CTAs after it.
    const int b0 = band * nks, t_end = (band + 1) * nks;
    const int slot_cta0 =
        b0 < extra * (per + 1) ? b0 / (per + 1) : extra + (b0 - extra * (per + 1)) / per;
    for (int i = tid; i < p.MB * (kTile / 4); i += kSmThreads) {
      const int m = i / (kTile / 4), nq = (i - m * (kTile / 4)) * 4;
      const int n = band * kTile + nq;
      if (n >= p.NA) continue;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      // Slot j of the band: its first tile, then the starts of the next CTAs.
      for (int j0 = 0;; j0 += 8) {
        float4 v[8];
        bool any = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int cta = slot_cta0 + j0 + j;
          const int ts = (j0 + j == 0) ? band * nks : cta * per + min(cta, extra);
          const bool in = (j0 + j == 0) || ts < t_end;
          any |= in;
          v[j] = in ? __ldcg(reinterpret_cast<const float4*>(
                          p.partials + static_cast<size_t>(ts) * kMN * kTile + m * kTile + nq))
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // in K order; absent slots add exact zeros
          acc.x += v[j].x;
          acc.y += v[j].y;
          acc.z += v[j].z;
          acc.w += v[j].w;
        }
        const int next = slot_cta0 + j0 + 8;
        if (!any || next * per + min(next, extra) >= t_end) break;
      }
      const float v0 = __fmul_rn(acc.x, alpha), v1 = __fmul_rn(acc.y, alpha);
      const float v2 = __fmul_rn(acc.z, alpha), v3 = __fmul_rn(acc.w, alpha);
      *reinterpret_cast<uint2*>(p.d + static_cast<int64_t>(m) * p.ldd + n) =
          make_uint2(cvt_bf16x2(v0, v1), cvt_bf16x2(v2, v3));
      vmax = fmaxf(vmax, fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3))));
    }
  }
  if (p.d_amax != nullptr && nb > 0) {
    // Rounding to bf16 is monotone: the bf16 of the largest |v| is the amax
    // of the stored D.  Every reduced band counts once on the ticket.
    sm_block_max(cvt_bf16x2(vmax, 0.0f) & 0xFFFFu, s_red, &s_d_bits);
    if (tid == 0) {
      atomicMax(p.d_amax_acc, s_d_bits);
      __threadfence();
      if (atomicAdd(p.d_amax_ticket, static_cast<uint32_t>(nb)) + nb ==
          static_cast<uint32_t>(nbands)) {
        __threadfence();
        *p.d_amax = atomicExch(p.d_amax_acc, 0u);
        atomicExch(p.d_amax_ticket, 0u);
      }
    }
  }
  if (kCastA && gtid == 0) bulk_wait_group<0>();  // W8 stores done before the smem goes away
  if (kDW && lane == 0) bulk_wait_group<0>();     // and dW's boxes
  if (!ok && a_issued && tid == 0) {
    // Copies in flight land before the shared memory goes away (bounded).
    volatile int never = 0;
    for (int k = 0; k < mine; ++k) mbar_wait_bounded(&loaded[k], 0, &never);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace fp8lin
