// gemm_kernels.cuh -- device code of the FP8 GEMM of the fp8 Linear on the
// 5th-generation tensor cores (sm_103a):
// D[m, n] = bf16((sum_k A[m, k] * B[n, k]) * inv_a * inv_b)
// with both operands K-major 8-bit (e4m3 or e5m2) and fp32 accumulation in
// tensor memory.  The three products of the Linear's forward and backward
// ("Why swapping nn.Linear with FP8Linear brings throughput decrease for 7B
// LLAMA2-like model?", pytorch/ao issue 1199: the FP8Linear that replaces
// nn.Linear) all take this form once the transposed fp8 copies exist.
//
// Two persistent, warp-specialised kernels (320 threads):
//   gemm_fp8_pair_kernel  clusters of 2 CTAs sharing a 256 x BN tile
//                         (tcgen05.mma.cta_group::2), for more than 128 rows;
//   gemm_fp8_kernel       one CTA per 128 x BN tile (cta_group::1), for up to
//                         128 rows; with at most 64 rows the operands are
//                         swapped (D^T = B . A^T) so the weight fills the
//                         128-row MMA, and the epilogue stores transposed.
// Roles: warp 0 is the TMA producer (128-byte-swizzled K-major boxes, 128
// bytes of K per stage, STAGES-deep mbarrier ring); warp 1 allocates TMEM
// (two BN-column fp32 accumulators) and one lane issues the MMAs; warps 2..9
// are the epilogue, two per TMEM lane quarter (tcgen05.ld of their 32 TMEM
// lanes, scale by alpha = inv_a * inv_b, bf16, TMA stores of 32 x 32 boxes
// staged in shared memory, optionally the amax of the stored output).  The
// double-buffered accumulator overlaps the epilogue of one work unit with the
// main loop of the next.
//
// Work units: the tiles are dealt round-robin to the persistent CTAs (pairs).
// When the tiles do not fill one wave (few rows: M = 16 or 256 against a
// 4096-wide weight) and the K loop is long, each of the R tiles is split into
// S slices of the K loop (S = floor(slots / R)), so the work runs on all slots;
// every slice writes its fp32 partial to the workspace, waits (bounded) until
// all S slices of its 32-row group have written theirs, then sums all S
// partials of its own 1/S share of the columns in slice order --
// deterministic -- and writes the bf16 result.
//
// Every wait on an mbarrier is bounded (kWaitLimitNs); a wait that runs out
// records an error code in the workspace, raises a CTA-wide abort flag, lets
// its own copies / MMAs in flight finish (bounded), frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace fp8lin {
namespace {

constexpr int kBM = 128;           // rows of A per CTA (MMA M per CTA)
constexpr int kBK = 128;           // bytes (= 8-bit elements) of K per stage
constexpr int kMmaK = 32;          // K of one kind::f8f6f4 MMA
constexpr int kGemmThreads = 320;  // 10 warps: producer, MMA, 8 epilogue
constexpr int kEpiWarps = 8;       // two per TMEM lane quarter, each on half the columns
constexpr int kBoxCols = 64;                          // epilogue box: 32 rows x 64 bf16 columns
constexpr int kBoxBytes = 32 * kBoxCols * 2;          // (128-byte rows: whole L2 lines)
constexpr int kBoxesPerWarp = 1;                      // staging boxes per epilogue warp
constexpr int kEpiStagingBytes = kEpiWarps * kBoxesPerWarp * kBoxBytes;

// The pair kernel runs EPI epilogue warps: 8 (two per TMEM lane quarter,
// each on half the columns) where the epilogue is on the critical path --
// tiles of few K blocks, or fewer tiles than pairs -- or 4 (one per quarter,
// on all the columns) where a tile's epilogue hides under the next tile's
// main loop: there the fewer warps took 0.5-3 % off the products (their
// issue slots and their draw on the SM are the main loop's).
template <int EPI>
constexpr int pair_threads() {
  return 64 + 32 * EPI;
}

// Epilogue warps split the BN columns of a tile in two halves when each half
// still holds whole 32-column chunks (and there are two warps a quarter).
template <int BN, int EPI = kEpiWarps>
struct EpiSplit {
  static constexpr int kHalves = EPI == 8 && BN >= 64 ? 2 : 1;
  static constexpr int kCols = BN / kHalves;
};
constexpr int kMaxSplit = 8;

struct GemmParams {
  int M, N, K;          // kernel view: A has M rows, B has N rows, contraction K
  uint32_t idesc;
  const float* inv_a;
  const float* inv_b;
  uint16_t* d;          // bf16 output
  int64_t ldd;          // elements
  int* err;
  // Schedule: tiles [0, t_full) run whole; tiles [t_full, tiles) run as
  // s_tail K slices each.
  int t_full;
  int s_tail;
  float* partials;      // fp32 partials of split tiles (workspace)
  int* tickets;         // per split tile and 32-row group counters (workspace, zero)
  // max |D| over the stored bf16 values, as fp32 bits (nullptr: not wanted),
  // published by the last epilogue warp through two self-cleaning words.
  uint32_t* amax_out;
  uint32_t* amax_acc;
  uint32_t* amax_ticket;
};

// What one work unit does with its accumulator.
enum Role : int {
  kWhole = 0,     // the whole K loop: store bf16
  kSlice = 1,     // one of nsplit K slices of a few-tile GEMM
};

struct Unit {
  int tile, split, nsplit, kb0, kb1, role;
  int prob;  // which GEMM of a two-GEMM launch (0 otherwise)
};

// The n-th work unit of persistent slot `slot` (a CTA, or a CTA pair) out of
// `slots` (round-robin over the units); false when the slot has no n-th
// unit.  All roles of a CTA walk the same sequence.
__device__ __forceinline__ bool unit_at(int slot, int slots, int n, const GemmParams& p,
                                        int num_tiles, int num_kb, Unit& u) {
  const int ui = slot + n * slots;
  if (ui >= p.t_full + (num_tiles - p.t_full) * p.s_tail) return false;
  u.prob = 0;
  if (ui < p.t_full) {
    u.tile = ui;
    u.split = 0;
    u.nsplit = 1;
    u.kb0 = 0;
    u.kb1 = num_kb;
    u.role = kWhole;
  } else {
    const int v = ui - p.t_full;
    u.tile = p.t_full + v / p.s_tail;
    u.split = v % p.s_tail;
    u.nsplit = p.s_tail;
    const int per = (num_kb + p.s_tail - 1) / p.s_tail;
    u.kb0 = u.split * per;
    u.kb1 = min(num_kb, u.kb0 + per);
    u.role = kSlice;
  }
  return true;
}

// Two GEMMs in one launch of the pair kernel, whole tiles only.  Problem 0
// is the one with the longer K loop (cost c0 K blocks a tile, tiles0 tiles),
// problem 1 the other (c1, tiles1).  Problem 0's tiles are dealt round-robin:
// pair p gets L_p = tiles0 / slots (+1 for the first tiles0 % slots pairs, the
// heavy ones).  Each light pair then gets up to `d` of problem 1's tiles
// first (tiles [0, E), E = min(tiles1, light pairs * d), round-robin over the
// light pairs), and the rest of problem 1's tiles go round-robin over all
// pairs, light pairs first.  The host picks d so that the busiest pair's
// K blocks are fewest (d = 0 is plain round-robin).  The same function deals
// the units on the device and checks the deal on the host.
struct GroupSched {
  int tiles0, tiles1, d;
};

__host__ __device__ inline bool unit_at_grouped(int p, int slots, int n, const GroupSched& gs,
                                                int num_kb0, int num_kb1, Unit& u) {
  const int ll = gs.tiles0 / slots, heavy = gs.tiles0 % slots, light = slots - heavy;
  const int e = gs.tiles1 < light * gs.d ? gs.tiles1 : light * gs.d;
  const int r = gs.tiles1 - e;
  u.split = 0;
  u.nsplit = 1;
  u.kb0 = 0;
  u.role = kWhole;
  const int lp = ll + (p < heavy ? 1 : 0);
  if (n < lp) {
    u.prob = 0;
    u.tile = p + n * slots;
    u.kb1 = num_kb0;
    return true;
  }
  int m = n - lp;
  u.prob = 1;
  u.kb1 = num_kb1;
  if (p >= heavy) {
    const int q = p - heavy;
    const int ep = e > q ? (e - q + light - 1) / light : 0;
    if (m < ep) {
      u.tile = q + light * m;
      return true;
    }
    m -= ep;
  }
  const int pos = p >= heavy ? p - heavy : light + p;
  const int rp = r > pos ? (r - pos + slots - 1) / slots : 0;
  if (m < rp) {
    u.tile = e + pos + slots * m;
    return true;
  }
  return false;
}

__device__ __forceinline__ void record_error(int* err, volatile int* abort_flag, int code) {
  atomicCAS(err, 0, code);
  *abort_flag = 1;
}

template <int kChunk>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, uint32_t (&r)[kChunk]) {
  if constexpr (kChunk == 32)
    tmem_load_32cols(taddr, r);
  else
    tmem_load_16cols(taddr, r);
  tmem_load_wait();
}

// Scale two 32-row x 32-column accumulator chunks (this lane's row in ra[]
// and rb[], columns col0..col0+63), convert to bf16, stage them in `box` and
// store the 32 x 64 box at (row0, col0) of D with TMA.  The box's rows are
// 128 bytes -- whole L2 lines of D -- with 16-byte chunks swizzled as the
// 128-byte TMA swizzle expects (chunk ^= row & 7), which also keeps the
// warp's shared-memory writes free of bank conflicts.  Columns beyond D are
// clipped by the store.
template <bool kTrack>
__device__ __forceinline__ void store_pair_tma(const uint32_t (&ra)[32], const uint32_t (&rb)[32],
                                               float alpha, uint8_t* box, const CUtensorMap* tmD,
                                               int row0, int col0, int lane, float& vmax) {
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float v0, v1;
    mul2_rn(ra[2 * j], ra[2 * j + 1], alpha, v0, v1);
    w[j] = cvt_bf16x2(v0, v1);
    if constexpr (kTrack) vmax = fmaxf(vmax, fmaxf(fabsf(v0), fabsf(v1)));
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float v0, v1;
    mul2_rn(rb[2 * j], rb[2 * j + 1], alpha, v0, v1);
    w[16 + j] = cvt_bf16x2(v0, v1);
    if constexpr (kTrack) vmax = fmaxf(vmax, fmaxf(fabsf(v0), fabsf(v1)));
  }
  if (lane == 0) bulk_wait_group_read<kBoxesPerWarp - 1>();  // this box's last store has read it
  __syncwarp();
  uint8_t* rowp = box + lane * 128;
  const int sw = lane & 7;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4*>(rowp + ((q ^ sw) << 4)) =
        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmD, box, col0, row0);
    bulk_commit_group();
  }
}

// One 32-column chunk of a K-split tile's reduced sums (this lane's row),
// scaled, rounded to bf16 and stored straight from registers: 16-byte
// stores, 16 columns at a time inside D (N is a multiple of 16).
template <bool kTrack>
__device__ __forceinline__ void store_chunk_direct(const float (&acc)[32], float alpha,
                                                   const GemmParams& p, int row, int col0,
                                                   float& vmax) {
  if (row >= p.M) return;
  uint16_t* dst = p.d + static_cast<int64_t>(row) * p.ldd + col0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (col0 + 16 * h >= p.N) break;
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float v0 = __fmul_rn(acc[16 * h + 2 * j], alpha);
      const float v1 = __fmul_rn(acc[16 * h + 2 * j + 1], alpha);
      w[j] = cvt_bf16x2(v0, v1);
      if constexpr (kTrack) vmax = fmaxf(vmax, fmaxf(fabsf(v0), fabsf(v1)));
    }
    *reinterpret_cast<uint4*>(dst + 16 * h) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(dst + 16 * h + 8) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// Final bf16 output of raw fp32 accumulators (this lane's row): two
// consecutive 32-column chunks ra, rb at col0 (TMA store of a 32 x 64 box),
// or, with kTransStore, one chunk ra of kChunk columns stored transposed.
// When D's amax is wanted (p.amax_out, warp-uniform), vmax collects the
// largest |v| of the fp32 values before their rounding to bf16: rounding to
// nearest even is monotone and odd, so max |bf16(v)| = bf16(max |v|), and one
// rounding at the end gives the amax of the stored bf16 D exactly.  Elements
// outside D come from zero-filled operand rows or columns, hence are zero and
// cannot raise it.
template <int kChunk, bool kTransStore>
__device__ __forceinline__ void emit(const uint32_t (&ra)[kChunk], const uint32_t (&rb)[kChunk],
                                     float alpha, const GemmParams& p, const CUtensorMap* tmD,
                                     uint8_t* boxes, uint32_t& box_no, int row0, int col0, int lane,
                                     float& vmax) {
  const bool track = p.amax_out != nullptr;
  if constexpr (!kTransStore) {
    static_assert(kChunk == 32, "TMA-store epilogue works on pairs of 32-column chunks");
    uint8_t* box = boxes + (box_no % kBoxesPerWarp) * kBoxBytes;
    if (track)  // warp-uniform; the untracked store carries no max at all
      store_pair_tma<true>(ra, rb, alpha, box, tmD, row0, col0, lane, vmax);
    else
      store_pair_tma<false>(ra, rb, alpha, box, tmD, row0, col0, lane, vmax);
    ++box_no;
  } else {
    // kernel element (row, col) is output element (col, row)
    const int row = row0 + lane;
    if (row < p.M) {
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        if (col0 + j < p.N) {
          const float v = __fmul_rn(__uint_as_float(ra[j]), alpha);
          const uint32_t b = cvt_bf16x2(v, 0.0f) & 0xFFFFu;
          p.d[static_cast<int64_t>(col0 + j) * p.ldd + row] = static_cast<uint16_t>(b);
          if (track) vmax = fmaxf(vmax, fabsf(v));
        }
      }
    }
  }
}

// Partial of one (slice, 32-row group): chunk c is stored as [c][q][lane][4]
// floats so a warp's 16-byte stores and loads are contiguous.
template <int kChunk>
__device__ __forceinline__ void store_partial(float* region, int c, const uint32_t (&r)[kChunk],
                                              int lane) {
#pragma unroll
  for (int q = 0; q < kChunk / 4; ++q)
    __stcg(reinterpret_cast<float4*>(region + ((c * (kChunk / 4) + q) * 32 + lane) * 4),
           make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                       __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
}

template <int kChunk>
__device__ __forceinline__ void add_partial(const float* region, int c, float (&acc)[kChunk],
                                            int lane) {
#pragma unroll
  for (int q = 0; q < kChunk / 4; ++q) {
    const float4 v =
        __ldcg(reinterpret_cast<const float4*>(region + ((c * (kChunk / 4) + q) * 32 + lane) * 4));
    acc[4 * q] += v.x;
    acc[4 * q + 1] += v.y;
    acc[4 * q + 2] += v.z;
    acc[4 * q + 3] += v.w;
  }
}

__device__ __forceinline__ int ld_acquire_int(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Epilogue of one work unit for one warp: 32 rows (row0..row0+31) x BN
// columns starting at col_base, accumulator at TMEM address t_row.  `group`
// identifies the 32-row group inside the tile (G groups per tile).  Arrives on
// the accumulator-empty barrier (via `release`) as soon as TMEM is read.
//
// A K slice of a split tail tile writes its raw fp32 partial, announces it on
// the group's ticket, waits (bounded) until all S slices have done so, then
// reduces its own 1/S share of the columns: every slice sums all S partials
// of those columns in slice order (deterministic) and stores the bf16
// result.  The slices of a tail tile run on distinct CTAs as their last unit,
// all resident at once, so the wait cannot block on itself.  The last slice to
// finish clears both counters for the next call.
template <int kCols, bool kTransStore, typename Release>
__device__ __forceinline__ void epilogue_unit(const GemmParams& p, const Unit& u, int G,
                                              int group, int row0, int col_base, uint32_t t_row,
                                              float alpha, const CUtensorMap* tmD, uint8_t* boxes,
                                              uint32_t& box_no, int lane,
                                              volatile int* abort_flag, float& vmax,
                                              Release release) {
  constexpr int kChunk = (kCols % 32 == 0) ? 32 : 16;
  const bool active = row0 < p.M;  // warp-uniform
  int nch = 0;                     // chunks with at least one column inside D
  while (nch < kCols / kChunk && col_base + nch * kChunk < p.N) ++nch;
  if (u.role == kWhole) {
    if (active && nch > 0) {
      // Two chunks per iteration, loaded from TMEM together.  The TMA store
      // takes them as one 32 x 64 box; a chunk past the last one inside D
      // (nch odd) is not loaded, and its half of the box is clipped.
      uint32_t ra[kChunk], rb[kChunk];
#pragma unroll 1
      for (int c = 0; c < nch; c += 2) {
        if (c + 1 < nch) {
          if constexpr (kChunk == 32) {
            tmem_load_32cols(t_row + c * kChunk, ra);
            tmem_load_32cols(t_row + (c + 1) * kChunk, rb);
          } else {
            tmem_load_16cols(t_row + c * kChunk, ra);
            tmem_load_16cols(t_row + (c + 1) * kChunk, rb);
          }
          tmem_load_wait();
          if constexpr (kTransStore) {
            emit<kChunk, true>(ra, ra, alpha, p, tmD, boxes, box_no, row0, col_base + c * kChunk,
                               lane, vmax);
            emit<kChunk, true>(rb, rb, alpha, p, tmD, boxes, box_no, row0,
                               col_base + (c + 1) * kChunk, lane, vmax);
          } else {
            emit<kChunk, false>(ra, rb, alpha, p, tmD, boxes, box_no, row0, col_base + c * kChunk,
                                lane, vmax);
          }
        } else {
          tmem_load_chunk<kChunk>(t_row + c * kChunk, ra);
#pragma unroll
          for (int j = 0; j < kChunk; ++j) rb[j] = 0u;
          emit<kChunk, kTransStore>(ra, rb, alpha, p, tmD, boxes, box_no, row0,
                                    col_base + c * kChunk, lane, vmax);
        }
      }
    }
    release();
    return;
  }
  const size_t region_floats = static_cast<size_t>(32) * kCols;
  const int tail_tile = u.tile - p.t_full;
  float* mine = p.partials + ((static_cast<size_t>(tail_tile) * u.nsplit + u.split) * G + group) *
                                 region_floats;
  if (active) {
    uint32_t ra[kChunk], rb[kChunk];
#pragma unroll 1
    for (int c = 0; c < nch; c += 2) {
      if (c + 1 < nch) {
        if constexpr (kChunk == 32) {
          tmem_load_32cols(t_row + c * kChunk, ra);
          tmem_load_32cols(t_row + (c + 1) * kChunk, rb);
        } else {
          tmem_load_16cols(t_row + c * kChunk, ra);
          tmem_load_16cols(t_row + (c + 1) * kChunk, rb);
        }
        tmem_load_wait();
        store_partial<kChunk>(mine, c, ra, lane);
        store_partial<kChunk>(mine, c + 1, rb, lane);
      } else {
        tmem_load_chunk<kChunk>(t_row + c * kChunk, ra);
        store_partial<kChunk>(mine, c, ra, lane);
      }
    }
  }
  release();
  if (!active) return;
  __threadfence();
  __syncwarp();
  int* ticket = p.tickets + 2 * (tail_tile * G + group);
  int* done = ticket + 1;
  bool all_in = true;
  if (lane == 0) {
    atomicAdd(ticket, 1);
    if (ld_acquire_int(ticket) < u.nsplit) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_int(ticket) < u.nsplit) {
        if (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs) {
          all_in = false;
          break;
        }
        __nanosleep(64);
      }
    }
  }
  all_in = __shfl_sync(0xFFFFFFFFu, all_in ? 1 : 0, 0) != 0;
  if (!all_in) {
    if (lane == 0) record_error(p.err, abort_flag, kErrGemmEpilogueWait);
    return;
  }
  __threadfence();
  // This slice's share of the chunks.
  const int share = (nch + u.nsplit - 1) / u.nsplit;
  const int c_lo = u.split * share;
  const int c_hi = min(nch, c_lo + share);
  const bool track = p.amax_out != nullptr;  // warp-uniform
#pragma unroll 1
  for (int c = c_lo; c < c_hi; ++c) {
    float acc[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) acc[j] = 0.0f;
    for (int s2 = 0; s2 < u.nsplit; ++s2) {  // fixed slice order: deterministic sums
      const float* region =
          p.partials + ((static_cast<size_t>(tail_tile) * u.nsplit + s2) * G + group) *
                           region_floats;
      add_partial<kChunk>(region, c, acc, lane);
    }
    if constexpr (kTransStore) {
      uint32_t r[kChunk];
#pragma unroll
      for (int j = 0; j < kChunk; ++j) r[j] = __float_as_uint(acc[j]);
      emit<kChunk, true>(r, r, alpha, p, tmD, boxes, box_no, row0, col_base + c * kChunk, lane,
                         vmax);
    } else if (track) {
      store_chunk_direct<true>(acc, alpha, p, row0 + lane, col_base + c * kChunk, vmax);
    } else {
      store_chunk_direct<false>(acc, alpha, p, row0 + lane, col_base + c * kChunk, vmax);
    }
  }
  __syncwarp();
  if (lane == 0) {
    // Everyone has read the ticket before anyone can finish: the last to
    // finish may clear both counters.
    if (atomicAdd(done, 1) == u.nsplit - 1) {
      atomicExch(ticket, 0);
      atomicExch(done, 0);
    }
  }
}

// Every epilogue warp of the grid arrives here once, after its last unit:
// the warp's maximum, rounded to bf16 as D was, joins the grid's through an
// atomic max on the workspace accumulator, and the last warp to arrive
// publishes it to p.amax_out and clears both words for the next call.  A bf16
// bit pattern shifted up by 16 is the fp32 bit pattern of the same value, and
// non-negative values order like their bits.
__device__ __forceinline__ void publish_amax(const GemmParams& p, float vmax, int lane,
                                             unsigned epi_warps = kEpiWarps) {
  if (p.amax_out == nullptr) return;
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, cvt_bf16x2(vmax, 0.0f) & 0xFFFFu);
  if (lane == 0) {
    atomicMax(p.amax_acc, m << 16);
    __threadfence();
    if (atomicAdd(p.amax_ticket, 1u) == gridDim.x * epi_warps - 1u) {
      __threadfence();
      *p.amax_out = atomicExch(p.amax_acc, 0u);
      atomicExch(p.amax_ticket, 0u);
    }
  }
}

// ------------------------------------------------------------------ one-CTA kernel

template <int BN, int STAGES>
struct Cfg {
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN <= 32    ? 32
                                   : 2 * BN <= 64  ? 64
                                   : 2 * BN <= 128 ? 128
                                   : 2 * BN <= 256 ? 256
                                                   : 512;
  static constexpr int kBarrierBytes = 256;
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(STAGES) * kStageBytes + kEpiStagingBytes + kBarrierBytes;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128");
  static_assert(kBBytes % 1024 == 0, "B tiles keep 1024-byte alignment");
};

template <int BN, int STAGES, bool kTransStore>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  using C = Cfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::kABytes;
  uint8_t* sEpi = sB + STAGES * C::kBBytes;  // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(sEpi + kEpiStagingBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* drain = acc_empty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_n = (p.N + BN - 1) / BN;
  const int num_tiles = ((p.M + kBM - 1) / kBM) * num_n;
  const int num_kb = (p.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    if (!kTransStore) tma_prefetch_map(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();               // operands, scales and D are ready / free
  griddep_launch_dependents();  // the next kernel may start its prologue on freed SMs

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t fills[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) fills[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Unit u;
      for (int n = 0; ok && unit_at(blockIdx.x, gridDim.x, n, p, num_tiles, num_kb, u); ++n) {
        const int m_blk = u.tile / num_n, n_blk = u.tile % num_n;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          tma_load_2d(sA + stage * C::kABytes, &tmA, &full[stage], kb * kBK, m_blk * kBM);
          tma_load_2d(sB + stage * C::kBBytes, &tmB, &full[stage], kb * kBK, n_blk * BN);
#pragma unroll
          for (int s = 0; s < STAGES; ++s)
            if (s == stage) ++fills[s];
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        record_error(p.err, abort_flag, kErrGemmProducerWait);
        // Let this thread's copies in flight land before the CTA exits.
        volatile int never = 0;
#pragma unroll
        for (int s = 0; s < STAGES; ++s)
          if (fills[s] > 0) mbar_wait_bounded(&full[s], (fills[s] - 1) & 1u, &never);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      Unit u;
      for (int n = 0; ok && unit_at(blockIdx.x, gridDim.x, n, p, num_tiles, num_kb, u); ++n) {
        if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t a_desc = smem_desc_k_sw128(smem_addr(sA + stage * C::kABytes));
          const uint64_t b_desc = smem_desc_k_sw128(smem_addr(sB + stage * C::kBBytes));
#pragma unroll
          for (int k = 0; k < kBK / kMmaK; ++k) {
            // advance the start address by k * 32 bytes (encoded >> 4)
            mma_f8f6f4(d_tmem, a_desc + static_cast<uint64_t>(k * (kMmaK >> 4)),
                       b_desc + static_cast<uint64_t>(k * (kMmaK >> 4)), p.idesc,
                       (kb > u.kb0 || k > 0) ? 1u : 0u);
          }
          issued = true;
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        record_error(p.err, abort_flag, kErrGemmMmaWait);
        if (issued) {
          // Wait for this thread's MMAs in flight before TMEM is freed.
          volatile int never = 0;
          mma_commit(drain);
          mbar_wait_bounded(drain, 0, &never);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    using E = EpiSplit<BN>;
    const int quarter = warp & 3;        // TMEM lanes this warp may read: 32*quarter..+31
    const int half = (warp - 2) >> 2;    // which half of the columns (0 or 1)
    const bool has_cols = half < E::kHalves;
    const float alpha = __fmul_rn(*p.inv_a, *p.inv_b);
    uint8_t* boxes = sEpi + (warp - 2) * kBoxesPerWarp * kBoxBytes;
    uint32_t box_no = 0;
    float vmax = 0.0f;
    int acc = 0;
    uint32_t acc_phase = 0;
    Unit u;
    for (int n = 0; unit_at(blockIdx.x, gridDim.x, n, p, num_tiles, num_kb, u); ++n) {
      const int m_blk = u.tile / num_n, n_blk = u.tile % num_n;
      // tcgen05.ld below is warp-collective: take the decision warp-uniformly.
      const bool ready = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&acc_full[acc], acc_phase,
                                                                  abort_flag));
      if (!ready) {
        if (lane == 0) record_error(p.err, abort_flag, kErrGemmEpilogueWait);
        break;
      }
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * BN + half * E::kCols);
      const int acc_now = acc;
      auto release = [&] {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc_now]);
      };
      if (has_cols)
        epilogue_unit<E::kCols, kTransStore>(p, u, 4 * E::kHalves, half * 4 + quarter,
                                             m_blk * kBM + quarter * 32,
                                             n_blk * BN + half * E::kCols, t_row, alpha, &tmD,
                                             boxes, box_no, lane, abort_flag, vmax, release);
      else
        release();
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    publish_amax(p, vmax, lane);
    if (lane == 0) bulk_wait_group<0>();  // stores done before the staging memory goes away
  }

  __syncwarp();  // reconverge the producer / MMA warps around their elected lane
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ CTA-pair kernel
//
// Two CTAs of a cluster share one 256 x BN tile: each CTA loads 128 rows of
// A and BN/2 rows of B per stage (so a stage is 16 KB + BN/2 * 128 B per
// CTA instead of 16 KB + BN * 128 B), and the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256) reading both CTAs' shared memory; each
// CTA's TMEM receives its 128 rows of the accumulator.
//   full[s]      lives in the even CTA; both CTAs' TMA loads count their
//                bytes on it (the even producer arms it for both);
//   empty[s]     one per CTA; the MMA commit arrives on both (multicast);
//   acc_full[a]  one per CTA; the MMA commit arrives on both (multicast);
//   acc_empty[a] lives in the even CTA; all 8 epilogue warps arrive on it.
// Every wait is a CTA-scope acquire, although peers arrive on full[] and
// acc_empty[]: what a wait orders is carried by other means.  TMA data is
// visible once the barrier's transaction count completes; MMA completion is
// what the tcgen05.commit arrive signals; and TMEM reuse is ordered by the
// tcgen05.fence before/after-thread-sync pair around the epilogue's release
// arrive.  A cluster-scope acquire would add a memory fence to each wait.

template <int BN, int STAGES>
struct PairCfg {
  static constexpr int kABytes = kBM * kBK;             // 128 rows of A per CTA
  static constexpr int kBBytes = (BN / 2) * kBK;        // BN/2 rows of B per CTA
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN <= 256 ? 256 : 512;
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(STAGES) * kStageBytes + kEpiStagingBytes + 256;
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "MMA N for M=256");
  static_assert(kBBytes % 1024 == 0, "B tiles keep 1024-byte alignment");
};

// The pair kernel's body; kGrouped runs two GEMMs in one launch (problem 1:
// tmA1 / tmB1 / tmD1 / p1, dealt with problem 0's tiles by unit_at_grouped).
template <int BN, int STAGES, bool kGrouped, int EPI>
__device__ __forceinline__ void pair_gemm_body(const CUtensorMap* tmA0, const CUtensorMap* tmB0,
                                               const CUtensorMap* tmD0, const GemmParams& p,
                                               const CUtensorMap* tmA1, const CUtensorMap* tmB1,
                                               const CUtensorMap* tmD1, const GemmParams& p1,
                                               const GroupSched& gs) {
  using C = PairCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::kABytes;
  uint8_t* sEpi = sB + STAGES * C::kBBytes;  // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(sEpi + kEpiStagingBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* drain = acc_empty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // Written by the peer CTA just before the closing cluster barrier: whether
  // it gave up anywhere, and (odd CTA -> even CTA) how many loads its
  // producer issued into each stage.
  volatile uint32_t* peer_abort = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
  volatile uint32_t* peer_fills = peer_abort + 1;       // [STAGES]
  volatile uint32_t* own_fills = peer_fills + STAGES;   // [STAGES] this CTA's producer's
  static_assert(sizeof(uint64_t) * (2 * STAGES + 5) + sizeof(uint32_t) * (3 + 2 * STAGES) <= 256,
                "barrier block");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();      // 0: issues the MMAs
  const int pair = static_cast<int>(cluster_id_x());
  const int num_pairs = static_cast<int>(cluster_count_x());
  const int num_n = (p.N + BN - 1) / BN;
  const int num_tiles = ((p.M + 2 * kBM - 1) / (2 * kBM)) * num_n;
  const int num_kb = (p.K + kBK - 1) / kBK;
  const int num_n1 = kGrouped ? (p1.N + BN - 1) / BN : num_n;
  const int num_kb1 = kGrouped ? (p1.K + kBK - 1) / kBK : num_kb;
  auto next_unit = [&](int n, Unit& u) -> bool {
    if constexpr (kGrouped)
      return unit_at_grouped(pair, num_pairs, n, gs, num_kb, num_kb1, u);
    else
      return unit_at(pair, num_pairs, n, p, num_tiles, num_kb, u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 2 * EPI);  // every epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *peer_abort = 0;
    for (int s = 0; s < STAGES; ++s) peer_fills[s] = own_fills[s] = 0;
    fence_barrier_init();
    tma_prefetch_map(tmA0);
    tma_prefetch_map(tmB0);
    tma_prefetch_map(tmD0);
    if (kGrouped) {
      tma_prefetch_map(tmA1);
      tma_prefetch_map(tmB1);
      tma_prefetch_map(tmD1);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();               // operands, scales and D are ready / free
  griddep_launch_dependents();  // the next kernel may start its prologue on freed SMs

  if (warp == 0) {
    // ------------------------------------------------------------ producers (both CTAs)
    if (lane == 0) {
      uint32_t fills[STAGES];  // loads issued into each stage
#pragma unroll
      for (int s = 0; s < STAGES; ++s) fills[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Unit u;
      for (int n = 0; ok && next_unit(n, u); ++n) {
        const bool second = kGrouped && u.prob != 0;
        const int nn = second ? num_n1 : num_n;
        const int m_blk = u.tile / nn, n_blk = u.tile % nn;
        const CUtensorMap* tmA = second ? tmA1 : tmA0;
        const CUtensorMap* tmB = second ? tmB1 : tmB0;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t full_even = map_to_cta(smem_addr(&full[stage]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
          tma_load_2d_pair(sA + stage * C::kABytes, tmA, full_even, kb * kBK,
                           m_blk * 2 * kBM + static_cast<int>(rank) * kBM);
          tma_load_2d_pair(sB + stage * C::kBBytes, tmB, full_even, kb * kBK,
                           n_blk * BN + static_cast<int>(rank) * (BN / 2));
#pragma unroll
          for (int s = 0; s < STAGES; ++s)
            if (s == stage) ++fills[s];
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) record_error(p.err, abort_flag, kErrGemmProducerWait);
      // The even CTA's full[] barriers count the odd CTA's loads too: only
      // the even CTA can tell that they have landed (see the end).
      if (rank == 1) {
        const uint32_t even_fills = map_to_cta(smem_addr(const_cast<uint32_t*>(peer_fills)), 0);
#pragma unroll
        for (int s = 0; s < STAGES; ++s) st_shared_cluster_u32(even_fills + 4u * s, fills[s]);
      } else {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) own_fills[s] = fills[s];
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      Unit u;
      for (int n = 0; ok && next_unit(n, u); ++n) {
        const uint32_t idesc = (kGrouped && u.prob != 0) ? p1.idesc : p.idesc;
        if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t a_desc = smem_desc_k_sw128(smem_addr(sA + stage * C::kABytes));
          const uint64_t b_desc = smem_desc_k_sw128(smem_addr(sB + stage * C::kBBytes));
#pragma unroll
          for (int k = 0; k < kBK / kMmaK; ++k) {
            mma_f8f6f4_pair(d_tmem, a_desc + static_cast<uint64_t>(k * (kMmaK >> 4)),
                            b_desc + static_cast<uint64_t>(k * (kMmaK >> 4)), idesc,
                            (kb > u.kb0 || k > 0) ? 1u : 0u);
          }
          issued = true;
          mma_commit_pair_multicast(&empty[stage], 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_multicast(&acc_full[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        record_error(p.err, abort_flag, kErrGemmMmaWait);
        if (issued) {
          volatile int never = 0;
          mma_commit_pair_multicast(drain, 0x1);
          mbar_wait_bounded(drain, 0, &never);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    using E = EpiSplit<BN, EPI>;
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // 0 for every warp when EPI == 4
    const float alpha0 = __fmul_rn(*p.inv_a, *p.inv_b);
    const float alpha1 = kGrouped ? __fmul_rn(*p1.inv_a, *p1.inv_b) : alpha0;
    const uint32_t acc_empty_even0 = map_to_cta(smem_addr(&acc_empty[0]), 0);
    uint8_t* boxes = sEpi + (warp - 2) * kBoxesPerWarp * kBoxBytes;
    uint32_t box_no = 0;
    float vmax0 = 0.0f, vmax1 = 0.0f;
    int acc = 0;
    uint32_t acc_phase = 0;
    Unit u;
    for (int n = 0; next_unit(n, u); ++n) {
      const bool second = kGrouped && u.prob != 0;
      const GemmParams& pu = second ? p1 : p;
      const int nn = second ? num_n1 : num_n;
      const int m_blk = u.tile / nn, n_blk = u.tile % nn;
      const bool ready = __all_sync(
          0xFFFFFFFFu, mbar_wait_bounded(&acc_full[acc], acc_phase, abort_flag));
      if (!ready) {
        if (lane == 0) record_error(p.err, abort_flag, kErrGemmEpilogueWait);
        break;
      }
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * BN + half * E::kCols);
      const int row_group = static_cast<int>(rank) * 4 + quarter;
      const uint32_t release_addr = acc_empty_even0 + static_cast<uint32_t>(acc * 8);
      epilogue_unit<E::kCols, false>(pu, u, 8 * E::kHalves, half * 8 + row_group,
                                     m_blk * 2 * kBM + row_group * 32, n_blk * BN + half * E::kCols,
                                     t_row, second ? alpha1 : alpha0, second ? tmD1 : tmD0, boxes,
                                     box_no, lane, abort_flag, second ? vmax1 : vmax0,
                                     [&] {
                                       tc_fence_before_sync();
                                       __syncwarp();
                                       if (lane == 0) mbar_arrive_cluster(release_addr);
                                     });
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    publish_amax(p, vmax0, lane, EPI);
    if (kGrouped) publish_amax(p1, vmax1, lane, EPI);  // (at most one of the two asks for it)
    if (lane == 0) bulk_wait_group<0>();  // stores done before the staging memory goes away
  }

  __syncwarp();
  __syncthreads();  // every role of this CTA is done: its abort flag is final
  if (threadIdx.x == 0)
    st_shared_cluster_u32(map_to_cta(smem_addr(const_cast<uint32_t*>(peer_abort)), rank ^ 1u),
                          *abort_flag != 0 ? 1u : 0u);
  tc_fence_before_sync();
  cluster_sync_all();  // no CTA leaves while its peer may still read its shared memory
  // Both CTAs take the same decision from the two flags.  Without a failure
  // every load has been consumed by an MMA, so it has landed.  After one, a
  // producer may have stopped with loads in flight, and the two producers
  // may have stopped one phase apart on a stage (each waits for the same MMA
  // commits, so neither gets further ahead).  The even CTA, whose full[]
  // barriers count both CTAs' bytes, balances each stage's last phase -- it
  // arms a phase only the odd CTA loaded into, and completes the bytes of one
  // the odd CTA never loaded -- then waits (bounded) for that phase; every
  // earlier phase of a stage has completed already.  The second cluster
  // barrier keeps the odd CTA until then.
  if (*abort_flag != 0 || *peer_abort != 0) {
    if (rank == 0 && threadIdx.x == 0) {
      volatile int never = 0;
#pragma unroll
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t fe = own_fills[s], fo = peer_fills[s];
        if (fo > fe) mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        if (fe > fo) mbar_complete_tx(&full[s], C::kStageBytes);
        const uint32_t last = fe > fo ? fe : fo;
        if (last > 0) mbar_wait_bounded(&full[s], (last - 1) & 1u, &never);
      }
    }
    cluster_sync_all();
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(pair_threads<EPI>(), 1)
    gemm_fp8_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmD,
                         const __grid_constant__ GemmParams p) {
  pair_gemm_body<BN, STAGES, false, EPI>(&tmA, &tmB, &tmD, p, &tmA, &tmB, &tmD, p,
                                         GroupSched{0, 0, 0});
}

// Two GEMMs of the same tile shape in one launch (see unit_at_grouped).
template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(pair_threads<EPI>(), 1)
    gemm_fp8_pair2_kernel(const __grid_constant__ CUtensorMap tmA0,
                          const __grid_constant__ CUtensorMap tmB0,
                          const __grid_constant__ CUtensorMap tmD0,
                          const __grid_constant__ GemmParams p0,
                          const __grid_constant__ CUtensorMap tmA1,
                          const __grid_constant__ CUtensorMap tmB1,
                          const __grid_constant__ CUtensorMap tmD1,
                          const __grid_constant__ GemmParams p1,
                          const __grid_constant__ GroupSched gs) {
  pair_gemm_body<BN, STAGES, true, EPI>(&tmA0, &tmB0, &tmD0, p0, &tmA1, &tmB1, &tmD1, p1, gs);
}

}  // namespace
}  // namespace fp8lin
