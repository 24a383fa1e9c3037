// gemm_tcgen05.cu -- FP8 GEMM of the fp8 Linear on the 5th-generation tensor
// cores (sm_103a): D[m, n] = bf16((sum_k A[m, k] * B[n, k]) * inv_a * inv_b)
// with both operands K-major 8-bit (e4m3 or e5m2) and fp32 accumulation in
// tensor memory.  The three products of the Linear's forward and backward
// ("Why swapping nn.Linear with FP8Linear brings throughput decrease for 7B
// LLAMA2-like model?", pytorch/ao issue 1199: the FP8Linear that replaces
// nn.Linear) all take this form once the transposed fp8 copies exist.
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: 128-byte-swizzled K-major tiles of A (128 rows)
//               and B (BN rows), 128 bytes of K per stage, STAGES-deep ring;
//   warp 1      allocates TMEM (two BN-column fp32 accumulators) and one
//               elected lane issues tcgen05.mma.kind::f8f6f4 (M=128, N=BN,
//               K=32 per instruction), committing each stage back to the
//               producer and each finished accumulator to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld of their 32 TMEM lanes, multiply by
//               alpha = inv_a * inv_b, convert to bf16, 16-byte stores.
// The double-buffered accumulator lets the epilogue of tile i overlap the
// main loop of tile i+1.  For a handful of rows (small token counts) the
// operands are swapped so the weight fills the 128-row MMA and the epilogue
// stores the transposed result.
//
// Every wait on an mbarrier is bounded (kWaitLimitNs); a wait that runs out
// records an error code in the workspace, raises a CTA-wide abort flag, lets
// its own copies / MMAs in flight finish (bounded), frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace fp8lin {
namespace {

constexpr int kBM = 128;           // tile rows (MMA M)
constexpr int kBK = 128;           // bytes (= 8-bit elements) of K per stage
constexpr int kMmaK = 32;          // K of one kind::f8f6f4 MMA
constexpr int kGemmThreads = 192;  // 6 warps

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
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * kStageBytes + kBarrierBytes;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128");
  static_assert(kBBytes % 1024 == 0, "B tiles keep 1024-byte alignment");
};

struct GemmParams {
  int M, N, K;          // kernel view: A has M rows, B has N rows, contraction K
  uint32_t idesc;
  const float* inv_a;
  const float* inv_b;
  uint16_t* d;          // bf16 output
  int64_t ldd;          // elements
  int* err;
};

__device__ __forceinline__ void record_error(int* err, volatile int* abort_flag, int code) {
  atomicCAS(err, 0, code);
  *abort_flag = 1;
}

template <int BN, int STAGES, bool kTransStore>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
  using C = Cfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * C::kBBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* drain = acc_empty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (p.M + kBM - 1) / kBM;
  const int num_n = (p.N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = (p.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t fills[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) fills[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int m_blk = tile / num_n, n_blk = tile % num_n;
        for (int kb = 0; kb < num_kb; ++kb) {
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
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
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
                       (kb > 0 || k > 0) ? 1u : 0u);
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
    const int quarter = warp & 3;  // TMEM lanes this warp may read: 32*quarter..+31
    const float alpha = __fmul_rn(*p.inv_a, *p.inv_b);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int m_blk = tile / num_n, n_blk = tile % num_n;
      // tcgen05.ld below is warp-collective: take the decision warp-uniformly.
      const bool ready = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&acc_full[acc], acc_phase,
                                                                  abort_flag));
      if (!ready) {
        if (lane == 0) record_error(p.err, abort_flag, kErrGemmEpilogueWait);
        break;
      }
      tc_fence_after_sync();
      const int row = m_blk * kBM + quarter * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      constexpr int kChunk = (BN % 32 == 0) ? 32 : 16;
#pragma unroll 1
      for (int c = 0; c < BN / kChunk; ++c) {
        float v[kChunk];
        if constexpr (kChunk == 32) {
          uint32_t r[32];
          tmem_load_32cols(t_row + c * 32, r);
          tmem_load_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), alpha);
        } else {
          uint32_t r[16];
          tmem_load_16cols(t_row + c * 16, r);
          tmem_load_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), alpha);
        }
        const int col0 = n_blk * BN + c * kChunk;
        if (row < p.M) {
          if constexpr (!kTransStore) {
            uint16_t* dst = p.d + static_cast<int64_t>(row) * p.ldd + col0;
#pragma unroll
            for (int g = 0; g < kChunk / 8; ++g) {
              if (col0 + g * 8 + 8 <= p.N) {
                uint4 w;
                w.x = cvt_bf16x2(v[g * 8 + 0], v[g * 8 + 1]);
                w.y = cvt_bf16x2(v[g * 8 + 2], v[g * 8 + 3]);
                w.z = cvt_bf16x2(v[g * 8 + 4], v[g * 8 + 5]);
                w.w = cvt_bf16x2(v[g * 8 + 6], v[g * 8 + 7]);
                *reinterpret_cast<uint4*>(dst + g * 8) = w;
              }
            }
          } else {
            // kernel element (row, col) is output element (col, row)
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
              if (col0 + j < p.N) {
                const uint32_t b = cvt_bf16x2(v[j], 0.0f) & 0xFFFFu;
                p.d[static_cast<int64_t>(col0 + j) * p.ldd + row] = static_cast<uint16_t>(b);
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
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

template <int BN, int STAGES>
struct PairCfg {
  static constexpr int kABytes = kBM * kBK;             // 128 rows of A per CTA
  static constexpr int kBBytes = (BN / 2) * kBK;        // BN/2 rows of B per CTA
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN <= 256 ? 256 : 512;
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * kStageBytes + 256;
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "MMA N for M=256");
  static_assert(kBBytes % 1024 == 0, "B tiles keep 1024-byte alignment");
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_fp8_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using C = PairCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * C::kBBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* drain = acc_empty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();      // 0: issues the MMAs
  const int pair = static_cast<int>(cluster_id_x());
  const int num_pairs = static_cast<int>(cluster_count_x());
  const int num_m = (p.M + 2 * kBM - 1) / (2 * kBM);
  const int num_n = (p.N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = (p.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 8);  // 4 epilogue warps x 2 CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producers (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs) {
        const int m_blk = tile / num_n, n_blk = tile % num_n;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_cluster_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t full_even = map_to_cta(smem_addr(&full[stage]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
          tma_load_2d_pair(sA + stage * C::kABytes, &tmA, full_even, kb * kBK,
                           m_blk * 2 * kBM + static_cast<int>(rank) * kBM);
          tma_load_2d_pair(sB + stage * C::kBBytes, &tmB, full_even, kb * kBK,
                           n_blk * BN + static_cast<int>(rank) * (BN / 2));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) record_error(p.err, abort_flag, kErrGemmProducerWait);
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
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs) {
        if (!mbar_wait_cluster_bounded(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_cluster_bounded(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t a_desc = smem_desc_k_sw128(smem_addr(sA + stage * C::kABytes));
          const uint64_t b_desc = smem_desc_k_sw128(smem_addr(sB + stage * C::kBBytes));
#pragma unroll
          for (int k = 0; k < kBK / kMmaK; ++k) {
            mma_f8f6f4_pair(d_tmem, a_desc + static_cast<uint64_t>(k * (kMmaK >> 4)),
                            b_desc + static_cast<uint64_t>(k * (kMmaK >> 4)), p.idesc,
                            (kb > 0 || k > 0) ? 1u : 0u);
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
    const int quarter = warp & 3;
    const float alpha = __fmul_rn(*p.inv_a, *p.inv_b);
    const uint32_t acc_empty_even0 = map_to_cta(smem_addr(&acc_empty[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs) {
      const int m_blk = tile / num_n, n_blk = tile % num_n;
      const bool ready = __all_sync(
          0xFFFFFFFFu, mbar_wait_cluster_bounded(&acc_full[acc], acc_phase, abort_flag));
      if (!ready) {
        if (lane == 0) record_error(p.err, abort_flag, kErrGemmEpilogueWait);
        break;
      }
      tc_fence_after_sync();
      const int row = m_blk * 2 * kBM + static_cast<int>(rank) * kBM + quarter * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_load_32cols(t_row + c * 32, r);
        tmem_load_wait();
        const int col0 = n_blk * BN + c * 32;
        if (row < p.M) {
          uint16_t* dst = p.d + static_cast<int64_t>(row) * p.ldd + col0;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (col0 + g * 8 + 8 <= p.N) {
              uint4 w;
              w.x = cvt_bf16x2(__fmul_rn(__uint_as_float(r[g * 8 + 0]), alpha),
                               __fmul_rn(__uint_as_float(r[g * 8 + 1]), alpha));
              w.y = cvt_bf16x2(__fmul_rn(__uint_as_float(r[g * 8 + 2]), alpha),
                               __fmul_rn(__uint_as_float(r[g * 8 + 3]), alpha));
              w.z = cvt_bf16x2(__fmul_rn(__uint_as_float(r[g * 8 + 4]), alpha),
                               __fmul_rn(__uint_as_float(r[g * 8 + 5]), alpha));
              w.w = cvt_bf16x2(__fmul_rn(__uint_as_float(r[g * 8 + 6]), alpha),
                               __fmul_rn(__uint_as_float(r[g * 8 + 7]), alpha));
              *reinterpret_cast<uint4*>(dst + g * 8) = w;
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_even0 + static_cast<uint32_t>(acc * 8));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncwarp();
  tc_fence_before_sync();
  cluster_sync_all();  // no CTA leaves while its peer may still read its shared memory
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

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

// 2-D map over an 8-bit [rows, k] matrix (row stride ld bytes), box
// [box_rows, 128 bytes], 128-byte swizzle, zero fill outside the matrix.
bool make_map_k_major(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t k, int64_t ld,
                      int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int STAGES, bool kTransStore>
cudaError_t run(const uint8_t* a, int64_t lda, const uint8_t* b, int64_t ldb, const GemmParams& p,
                const DeviceInfo& dev, cudaStream_t stream) {
  using C = Cfg<BN, STAGES>;
  auto kernel = gemm_fp8_kernel<BN, STAGES, kTransStore>;
  static int configured_device = -1;
  if (configured_device != dev.device) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    configured_device = dev.device;
  }
  CUtensorMap ma, mb;
  if (!make_map_k_major(&ma, a, p.M, p.K, lda, kBM)) return cudaErrorInvalidValue;
  if (!make_map_k_major(&mb, b, p.N, p.K, ldb, BN)) return cudaErrorInvalidValue;
  const int tiles = ((p.M + kBM - 1) / kBM) * ((p.N + BN - 1) / BN);
  const int grid = tiles < dev.num_sms ? tiles : dev.num_sms;
  kernel<<<grid, kGemmThreads, C::kSmemBytes, stream>>>(ma, mb, p);
  return cudaGetLastError();
}

template <int BN, int STAGES>
cudaError_t run_pair(const uint8_t* a, int64_t lda, const uint8_t* b, int64_t ldb,
                     const GemmParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  using C = PairCfg<BN, STAGES>;
  auto kernel = gemm_fp8_pair_kernel<BN, STAGES>;
  static int configured_device = -1;
  static int max_pairs = 0;
  if (configured_device != dev.device) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    (void)e;
    cudaLaunchConfig_t probe = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    probe.gridDim = dim3(2 * (dev.num_sms / 2));
    probe.blockDim = dim3(kGemmThreads);
    probe.dynamicSmemBytes = C::kSmemBytes;
    probe.attrs = attr;
    probe.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &probe) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = dev.num_sms / 2;
    }
    max_pairs = n;
    configured_device = dev.device;
  }
  CUtensorMap ma, mb;
  if (!make_map_k_major(&ma, a, p.M, p.K, lda, kBM)) return cudaErrorInvalidValue;
  if (!make_map_k_major(&mb, b, p.N, p.K, ldb, BN / 2)) return cudaErrorInvalidValue;
  const int tiles = ((p.M + 2 * kBM - 1) / (2 * kBM)) * ((p.N + BN - 1) / BN);
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, ma, mb, p);
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
  if (g.M <= 64) {
    // Few rows: D^T = B . A^T, the weight-side operand fills the 128-row MMA.
    p.M = static_cast<int>(g.N);
    p.N = static_cast<int>(g.M);
    p.idesc = 0;
    if (g.M <= 16) {
      p.idesc = make_idesc_f8(g.fmt_b, g.fmt_a, kBM, 16);
      return run<16, 8, true>(g.b, g.ldb, g.a, g.lda, p, dev, stream);
    }
    if (g.M <= 32) {
      p.idesc = make_idesc_f8(g.fmt_b, g.fmt_a, kBM, 32);
      return run<32, 8, true>(g.b, g.ldb, g.a, g.lda, p, dev, stream);
    }
    p.idesc = make_idesc_f8(g.fmt_b, g.fmt_a, kBM, 64);
    return run<64, 8, true>(g.b, g.ldb, g.a, g.lda, p, dev, stream);
  }
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  // BN = 256 unless 128 pads the N edge clearly less (e.g. N = 1600).
  const int64_t pad256 = (g.N + 255) / 256 * 256, pad128 = (g.N + 127) / 128 * 128;
  const bool narrow = pad256 * 100 > pad128 * 105;
  if (g.M > kBM) {
    // CTA pairs: 256-row tiles.
    if (narrow) {
      p.idesc = make_idesc_f8(g.fmt_a, g.fmt_b, 2 * kBM, 128);
      return run_pair<128, 8>(g.a, g.lda, g.b, g.ldb, p, dev, stream);
    }
    p.idesc = make_idesc_f8(g.fmt_a, g.fmt_b, 2 * kBM, 256);
    return run_pair<256, 6>(g.a, g.lda, g.b, g.ldb, p, dev, stream);
  }
  if (narrow) {
    p.idesc = make_idesc_f8(g.fmt_a, g.fmt_b, kBM, 128);
    return run<128, 6, false>(g.a, g.lda, g.b, g.ldb, p, dev, stream);
  }
  p.idesc = make_idesc_f8(g.fmt_a, g.fmt_b, kBM, 256);
  return run<256, 4, false>(g.a, g.lda, g.b, g.ldb, p, dev, stream);
}

}  // namespace fp8lin
