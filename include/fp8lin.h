/*
 * fp8lin.h -- C ABI of libfp8lin, the float8 training Linear with tensorwise
 * scaling on one GB300 (sm_103a).
 *
 * What the library computes (the hot path of the float8 training Linear that
 * replaces nn.Linear in "Why swapping nn.Linear with FP8Linear brings
 * throughput decrease for 7B LLAMA2-like model?" (pytorch/ao issue 1199)):
 *
 *   amax   a     = max |t|                      over a bf16 tensor t
 *   scale  s     = fl32(F / max(a, eps)),  inv = fl32(1 / s)
 *                  F = 448 (e4m3: input, weight) or 57344 (e5m2: grad_output)
 *   cast   q     = sat_rne_fp8(fl32(t * s)), plus the transposed copy q^T
 *   GEMMs  y     = (x8  . W8^T)  * inv_x  * inv_w     -> bf16 [M, N]
 *          dX    = (dY8 . W8)    * inv_dy * inv_w     -> bf16 [M, K]
 *          dW    = (dY8^T . x8)  * inv_dy * inv_x     -> bf16 [N, K]
 *   with fp32 accumulation on the tensor cores.
 *
 * Sources, by page and section:
 *   - "Integrate float8nocompile, an experimental feature for high
 *     performance" (pytorch/torchtitan PR 778), Summary: tensorwise dynamic
 *     scaling with hand-written conversion kernels; "Benchmarking single
 *     linear layer forward+backward performance": the two amax algorithms
 *     (KernelAlgorithm.ATOMIC_MAX, KernelAlgorithm.REDUCTION) and the
 *     forward+backward scope of one Linear.
 *   - "[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than BF16"
 *     (pytorch/ao issue 1297), repro script: Float8LinearConfig with
 *     CastConfig(scaling_type=ScalingType.DELAYED) per tensor role,
 *     enable_amax_init, and sync_float8_amax_and_scale_history(model) after
 *     loss.backward().
 * The pages print no numerics; the formulas above are the plain reading
 * (formats e4m3/e5m2 with saturation to the largest finite value,
 * round-to-nearest-even, no power-of-two rounding of the scale).
 *
 * Conventions for every entry point:
 *   - Layout: row-major. A "[R, C] bf16 tensor with row stride ld" has
 *     element (i, j) at ((const uint16_t*)p)[i * ld + j].  fp8 outputs are
 *     dense row-major bytes (row stride = number of columns).  W is [N, K]
 *     (out_features x in_features) as in nn.Linear.
 *   - Ownership: every pointer is a caller-owned DEVICE pointer (except the
 *     fp8lin_scaling_state struct itself, which lives in host memory).  The
 *     library allocates no device memory and keeps no per-call state.
 *   - Asynchrony: every call enqueues work on `stream` and returns without
 *     synchronising; scalars (amax, scale, ...) stay on the device.
 *   - Errors: arguments are checked before anything is enqueued; a bad call
 *     returns FP8LIN_EINVAL (null/misaligned pointer, negative size, stride
 *     smaller than the row) or FP8LIN_EUNSUPPORTED (shape or format the
 *     kernels do not take) and enqueues nothing.  A failed launch returns
 *     FP8LIN_ECUDA (fp8lin_last_cuda_error() gives the cudaError_t).
 *     Device-side waits are bounded: a wait that runs out records a code in
 *     the workspace and the kernel returns; fp8lin_check() reports it as
 *     FP8LIN_ETIMEOUT.  Nothing traps on the device.
 *   - Alignment: every device pointer 16-byte aligned; bf16 row strides a
 *     multiple of 8 elements; columns a multiple of 16; rows a multiple of 16
 *     wherever a transposed copy (or a GEMM operand) has them as its row
 *     length.  In practice: M, K, N multiples of 16.
 *   - Inputs are NaN-free by contract; NaN propagation is not specified.
 *   - Per-device set-up (kernel shared-memory attributes, occupancy counts,
 *     the device address of fp8lin_amax_noalloc's static array) is done by
 *     the first call on each device and kept for the life of the process,
 *     for that device's primary context.  cudaDeviceReset() ends that
 *     context and with it the set-up: do not call the library on a device
 *     after resetting it in the same process.
 */
#ifndef FP8LIN_H
#define FP8LIN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8LIN_OK = 0,
  FP8LIN_EINVAL = 1,        /* bad argument; nothing enqueued */
  FP8LIN_EUNSUPPORTED = 2,  /* valid but not handled (shape/format/size); nothing enqueued */
  FP8LIN_ECUDA = 3,         /* a CUDA call failed; see fp8lin_last_cuda_error() */
  FP8LIN_ETIMEOUT = 4       /* a bounded device wait ran out (reported by fp8lin_check) */
} fp8lin_status;

/* 8-bit formats: e4m3 (max 448, no infinity) for input and weight, e5m2 (max
 * 57344) for grad_output. */
typedef enum { FP8LIN_E4M3 = 0, FP8LIN_E5M2 = 1 } fp8lin_fmt;

/* amax algorithms, after the KernelAlgorithm choice of the single-linear
 * benchmark table in "Integrate float8nocompile ..." (torchtitan PR 778):
 *   ATOMIC      one pass; each CTA folds its block maximum into the result
 *               with one atomic max (through self-cleaning workspace words
 *               when a workspace is given, so no memset precedes it);
 *   REDUCTION   each CTA writes its partial maximum to the workspace and a
 *               second, one-CTA kernel reduces them;
 *   SINGLE_PASS (dynamic scaling only: fp8lin_forward, fp8lin_backward,
 *               fp8lin_cast_dynamic)
 *               amax -> scale -> cast (+transpose) in one cooperative launch
 *               that keeps the bf16 tensor on chip between the phases; only
 *               for tensors that fit (fp8lin_single_pass_max_elems()); larger
 *               tensors fall back to ATOMIC inside forward/backward;
 *   PRECOMPUTED (dynamic scaling only, not fp8lin_amax) *amax already holds
 *               the tensor's amax -- the GEMM that produced the tensor wrote
 *               it from its epilogue (the y_amax / dx_amax outputs below)
 *               -- so the cast reads the tensor once: scale, then cast
 *               (+transpose).  This moves the amax into the producer: the
 *               diagnosis in "Why swapping nn.Linear with FP8Linear brings
 *               throughput decrease ..." (pytorch/ao issue 1199) is that the
 *               eager float8 casts run as kernels of their own, apart from
 *               the ops around them. */
typedef enum {
  FP8LIN_AMAX_ATOMIC = 0,
  FP8LIN_AMAX_REDUCTION = 1,
  FP8LIN_AMAX_SINGLE_PASS = 2,
  FP8LIN_AMAX_AUTO = 3,      /* SINGLE_PASS where the tensor fits, else ATOMIC */
  FP8LIN_AMAX_PRECOMPUTED = 4
} fp8lin_amax_algo;

/* Scaling type per tensor, after CastConfig(scaling_type=...) in the repro
 * script of "[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than BF16". */
typedef enum { FP8LIN_DYNAMIC = 0, FP8LIN_DELAYED = 1 } fp8lin_scaling;

/* Per-tensor scaling state.  The struct is host memory; the pointers in it
 * are caller-owned device buffers (fp32 / int32).
 *   amax          fp32[1]  amax of the tensor last cast with this state
 *   scale         fp32[1]  scale the next cast uses (delayed) / last used (dynamic)
 *   inv_scale     fp32[1]  fl32(1 / scale), folded into the GEMM epilogues
 *   amax_history  fp32[history_len]  delayed only: ring of past amaxes, zero-filled
 *                 by the caller before the first step
 *   head          int32[1] delayed only: next ring slot, 0 before the first step
 *   history_len   delayed only: ring length H >= 1
 *   fmt           fp8lin_fmt of the cast
 *   kind          fp8lin_scaling
 *   amax_algo     fp8lin_amax_algo used by fp8lin_forward/backward
 *   needs_init    delayed only, host flag: when nonzero the next forward or
 *                 backward cast first takes the scale from the tensor's own
 *                 amax (enable_amax_init in the repro script) without
 *                 touching the ring, and the library then sets it to 0
 *   eps           floor of the amax in the scale (1e-12 is the usual value) */
typedef struct fp8lin_scaling_state {
  float* amax;
  float* scale;
  float* inv_scale;
  float* amax_history;
  int32_t* head;
  int32_t history_len;
  int32_t fmt;
  int32_t kind;
  int32_t amax_algo;
  int32_t needs_init;
  float eps;
} fp8lin_scaling_state;

/* ---- library information ------------------------------------------- */

/* Human-readable name of a status code (static string). */
const char* fp8lin_status_string(int status);

/* cudaError_t of the last failed CUDA call made by this thread (0 if none). */
int fp8lin_last_cuda_error(void);

/* Which operation the last failed CUDA call of this thread was in, with the
 * error's name (static per-thread string; "" if none). */
const char* fp8lin_last_error_detail(void);

/* ABI version: 100 * major + minor. */
int fp8lin_version(void);

/* Bytes of workspace `ws` the calls below need for these Linear sizes.  The
 * workspace is caller-owned device memory, 256-byte aligned, zero-filled by
 * the caller ONCE after allocation; the library keeps it consistent after
 * that.  Calls that share one workspace must not overlap on the GPU. */
size_t fp8lin_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* Largest tensor (elements) FP8LIN_AMAX_SINGLE_PASS handles on the current
 * device (0 if the device cannot run it). */
int64_t fp8lin_single_pass_max_elems(void);

/* Synchronise `stream`, then read and clear the workspace's device error
 * record.  Returns FP8LIN_OK, FP8LIN_ETIMEOUT (a bounded wait ran out) or
 * FP8LIN_ECUDA. */
fp8lin_status fp8lin_check(void* ws, cudaStream_t stream);

/* ---- steps of the path ---------------------------------------------- */

/* amax (row a1 of the path): *amax_out = max |x[i, j]| over the bf16
 * [rows, cols] tensor x with row stride ld, as fp32 (exact: the maximum of
 * bf16 magnitudes widened to fp32).  An empty tensor gives 0.
 * algo: FP8LIN_AMAX_ATOMIC or FP8LIN_AMAX_REDUCTION (same bits).
 * ws: workspace (REDUCTION keeps its partial maxima there).
 * Source: "Integrate float8nocompile ..." (torchtitan PR 778), Summary and
 * the single-linear benchmark table (ATOMIC_MAX / REDUCTION). */
fp8lin_status fp8lin_amax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                          float* amax_out, int32_t algo, void* ws, cudaStream_t stream);

/* amax without workspace or allocation.  The pages have no counterpart of
 * this entry point; it exists for callers that cannot call cudaMalloc and
 * have no workspace to pass -- for example a plug-in running inside a host
 * framework that owns all device memory through its own pool (a direct
 * cudaMalloc would bypass that pool's accounting, or fail because the pool
 * has reserved the memory), or a tool allowed to touch only the buffers it
 * was handed.
 * Computes exactly what fp8lin_amax(..., FP8LIN_AMAX_REDUCTION, ws, ...)
 * computes (same bits), with the partial maxima kept in a static device
 * array of the library instead of `ws`: 4096 slots of 4 bytes (16 KiB),
 * one per CTA, held on every GPU that loads the library until the process
 * exits.  It allocates nothing and calls no allocating routine.
 * Limits: the shape rules of fp8lin_amax; a launch that would need more
 * than 4096 CTAs (a device with more than 512 SMs) returns
 * FP8LIN_EUNSUPPORTED with nothing enqueued.
 * Each call looks up the array's device address (cudaGetSymbolAddress) with
 * the device current, so the address stays right after a device reset; the
 * first lookup on a device may load the library's device code, so make the
 * first call before any stream capture.  All calls on a device share the one array,
 * which keeps the last call's contents (nothing in it needs clearing: each
 * call writes every slot it reads); calls that overlap on the GPU -- on two
 * streams, or from two host threads -- race on it and must be serialised
 * by the caller. */
fp8lin_status fp8lin_amax_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                  float* amax_out, cudaStream_t stream);

/* scale (rows a2 / a2' of the path).  Dynamic: reads *st->amax and writes
 * scale = fl32(F / max(amax, eps)) and inv_scale = fl32(1 / scale).
 * Delayed: ring[head] = *amax; head = (head + 1) % H; then the same formula
 * on max(ring) -- the per-tensor work of sync_float8_amax_and_scale_history
 * after backward in "[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than
 * BF16" (pytorch/ao issue 1297), repro script. */
fp8lin_status fp8lin_scale(const fp8lin_scaling_state* st, cudaStream_t stream);

/* fp8lin_scale of each of n states (0 <= n <= 8) in ONE launch, one thread a
 * state: the history updates and rescales of a Linear's x, W and dY states
 * after its backward, which sync_float8_amax_and_scale_history performs one
 * tensor at a time in "[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than
 * BF16" (pytorch/ao issue 1297), repro script.  `states` points to n states
 * in host memory (read during the call only), each checked as fp8lin_scale
 * checks it.  No buffer a state's update writes (scale, inv_scale and,
 * delayed, amax_history[0..H) and head) may overlap any buffer of another
 * state; states may share an amax, which is only read.  The results are
 * those of n fp8lin_scale calls, bit for bit.  EINVAL for n < 0 or n > 8,
 * for states NULL with n > 0, for any state fp8lin_scale rejects and for
 * overlapping states (nothing enqueued); n == 0 enqueues nothing. */
fp8lin_status fp8lin_scale_many(const fp8lin_scaling_state* states, int32_t n,
                                cudaStream_t stream);

/* cast (row a3): out[i, j] = sat_rne_fp8(fl32(x[i, j] * (*scale))) into the
 * dense [rows, cols] byte array out; if out_t is not NULL also
 * out_t[j, i] = out[i, j] (dense [cols, rows]).  If amax_out is not NULL the
 * amax of x is recorded in the same pass (delayed scaling's single pass).
 * fmt: fp8lin_fmt.  out may be NULL when out_t is not.
 * Source: "Integrate float8nocompile ..." (torchtitan PR 778), Summary
 * (float8 conversion kernels). */
fp8lin_status fp8lin_cast(const void* x, int64_t rows, int64_t cols, int64_t ld,
                          int32_t fmt, const float* scale, uint8_t* out, uint8_t* out_t,
                          float* amax_out, cudaStream_t stream);

/* Dynamic scaling in one call: amax -> scale -> cast (+ transpose) with
 * st->amax_algo (ATOMIC, REDUCTION, SINGLE_PASS or AUTO); writes *st->amax,
 * *st->scale, *st->inv_scale, out and (if not NULL) out_t.  st->kind must
 * be FP8LIN_DYNAMIC.  ws is the caller's workspace (fp8lin_workspace_bytes
 * of any shape): REDUCTION's partial maxima and the single pass's barrier
 * words live there.  SINGLE_PASS returns FP8LIN_EUNSUPPORTED (nothing
 * enqueued) for tensors above fp8lin_single_pass_max_elems().  Source:
 * "Integrate float8nocompile ..." (torchtitan PR 778), Summary (tensorwise
 * dynamic scaling with hand-written conversion kernels) and "Benchmarking
 * single linear layer forward+backward performance" (the ATOMIC_MAX and
 * REDUCTION amax algorithms). */
fp8lin_status fp8lin_cast_dynamic(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                  const fp8lin_scaling_state* st, uint8_t* out,
                                  uint8_t* out_t, void* ws, cudaStream_t stream);

/* Delayed scaling's cast of one tensor, as fp8lin_forward / fp8lin_backward
 * run it: cast with the stored *st->scale into out (+ out_t) and record the
 * tensor's amax into *st->amax in the same pass -- one read of the tensor.
 * If st->needs_init is set, the scale is first taken from the tensor's own
 * amax (enable_amax_init), without touching the ring, and needs_init is
 * cleared.  st->kind must be FP8LIN_DELAYED; the ring update is
 * fp8lin_scale's, after backward.  Source: "[float8] FP8 GPT 1.5B Delayed
 * Scaling 2x Slower than BF16" (pytorch/ao issue 1297), repro script
 * (ScalingType.DELAYED, enable_amax_init). */
fp8lin_status fp8lin_cast_delayed(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                  fp8lin_scaling_state* st, uint8_t* out, uint8_t* out_t,
                                  void* ws, cudaStream_t stream);

/* FP8 GEMM (rows a4-a6): d[m, n] = bf16( (sum_k A[m, k] * B[n, k]) *
 * fl32(inv_a * inv_b) ), accumulated in fp32 on the tensor cores -- the form
 * every product of the FP8Linear of "Why swapping nn.Linear with FP8Linear
 * brings throughput decrease for 7B LLAMA2-like model?" (pytorch/ao issue
 * 1199) takes once the transposed fp8 copies exist: y = x8 . W8^T,
 * dX = dY8 . (W8^T)^T, dW = dY8^T . (x8^T)^T.
 * a: fp8 [M, K] row stride lda bytes; b: fp8 [N, K] row stride ldb bytes
 * (both with the contraction index fastest); fmt_a, fmt_b: fp8lin_fmt;
 * inv_a, inv_b: device fp32[1]; d: bf16 [M, N] row stride ldd elements.
 * d_amax: NULL, or device fp32[1] that receives max |d| over the stored
 * bf16 values, computed in the epilogue (no extra pass over d); 0 when d is
 * empty or K == 0.
 * K == 0 writes zeros.  Requires lda, ldb multiples of 16, ldd a multiple
 * of 8, N and K multiples of 16. */
fp8lin_status fp8lin_gemm(const uint8_t* a, const uint8_t* b, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int32_t fmt_a, int32_t fmt_b,
                          const float* inv_a, const float* inv_b, void* d, int64_t ldd,
                          float* d_amax, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Names the kernel, tile shape and schedule fp8lin_gemm uses on the current
 * device for an M x N x K GEMM with a workspace of fp8lin_workspace_bytes,
 * as one NUL-terminated line written into buf (caller-owned host memory of
 * buf_len bytes; truncated to fit).  The kernel name is spelled as profilers
 * list it, e.g. "gemm_fp8_pair_kernel<256, 6, 4>".  Enqueues nothing.  Returns
 * FP8LIN_EINVAL for negative sizes or a NULL / empty buffer, FP8LIN_ECUDA
 * without a usable device. */
fp8lin_status fp8lin_gemm_describe(int64_t M, int64_t N, int64_t K, char* buf, size_t buf_len);

/* The line fp8lin_gemm_describe writes, for a device of num_sms SMs that
 * holds one GEMM CTA per SM (num_sms / 2 CTA pairs), as the kernels are
 * sized for: the same kernel choice and the same K-split rules, computed on
 * the host without touching a device (planning, and tests on a machine
 * without a GPU).  On a GB300 (152 SMs) it matches fp8lin_gemm_describe.
 * Returns FP8LIN_EINVAL for negative sizes, num_sms < 2 or a NULL / empty
 * buffer. */
fp8lin_status fp8lin_gemm_describe_for(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                                       char* buf, size_t buf_len);

/* How fp8lin_backward would run its two GEMMs (dX: Ma x Na x Ka, dW:
 * Mb x Nb x Kb) on a device of num_sms SMs, computed on the host: "grouped"
 * when both take 256-wide CTA-pair tiles and one launch that deals the tiles
 * of both by their K loops is expected to take at most 0.92 of the time of
 * two, else "separate"; then the tile counts (problem 0: the longer K loop),
 * K blocks, the deal's parameter d, the estimated K blocks of the busiest
 * CTA pair both ways, the grouped launch's epilogue warps (4 or 8), and
 * "DEAL BROKEN" if the deal would not hand out every
 * tile exactly once (a self-check of the same function the kernel deals
 * with).  This is the plan's decision; FP8LIN_GROUP in the environment
 * overrides it in fp8lin_backward (0: never group, 2: group whenever both
 * qualify).  Returns FP8LIN_EINVAL for sizes < 1, num_sms < 2 or a NULL /
 * empty buffer. */
fp8lin_status fp8lin_gemm_group_describe_for(int64_t Ma, int64_t Na, int64_t Ka, int64_t Mb,
                                             int64_t Nb, int64_t Kb, int32_t num_sms, char* buf,
                                             size_t buf_len);

/* Forward of the Linear -- the forward half of the "forward+backward" of one
 * Linear timed in "Integrate float8nocompile, an experimental feature for
 * high performance" (torchtitan PR 778), "Benchmarking single linear layer
 * forward+backward performance"; the FP8Linear of pytorch/ao issue 1199:
 * amax/scale/cast of x ([M, K], e4m3, state sx) and W ([N, K], e4m3, state
 * sw), then y = x8 . W8^T * inv_x * inv_w (bf16 [M, N]).  Writes the fp8 copies x8 [M, K], x8t [K, M], w8 [N, K],
 * w8t [K, N]; x8t and w8t are what fp8lin_backward needs.  Dynamic states
 * take their scale from this call's amax; delayed states cast with their
 * stored scale and record this call's amax (and do the amax init first when
 * needs_init is set).  All buffers dense row-major.
 * y_amax: NULL, or device fp32[1] that receives max |y| from the GEMM
 * epilogue -- point it at the amax of the next layer's input state and give
 * that state FP8LIN_AMAX_PRECOMPUTED to cast y in one pass.
 * w == NULL skips W's cast and uses w8, w8t and sw as an earlier call left
 * them: the weight cached across calls while it is unchanged, e.g. over the
 * micro-batches of one optimizer step (the few-token case, where W's cast
 * dominates the step).  The result is the one a fresh cast would give as long
 * as sw's scale has not moved since: always for dynamic scaling, and until
 * the next fp8lin_scale of sw for delayed scaling.  EINVAL if sw is delayed
 * and still needs its first (amax-init) cast.
 * A few tokens (M <= 32) with dynamic scaling of x (amax_algo AUTO,
 * SINGLE_PASS or PRECOMPUTED) and, when W is cast, of W (AUTO or
 * SINGLE_PASS): x's cast, W's cast and y run as one fused launch (same
 * results: casts and scales bit for bit, y within the GEMM's bound; only the
 * order in which y's fp32 partial sums are added differs).
 * FP8LIN_SMALL_M=0 in the environment turns this off.
 * More tokens, with both states dynamic (AUTO or SINGLE_PASS) and W cast by
 * the cooperative single pass: where x has at most one 128 x 128 tile for
 * each CTA of W's launch, x's cast runs inside W's (one launch; the same
 * bits).  FP8LIN_PAIR_CAST=0 in the environment casts them apart. */
fp8lin_status fp8lin_forward(const void* x, const void* w, int64_t M, int64_t K, int64_t N,
                             fp8lin_scaling_state* sx, fp8lin_scaling_state* sw,
                             void* y, float* y_amax, uint8_t* x8, uint8_t* x8t, uint8_t* w8,
                             uint8_t* w8t, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Backward of the Linear -- the backward half of the single-linear
 * "forward+backward" of torchtitan PR 778; the FP8Linear's backward of
 * pytorch/ao issue 1199: amax/scale/cast of dY ([M, N], e5m2, state sdy)
 * into dy8 [M, N] and dy8t [N, M], then
 *   dX = dY8 . W8 * inv_dy * inv_w     (bf16 [M, K], skipped if dx == NULL)
 *   dW = dY8^T . x8 * inv_dy * inv_x   (bf16 [N, K], skipped if dw == NULL)
 * from the x8t / w8t written by fp8lin_forward and the inv_scale of sx, sw.
 * dx_amax, dw_amax: NULL, or device fp32[1] receiving max |dX| / max |dW|
 * from the GEMM epilogues (each needs its GEMM: dx / dw not NULL); dx_amax
 * can feed the previous layer's grad_output state as PRECOMPUTED.
 * A few tokens (M <= 32) with dynamic scaling of dY (AUTO, SINGLE_PASS or
 * PRECOMPUTED) and dx not NULL: dY's cast and dX run as one fused launch
 * (as in fp8lin_forward), and dW in the same launch when dw is not NULL and
 * dw_amax is NULL (dW equals the GEMM's value for value; an exact zero may
 * differ in sign).  Otherwise dW follows as its own GEMM; so it does with
 * FP8LIN_SMALL_M_DW=0 in the environment.
 * When dX and dW both run on the 256-wide pair tiles, at most one of dx_amax
 * and dw_amax is given, and the host plan expects one launch over both GEMMs'
 * tiles to take at most 0.92 of the time of two (fp8lin_gemm_group_describe_for
 * prints the decision), they run as one launch; it computes every tile whole,
 * as the separate GEMM does where it splits no K loop.  FP8LIN_GROUP=0 in the
 * environment never groups them, FP8LIN_GROUP=2 groups them whenever they
 * qualify. */
fp8lin_status fp8lin_backward(const void* dy, int64_t M, int64_t K, int64_t N,
                              const uint8_t* x8t, const uint8_t* w8t,
                              const fp8lin_scaling_state* sx, const fp8lin_scaling_state* sw,
                              fp8lin_scaling_state* sdy, uint8_t* dy8, uint8_t* dy8t,
                              void* dx, void* dw, float* dx_amax, float* dw_amax, void* ws,
                              size_t ws_bytes, cudaStream_t stream);

/* ---- one step from host buffers --------------------------------------- */

/* Caller-owned device side of one slot of fp8lin_step_host.  x, w, dy receive
 * the step's inputs (bf16 [M, K], [N, K], [M, N]); y, dx, dw hold its outputs
 * (bf16 [M, N], [M, K], [N, K]) until they are copied out; x8 ... dy8t and
 * ws are as for fp8lin_forward / fp8lin_backward.  ev[0..4] are caller-created
 * events (cudaEventCreateWithFlags(..., cudaEventDisableTiming)) that order
 * this slot's copies against its compute; the library only records and waits
 * on them.  Two slots used in turn let one step's copies run while the other
 * slot's step computes: their bf16 buffers and events must be distinct, their
 * fp8 buffers and workspace may be shared (all compute runs on one stream). */
typedef struct fp8lin_step_slot {
  void* x;
  void* w;
  void* dy;
  void* y;
  void* dx;
  void* dw;
  uint8_t* x8;
  uint8_t* x8t;
  uint8_t* w8;
  uint8_t* w8t;
  uint8_t* dy8;
  uint8_t* dy8t;
  void* ws;
  size_t ws_bytes;
  cudaEvent_t ev[5];
} fp8lin_step_slot;

/* One training step of the Linear from host memory: copies x_h, w_h, dy_h
 * (host bf16, dense, pinned for the copies to be asynchronous) into the
 * slot, runs fp8lin_forward and fp8lin_backward on `compute` (and, for each
 * delayed state, the fp8lin_scale of sync_float8_amax_and_scale_history
 * after backward, as in the repro script of "[float8] FP8 GPT 1.5B Delayed
 * Scaling 2x Slower than BF16", pytorch/ao issue 1297), and copies y, dX, dW
 * back into y_h, dx_h, dw_h.  Uploads run on `h2d`, downloads on `d2h`
 * (one cudaMemcpyAsync per tensor), ordered by the slot's events:
 *   - the uploads of x, W wait until this slot's previous forward has read
 *     them, the upload of dY until its previous backward has;
 *   - the forward waits for x, W and for this slot's previous downloads;
 *     the backward waits for dY; y's download follows the forward (it
 *     overlaps the backward), dX's and dW's the backward.
 * With wait != 0, `compute` then waits for this step's downloads: the host
 * buffers hold the results once `compute` has reached this point.  With
 * wait == 0 the next step's compute may run while the downloads are in
 * flight; make `compute` wait on slot->ev[4] (downloads done) before reading
 * the host outputs.  Every argument is checked before anything is enqueued.
 * The library allocates nothing; the host buffers and the slot are the
 * caller's. */
fp8lin_status fp8lin_step_host(const void* x_h, const void* w_h, const void* dy_h, void* y_h,
                               void* dx_h, void* dw_h, int64_t M, int64_t K, int64_t N,
                               fp8lin_scaling_state* sx, fp8lin_scaling_state* sw,
                               fp8lin_scaling_state* sdy, const fp8lin_step_slot* slot,
                               cudaStream_t compute, cudaStream_t h2d, cudaStream_t d2h,
                               int wait);

/* ---- measurement hooks ------------------------------------------------ */

/* Count of kernels this library has launched in the process. */
uint64_t fp8lin_launch_count(void);

/* Kernel timing: while enabled, every kernel launch of the library is
 * bracketed by a pair of CUDA events on its stream (up to a fixed number of
 * pairs).  fp8lin_profile_collect() synchronises those events, adds up the
 * milliseconds per kernel kind into ms[kind] and launches into count[kind]
 * (arrays of FP8LIN_PROF_KINDS entries), and clears the record.  Not
 * thread-safe; not for use under CUDA graph capture. */
enum {
  FP8LIN_PROF_AMAX = 0, FP8LIN_PROF_SCALE = 1, FP8LIN_PROF_CAST = 2,
  FP8LIN_PROF_CAST_FUSED = 3, FP8LIN_PROF_GEMM = 4,
  FP8LIN_PROF_SMALL_M = 5,   /* a few-token product fused with its casts */
  FP8LIN_PROF_KINDS = 6
};
void fp8lin_profile_enable(int on);
fp8lin_status fp8lin_profile_collect(double* ms, int64_t* count);

/* The same record launch by launch, in launch order: synchronises the
 * events, writes the milliseconds and the FP8LIN_PROF_* kind of the first
 * min(recorded, capacity) launches into ms[] / kind[] (host arrays), clears
 * the record and returns how many it wrote; a negative value is -status. */
int64_t fp8lin_profile_launches(double* ms, int32_t* kind, int64_t capacity);

#ifdef __cplusplus
}
#endif

#endif /* FP8LIN_H */
