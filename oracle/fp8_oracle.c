/*
 * fp8_oracle.c -- plain CPU oracle for the float8 training Linear with
 * tensorwise scaling.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA library: every rule below is written out from its definition.
 *
 * Sources:
 *  - "Integrate float8nocompile, an experimental feature for high performance"
 *    (pytorch/torchtitan PR 778), Summary: float8 conversion with tensorwise
 *    dynamic scaling (one scale per tensor, from that tensor's amax), and the
 *    "Benchmarking single linear layer forward+backward" table, whose two
 *    kernel algorithms (ATOMIC_MAX, REDUCTION) both compute the same amax.
 *  - "[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than BF16"
 *    (pytorch/ao issue 1297), repro script: CastConfig(ScalingType.DELAYED)
 *    for input, weight and grad_output, the enable_amax_init option, and
 *    sync_float8_amax_and_scale_history(model) after loss.backward().
 *  - The pages never print the numerics.  The readings used here (all plain):
 *      scale  = fl32(F / max(amax, eps)), F = 448 (e4m3) or 57344 (e5m2);
 *      inv    = fl32(1 / scale);
 *      cast   = sat_rne_fp8(fl32(x * scale)), saturating to +-F, ties to even;
 *      e4m3   = 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinity,
 *               NaN only at S.1111.111 (so the largest finite is 448);
 *      e5m2   = 1 sign, 5 exponent (bias 15), 2 mantissa bits, IEEE-style
 *               infinity and NaN (largest finite 57344);
 *      delayed: ring[head] = amax; head = (head+1) % H;
 *               scale = fl32(F / max(max(ring), eps)).
 *
 * Every function here is scalar and written for clarity, not speed; the only
 * concession is an OpenMP loop over independent rows.
 *
 * Compile with -ffp-contract=off and without -ffast-math: the fp32 products
 * and quotients below must each be one IEEE round-to-nearest-even operation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_E4M3 0
#define ORACLE_E5M2 1

typedef struct {
  int mbits;       /* mantissa (fraction) bits */
  int bias;        /* exponent bias */
  double maxval;   /* largest finite magnitude */
} fp8_format;

static fp8_format format_of(int fmt) {
  fp8_format f;
  if (fmt == ORACLE_E4M3) { f.mbits = 3; f.bias = 7;  f.maxval = 448.0;   }
  else                    { f.mbits = 2; f.bias = 15; f.maxval = 57344.0; }
  return f;
}

/* Threads an OpenMP loop of this oracle uses (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Largest finite magnitude of the format: (2 - 2^-m) * 2^emax. */
double oracle_fp8_max(int fmt) { return format_of(fmt).maxval; }

/* Decode one 8-bit code to its real value (NaN / +-inf where the format
 * defines them). */
double oracle_fp8_decode(uint8_t code, int fmt) {
  fp8_format f = format_of(fmt);
  int ebits = 7 - f.mbits;
  int sign = code >> 7;
  int e = (code >> f.mbits) & ((1 << ebits) - 1);
  int m = code & ((1 << f.mbits) - 1);
  double v;
  if (fmt == ORACLE_E4M3 && e == 15 && m == 7) return NAN;
  if (fmt == ORACLE_E5M2 && e == 31) {
    if (m != 0) return NAN;
    return sign ? -INFINITY : INFINITY;
  }
  if (e == 0)  /* subnormal: m * 2^(1 - bias - mbits) */
    v = ldexp((double)m, 1 - f.bias - f.mbits);
  else         /* normal: (1 + m / 2^mbits) * 2^(e - bias) */
    v = ldexp((double)((1 << f.mbits) + m), e - f.bias - f.mbits);
  return sign ? -v : v;
}

/* Bits of a finite magnitude v that is exactly representable and <= max. */
static uint8_t pack_magnitude(double v, fp8_format f) {
  double min_normal = ldexp(1.0, 1 - f.bias);
  int e2;
  if (v == 0.0) return 0;
  if (v < min_normal) {
    /* subnormal: exponent field 0, mantissa = v / 2^(1 - bias - mbits) */
    return (uint8_t)ldexp(v, f.bias + f.mbits - 1);
  }
  frexp(v, &e2);              /* v = frac * 2^e2, frac in [0.5, 1) */
  {
    int E = e2 - 1;           /* v in [2^E, 2^(E+1)) */
    int mant = (int)(ldexp(v, f.mbits - E) - (double)(1 << f.mbits));
    return (uint8_t)(((E + f.bias) << f.mbits) | mant);
  }
}

/* Saturating round-to-nearest-even encode of an fp32 value:
 *   round r to the nearest value of the format (ties to the even mantissa,
 *   subnormals included); if the rounded magnitude exceeds the largest finite
 *   F, or r is infinite, the result is +-F.  The sign of zero is kept.
 *   NaN (outside the contract) maps to the format's NaN code 0x7F. */
uint8_t oracle_fp8_encode(float r, int fmt) {
  fp8_format f = format_of(fmt);
  uint8_t sign = signbit(r) ? 0x80 : 0x00;
  double a, quantum, n, v;
  if (isnan(r)) return 0x7F;
  a = fabs((double)r);
  if (isinf(a)) return sign | pack_magnitude(f.maxval, f);
  if (a < ldexp(1.0, 1 - f.bias)) {
    quantum = ldexp(1.0, 1 - f.bias - f.mbits);      /* subnormal spacing */
  } else {
    int e2;
    frexp(a, &e2);                                   /* a in [2^(e2-1), 2^e2) */
    quantum = ldexp(1.0, e2 - 1 - f.mbits);          /* spacing in that binade */
  }
  n = nearbyint(a / quantum);   /* exact quotient; default mode is ties-to-even */
  v = n * quantum;
  if (v > f.maxval) v = f.maxval;                    /* saturate */
  return sign | pack_magnitude(v, f);
}

/* bf16 bits -> fp32 (exact widening). */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

/* amax = max_i |x_i| over a bf16 [rows, cols] tensor with row stride ld
 * (elements).  An empty tensor has amax 0. */
float oracle_amax_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld) {
  float best = 0.0f;
  int64_t i;
#pragma omp parallel for reduction(max : best) schedule(static)
  for (i = 0; i < rows; ++i) {
    int64_t j;
    for (j = 0; j < cols; ++j) {
      float a = fabsf(bf16_to_f32(x[i * ld + j]));
      if (a > best) best = a;
    }
  }
  return best;
}

/* Dynamic scale: scale = fl32(F / max(amax, eps)), inv = fl32(1 / scale). */
void oracle_scale_dynamic(float amax, float eps, int fmt, float* scale, float* inv) {
  float F = (float)format_of(fmt).maxval;
  float denom = amax > eps ? amax : eps;
  float s = F / denom;
  *scale = s;
  *inv = 1.0f / s;
}

/* Delayed scaling update (the step the pages run after backward):
 *   ring[head] = amax; head = (head + 1) % H;
 *   scale = fl32(F / max(max_h ring[h], eps)); inv = fl32(1 / scale).
 * The max runs over all H slots; unfilled slots hold 0 and never win. */
void oracle_scale_delayed(float* ring, int32_t H, int32_t* head, float amax,
                          float eps, int fmt, float* scale, float* inv) {
  float m = 0.0f;
  int32_t h;
  ring[*head] = amax;
  *head = (*head + 1) % H;
  for (h = 0; h < H; ++h)
    if (ring[h] > m) m = ring[h];
  oracle_scale_dynamic(m, eps, fmt, scale, inv);
}

/* Cast: q[i,j] = encode(fl32(x[i,j] * scale)), written row-major dense
 * [rows, cols] into out; if out_t is not NULL also qT[j,i] = q[i,j] dense
 * [cols, rows].  Returns the amax of x seen in the same pass. */
float oracle_cast_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                       float scale, int fmt, uint8_t* out, uint8_t* out_t) {
  float best = 0.0f;
  int64_t i;
#pragma omp parallel for reduction(max : best) schedule(static)
  for (i = 0; i < rows; ++i) {
    int64_t j;
    for (j = 0; j < cols; ++j) {
      float xv = bf16_to_f32(x[i * ld + j]);
      float r = xv * scale;
      uint8_t q = oracle_fp8_encode(r, fmt);
      if (fabsf(xv) > best) best = fabsf(xv);
      if (out) out[i * cols + j] = q;
      if (out_t) out_t[j * rows + i] = q;
    }
  }
  return best;
}

/* Encode a plain array of fp32 values (no scaling), for codec checks. */
void oracle_encode_f32(const float* r, int64_t n, int fmt, uint8_t* out) {
  int64_t i;
#pragma omp parallel for schedule(static)
  for (i = 0; i < n; ++i) out[i] = oracle_fp8_encode(r[i], fmt);
}

/* Decode a byte array to fp64 through the format definition. */
void oracle_decode_array(const uint8_t* q, int64_t n, int fmt, double* out) {
  double table[256];
  int c;
  int64_t i;
  for (c = 0; c < 256; ++c) table[c] = oracle_fp8_decode((uint8_t)c, fmt);
#pragma omp parallel for schedule(static)
  for (i = 0; i < n; ++i) out[i] = table[q[i]];
}

/* One GEMM entry, straight from the definition:
 *   y[m,n] = sum_k dec(A[m,k]) * dec(B[n,k]) / (scale_a * scale_b)
 *   s[m,n] = sum_k |dec(A[m,k]) * dec(B[n,k])| / (scale_a * scale_b)
 * with A [*, K] and B [*, K] both stored with the contraction index fastest
 * (row strides lda, ldb bytes), accumulated in fp64. */
void oracle_gemm_entries(const uint8_t* A, const uint8_t* B, int64_t K,
                         int64_t lda, int64_t ldb, int fmt_a, int fmt_b,
                         float scale_a, float scale_b,
                         const int64_t* rows_m, const int64_t* cols_n, int64_t count,
                         double* y, double* s) {
  double ta[256], tb[256];
  double denom = (double)scale_a * (double)scale_b;
  int c;
  int64_t e;
  for (c = 0; c < 256; ++c) {
    ta[c] = oracle_fp8_decode((uint8_t)c, fmt_a);
    tb[c] = oracle_fp8_decode((uint8_t)c, fmt_b);
  }
#pragma omp parallel for schedule(dynamic, 16)
  for (e = 0; e < count; ++e) {
    const uint8_t* a = A + rows_m[e] * lda;
    const uint8_t* b = B + cols_n[e] * ldb;
    double acc = 0.0, acc_abs = 0.0;
    int64_t k;
    for (k = 0; k < K; ++k) {
      double p = ta[a[k]] * tb[b[k]];
      acc += p;
      acc_abs += fabs(p);
    }
    y[e] = acc / denom;
    s[e] = acc_abs / denom;
  }
}
