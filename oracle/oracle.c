/*
 * oracle.c -- plain, slow CPU oracle for symmetric w8a8 scaled quantisation
 * and the scaled matrix multiply with a dequantising epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * reads this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant generator with the CUDA path.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -shared -fPIC.
 * Every floating-point step is a single IEEE operation in the stated
 * precision; OpenMP only splits independent output rows between threads and
 * never changes the order of any per-element arithmetic.
 *
 * Sources (web pages, cited by title and section):
 *  [P1] "[Kernel] Add w8a8 CUTLASS kernels" -- the cutlass_scaled_mm_dq
 *       feature list (symmetric activations and weights; per-tensor or
 *       per-token activation scales; per-tensor or per-output-channel weight
 *       scales; bf16/fp16 outputs), the per_tensor_quantize example in the
 *       review thread (divide, clamp to the e4m3 finite range, cast), and the
 *       column-major-B remark in the same thread.
 *  [P2] "[Kernel] Support Fp8 Checkpoints (Dynamic + Static)" -- dynamic
 *       (runtime absmax) vs static (given) activation scales; one shared
 *       weight scale for merged QKV / gate-up layers (review discussion).
 *  [P3] "Enable scaled FP8 (e4m3fn) KV cache on ROCm (AMD GPU)" -- section
 *       "Scaling semantics": scale = AbsMax / 448 (OCP e4m3 MAXNORM),
 *       quant = fp8(x / scale), dequant = fp8_dequant(q) * scale; and the
 *       answer that a missing scale means a scale of 1.0.
 *
 * Readings where the pages are silent (each one also pinned by a test):
 *  - division is a correctly rounded fp32 x / scale (not x * (1/scale));
 *  - e4m3 rounding is round-to-nearest, ties to the even code; |v| >= 448
 *    (and +-inf) saturates to +-448; NaN encodes as 0x7F; the sign of zero
 *    is kept (a negative value that rounds to zero gives 0x80);
 *  - int8 rounding is round-to-nearest-even, saturated to [-128, 127], NaN
 *    gives 0; the int8 scale divisor is 127;
 *  - absmax ignores NaN and starts at 0; absmax == 0 gives scale 1.0;
 *  - epilogue: y = ((float)acc * scale_a) * scale_b in fp32, in that order,
 *    then one round-to-nearest-even to bf16 or fp16.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_E4M3 = 0, ORC_INT8 = 1, ORC_BF16 = 2, ORC_FP16 = 3 };
enum { ORC_PER_TENSOR = 0, ORC_PER_ROW = 1 };

/* ------------------------------------------------------------------ */
/* 16-bit float decode (exact)                                        */
/* ------------------------------------------------------------------ */

float orc_bf16_to_f32(uint16_t h) {
  /* bf16 is the upper half of an fp32 word. */
  uint32_t w = (uint32_t)h << 16;
  float f;
  memcpy(&f, &w, 4);
  return f;
}

float orc_f16_to_f32(uint16_t h) {
  /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return (float)(sign ? -v : v);
}

static float load16(const uint16_t* p, int dtype) {
  return dtype == ORC_BF16 ? orc_bf16_to_f32(*p) : orc_f16_to_f32(*p);
}

/* ------------------------------------------------------------------ */
/* fp32 -> 16-bit float, round to nearest even (own implementation)   */
/* ------------------------------------------------------------------ */

/* Round a finite non-negative double a to the nearest multiple of 2^q_exp,
 * ties to even (rint under the default rounding mode), exactly. */
static double round_to_quantum(double a, int q_exp) {
  return ldexp(rint(ldexp(a, -q_exp)), q_exp);
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t w;
  memcpy(&w, &f, 4);
  uint16_t sign = (uint16_t)((w >> 16) & 0x8000);
  if (isnan(f)) return (uint16_t)(sign | 0x7FC0);
  double a = fabs((double)f);
  if (a == 0.0) return sign;
  if (isinf(f)) return (uint16_t)(sign | 0x7F80);
  /* bf16: 8 significant bits, min normal 2^-126, subnormal quantum 2^-133. */
  int e;
  frexp(a, &e);            /* a = fr * 2^e, fr in [0.5, 1) -> unbiased exp e-1 */
  int ue = e - 1;
  int q_exp = (ue < -126 ? -126 : ue) - 7;
  double r = round_to_quantum(a, q_exp);
  /* Largest finite bf16 is (2 - 2^-7) * 2^127; anything that rounds above it
   * is infinity. */
  if (r > ldexp(255.0, 120)) return (uint16_t)(sign | 0x7F80);
  if (r == 0.0) return sign; /* underflow to a signed zero */
  frexp(r, &e);
  ue = e - 1;
  uint16_t bits;
  if (ue < -126) {
    bits = (uint16_t)ldexp(r, 133); /* subnormal fraction */
  } else {
    uint16_t frac = (uint16_t)(ldexp(r, 7 - ue) - 128.0);
    bits = (uint16_t)(((ue + 127) << 7) | frac);
  }
  return (uint16_t)(sign | bits);
}

uint16_t orc_f32_to_f16(float f) {
  uint32_t w;
  memcpy(&w, &f, 4);
  uint16_t sign = (uint16_t)((w >> 16) & 0x8000);
  if (isnan(f)) return (uint16_t)(sign | 0x7E00);
  double a = fabs((double)f);
  if (a == 0.0) return sign;
  if (isinf(f)) return (uint16_t)(sign | 0x7C00);
  /* binary16: 11 significant bits, min normal 2^-14, subnormal quantum 2^-24,
   * max finite 65504. */
  int e;
  frexp(a, &e);
  int ue = e - 1;
  int q_exp = (ue < -14 ? -14 : ue) - 10;
  double r = round_to_quantum(a, q_exp);
  if (r > 65504.0) return (uint16_t)(sign | 0x7C00);
  if (r == 0.0) return sign;
  frexp(r, &e);
  ue = e - 1;
  uint16_t bits;
  if (ue < -14) {
    bits = (uint16_t)ldexp(r, 24);
  } else {
    uint16_t frac = (uint16_t)(ldexp(r, 10 - ue) - 1024.0);
    bits = (uint16_t)(((ue + 15) << 10) | frac);
  }
  return (uint16_t)(sign | bits);
}

static uint16_t store16(float f, int dtype) {
  return dtype == ORC_BF16 ? orc_f32_to_bf16(f) : orc_f32_to_f16(f);
}

/* ------------------------------------------------------------------ */
/* OCP e4m3fn: value table and table-driven encoder                    */
/* ------------------------------------------------------------------ */

/* Value of a non-negative e4m3fn code 0x00..0x7E: 4 exponent bits (bias 7),
 * 3 fraction bits, no infinities; 0x7F is NaN.  Exponent field 0 is
 * subnormal: m/8 * 2^-6.  Otherwise (1 + m/8) * 2^(e-7).  The largest code
 * 0x7E is 1.75 * 2^8 = 448, the MAXNORM of the KV-cache page. */
double orc_e4m3_value(int code) {
  int s = (code >> 7) & 1;
  int c = code & 0x7F;
  if (c == 0x7F) return NAN;
  int e = c >> 3, m = c & 7;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

static double g_e4m3_table[127];  /* ascending values of codes 0x00..0x7E */
static double g_e4m3_decode[256]; /* value of every code, NaN for 0x7F/0xFF */
static int g_table_ready = 0;

static void build_table(void) {
  if (g_table_ready) return;
  for (int c = 0; c < 127; ++c) g_e4m3_table[c] = orc_e4m3_value(c);
  for (int c = 0; c < 256; ++c) g_e4m3_decode[c] = orc_e4m3_value(c);
  g_table_ready = 1;
}

void orc_init(void) { build_table(); }

/* Nearest table entry to v, ties to the even code, saturating at 448. */
uint8_t orc_encode_e4m3(float v) {
  if (isnan(v)) return 0x7F;
  int s = signbit(v) ? 1 : 0;
  double a = fabs((double)v);
  int idx;
  if (a >= 448.0) {
    idx = 126;
  } else {
    /* largest i with table[i] <= a (table[0] = 0 <= a always) */
    int lo = 0, hi = 126;
    while (lo < hi) {
      int mid = (lo + hi + 1) / 2;
      if (g_e4m3_table[mid] <= a) lo = mid; else hi = mid - 1;
    }
    idx = lo;
    if (g_e4m3_table[idx] != a) {
      /* a lies strictly between table[idx] and table[idx+1]; both
       * differences are exact in double. */
      double dlo = a - g_e4m3_table[idx];
      double dhi = g_e4m3_table[idx + 1] - a;
      if (dhi < dlo || (dhi == dlo && ((idx + 1) % 2 == 0))) idx = idx + 1;
    }
  }
  return (uint8_t)(idx | (s << 7));
}

int8_t orc_encode_int8(float v) {
  if (isnan(v)) return 0;
  double r = rint((double)v); /* round half to even */
  if (r > 127.0) r = 127.0;
  if (r < -128.0) r = -128.0;
  return (int8_t)r;
}

static double decode_q(uint8_t c, int qdtype) {
  return qdtype == ORC_E4M3 ? g_e4m3_decode[c] : (double)(int8_t)c;
}

/* ------------------------------------------------------------------ */
/* absmax, scale, quantise, dequantise                                 */
/* ------------------------------------------------------------------ */

/* Max of |x| over one row, ignoring NaN, starting from 0. */
static float row_absmax(const uint16_t* x, int dtype, int64_t cols) {
  float m = 0.0f;
  for (int64_t j = 0; j < cols; ++j) {
    float a = fabsf(load16(x + j, dtype));
    if (a > m) m = a; /* false for NaN */
  }
  return m;
}

void orc_absmax(const uint16_t* x, int dtype, int64_t rows, int64_t cols,
                int64_t ld, int gran, float* out) {
  if (gran == ORC_PER_ROW) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) out[i] = row_absmax(x + i * ld, dtype, cols);
  } else {
    float m = 0.0f;
    for (int64_t i = 0; i < rows; ++i) {
      float r = row_absmax(x + i * ld, dtype, cols);
      if (r > m) m = r;
    }
    out[0] = m;
  }
}

float orc_scale_from_absmax(float amax, int qdtype) {
  float qmax = qdtype == ORC_E4M3 ? 448.0f : 127.0f;
  return amax > 0.0f ? amax / qmax : 1.0f;
}

/* q[i, j] = encode(x[i, j] / scale[i or 0]).  With dynamic=1 the scales are
 * computed first (absmax / qmax per row or over the tensor) and written to
 * `scale`; with dynamic=0 they are read from it. */
void orc_quant(const uint16_t* x, int x_dtype, int64_t rows, int64_t cols,
               int64_t ld_x, uint8_t* q, int q_dtype, int64_t ld_q,
               float* scale, int gran, int dynamic) {
  build_table();
  if (dynamic) {
    int64_t n = gran == ORC_PER_ROW ? rows : 1;
    orc_absmax(x, x_dtype, rows, cols, ld_x, gran, scale);
    for (int64_t i = 0; i < n; ++i) scale[i] = orc_scale_from_absmax(scale[i], q_dtype);
  }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows; ++i) {
    float s = scale[gran == ORC_PER_ROW ? i : 0];
    for (int64_t j = 0; j < cols; ++j) {
      float v = load16(x + i * ld_x + j, x_dtype) / s;
      q[i * ld_q + j] = q_dtype == ORC_E4M3 ? orc_encode_e4m3(v)
                                            : (uint8_t)orc_encode_int8(v);
    }
  }
}

/* y[i, j] = round16(float(decode(q[i, j])) * scale[i or 0]). */
void orc_dequant(const uint8_t* q, int q_dtype, int64_t rows, int64_t cols,
                 int64_t ld_q, const float* scale, int gran, uint16_t* y,
                 int y_dtype, int64_t ld_y) {
  build_table();
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows; ++i) {
    float s = scale[gran == ORC_PER_ROW ? i : 0];
    for (int64_t j = 0; j < cols; ++j) {
      float d = (float)decode_q(q[i * ld_q + j], q_dtype);
      y[i * ld_y + j] = store16(d * s, y_dtype);
    }
  }
}

/* ------------------------------------------------------------------ */
/* scaled matmul                                                       */
/* ------------------------------------------------------------------ */

/* One output element.  A is [M, K] row-major with leading dim lda; B is
 * stored [N, K] with K contiguous (the "column-major B" of the CUTLASS
 * review thread).  The e4m3 dot product is accumulated in double, which is
 * exact: every e4m3 value is a multiple of 2^-9 below 2^9 in magnitude, so
 * each product is a multiple of 2^-18 below 2^18, and fewer than 2^17 such
 * terms sum exactly in 53 bits.  The int8 dot product is accumulated in
 * int64 and is exact. */
static void one_element(const uint8_t* A, int64_t lda, const uint8_t* B,
                        int64_t ldb, const float* sa, int a_gran,
                        const float* sb, int b_gran, int64_t m, int64_t n,
                        int64_t K, int q_dtype, int out_dtype, double* acc_out,
                        int64_t* iacc_out, float* y_out, uint16_t* out16) {
  const uint8_t* a = A + m * lda;
  const uint8_t* b = B + n * ldb;
  float accf;
  if (q_dtype == ORC_E4M3) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += g_e4m3_decode[a[k]] * g_e4m3_decode[b[k]];
    if (acc_out) *acc_out = acc;
    if (iacc_out) *iacc_out = 0;
    accf = (float)acc;
  } else {
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k) acc += (int64_t)(int8_t)a[k] * (int64_t)(int8_t)b[k];
    if (iacc_out) *iacc_out = acc;
    if (acc_out) *acc_out = (double)acc;
    accf = (float)acc;
  }
  float ya = sa[a_gran == ORC_PER_ROW ? m : 0];
  float yb = sb[b_gran == ORC_PER_ROW ? n : 0];
  float y = (accf * ya) * yb;
  if (y_out) *y_out = y;
  if (out16) *out16 = store16(y, out_dtype);
}

/* Full M x N product.  Any of acc / iacc / y / out may be NULL; when given
 * they are dense [M, N] row-major. */
void orc_scaled_mm(const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                   const float* sa, int a_gran, const float* sb, int b_gran,
                   int64_t M, int64_t N, int64_t K, int q_dtype, int out_dtype,
                   double* acc, int64_t* iacc, float* y, uint16_t* out) {
  build_table();
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      int64_t o = m * N + n;
      one_element(A, lda, B, ldb, sa, a_gran, sb, b_gran, m, n, K, q_dtype,
                  out_dtype, acc ? acc + o : 0, iacc ? iacc + o : 0,
                  y ? y + o : 0, out ? out + o : 0);
    }
  }
}

/* Selected elements (idx_m[i], idx_n[i]) for i < count; outputs have length
 * count. */
void orc_scaled_mm_sample(const uint8_t* A, int64_t lda, const uint8_t* B,
                          int64_t ldb, const float* sa, int a_gran,
                          const float* sb, int b_gran, int64_t K, int q_dtype,
                          int out_dtype, const int64_t* idx_m,
                          const int64_t* idx_n, int64_t count, double* acc,
                          int64_t* iacc, float* y, uint16_t* out) {
  build_table();
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t i = 0; i < count; ++i) {
    one_element(A, lda, B, ldb, sa, a_gran, sb, b_gran, idx_m[i], idx_n[i], K,
                q_dtype, out_dtype, acc ? acc + i : 0, iacc ? iacc + i : 0,
                y ? y + i : 0, out ? out + i : 0);
  }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------ */
/* merged-layer shards: requantise to one shared scale                 */
/* ------------------------------------------------------------------ */

/* A merged weight (QKV or gate-up) stored [rows, cols] whose consecutive row
 * shards i = 0..nshards-1 (shard_rows[i] rows each) were quantised with their
 * own scales shard_scales[i] is rewritten to one shared scale
 * s_max = max_i shard_scales[i] ("[Kernel] Support Fp8 Checkpoints (Dynamic
 * + Static)", review discussion: w_scale = max(wq_scale, wk_scale,
 * wv_scale); wq' = (wq_scale / w_scale) * wq):
 *   r_i = s_i / s_max                      (one fp32 division)
 *   q'[row, j] = encode(decode(q) * r_i)    (one fp32 multiplication, then
 *                                            the same encoder as quantise)
 * scale_out[0] = s_max. */
void orc_requant_shards(const uint8_t* q, int q_dtype, int64_t cols, int64_t ld,
                        const float* shard_scales, const int64_t* shard_rows,
                        int nshards, uint8_t* out, int64_t ld_out,
                        float* scale_out) {
  build_table();
  float smax = shard_scales[0];
  for (int i = 1; i < nshards; ++i)
    if (shard_scales[i] > smax) smax = shard_scales[i];
  scale_out[0] = smax;
  int64_t row0 = 0;
  for (int i = 0; i < nshards; ++i) {
    float r = shard_scales[i] / smax;
#pragma omp parallel for schedule(static)
    for (int64_t rr = 0; rr < shard_rows[i]; ++rr) {
      int64_t row = row0 + rr;
      for (int64_t j = 0; j < cols; ++j) {
        float v = (float)decode_q(q[row * ld + j], q_dtype) * r;
        out[row * ld_out + j] = q_dtype == ORC_E4M3 ? orc_encode_e4m3(v)
                                                    : (uint8_t)orc_encode_int8(v);
      }
    }
    row0 += shard_rows[i];
  }
}
