/*
 * dit_oracle.c -- plain CPU oracle for the DiT elementwise hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see dit_oracle.h).  Build with
 *     gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared
 * and never with -ffast-math: every `float` operation below must be one IEEE
 * fp32 operation rounded to nearest-even, and `a * b + c` must stay two
 * roundings.  (GCC contracts to FMA by default in GNU C mode, hence the flag.)
 *
 * Readings taken where the pages leave a step open (each is listed with its
 * justification in the repository's design notes):
 *   R1  residual gate: p = fl(update * gate), s = fl(hidden + p), then one
 *       rounding of s to the storage dtype.  No FMA.
 *   R2  RMS statistic ("fp32 statistics", and the pages' bound of one
 *       bf16 ulp per output element): ms = RN32(sum x^2 / D), the exact mean
 *       of the squares rounded once to fp32 (the sum taken exactly, as a
 *       big integer); v = fl(ms + eps); r = RN32(1 / sqrt(v)), the correctly
 *       rounded fp32 inverse root of the fp32 v.  Both are single roundings
 *       of exact values, so they do not depend on a summation order.  eps
 *       sits inside the root, added to the mean square (the standard
 *       weightless RMSNorm).
 *   R3  modulation order, left to right as the expression is written:
 *       n = fl(x * r); one = fl(1 + scale); t = fl(n * one); y = fl(t + shift);
 *       then one rounding of y to the storage dtype.  1 + scale is formed in
 *       fp32, not in the storage dtype.
 *   R4  fused op: the RMS of the fused op is taken over the residual as
 *       stored (rounded to the dtype), so the fused result equals the
 *       residual gate followed by the modulation.
 *   R5  a [B, 1, D] operand serves rows b*L .. b*L+L-1 of batch b.
 *   R6  fp32 -> bf16/fp16 rounding is round-to-nearest-even, overflow gives
 *       +-inf, subnormals are kept, NaN stays NaN.
 *   R7  FP8 output (the RMSNorm + FP8 quantisation family the prhub summary
 *       of sglang PR #34172 names among its related PRs): OCP E4M3 with no
 *       infinities (bias 7, 3 fraction bits, largest finite 448); a static
 *       per-tensor scale s, applied as q = fl(y * fl(1 / s)) to the fp32
 *       modulation value y (before any rounding to the activation dtype);
 *       q rounded to nearest-even on the E4M3 grid, saturating at +-448
 *       (infinities included), NaN stays NaN.
 */
#include "dit_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* dtype codecs                                                              */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

static float bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* bf16 is the upper half of an fp32 word: widening is exact. */
float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* Round to nearest, ties to even, by adding just under half an ulp of bf16
 * (0x7FFF) plus the lowest kept bit, then truncating.  A carry out of the
 * fraction bumps the exponent, which is the correct rounding up to the next
 * binade (and to infinity past the largest finite bf16). */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t x = f32_bits(f);
  if (isnan(f)) return (uint16_t)((x >> 16) | 0x0040u); /* quiet NaN */
  uint32_t lsb = (x >> 16) & 1u;
  x += 0x7FFFu + lsb;
  return (uint16_t)(x >> 16);
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float orc_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int frac = h & 0x3FF;
  float v;
  if (e == 0)
    v = ldexpf((float)frac, -24); /* zero or subnormal: frac * 2^-24 */
  else if (e == 31)
    v = frac ? NAN : INFINITY;
  else
    v = ldexpf((float)(frac + 1024), e - 25); /* (1.frac) * 2^(e-15) */
  return sign ? -v : v;
}

/* Round |f| to the binary16 grid.  In the binade [2^E, 2^(E+1)) the spacing
 * is 2^(E-10); below 2^-14 (subnormals) it is 2^-24.  Dividing by the spacing
 * (a power of two, so exactly) gives a real number whose nearest integer,
 * ties to even (nearbyintf in the default rounding mode), is the rounded
 * significand. */
uint16_t orc_f32_to_f16(float f) {
  uint16_t sign = (uint16_t)((f32_bits(f) >> 16) & 0x8000u);
  if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
  float a = fabsf(f);
  if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
  if (a < 0x1p-14f) {
    /* k in [0, 1024]; k = 1024 is the smallest normal, whose bit pattern is
     * exactly 0x0400 = exponent field 1, fraction 0. */
    float k = nearbyintf(a * 0x1p24f);
    return (uint16_t)(sign | (uint16_t)k);
  }
  int e2;
  (void)frexpf(a, &e2); /* a = m * 2^e2 with m in [0.5, 1) */
  int E = e2 - 1;       /* a in [2^E, 2^(E+1)) */
  float m = nearbyintf(a / ldexpf(1.0f, E - 10)); /* in [1024, 2048] */
  if (m == 2048.0f) {
    m = 1024.0f;
    E += 1;
  }
  if (E > 15) return (uint16_t)(sign | 0x7C00u); /* past 65504: infinity */
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) |
                    (uint16_t)((int)m - 1024));
}

float orc_load(const void* p, int64_t i, int dtype) {
  switch (dtype) {
    case ORC_BF16: return orc_bf16_to_f32(((const uint16_t*)p)[i]);
    case ORC_FP16: return orc_f16_to_f32(((const uint16_t*)p)[i]);
    default:       return ((const float*)p)[i];
  }
}

void orc_store(void* p, int64_t i, float v, int dtype) {
  switch (dtype) {
    case ORC_BF16: ((uint16_t*)p)[i] = orc_f32_to_bf16(v); break;
    case ORC_FP16: ((uint16_t*)p)[i] = orc_f32_to_f16(v); break;
    default:       ((float*)p)[i] = v; break;
  }
}

/* One rounding of a double to the dtype.  fp32: the C conversion (round to
 * nearest even).  bf16/fp16: first to fp32 by rounding to odd -- truncate
 * toward zero, then set the last bit if anything was discarded -- then to the
 * 16-bit format by round-to-nearest-even.  fp32 keeps at least two bits more
 * than either 16-bit format, so the two steps give the correctly rounded
 * result (Boldo and Melquiond, "When double rounding is odd", 2005). */
void orc_store_double(void* p, int64_t i, double v, int dtype) {
  if (dtype == ORC_FP32 || isnan(v) || isinf(v)) {
    orc_store(p, i, (float)v, dtype);
    return;
  }
  float f = (float)v;
  if (fabs((double)f) > fabs(v)) f = nextafterf(f, 0.0f); /* toward zero */
  if ((double)f != v && !isinf(f)) {
    uint32_t b = f32_bits(f);
    b |= 1u; /* sticky: odd */
    f = bits_f32(b);
  }
  orc_store(p, i, f, dtype);
}

void orc_decode_array(float* dst_f32, const void* src, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) dst_f32[i] = orc_load(src, i, dtype);
}

void orc_encode_array(void* dst, const float* src_f32, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) orc_store(dst, i, src_f32[i], dtype);
}

/* OCP E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; no
 * infinities; exponent 15 with fraction 7 is NaN.  Codes 0..7 are
 * subnormal, k * 2^-9. */
float orc_e4m3_to_f32(uint8_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  float v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexpf((float)m, -9);
  else
    v = ldexpf((float)(8 + m), e - 10);
  return (b & 0x80) ? -v : v;
}

/* Reading R7.  |f| is rounded to the E4M3 grid of its binade with
 * nearbyint (round to nearest, ties to even, in the default rounding mode):
 * spacing 2^-9 below 2^-6 (subnormals), 2^(E-3) in [2^E, 2^(E+1)).  The
 * grid multiple k then maps to the code directly: codes grow with the value,
 * and a binade's 8 steps are the 8 fraction values. */
uint8_t orc_f32_to_e4m3(float f) {
  if (isnan(f)) return 0x7F;
  const uint8_t sign = signbit(f) ? 0x80 : 0;
  const double a = fabs((double)f);
  if (a >= 448.0) return sign | 0x7E; /* saturate, infinities included */
  if (a < ldexp(1.0, -6)) {
    const double k = nearbyint(a / ldexp(1.0, -9)); /* 0..8; 8 is 2^-6 */
    return sign | (uint8_t)k;
  }
  int E;
  (void)frexp(a, &E); /* a = m * 2^E with m in [0.5, 1): binade 2^(E-1) */
  E -= 1;
  double k = nearbyint(a / ldexp(1.0, E - 3)); /* 8..16 */
  int ex = E + 7;
  if (k == 16.0) {
    k = 8.0;
    ex += 1;
  }
  return sign | (uint8_t)((ex << 3) | ((int)k - 8));
}

/* ------------------------------------------------------------------------ */
/* one row of each operation                                                 */
/* ------------------------------------------------------------------------ */

/* Row r of  out = hidden + update * gate  (reading R1).  The gate row is r
 * itself for a full gate and the batch index b = r / L for a [B, 1, D] gate
 * (reading R5). */
static void residual_gate_row(void* out, const void* hidden, const void* update,
                              const void* gate, int64_t r, int64_t L, int64_t D,
                              int dtype, int gate_layout) {
  int64_t grow = (gate_layout == ORC_FULL) ? r : r / L;
  for (int64_t d = 0; d < D; ++d) {
    float h = orc_load(hidden, r * D + d, dtype);
    float u = orc_load(update, r * D + d, dtype);
    float g = orc_load(gate, grow * D + d, dtype);
    float p = u * g;
    float s = h + p;
    orc_store(out, r * D + d, s, dtype);
  }
}

/* ------------------------------------------------------------------------ */
/* the row statistic (reading R2)                                            */
/* ------------------------------------------------------------------------ */

/* Every fp32 value is M * 2^e with M an integer below 2^24 and e >= -149, so
 * its square M^2 * 2^(2e) is an integer multiple of 2^-298 below 2^256.  A
 * row's sum of squares times 2^298 is therefore an integer below 2^585 for
 * rows of fewer than 2^31 elements: SQ_DIGITS base-2^32 digits hold it
 * exactly. */
#define SQ_SCALE 298
#define SQ_DIGITS 19

/* The exact sum of squares of a row (times 2^SQ_SCALE) as base-2^32 digits,
 * least significant first.  Each square is added as 32-bit parts into 64-bit
 * per-digit accumulators; the carries are propagated once at the end. */
static void exact_sum_of_squares(const void* x_row, int64_t D, int dtype,
                                 uint32_t digit[SQ_DIGITS]) {
  uint64_t acc[SQ_DIGITS];
  memset(acc, 0, sizeof acc);
  for (int64_t d = 0; d < D; ++d) {
    const float v = fabsf(orc_load(x_row, d, dtype));
    if (v == 0.0f) continue;
    int e2;
    (void)frexpf(v, &e2);            /* v in [2^(e2-1), 2^e2) */
    int e = e2 - 24;                 /* v = M * 2^e with M < 2^24 ... */
    if (e < -149) e = -149;          /* ... or, below 2^-126, M * 2^-149 */
    const uint64_t M = (uint64_t)ldexpf(v, -e); /* exact: an integer */
    const uint64_t sq = M * M;       /* < 2^48 */
    const int pos = 2 * e + SQ_SCALE; /* bit of the scaled sum where sq starts */
    const int k = pos / 32, s = pos % 32;
    const uint64_t t0 = (sq & 0xFFFFFFFFu) << s; /* < 2^63 */
    const uint64_t t1 = (sq >> 32) << s;          /* < 2^47, weight 2^32 more */
    acc[k] += t0 & 0xFFFFFFFFu;
    acc[k + 1] += (t0 >> 32) + (t1 & 0xFFFFFFFFu);
    acc[k + 2] += t1 >> 32;
  }
  uint64_t carry = 0;
  for (int i = 0; i < SQ_DIGITS; ++i) {
    const uint64_t t = acc[i] + carry;
    digit[i] = (uint32_t)t;
    carry = t >> 32;
  }
}

/* bit b of a little-endian base-2^32 number of n digits (0 outside it) */
static int bit_at(const uint32_t* q, int n, int b) {
  if (b < 0 || b >= 32 * n) return 0;
  return (int)((q[b / 32] >> (b % 32)) & 1u);
}

/* The fp32 value nearest (ties to even) to (digits * 2^-SQ_SCALE) / D.  The
 * digits, with 64 zero bits appended below them, are divided by D by long
 * division; the quotient then has at least 33 bits for any nonzero sum, and
 * the remainder says whether anything lies below it.  The result keeps 24
 * bits from the quotient's leading one, or the bits down to 2^-149 when it is
 * below 2^-126 (subnormal); the bit after the kept ones and the "sticky" OR
 * of everything below decide the rounding. */
static float rn32_mean(const uint32_t digit[SQ_DIGITS], uint32_t D) {
  enum { N = SQ_DIGITS + 2 };
  uint32_t num[N], q[N];
  num[0] = num[1] = 0;
  for (int i = 0; i < SQ_DIGITS; ++i) num[i + 2] = digit[i];
  uint64_t rem = 0;
  for (int i = N - 1; i >= 0; --i) {
    const uint64_t cur = (rem << 32) | num[i];
    q[i] = (uint32_t)(cur / D);
    rem = cur % D;
  }
  const int w0 = SQ_SCALE + 64; /* bit b of q weighs 2^(b - w0) */
  int top = -1;
  for (int b = 32 * N - 1; b >= 0; --b)
    if (bit_at(q, N, b)) {
      top = b;
      break;
    }
  if (top < 0) return 0.0f; /* every element was zero */
  int lsb = top - 23;
  if (lsb - w0 < -149) lsb = w0 - 149;
  uint64_t mant = 0;
  for (int b = top; b >= lsb; --b) mant = 2 * mant + (uint64_t)bit_at(q, N, b);
  const int guard = bit_at(q, N, lsb - 1);
  int sticky = rem != 0;
  for (int b = lsb - 2; b >= 0 && !sticky; --b) sticky = bit_at(q, N, b);
  if (guard && (sticky || (mant & 1u))) mant += 1;
  return (float)ldexp((double)mant, lsb - w0); /* exact, or +inf past FLT_MAX */
}

/* ms = RN32(mean(x^2)) of one row (reading R2): NaN if the row holds a NaN,
 * +inf if it holds an infinity, else the exact mean of the squares rounded
 * once to fp32 (+inf when that passes FLT_MAX). */
float orc_row_mean_square(const void* x_row, int64_t D, int dtype) {
  if (D <= 0 || D > 0x7FFFFFFF) return NAN;
  int inf = 0;
  for (int64_t d = 0; d < D; ++d) {
    const float v = orc_load(x_row, d, dtype);
    if (isnan(v)) return NAN;
    if (isinf(v)) inf = 1;
  }
  if (inf) return INFINITY;
  uint32_t digit[SQ_DIGITS];
  exact_sum_of_squares(x_row, D, dtype, digit);
  return rn32_mean(digit, (uint32_t)D);
}

/* RN32(1 / sqrt(v)): the root and the quotient in double, then one rounding
 * to fp32.  That is the correctly rounded fp32 value for every fp32 v (an
 * exhaustive check over one binade pair, [1, 4), covers all others, since
 * v * 4^k only scales the result by 2^-k). */
static float inverse_root(float v) { return (float)(1.0 / sqrt((double)v)); }

void orc_inverse_root_array(const float* v, float* r, int64_t n) {
  for (int64_t i = 0; i < n; ++i) r[i] = inverse_root(v[i]);
}

/* r = 1 / sqrt(mean(x^2) + eps) for one row (reading R2). */
float orc_row_rms_inverse(const void* x_row, int64_t D, float eps, int dtype) {
  float ms = orc_row_mean_square(x_row, D, dtype);
  float v = ms + eps;
  return inverse_root(v);
}

/* Row r of  out = rms_norm(x, eps) * (1 + scale) + shift  (reading R3). */
static void rmsnorm_modulate_row(void* out, float* t_out, const void* x,
                                 const void* scale, const void* shift,
                                 int64_t r, int64_t L, int64_t D, float eps,
                                 int dtype, int mod_layout, int fp8, float qinv) {
  if (D == 0) return;
  const size_t esize = (dtype == ORC_FP32) ? 4 : 2;
  const void* x_row = (const char*)x + (size_t)(r * D) * esize;
  float rinv = orc_row_rms_inverse(x_row, D, eps, dtype);
  int64_t mrow = (mod_layout == ORC_FULL) ? r : r / L;
  for (int64_t d = 0; d < D; ++d) {
    float xv = orc_load(x, r * D + d, dtype);
    float sc = orc_load(scale, mrow * D + d, dtype);
    float sh = orc_load(shift, mrow * D + d, dtype);
    float n = xv * rinv;
    float one = 1.0f + sc;
    float t = n * one;
    float y = t + sh;
    if (t_out) t_out[r * D + d] = t;
    if (fp8) /* reading R7 */
      ((uint8_t*)out)[r * D + d] = orc_f32_to_e4m3(y * qinv);
    else
      orc_store(out, r * D + d, y, dtype);
  }
}

/* gelu(x) = 0.5 * x * (1 + tanh(z)), z = sqrt(2/pi) * (x + 0.044715 * x^3),
 * in double.  1 + tanh(z) = 2 / (1 + exp(-2z)) exactly, so the value is
 * computed as x / (1 + exp(-2z)): the same function, without the cancellation
 * of 1 + tanh(z) when tanh(z) is close to -1 (x below about -4), where even a
 * double evaluation of the tanh form loses most of its digits. */
int orc_gelu_tanh(void* out, const void* x, int64_t n, int dtype) {
  if (n < 0 || (dtype != ORC_BF16 && dtype != ORC_FP16 && dtype != ORC_FP32)) return -1;
  if (n > 0 && (!out || !x)) return -1;
  const double k = sqrt(2.0 / 3.14159265358979323846);
  for (int64_t i = 0; i < n; ++i) {
    const double v = (double)orc_load(x, i, dtype);
    const double z = k * (v + 0.044715 * v * v * v);
    orc_store_double(out, i, v / (1.0 + exp(-2.0 * z)), dtype);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* argument checks and row iteration                                         */
/* ------------------------------------------------------------------------ */

static int bad_common(int64_t B, int64_t L, int64_t D, int dtype,
                      const int64_t* rows, int64_t nrows) {
  if (B < 0 || L < 0 || D < 0 || nrows < 0) return 1;
  if (dtype != ORC_BF16 && dtype != ORC_FP16 && dtype != ORC_FP32) return 1;
  if (rows) {
    for (int64_t i = 0; i < nrows; ++i)
      if (rows[i] < 0 || rows[i] >= B * L) return 1;
  }
  return 0;
}

static int bad_layout(int layout) {
  return layout != ORC_FULL && layout != ORC_ROW_BCAST;
}

/* Row at position i of the selection: rows[i], or i itself when rows is NULL. */
static int64_t row_at(const int64_t* rows, int64_t i) { return rows ? rows[i] : i; }

static int64_t selection_size(int64_t B, int64_t L, const int64_t* rows,
                              int64_t nrows) {
  return rows ? nrows : B * L;
}

typedef struct {
  int op; /* 0 residual gate, 1 modulate, 2 fused */
  void* out;
  void* out2;
  float* t_out;
  const void *hidden, *update, *gate, *scale, *shift;
  int64_t B, L, D;
  float eps;
  int dtype, layout1, layout2;
  int fp8;    /* modulated output in E4M3 (reading R7) */
  float qinv; /* fl(1 / quant_scale) */
  const int64_t* rows;
  int64_t begin, end; /* positions in the row selection */
} orc_job;

static void run_job(const orc_job* j) {
  for (int64_t i = j->begin; i < j->end; ++i) {
    int64_t r = row_at(j->rows, i);
    if (j->op == 0) {
      residual_gate_row(j->out, j->hidden, j->update, j->gate, r, j->L, j->D,
                        j->dtype, j->layout1);
    } else if (j->op == 1) {
      rmsnorm_modulate_row(j->out, j->t_out, j->hidden, j->scale, j->shift, r,
                           j->L, j->D, j->eps, j->dtype, j->layout1, j->fp8, j->qinv);
    } else {
      /* reading R4: the stored (rounded) residual is the modulation input */
      residual_gate_row(j->out, j->hidden, j->update, j->gate, r, j->L, j->D,
                        j->dtype, j->layout1);
      rmsnorm_modulate_row(j->out2, j->t_out, j->out, j->scale, j->shift, r,
                           j->L, j->D, j->eps, j->dtype, j->layout2, j->fp8, j->qinv);
    }
  }
}

static void* job_thread(void* arg) {
  run_job((const orc_job*)arg);
  return NULL;
}

/* Split the selection into nthreads contiguous parts; part 0 runs on the
 * calling thread. */
static int run_threads(int nthreads, orc_job base) {
  int64_t n = base.end;
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  orc_job* jobs = (orc_job*)calloc((size_t)nthreads, sizeof(orc_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].begin = n * t / nthreads;
    jobs[t].end = n * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, job_thread, &jobs[t]) != 0) break;
    started = t;
  }
  run_job(&jobs[0]);
  /* parts whose thread could not be started run here */
  for (int t = started + 1; t < nthreads; ++t) run_job(&jobs[t]);
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  free(jobs);
  free(tids);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* public entry points                                                       */
/* ------------------------------------------------------------------------ */

int orc_residual_gate_add_mt(int nthreads, void* out, const void* hidden,
                             const void* update, const void* gate, int64_t B,
                             int64_t L, int64_t D, int dtype, int gate_layout,
                             const int64_t* rows, int64_t nrows) {
  if (bad_common(B, L, D, dtype, rows, nrows) || bad_layout(gate_layout)) return -1;
  if (B * L * D > 0 && (!out || !hidden || !update || !gate)) return -1;
  orc_job j = {0};
  j.op = 0;
  j.out = out;
  j.hidden = hidden;
  j.update = update;
  j.gate = gate;
  j.B = B;
  j.L = L;
  j.D = D;
  j.dtype = dtype;
  j.layout1 = gate_layout;
  j.rows = rows;
  j.end = selection_size(B, L, rows, nrows);
  return run_threads(nthreads, j);
}

int orc_residual_gate_add(void* out, const void* hidden, const void* update,
                          const void* gate, int64_t B, int64_t L, int64_t D,
                          int dtype, int gate_layout, const int64_t* rows,
                          int64_t nrows) {
  return orc_residual_gate_add_mt(1, out, hidden, update, gate, B, L, D, dtype,
                                  gate_layout, rows, nrows);
}

static int modulate_impl(int nthreads, void* out, float* t_out, const void* x,
                         const void* scale, const void* shift, int64_t B,
                         int64_t L, int64_t D, float eps, int dtype,
                         int mod_layout, const int64_t* rows, int64_t nrows,
                         int fp8, float qinv) {
  if (bad_common(B, L, D, dtype, rows, nrows) || bad_layout(mod_layout)) return -1;
  if (D > 0x7FFFFFFF) return -1; /* the statistic's divisor is 32-bit */
  if (B * L * D > 0 && (!out || !x || !scale || !shift)) return -1;
  orc_job j = {0};
  j.op = 1;
  j.out = out;
  j.t_out = t_out;
  j.fp8 = fp8;
  j.qinv = qinv;
  j.hidden = x;
  j.scale = scale;
  j.shift = shift;
  j.B = B;
  j.L = L;
  j.D = D;
  j.eps = eps;
  j.dtype = dtype;
  j.layout1 = mod_layout;
  j.rows = rows;
  j.end = selection_size(B, L, rows, nrows);
  return run_threads(nthreads, j);
}

int orc_rmsnorm_modulate(void* out, float* t_out, const void* x,
                         const void* scale, const void* shift, int64_t B,
                         int64_t L, int64_t D, float eps, int dtype,
                         int mod_layout, const int64_t* rows, int64_t nrows) {
  return modulate_impl(1, out, t_out, x, scale, shift, B, L, D, eps, dtype,
                       mod_layout, rows, nrows, 0, 1.0f);
}

int orc_rmsnorm_modulate_mt(int nthreads, void* out, const void* x,
                            const void* scale, const void* shift, int64_t B,
                            int64_t L, int64_t D, float eps, int dtype,
                            int mod_layout, const int64_t* rows, int64_t nrows) {
  return modulate_impl(nthreads, out, NULL, x, scale, shift, B, L, D, eps,
                       dtype, mod_layout, rows, nrows, 0, 1.0f);
}

static int fused_impl(int nthreads, void* residual_out, void* modulated_out,
                      float* t_out, const void* hidden, const void* update,
                      const void* gate, const void* scale, const void* shift,
                      int64_t B, int64_t L, int64_t D, float eps, int dtype,
                      int gate_layout, int mod_layout, const int64_t* rows,
                      int64_t nrows, int fp8, float qinv) {
  if (bad_common(B, L, D, dtype, rows, nrows) || bad_layout(gate_layout) ||
      bad_layout(mod_layout) || D > 0x7FFFFFFF)
    return -1;
  if (B * L * D > 0 && (!residual_out || !modulated_out || !hidden || !update ||
                        !gate || !scale || !shift))
    return -1;
  orc_job j = {0};
  j.op = 2;
  j.out = residual_out;
  j.out2 = modulated_out;
  j.t_out = t_out;
  j.fp8 = fp8;
  j.qinv = qinv;
  j.hidden = hidden;
  j.update = update;
  j.gate = gate;
  j.scale = scale;
  j.shift = shift;
  j.B = B;
  j.L = L;
  j.D = D;
  j.eps = eps;
  j.dtype = dtype;
  j.layout1 = gate_layout;
  j.layout2 = mod_layout;
  j.rows = rows;
  j.end = selection_size(B, L, rows, nrows);
  return run_threads(nthreads, j);
}

int orc_gate_add_rmsnorm_modulate(void* residual_out, void* modulated_out,
                                  float* t_out, const void* hidden,
                                  const void* update, const void* gate,
                                  const void* scale, const void* shift,
                                  int64_t B, int64_t L, int64_t D, float eps,
                                  int dtype, int gate_layout, int mod_layout,
                                  const int64_t* rows, int64_t nrows) {
  return fused_impl(1, residual_out, modulated_out, t_out, hidden, update, gate,
                    scale, shift, B, L, D, eps, dtype, gate_layout, mod_layout,
                    rows, nrows, 0, 1.0f);
}

int orc_gate_add_rmsnorm_modulate_mt(int nthreads, void* residual_out,
                                     void* modulated_out, const void* hidden,
                                     const void* update, const void* gate,
                                     const void* scale, const void* shift,
                                     int64_t B, int64_t L, int64_t D, float eps,
                                     int dtype, int gate_layout, int mod_layout,
                                     const int64_t* rows, int64_t nrows) {
  return fused_impl(nthreads, residual_out, modulated_out, NULL, hidden, update,
                    gate, scale, shift, B, L, D, eps, dtype, gate_layout,
                    mod_layout, rows, nrows, 0, 1.0f);
}

/* Reading R7: the modulation (or the fused op) with its modulated output in
 * E4M3, q = fl(y * fl(1 / quant_scale)). */
int orc_rmsnorm_modulate_fp8(uint8_t* out, float* t_out, const void* x,
                             const void* scale, const void* shift, int64_t B,
                             int64_t L, int64_t D, float eps, int dtype,
                             int mod_layout, float quant_scale,
                             const int64_t* rows, int64_t nrows) {
  const float qinv = 1.0f / quant_scale;
  return modulate_impl(1, out, t_out, x, scale, shift, B, L, D, eps, dtype,
                       mod_layout, rows, nrows, 1, qinv);
}

int orc_gate_add_rmsnorm_modulate_fp8(void* residual_out, uint8_t* out,
                                      float* t_out, const void* hidden,
                                      const void* update, const void* gate,
                                      const void* scale, const void* shift,
                                      int64_t B, int64_t L, int64_t D, float eps,
                                      int dtype, int gate_layout, int mod_layout,
                                      float quant_scale, const int64_t* rows,
                                      int64_t nrows) {
  const float qinv = 1.0f / quant_scale;
  return fused_impl(1, residual_out, out, t_out, hidden, update, gate, scale,
                    shift, B, L, D, eps, dtype, gate_layout, mod_layout, rows,
                    nrows, 1, qinv);
}
