/*
 * dit_oracle.h -- plain CPU oracle for the DiT elementwise hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library (whose interface is include/dit_elementwise.h).
 *
 * Every function computes its outputs element by element, in IEEE fp32 with
 * round-to-nearest-even, with no fused multiply-add (build with
 * -ffp-contract=off and without -ffast-math) and with one final rounding to the
 * storage dtype.  The operations are:
 *
 *   residual gate      out = hidden + update * gate
 *       sglang PR #29361 "Add diffusion residual-gate CUDA fast path for LTX2",
 *       section Motivation (the hot pattern, for contiguous [B, L, D] tensors
 *       with a full gate or a [B, 1, D] gate).
 *   adaLN modulation   out = rms_norm(x, eps) * (1 + scale) + shift
 *       prhub summary of sglang PR #34172 (LTX-2 quality=high fused
 *       RMSNorm+modulate), section "key source snippet", the eager branch of
 *       _ltx2_rms_norm_modulate; the norm is the weightless RMSNormNoWeight of
 *       section "implementation breakdown", item 2.
 *   fused              the residual gate, rounded to the dtype and stored, then
 *       the modulation of that stored residual (one pass; the readings used
 *       where the pages are silent are listed in the file header of
 *       dit_oracle.c).
 *
 * Tensors are contiguous, row-major [B, L, D]; a "row" is one (b, l) pair and
 * has D elements.  A [B, 1, D] operand (layout ORC_ROW_BCAST) is used for every
 * row of batch b, i.e. for rows b*L .. b*L+L-1.
 *
 * Row selection: `rows` lists the rows to compute (each in [0, B*L)), `nrows`
 * their count.  rows == NULL means every row.  Outputs are written at the same
 * positions as in a full [B, L, D] output, so the caller passes full-size
 * output buffers and reads back the rows it asked for.
 *
 * Return value: 0 on success, -1 on a bad argument (nothing written).
 */
#ifndef DIT_ORACLE_H
#define DIT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_FP32 = 2 };
enum { ORC_FULL = 0, ORC_ROW_BCAST = 1 };

/* dtype codecs (textbook IEEE-754 round-to-nearest-even, subnormals kept) */
float    orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);
float    orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float f);
/* element i of a buffer of dtype `dtype`, as fp32 (exact) */
float    orc_load(const void* p, int64_t i, int dtype);
/* round v once to `dtype` and store it as element i */
void     orc_store(void* p, int64_t i, float v, int dtype);
/* n elements at a time: dst_f32[i] = orc_load(src, i); orc_store(dst, i, src_f32[i]) */
void     orc_decode_array(float* dst_f32, const void* src, int64_t n, int dtype);
void     orc_encode_array(void* dst, const float* src_f32, int64_t n, int dtype);

int orc_residual_gate_add(void* out, const void* hidden, const void* update,
                          const void* gate, int64_t B, int64_t L, int64_t D,
                          int dtype, int gate_layout,
                          const int64_t* rows, int64_t nrows);

/* t_out (optional, fp32, full [B, L, D] size) receives t = n * (1 + scale)
 * before the shift is added; tests use |t| as the scale of the rounding error
 * when the final add cancels. */
int orc_rmsnorm_modulate(void* out, float* t_out, const void* x,
                         const void* scale, const void* shift,
                         int64_t B, int64_t L, int64_t D, float eps,
                         int dtype, int mod_layout,
                         const int64_t* rows, int64_t nrows);

int orc_gate_add_rmsnorm_modulate(void* residual_out, void* modulated_out,
                                  float* t_out, const void* hidden,
                                  const void* update, const void* gate,
                                  const void* scale, const void* shift,
                                  int64_t B, int64_t L, int64_t D, float eps,
                                  int dtype, int gate_layout, int mod_layout,
                                  const int64_t* rows, int64_t nrows);

/* tanh-approximated GELU, elementwise over n elements:
 *   gelu(x) = 0.5 * x * (1 + tanh(sqrt(2/pi) * (x + 0.044715 * x^3)))
 * (the FFN activation of the LTX-2 blocks: prhub summary of sglang PR
 * #34172, "implementation breakdown" item 3, LTX2FeedForward's tanh-GELU),
 * evaluated in double and rounded once to the dtype. */
int orc_gelu_tanh(void* out, const void* x, int64_t n, int dtype);
/* one rounding of a double to the dtype (round-to-nearest-even) */
void orc_store_double(void* p, int64_t i, double v, int dtype);

/* OCP E4M3 (no infinities, largest finite 448): exact decoding, and one
 * rounding of an fp32 value to nearest-even with saturation at +-448; NaN
 * gives 0x7F. */
float   orc_e4m3_to_f32(uint8_t b);
uint8_t orc_f32_to_e4m3(float f);

/* The modulation and the fused op with the modulated output quantised to
 * E4M3: q = fl(y * fl(1 / quant_scale)) of the fp32 value y, rounded once
 * to E4M3 (RMSNorm + FP8 quantisation: the fusion family that the prhub
 * summary of sglang PR #34172 lists among its related PRs).  `out` holds
 * one byte per element. */
int orc_rmsnorm_modulate_fp8(uint8_t* out, float* t_out, const void* x,
                             const void* scale, const void* shift, int64_t B,
                             int64_t L, int64_t D, float eps, int dtype,
                             int mod_layout, float quant_scale,
                             const int64_t* rows, int64_t nrows);
int orc_gate_add_rmsnorm_modulate_fp8(void* residual_out, uint8_t* out,
                                      float* t_out, const void* hidden,
                                      const void* update, const void* gate,
                                      const void* scale, const void* shift,
                                      int64_t B, int64_t L, int64_t D, float eps,
                                      int dtype, int gate_layout, int mod_layout,
                                      float quant_scale, const int64_t* rows,
                                      int64_t nrows);

/* The per-row statistic, exposed for the tests: ms = RN32(mean(x^2)), the
 * exact mean of the squares of one row of D elements (0 < D < 2^31) rounded
 * once to fp32 (NaN if the row holds a NaN, +inf if it holds an infinity);
 * r = RN32(1/sqrt(fl(ms + eps))); and the inverse-root step alone, r[i] =
 * RN32(1/sqrt(v[i])) for n fp32 values. */
float orc_row_mean_square(const void* x_row, int64_t D, int dtype);
float orc_row_rms_inverse(const void* x_row, int64_t D, float eps, int dtype);
void  orc_inverse_root_array(const float* v, float* r, int64_t n);

/* Multi-threaded drivers for the CPU baseline: the same functions, with the
 * selected rows split into `nthreads` contiguous parts, one POSIX thread each.
 * They add no arithmetic of their own. */
int orc_residual_gate_add_mt(int nthreads, void* out, const void* hidden,
                             const void* update, const void* gate, int64_t B,
                             int64_t L, int64_t D, int dtype, int gate_layout,
                             const int64_t* rows, int64_t nrows);
int orc_rmsnorm_modulate_mt(int nthreads, void* out, const void* x,
                            const void* scale, const void* shift, int64_t B,
                            int64_t L, int64_t D, float eps, int dtype,
                            int mod_layout, const int64_t* rows, int64_t nrows);
int orc_gate_add_rmsnorm_modulate_mt(int nthreads, void* residual_out,
                                     void* modulated_out, const void* hidden,
                                     const void* update, const void* gate,
                                     const void* scale, const void* shift,
                                     int64_t B, int64_t L, int64_t D, float eps,
                                     int dtype, int gate_layout, int mod_layout,
                                     const int64_t* rows, int64_t nrows);

#ifdef __cplusplus
}
#endif
#endif /* DIT_ORACLE_H */
