/*
 * CPU oracle for the fused N-way partial reduce + residual add + RMSNorm
 * (+ per-token FP8 e4m3) path.  TEST INFRASTRUCTURE ONLY: the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * library never does, and this code shares nothing with it.
 *
 * What it computes is the *unfused* composition that the fused kernels must
 * reproduce:
 *   1. sum-reduce of the N partials in fp32, rank order 0..N-1, one rounding
 *      to the storage type (page "[OUTDATED] perf: optimize fused AllReduce +
 *      RMSNorm (custom_all_reduce)", Technical Details / 2stage, the flat
 *      reduce-scatter paragraph);
 *   2. rmsnorm2d_fwd_with_add(out, x, res, res_out, w, eps, gemma): residual
 *      add rounded to the storage type, then RMSNorm (page "[HIP]
 *      fix(custom-ar): gfx1250 fused all-reduce + RMSNorm", Changes and the
 *      bench_ar_rms.py listing, which calls the unfused op);
 *   3. dynamic per-token FP8 quantisation of the *rounded* output (same page,
 *      Changes, "Per-token FP8 output").
 *
 * Storage formats are handled from their definitions (IEEE 754 binary16,
 * bfloat16 = the top half of binary32, OCP OFP8 E4M3): no CUDA header, no
 * compiler intrinsic, no hardware conversion.
 *
 * Buffers: 16-bit element types are passed as raw uint16 bit patterns,
 * fp32 as float; all arrays are contiguous row-major.  Functions return 0 on
 * success and a negative number on an invalid argument.
 */
#ifndef AR_ORACLE_H
#define AR_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type codes (the oracle's own numbering). */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ---- storage-format conversions (round-to-nearest-even) ---- */
uint16_t orc_f32_to_bf16(float x);
float orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float x);
float orc_f16_to_f32(uint16_t h);
/* binary64 -> 16-bit format with a single rounding (used for the norm output) */
uint16_t orc_f64_to_bf16(double x);
uint16_t orc_f64_to_f16(double x);
/* OCP OFP8 E4M3 with saturation to +-448 for finite overflow, NaN -> S.1111.111 */
uint8_t orc_f32_to_e4m3(float x);
float orc_e4m3_to_f32(uint8_t c);

/* Array forms (n elements) so the Python side converts without loops. */
void orc_f32_to_bf16_n(uint16_t* out, const float* in, int64_t n);
void orc_bf16_to_f32_n(float* out, const uint16_t* in, int64_t n);
void orc_f32_to_f16_n(uint16_t* out, const float* in, int64_t n);
void orc_f16_to_f32_n(float* out, const uint16_t* in, int64_t n);
void orc_f32_to_e4m3_n(uint8_t* out, const float* in, int64_t n);
void orc_e4m3_to_f32_n(float* out, const uint8_t* in, int64_t n);

/* ---- the method ---- */

/* out[i] = round_T( (((float)x_0[i] + (float)x_1[i]) + ...) + (float)x_{n-1}[i] ),
 * i in [0, numel).  For ORC_F32 the fp32 sum is stored as is.  `out` may be
 * one of the partials. */
int orc_reduce_sum(void* out, const void* const* partials, int n, int64_t numel, int dtype);

/* rmsnorm2d_fwd_with_add on [m, h] rows, dtype ORC_BF16 or ORC_F16:
 *   z = round_T((float)s + (float)res_in)        (z = s when res_in is NULL)
 *   res_out = z                                  (skipped when NULL)
 *   inv = 1 / sqrt(sum_j z_j^2 / h + eps)        (binary64, j ascending)
 *   y = round_T(z * inv * w')  w' = w, or 1 + w when gemma != 0 (binary64)
 * y may be NULL. */
int orc_add_rmsnorm(void* y, void* res_out, const void* s, const void* res_in, const void* w,
                    int64_t m, int64_t h, float eps, int gemma, int dtype);

/* dynamic per-token quantisation of rounded rows y [m, h]:
 *   amax = max_j |y_j|; scale = amax / 448 (binary32);
 *   q_j = e4m3((float)y_j / scale) (binary32 quotient); amax == 0 -> scale 0, q 0. */
int orc_per_token_quant(uint8_t* q, float* scale, const void* y, int64_t m, int64_t h, int dtype);

/* The whole path, composed from the three steps above, row by row.
 * y may be NULL only when quant != 0; res_out, res_in may be NULL;
 * q and scale are required when quant != 0. */
int orc_fused_reduce_rmsnorm(void* y, void* res_out, uint8_t* q, float* scale,
                             const void* const* partials, int n, const void* res_in, const void* w,
                             int64_t m, int64_t h, float eps, int gemma, int quant, int dtype);

/* dynamic per-group quantisation of rounded rows y [m, h] in groups of `group`
 * consecutive elements (h a multiple of group): scale [m, h / group], each group with the
 * per-token rules (amax / 448, binary32 quotient, zero group -> scale 0, codes 0). */
int orc_per_group_quant(uint8_t* q, float* scale, const void* y, int64_t m, int64_t h, int64_t group, int dtype);

/* The whole path with its two options.
 *   y32 (may be NULL): the normalised row as binary32, RN_f32 of the binary64 value
 *       z * inv * w' (no rounding to the 16-bit type first);
 *   skip_norm: no normalisation, the output is z itself (the rounded sum plus residual);
 *       w may then be NULL and eps, gemma are unused.
 * The FP8 epilogue always quantises the 16-bit output (z with skip_norm); group > 0 makes
 * it per-group (scale [m, h / group]) instead of per-token (scale [m]). */
int orc_fused_ex(void* y, float* y32, void* res_out, uint8_t* q, float* scale, const void* const* partials,
                 int n, const void* res_in, const void* w, int64_t m, int64_t h, float eps, int gemma,
                 int quant, int skip_norm, int64_t group, int dtype);

#ifdef __cplusplus
}
#endif
#endif /* AR_ORACLE_H */
