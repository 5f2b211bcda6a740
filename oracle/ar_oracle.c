/*
 * CPU oracle, plain serial C.  TEST INFRASTRUCTURE ONLY (see ar_oracle.h):
 * nothing in the product library includes, links or calls this file.
 *
 * Build with strict IEEE arithmetic: -std=c11 -O2 -ffp-contract=off and no
 * -ffast-math.  All fp32 additions below are single binary32 operations;
 * the norm is evaluated in binary64 and rounded once.
 *
 * Every rounding to a storage format goes through round_grid(), which is the
 * definition of round-to-nearest-even on a binary floating grid with p
 * significand bits and a minimum normal exponent: the magnitude is divided by
 * the grid spacing of its binade (exact, a power of two), rounded to the
 * nearest integer with ties to even, and multiplied back.
 */
#include "ar_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* rounding on a binary grid                                               */
/* ---------------------------------------------------------------------- */

/* nearest integer, ties to even; v >= 0 and small enough that v - floor(v)
 * is exact in binary64 (always true here: v < 2^30). */
static double rne_int(double v) {
  double fl = floor(v);
  double d = v - fl;
  if (d > 0.5) return fl + 1.0;
  if (d < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* floor(log2(a)) for finite a > 0 */
static int ilog2(double a) {
  int ex;
  (void)frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
  return ex - 1;
}

/* Round a >= 0 to the grid of a format with p significand bits (hidden bit
 * included) whose smallest normal binade is 2^emin.  Below 2^emin the
 * spacing stays 2^(emin - p + 1) (gradual underflow). */
static double round_grid(double a, int p, int emin) {
  if (a == 0.0) return 0.0;
  int e = ilog2(a);
  if (e < emin) e = emin;
  double spacing = ldexp(1.0, e - (p - 1));
  return rne_int(a / spacing) * spacing;
}

/* Bit fields (exponent << (p-1) | fraction) of a grid value v >= 0 that is
 * representable and below the format's overflow threshold. */
static uint32_t encode_fields(double v, int p, int emin, int bias) {
  if (v == 0.0) return 0;
  int e = ilog2(v);
  if (e < emin) { /* subnormal: exponent field 0, fraction = v / spacing */
    return (uint32_t)(v / ldexp(1.0, emin - (p - 1)));
  }
  double frac = v / ldexp(1.0, e) - 1.0; /* in [0, 1) */
  uint32_t f = (uint32_t)(frac * (double)(1u << (p - 1)));
  return ((uint32_t)(e + bias) << (p - 1)) | f;
}

/* Value of the bit fields (no sign): exponent field E, fraction f. */
static double decode_fields(uint32_t E, uint32_t f, int p, int emin, int bias) {
  if (E == 0) return (double)f * ldexp(1.0, emin - (p - 1));
  return (1.0 + (double)f / (double)(1u << (p - 1))) * ldexp(1.0, (int)E - bias);
}

/* ---------------------------------------------------------------------- */
/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits; p = 8,         */
/* emin = -126; overflow (rounded magnitude >= 2^128) gives infinity.       */
/* ---------------------------------------------------------------------- */

static uint16_t bf16_from_double(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
  double r = round_grid(a, 8, -126);
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
  return (uint16_t)(sign | encode_fields(r, 8, -126, 127));
}

uint16_t orc_f32_to_bf16(float x) { return bf16_from_double((double)x); }
uint16_t orc_f64_to_bf16(double x) { return bf16_from_double(x); }

float orc_bf16_to_f32(uint16_t h) {
  uint32_t E = (h >> 7) & 0xFFu, f = h & 0x7Fu;
  double s = (h & 0x8000u) ? -1.0 : 1.0;
  if (E == 0xFFu) return (float)(f ? NAN : s * INFINITY);
  return (float)(s * decode_fields(E, f, 8, -126, 127));
}

/* ---------------------------------------------------------------------- */
/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits; p = 11,   */
/* emin = -14; rounded magnitude >= 2^16 gives infinity.                    */
/* ---------------------------------------------------------------------- */

static uint16_t f16_from_double(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
  double r = round_grid(a, 11, -14);
  if (r >= 65536.0) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | encode_fields(r, 11, -14, 15));
}

uint16_t orc_f32_to_f16(float x) { return f16_from_double((double)x); }
uint16_t orc_f64_to_f16(double x) { return f16_from_double(x); }

float orc_f16_to_f32(uint16_t h) {
  uint32_t E = (h >> 10) & 0x1Fu, f = h & 0x3FFu;
  double s = (h & 0x8000u) ? -1.0 : 1.0;
  if (E == 0x1Fu) return (float)(f ? NAN : s * INFINITY);
  return (float)(s * decode_fields(E, f, 11, -14, 15));
}

/* ---------------------------------------------------------------------- */
/* OCP OFP8 E4M3: 1 sign, 4 exponent (bias 7), 3 fraction bits; p = 4,      */
/* emin = -6; no infinities; S.1111.111 is NaN, so the largest finite value */
/* is 1.75 * 2^8 = 448.  Saturating conversion: finite magnitudes that      */
/* round above 448, and infinities, become +-448.                           */
/* ---------------------------------------------------------------------- */

uint8_t orc_f32_to_e4m3(float x) {
  uint8_t sign = signbit(x) ? 0x80u : 0u;
  if (isnan(x)) return (uint8_t)(sign | 0x7Fu);
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
  double r = round_grid(a, 4, -6);
  if (r > 448.0) r = 448.0; /* not reachable for a < 448; kept for clarity */
  return (uint8_t)(sign | encode_fields(r, 4, -6, 7));
}

float orc_e4m3_to_f32(uint8_t c) {
  uint32_t E = (c >> 3) & 0xFu, f = c & 0x7u;
  double s = (c & 0x80u) ? -1.0 : 1.0;
  if (E == 0xFu && f == 0x7u) return NAN;
  return (float)(s * decode_fields(E, f, 4, -6, 7));
}

void orc_f32_to_bf16_n(uint16_t* out, const float* in, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}
void orc_bf16_to_f32_n(float* out, const uint16_t* in, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(in[i]);
}
void orc_f32_to_f16_n(uint16_t* out, const float* in, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(in[i]);
}
void orc_f16_to_f32_n(float* out, const uint16_t* in, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(in[i]);
}
void orc_f32_to_e4m3_n(uint8_t* out, const float* in, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(in[i]);
}
void orc_e4m3_to_f32_n(float* out, const uint8_t* in, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_f32(in[i]);
}

/* ---------------------------------------------------------------------- */
/* element access                                                         */
/* ---------------------------------------------------------------------- */

static float load_elem(const void* p, int64_t i, int dtype) {
  if (dtype == ORC_F32) return ((const float*)p)[i];
  uint16_t h = ((const uint16_t*)p)[i];
  return dtype == ORC_BF16 ? orc_bf16_to_f32(h) : orc_f16_to_f32(h);
}

/* round a binary32 value to the element type and store it */
static void store_elem(void* p, int64_t i, float v, int dtype) {
  if (dtype == ORC_F32) {
    ((float*)p)[i] = v;
  } else {
    ((uint16_t*)p)[i] = dtype == ORC_BF16 ? orc_f32_to_bf16(v) : orc_f32_to_f16(v);
  }
}

/* round a binary64 value once to the 16-bit element type and store it */
static void store_elem_f64(void* p, int64_t i, double v, int dtype) {
  ((uint16_t*)p)[i] = dtype == ORC_BF16 ? orc_f64_to_bf16(v) : orc_f64_to_f16(v);
}

static int elem_size(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* ---------------------------------------------------------------------- */
/* step 1: sum-reduce in fp32, rank order, one rounding                     */
/* ---------------------------------------------------------------------- */

int orc_reduce_sum(void* out, const void* const* partials, int n, int64_t numel, int dtype) {
  if (!out || !partials || n < 1 || numel < 0) return -1;
  if (dtype != ORC_F32 && dtype != ORC_F16 && dtype != ORC_BF16) return -1;
  for (int r = 0; r < n; ++r)
    if (!partials[r]) return -1;
  for (int64_t i = 0; i < numel; ++i) {
    float acc = load_elem(partials[0], i, dtype);
    for (int r = 1; r < n; ++r) acc = acc + load_elem(partials[r], i, dtype);
    store_elem(out, i, acc, dtype);
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* step 2: residual add + RMSNorm (the unfused rmsnorm2d_fwd_with_add)      */
/* ---------------------------------------------------------------------- */

/* One row.  z_row receives the rounded residual sum as 16-bit bits.  With y32 non-NULL
 * the normalised row is also written as binary32 (one rounding of the binary64 value);
 * with skip_norm the output is z itself (no normalisation, weight unused). */
static void add_rmsnorm_row_ex(void* y, float* y32, void* res_out, uint16_t* z_row, const void* s,
                               const void* res_in, const void* w, int64_t row, int64_t h, float eps,
                               int gemma, int skip_norm, int dtype) {
  int64_t base = row * h;
  for (int64_t j = 0; j < h; ++j) {
    float sv = load_elem(s, base + j, dtype);
    if (res_in) {
      float zv = sv + load_elem(res_in, base + j, dtype);
      store_elem(z_row, j, zv, dtype);
    } else {
      z_row[j] = ((const uint16_t*)s)[base + j];
    }
    if (res_out) ((uint16_t*)res_out)[base + j] = z_row[j];
  }
  if (!y && !y32) return;
  if (skip_norm) {
    for (int64_t j = 0; j < h; ++j) {
      if (y) ((uint16_t*)y)[base + j] = z_row[j];
      if (y32) y32[base + j] = load_elem(z_row, j, dtype);
    }
    return;
  }
  double sumsq = 0.0;
  for (int64_t j = 0; j < h; ++j) {
    double zv = (double)load_elem(z_row, j, dtype);
    sumsq += zv * zv;
  }
  double mean_sq = sumsq / (double)h;
  double inv_rms = 1.0 / sqrt(mean_sq + (double)eps);
  for (int64_t j = 0; j < h; ++j) {
    double zv = (double)load_elem(z_row, j, dtype);
    double wv = (double)load_elem(w, j, dtype);
    double factor = gemma ? 1.0 + wv : wv;
    double yv = zv * inv_rms * factor;
    if (y) store_elem_f64(y, base + j, yv, dtype);
    if (y32) y32[base + j] = (float)yv;
  }
}

static void add_rmsnorm_row(void* y, void* res_out, uint16_t* z_row, const void* s, const void* res_in,
                            const void* w, int64_t row, int64_t h, float eps, int gemma, int dtype) {
  add_rmsnorm_row_ex(y, NULL, res_out, z_row, s, res_in, w, row, h, eps, gemma, 0, dtype);
}

int orc_add_rmsnorm(void* y, void* res_out, const void* s, const void* res_in, const void* w,
                    int64_t m, int64_t h, float eps, int gemma, int dtype) {
  if (!s || !w || m < 0 || h < 1) return -1;
  if (dtype != ORC_F16 && dtype != ORC_BF16) return -1;
  uint16_t* z_row = (uint16_t*)malloc((size_t)h * sizeof(uint16_t));
  if (!z_row) return -2;
  for (int64_t r = 0; r < m; ++r) add_rmsnorm_row(y, res_out, z_row, s, res_in, w, r, h, eps, gemma, dtype);
  free(z_row);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* step 3: dynamic per-token FP8 quantisation of the rounded output         */
/* ---------------------------------------------------------------------- */

static void quant_row(uint8_t* q, float* scale, const void* y, int64_t row, int64_t h, int dtype) {
  int64_t base = row * h;
  float amax = 0.0f;
  for (int64_t j = 0; j < h; ++j) {
    float a = fabsf(load_elem(y, base + j, dtype));
    if (a > amax) amax = a;
  }
  float sc = amax / 448.0f;
  scale[row] = sc;
  for (int64_t j = 0; j < h; ++j) {
    if (amax == 0.0f) {
      q[base + j] = 0;
    } else {
      float v = load_elem(y, base + j, dtype) / sc;
      q[base + j] = orc_f32_to_e4m3(v);
    }
  }
}

int orc_per_token_quant(uint8_t* q, float* scale, const void* y, int64_t m, int64_t h, int dtype) {
  if (!q || !scale || !y || m < 0 || h < 1) return -1;
  if (dtype != ORC_F16 && dtype != ORC_BF16) return -1;
  for (int64_t r = 0; r < m; ++r) quant_row(q, scale, y, r, h, dtype);
  return 0;
}

/* Dynamic per-group quantisation of one rounded row of h elements: every run of g
 * consecutive elements (h a multiple of g) gets its own scale amax_group / 448 and its
 * codes, with the per-token rules inside the group. */
static void quant_row_groups(uint8_t* q, float* scale, const void* y, int64_t h, int64_t g, int dtype) {
  for (int64_t k = 0; k < h / g; ++k) {
    const int64_t j0 = k * g, j1 = j0 + g;
    float amax = 0.0f;
    for (int64_t j = j0; j < j1; ++j) {
      float a = fabsf(load_elem(y, j, dtype));
      if (a > amax) amax = a;
    }
    float sc = amax / 448.0f;
    scale[k] = sc;
    for (int64_t j = j0; j < j1; ++j) q[j] = amax == 0.0f ? 0 : orc_f32_to_e4m3(load_elem(y, j, dtype) / sc);
  }
}

int orc_per_group_quant(uint8_t* q, float* scale, const void* y, int64_t m, int64_t h, int64_t group, int dtype) {
  if (!q || !scale || !y || m < 0 || h < 1 || group < 1 || h % group != 0) return -1;
  if (dtype != ORC_F16 && dtype != ORC_BF16) return -1;
  for (int64_t r = 0; r < m; ++r)
    quant_row_groups(q + r * h, scale + r * (h / group), (const uint16_t*)y + r * h, h, group, dtype);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* the composition                                                         */
/* ---------------------------------------------------------------------- */

int orc_fused_reduce_rmsnorm(void* y, void* res_out, uint8_t* q, float* scale,
                             const void* const* partials, int n, const void* res_in, const void* w,
                             int64_t m, int64_t h, float eps, int gemma, int quant, int dtype) {
  return orc_fused_ex(y, NULL, res_out, q, scale, partials, n, res_in, w, m, h, eps, gemma, quant, 0, 0, dtype);
}

int orc_fused_ex(void* y, float* y32, void* res_out, uint8_t* q, float* scale, const void* const* partials,
                 int n, const void* res_in, const void* w, int64_t m, int64_t h, float eps, int gemma,
                 int quant, int skip_norm, int64_t group, int dtype) {
  if (!partials || n < 1 || (!w && !skip_norm) || m < 0 || h < 1) return -1;
  if (group < 0 || (group > 0 && h % group != 0)) return -1;
  if (dtype != ORC_F16 && dtype != ORC_BF16) return -1;
  if (quant && (!q || !scale)) return -1;
  if (!quant && !y && !y32) return -1;
  for (int r = 0; r < n; ++r)
    if (!partials[r]) return -1;

  size_t row_bytes = (size_t)h * (size_t)elem_size(dtype);
  uint16_t* s_row = (uint16_t*)malloc(row_bytes);
  uint16_t* z_row = (uint16_t*)malloc(row_bytes);
  uint16_t* y_row = (uint16_t*)malloc(row_bytes);
  uint16_t* ro_row = (uint16_t*)malloc(row_bytes);
  const void** row_ptrs = (const void**)malloc((size_t)n * sizeof(void*));
  if (!s_row || !z_row || !y_row || !ro_row || !row_ptrs) {
    free(s_row); free(z_row); free(y_row); free(ro_row); free(row_ptrs);
    return -2;
  }
  for (int64_t r = 0; r < m; ++r) {
    int64_t base = r * h;
    for (int k = 0; k < n; ++k) row_ptrs[k] = (const uint16_t*)partials[k] + base;
    orc_reduce_sum(s_row, row_ptrs, n, h, dtype);
    const void* res_row = res_in ? (const void*)((const uint16_t*)res_in + base) : NULL;
    add_rmsnorm_row_ex(y_row, y32 ? y32 + base : NULL, ro_row, z_row, s_row, res_row, w, 0, h, eps, gemma,
                       skip_norm, dtype);
    if (res_out) memcpy((uint16_t*)res_out + base, ro_row, row_bytes);
    if (y) memcpy((uint16_t*)y + base, y_row, row_bytes);
    if (quant && group) quant_row_groups(q + base, scale + r * (h / group), y_row, h, group, dtype);
    else if (quant) quant_row(q + base, scale + r, y_row, 0, h, dtype);
  }
  free(s_row); free(z_row); free(y_row); free(ro_row); free(row_ptrs);
  return 0;
}
