/*
 * mla_oracle.c -- plain CPU oracle for the MLA latent-KV data-movement path.
 *
 * TEST INFRASTRUCTURE ONLY (see mla_oracle.h).  Single-threaded, no blocking,
 * no fusion, no reordering beyond what each definition states.  Every loop runs
 * in the order the definition is written: tokens, then heads, then elements.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared mla_oracle.c -lm
 * (-ffp-contract=off keeps every fp32 division/multiplication a separately
 * rounded IEEE operation, as the definitions below require).
 */
#include "mla_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================== */
/* Rounding to a binary floating-point format.                              */
/* ======================================================================== */

/*
 * Round a finite double |x| to the nearest number that has `p` significant bits
 * and an exponent of at least `emin`; ties go to the even last bit.  Numbers
 * below 2^emin are therefore rounded on the fixed grid 2^(emin-p+1) (the
 * subnormal grid of the format).  The exponent is unbounded above; overflow is
 * the caller's business.
 *
 * Method: pick the quantum q = 2^(max(floor(log2|x|), emin) - (p-1)); x/q is
 * exact (power-of-two scaling); rint() in the default rounding mode rounds it
 * to the nearest integer with ties to even; multiply back (exact).
 */
static double round_to_precision(double x, int p, int emin) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  (void)frexp(x, &e); /* |x| = m * 2^e with 0.5 <= m < 1, so floor(log2|x|) = e-1 */
  int ex = e - 1;
  if (ex < emin) ex = emin;
  double quantum = ldexp(1.0, ex - (p - 1));
  double n = rint(x / quantum);
  return n * quantum;
}

/* ---- bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits ----------- */

uint16_t orc_bf16_from_f64(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
  /* 8 significant bits; smallest normal 2^-126. */
  double r = round_to_precision(x, 8, -126);
  if (fabs(r) > (double)FLT_MAX) return (uint16_t)(sign | 0x7F80u); /* overflow -> inf */
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

uint16_t orc_bf16_from_f32(float x) { return orc_bf16_from_f64((double)x); }

double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---- IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits ------ */

/* Round to nearest even with 11 significant bits, smallest normal 2^-14
 * (subnormal quantum 2^-24); a rounded magnitude above the largest finite
 * value 65504 is an infinity (IEEE overflow under round to nearest). */
uint16_t orc_f16_from_f64(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
  double r = round_to_precision(x, 11, -14);
  double a = fabs(r);
  if (a > 65504.0) return (uint16_t)(sign | 0x7C00u);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1: unbiased exponent e - 1 */
  if (e - 1 < -14) /* subnormal: a = n * 2^-24 exactly */
    return (uint16_t)(sign | (uint16_t)ldexp(a, 24));
  uint16_t exp_field = (uint16_t)(e - 1 + 15);
  uint16_t mant = (uint16_t)(ldexp(a, 10 - (e - 1)) - 1024.0); /* a / 2^(e-1) * 2^10 - 2^10 */
  return (uint16_t)(sign | (exp_field << 10) | mant);
}

double orc_f16_to_f64(uint16_t h) {
  double sign = (h & 0x8000u) ? -1.0 : 1.0;
  int ef = (h >> 10) & 0x1F, m = h & 0x3FF;
  if (ef == 0x1F) return m ? NAN : sign * INFINITY;
  if (ef == 0) return sign * ldexp((double)m, -24);
  return sign * ldexp(1024.0 + m, ef - 15 - 10);
}

/* ---- OCP OFP8 formats --------------------------------------------------- */

typedef struct {
  int p;         /* significant bits including the implicit one */
  int emin;      /* exponent of the smallest normal */
  int bias;      /* exponent bias */
  int mbits;     /* stored mantissa bits */
  double maxfin; /* largest finite magnitude */
} fp8_format;

/* [OFP8] Table 1: E4M3 bias 7, max normal 1.75*2^8 = 448, min normal 2^-6,
 * min subnormal 2^-9, no infinities, NaN = S.1111.111.
 * E5M2 bias 15, max normal 1.75*2^15 = 57344, min normal 2^-14, min subnormal
 * 2^-16, infinities S.11111.00, NaN = S.11111.{01,10,11}. */
static fp8_format fp8_params(int fmt) {
  fp8_format f;
  if (fmt == ORC_FP8_E4M3) {
    f.p = 4; f.emin = -6; f.bias = 7; f.mbits = 3; f.maxfin = 448.0;
  } else {
    f.p = 3; f.emin = -14; f.bias = 15; f.mbits = 2; f.maxfin = 57344.0;
  }
  return f;
}

/*
 * fp32 -> fp8 with round-to-nearest-even and saturation of finite overflow
 * (and of +-inf) to +-max: the conversion the grouped insert applies to
 * value/k_scale and the pack applies to value/out_scale ("PR #55356" Source
 * snippets, the scaled_convert branch; "PR #51772" Implementation item 1, the
 * pairwise fp8 cast).  Every NaN, whatever its sign, becomes the canonical
 * NaN code 0x7F: the pages route the cast through the native pairwise
 * converters ("PR #51772" Implementation item 1), which produce that code for
 * a NaN input, and the OFP8 definition leaves the NaN sign open.  The rounding
 * is done on the exact fp32 value, never through an intermediate format.
 */
uint8_t orc_fp8_from_f32(float xf, int fmt) {
  fp8_format F = fp8_params(fmt);
  double x = (double)xf;
  if (isnan(x)) return 0x7Fu;
  uint8_t sign = signbit(x) ? 0x80u : 0u;
  double a = fabs(x);
  double r = isinf(a) ? a : round_to_precision(a, F.p, F.emin);
  if (r > F.maxfin) r = F.maxfin; /* saturate */
  if (r == 0.0) return sign;
  int e;
  (void)frexp(r, &e);
  int ex = e - 1;
  unsigned expf, mant;
  if (ex < F.emin) { /* subnormal: r = mant * 2^(emin - mbits) */
    expf = 0;
    mant = (unsigned)(r / ldexp(1.0, F.emin - F.mbits));
  } else { /* normal: r = (1 + mant/2^mbits) * 2^ex */
    expf = (unsigned)(ex + F.bias);
    mant = (unsigned)((r / ldexp(1.0, ex) - 1.0) * (double)(1u << F.mbits));
  }
  return (uint8_t)(sign | (expf << F.mbits) | mant);
}

/* Exact value of an fp8 code, from the field definitions in [OFP8]. */
double orc_fp8_to_f64(uint8_t c, int fmt) {
  fp8_format F = fp8_params(fmt);
  int neg = (c >> 7) & 1;
  unsigned expf = ((unsigned)c >> F.mbits) & ((1u << (7 - F.mbits)) - 1u);
  unsigned mant = (unsigned)c & ((1u << F.mbits) - 1u);
  double v;
  if (fmt == ORC_FP8_E4M3) {
    if (expf == 15u && mant == 7u) return neg ? -NAN : NAN;
  } else if (expf == 31u) {
    if (mant != 0u) return neg ? -NAN : NAN;
    return neg ? -INFINITY : INFINITY;
  }
  if (expf == 0u)
    v = ldexp((double)mant, F.emin - F.mbits);
  else
    v = ldexp(1.0 + (double)mant / (double)(1u << F.mbits), (int)expf - F.bias);
  return neg ? -v : v;
}

/* fp8 -> bf16 widening with no scale: every finite fp8 value (of either
 * format) is exactly representable in bf16, so this is exact.  This is the
 * plain dtype cast the chunked-context loop applies to a gathered fp8 latent
 * ("PR #51772" Implementation item 5: the conditional cast to the kv_b_proj
 * input dtype). */
uint16_t orc_bf16_from_fp8(uint8_t c, int fmt) {
  double v = orc_fp8_to_f64(c, fmt);
  uint16_t sign = (c & 0x80u) ? 0x8000u : 0u;
  if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
  if (isinf(v)) return (uint16_t)(sign | 0x7F80u);
  return orc_bf16_from_f64(v);
}

/* fp8 -> fp16, exact (every e4m3 and e5m2 value is an fp16 value); a NaN code
 * gives the quiet NaN with the code's sign. */
uint16_t orc_f16_from_fp8(uint8_t c, int fmt) {
  double v = orc_fp8_to_f64(c, fmt);
  if (isnan(v)) return (uint16_t)(((c & 0x80u) ? 0x8000u : 0u) | 0x7E00u);
  return orc_f16_from_f64(v);
}

void orc_fp8_encode_f32_array(const float* x, int64_t n, int fmt, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_from_f32(x[i], fmt);
}

void orc_fp8_decode_array(const uint8_t* c, int64_t n, int fmt, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_to_f64(c[i], fmt);
}

void orc_bf16_from_f64_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_f64(x[i]);
}

void orc_bf16_from_f32_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_f32(x[i]);
}

/* ======================================================================== */
/* RMSNorm and RoPE ("PR #50585" Source snippets, _precompute_fused_context_kv:
 * a grouped RMSNorm of kv_c with one weight row per layer, then a RoPE of k_pe
 * with the same positions for every layer).                                 */
/* ======================================================================== */

/*
 * cos/sin table of a rotary embedding: row p holds cos(p*f_i) for i < rot/2,
 * then sin(p*f_i), with f_i = base^(-2i/rot).  Computed in double and rounded
 * once to fp32.
 */
void orc_rope_cos_sin_cache(int64_t max_position, int32_t rot_dim, double base, float* out) {
  int32_t half = rot_dim / 2;
  for (int64_t p = 0; p < max_position; ++p) {
    for (int32_t i = 0; i < half; ++i) {
      double inv_freq = pow(base, -2.0 * (double)i / (double)rot_dim);
      double theta = (double)p * inv_freq;
      out[p * rot_dim + i] = (float)cos(theta);
      out[p * rot_dim + half + i] = (float)sin(theta);
    }
  }
}

/*
 * RMSNorm of one row: y_i = x_i / sqrt(mean_j(x_j^2) + eps) * gamma_i, computed
 * in double from the bf16 inputs and rounded once to bf16.  eps is the fp32
 * value the caller passes.
 */
void orc_rms_norm_row(const uint16_t* x, const uint16_t* gamma, int32_t n, float eps,
                      uint16_t* y) {
  double sum_sq = 0.0;
  for (int32_t i = 0; i < n; ++i) {
    double v = orc_bf16_to_f64(x[i]);
    sum_sq += v * v;
  }
  double inv_rms = 1.0 / sqrt(sum_sq / (double)n + (double)eps);
  for (int32_t i = 0; i < n; ++i) {
    double v = orc_bf16_to_f64(x[i]);
    y[i] = orc_bf16_from_f64(v * inv_rms * orc_bf16_to_f64(gamma[i]));
  }
}

/*
 * Neox-style rotation of one row over rot_dim elements: element i is paired with
 * element i + rot/2 (i < rot/2) and the pair is rotated by the angle whose
 * cos/sin sit in cos_sin_row[i] and cos_sin_row[rot/2 + i]:
 *   y_i         = x_i * cos - x_{i+rot/2} * sin
 *   y_{i+rot/2} = x_{i+rot/2} * cos + x_i * sin
 * computed in double and rounded once to bf16.
 */
void orc_rope_neox_row(const uint16_t* x, const float* cos_sin_row, int32_t rot_dim,
                       uint16_t* y) {
  int32_t half = rot_dim / 2;
  for (int32_t i = 0; i < half; ++i) {
    double c = (double)cos_sin_row[i];
    double s = (double)cos_sin_row[half + i];
    double x1 = orc_bf16_to_f64(x[i]);
    double x2 = orc_bf16_to_f64(x[half + i]);
    y[i] = orc_bf16_from_f64(x1 * c - x2 * s);
    y[half + i] = orc_bf16_from_f64(x2 * c + x1 * s);
  }
}

/* ======================================================================== */
/* Grouped multi-layer cache insert ("PR #55356" Implementation items 2-3,  */
/* Source snippets: concat_and_cache_mla_grouped_kernel).                   */
/* ======================================================================== */

/*
 * One layer's insert, the per-layer operation the grouped insert must equal
 * ("PR #55356" test_concat_and_cache_mla_grouped: the reference is one
 * single-layer insert per layer).  For each token t in order:
 *   slot s = slot_mapping[t]; s < 0 is padding and is skipped;
 *   s >= num_blocks*block_size is skipped and reported (ORC_ERR_SLOT_OOB);
 *   with RoPE on, a position outside [0, max_position) is skipped and reported;
 *   row = [RMSNorm(kv_c[t]) or kv_c[t] | RoPE(k_pe[t]) or k_pe[t]]  (bf16);
 *   destination = cache + (s / block_size) * block_stride
 *                       + (s % block_size) * entry_stride   (elements),
 *   kv_c at element 0 and k_pe at element kv_lora_rank;
 *   a bf16 cache stores the bf16 bits, an fp8 cache stores
 *   fp8(float(element) / k_scale) for every element.
 */
uint32_t orc_insert_layer(const uint16_t* kv_c, int64_t kvc_token_stride,
                          const uint16_t* k_pe, int64_t kpe_token_stride, int32_t num_tokens,
                          int32_t kv_lora_rank, int32_t pe_dim, const int64_t* slot_mapping,
                          void* cache, int32_t cache_dtype, int64_t num_blocks,
                          int32_t block_size, int64_t block_stride, int64_t entry_stride,
                          float k_scale, const uint16_t* gamma, float eps,
                          const int64_t* positions, const float* cos_sin_cache,
                          int64_t max_position) {
  uint32_t err = 0;
  int32_t entry = kv_lora_rank + pe_dim;
  uint16_t* row = (uint16_t*)malloc((size_t)entry * sizeof(uint16_t));
  if (!row) return 0xFFFFFFFFu;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= num_blocks * (int64_t)block_size) {
      err |= ORC_ERR_SLOT_OOB;
      continue;
    }
    const float* cs = NULL;
    if (positions) {
      int64_t pos = positions[t];
      if (pos < 0 || pos >= max_position) {
        err |= ORC_ERR_POS_OOB;
        continue;
      }
      cs = cos_sin_cache + pos * (int64_t)pe_dim;
    }
    const uint16_t* x = kv_c + (int64_t)t * kvc_token_stride;
    const uint16_t* r = k_pe + (int64_t)t * kpe_token_stride;
    if (gamma)
      orc_rms_norm_row(x, gamma, kv_lora_rank, eps, row);
    else
      memcpy(row, x, (size_t)kv_lora_rank * sizeof(uint16_t));
    if (positions)
      orc_rope_neox_row(r, cs, pe_dim, row + kv_lora_rank);
    else
      memcpy(row + kv_lora_rank, r, (size_t)pe_dim * sizeof(uint16_t));

    int64_t dst = (s / block_size) * block_stride + (s % block_size) * entry_stride;
    if (cache_dtype == ORC_BF16) {
      uint16_t* c = (uint16_t*)cache + dst;
      for (int32_t i = 0; i < entry; ++i) c[i] = row[i];
    } else {
      uint8_t* c = (uint8_t*)cache + dst;
      for (int32_t i = 0; i < entry; ++i) {
        float v = (float)orc_bf16_to_f64(row[i]);
        float q = v / k_scale;
        c[i] = orc_fp8_from_f32(q, cache_dtype);
      }
    }
  }
  free(row);
  return err;
}

/*
 * The grouped insert, by definition one orc_insert_layer per layer, in layer
 * order.  Layer l reads kv_c/k_pe at l * layer stride, slots at
 * l * slot_layer_stride (0 = one mapping shared by every layer, the aliased
 * "shared_slot_mapping" case), gamma row l, k_scales[l] (fp8 only), and writes
 * caches[l].
 */
uint32_t orc_insert_grouped(const uint16_t* kv_c, int64_t kvc_token_stride,
                            int64_t kvc_layer_stride, const uint16_t* k_pe,
                            int64_t kpe_token_stride, int64_t kpe_layer_stride,
                            int32_t num_tokens, int32_t num_layers, int32_t kv_lora_rank,
                            int32_t pe_dim, const int64_t* slot_mapping,
                            int64_t slot_layer_stride, void* const* caches,
                            const float* k_scales, int32_t cache_dtype, int64_t num_blocks,
                            int32_t block_size, int64_t block_stride, int64_t entry_stride,
                            const uint16_t* gamma, int64_t gamma_layer_stride, float eps,
                            const int64_t* positions, const float* cos_sin_cache,
                            int64_t max_position) {
  uint32_t err = 0;
  for (int32_t l = 0; l < num_layers; ++l) {
    err |= orc_insert_layer(
        kv_c + (int64_t)l * kvc_layer_stride, kvc_token_stride,
        k_pe + (int64_t)l * kpe_layer_stride, kpe_token_stride, num_tokens, kv_lora_rank,
        pe_dim, slot_mapping + (int64_t)l * slot_layer_stride, caches[l], cache_dtype,
        num_blocks, block_size, block_stride, entry_stride,
        cache_dtype == ORC_BF16 ? 1.0f : k_scales[l],
        gamma ? gamma + (int64_t)l * gamma_layer_stride : NULL, eps, positions,
        cos_sin_cache, max_position);
  }
  return err;
}

/*
 * The grouped RMSNorm + RoPE of the DSpark context projection on its own
 * ("PR #50585", Implementation item 3 and Source snippets,
 * _precompute_fused_context_kv: the [num_ctx, L, kv_width] projection output
 * split into kv_c and k_pe, each made layer-major, kv_c RMS-normalised with
 * layer l's weight row, k_pe rotated with the token's position, the same
 * positions for every layer).  For every layer l and token t, in order: if a
 * rotation is asked for and the position lies outside [0, max_position), the
 * row is skipped (both outputs untouched, ORC_ERR_POS_OOB); otherwise
 *   kv_c_out[t, l] = rms_norm_row(kv_c[t, l], gamma[l])   (copy when gamma is NULL)
 *   k_pe_out[t, l] = rope_neox_row(k_pe[t, l], table[pos[t]])  (copy when positions is NULL)
 * with element (t, l, i) of each buffer at t * token stride + l * layer stride + i.
 */
uint32_t orc_norm_rope_grouped(const uint16_t* kv_c, int64_t kvc_token_stride,
                               int64_t kvc_layer_stride, const uint16_t* k_pe,
                               int64_t kpe_token_stride, int64_t kpe_layer_stride,
                               int32_t num_tokens, int32_t num_layers, int32_t kv_lora_rank,
                               int32_t pe_dim, const uint16_t* gamma, int64_t gamma_layer_stride,
                               float eps, const int64_t* positions, const float* cos_sin_cache,
                               int64_t max_position, uint16_t* kv_c_out, int64_t oc_token_stride,
                               int64_t oc_layer_stride, uint16_t* k_pe_out,
                               int64_t op_token_stride, int64_t op_layer_stride) {
  uint32_t err = 0;
  for (int32_t l = 0; l < num_layers; ++l) {
    for (int32_t t = 0; t < num_tokens; ++t) {
      const float* cs = NULL;
      if (positions) {
        int64_t pos = positions[t];
        if (pos < 0 || pos >= max_position) {
          err |= ORC_ERR_POS_OOB;
          continue;
        }
        cs = cos_sin_cache + pos * (int64_t)pe_dim;
      }
      const uint16_t* x = kv_c + (int64_t)t * kvc_token_stride + (int64_t)l * kvc_layer_stride;
      const uint16_t* r = k_pe + (int64_t)t * kpe_token_stride + (int64_t)l * kpe_layer_stride;
      uint16_t* yc = kv_c_out + (int64_t)t * oc_token_stride + (int64_t)l * oc_layer_stride;
      uint16_t* yp = k_pe_out + (int64_t)t * op_token_stride + (int64_t)l * op_layer_stride;
      if (gamma)
        orc_rms_norm_row(x, gamma + (int64_t)l * gamma_layer_stride, kv_lora_rank, eps, yc);
      else
        memcpy(yc, x, (size_t)kv_lora_rank * sizeof(uint16_t));
      if (positions)
        orc_rope_neox_row(r, cs, pe_dim, yp);
      else
        memcpy(yp, r, (size_t)pe_dim * sizeof(uint16_t));
    }
  }
  return err;
}

/* ======================================================================== */
/* Context gather and cast ("PR #51772" Implementation item 2:              */
/* _gather_context_latent then the conditional cast to the kv_b_proj dtype). */
/* ======================================================================== */

/* Copy one element, widening fp8 -> bf16 exactly when the formats differ. */
static int is16(int32_t d) { return d == ORC_BF16 || d == ORC_F16; }

/* Copy one element, widening fp8 -> bf16 / fp16 exactly when the formats differ. */
static void copy_elt(const void* src, int32_t sd, int64_t si, void* dst, int32_t dd,
                     int64_t di) {
  if (sd == dd) {
    if (is16(sd))
      ((uint16_t*)dst)[di] = ((const uint16_t*)src)[si];
    else
      ((uint8_t*)dst)[di] = ((const uint8_t*)src)[si];
  } else if (dd == ORC_BF16) {
    ((uint16_t*)dst)[di] = orc_bf16_from_fp8(((const uint8_t*)src)[si], sd);
  } else { /* fp8 -> fp16 */
    ((uint16_t*)dst)[di] = orc_f16_from_fp8(((const uint8_t*)src)[si], sd);
  }
}

/*
 * Gather the latent rows of a chunk of context from the paged cache.
 * Sequence s owns output rows [cu_chunk_lens[s], cu_chunk_lens[s+1]); output row
 * i of sequence s holds context position p = chunk_starts[s] + (i -
 * cu_chunk_lens[s]), which lives in physical block block_table[s][p /
 * block_size] at offset p % block_size.  The row's first entry_dim elements are
 * copied raw (out_dtype == cache_dtype) or widened exactly to bf16.  A position
 * whose table index is negative or >= block_table_stride (the table's row
 * width), or whose block id is outside [0, num_blocks), is skipped and
 * reported (ORC_ERR_BLOCK_OOB).  Output rows not owned by any sequence are left
 * untouched.
 */
uint32_t orc_context_gather(const void* cache, int32_t cache_dtype, int64_t num_blocks,
                            int32_t block_size, int64_t block_stride, int64_t entry_stride,
                            int32_t entry_dim, const int32_t* block_table,
                            int64_t block_table_stride, const int32_t* cu_chunk_lens,
                            const int32_t* chunk_starts, int32_t num_seqs, int32_t num_tokens,
                            void* out, int64_t out_row_stride, int32_t out_dtype) {
  uint32_t err = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    for (int64_t i = cu_chunk_lens[s]; i < cu_chunk_lens[s + 1]; ++i) {
      if (i < 0 || i >= num_tokens) continue;
      int64_t p = (int64_t)chunk_starts[s] + (i - cu_chunk_lens[s]);
      int64_t k = p >= 0 ? p / block_size : -1;
      if (k < 0 || k >= block_table_stride) {
        err |= ORC_ERR_BLOCK_OOB;
        continue;
      }
      int32_t blk = block_table[(int64_t)s * block_table_stride + k];
      if (blk < 0 || (int64_t)blk >= num_blocks) {
        err |= ORC_ERR_BLOCK_OOB;
        continue;
      }
      int64_t src = (int64_t)blk * block_stride + (p % block_size) * entry_stride;
      for (int32_t e = 0; e < entry_dim; ++e)
        copy_elt(cache, cache_dtype, src + e, out, out_dtype, i * out_row_stride + e);
    }
  }
  return err;
}

/* Row-wise dtype cast used by the step-by-step reference: a copy when the
 * formats agree, the exact fp8 -> bf16 widening otherwise. */
void orc_cast_rows(const void* src, int32_t src_dtype, int64_t src_row_stride, int64_t rows,
                   int64_t cols, void* dst, int32_t dst_dtype, int64_t dst_row_stride) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      copy_elt(src, src_dtype, r * src_row_stride + c, dst, dst_dtype,
               r * dst_row_stride + c);
}

/* ======================================================================== */
/* Chunked-context K/V pack ("PR #51772" Source snippets:                   */
/* fused_mla_kv_concat and fused_mla_kv_concat_quant_fp8).                  */
/* ======================================================================== */

/* bf16 key concat: key[t, h, 0:nope] = k_nope[t, h, :], key[t, h, nope:nope+rope]
 * = k_pe[t, :] (the same k_pe for every head).  Output contiguous [T, H, nope+rope]. */
void orc_concat_key(const uint16_t* k_nope, int64_t kn_token_stride, int64_t kn_head_stride,
                    const uint16_t* k_pe, int64_t kpe_token_stride, int32_t num_tokens,
                    int32_t num_heads, int32_t nope_dim, int32_t rope_dim, uint16_t* key) {
  int64_t kd = (int64_t)nope_dim + rope_dim;
  for (int32_t t = 0; t < num_tokens; ++t)
    for (int32_t h = 0; h < num_heads; ++h) {
      uint16_t* dst = key + ((int64_t)t * num_heads + h) * kd;
      for (int32_t i = 0; i < nope_dim; ++i)
        dst[i] = k_nope[(int64_t)t * kn_token_stride + (int64_t)h * kn_head_stride + i];
      for (int32_t i = 0; i < rope_dim; ++i)
        dst[nope_dim + i] = k_pe[(int64_t)t * kpe_token_stride + i];
    }
}

/* One bf16 element into the output format: the bits themselves for bf16, else
 * fp8(float(e) / out_scale). */
/* One 16-bit input element (bf16 or fp16, in_dtype) to the output: its bits
 * for a 16-bit output (of the same type), else fp8(float(e) / out_scale). */
static void put_from_16(uint16_t e, int32_t in_dtype, void* out, int32_t out_dtype, int64_t i,
                        float out_scale) {
  if (is16(out_dtype)) {
    ((uint16_t*)out)[i] = e;
  } else {
    float v = (float)(in_dtype == ORC_F16 ? orc_f16_to_f64(e) : orc_bf16_to_f64(e));
    ((uint8_t*)out)[i] = orc_fp8_from_f32(v / out_scale, out_dtype);
  }
}

/*
 * The fused pack.  key_out is contiguous [T, H, nope+rope] and v_out (may be
 * NULL) contiguous [T, H, v_dim], both in out_dtype:
 *   key[t,h,i]        = conv(k_nope[t,h,i])            i < nope
 *   key[t,h,nope + j] = k_pe term                      j < rope
 *   V[t,h,i]          = conv(v[t,h,i])                 i < v_dim
 * where conv is the identity for a 16-bit output and fp8(float(e)/out_scale) for
 * fp8 output.  k_nope and v are 16-bit of in_dtype (bf16 or fp16; "PR #51772"
 * Review: bf16 and fp16 inputs), and a 16-bit output has the input's type.
 * The k_pe term: a 16-bit k_pe (of in_dtype) goes through conv; an fp8 k_pe is
 * copied byte for byte into an fp8 key of the same format (the KPE_FP8 branch:
 * no rescale) and widened exactly, with no scale, into a 16-bit key.
 */
void orc_context_kv_pack(const uint16_t* k_nope, int64_t kn_token_stride,
                         int64_t kn_head_stride, const uint16_t* v, int64_t v_token_stride,
                         int64_t v_head_stride, const void* k_pe, int64_t kpe_token_stride,
                         int32_t kpe_dtype, int32_t num_tokens, int32_t num_heads,
                         int32_t nope_dim, int32_t rope_dim, int32_t v_dim, void* key_out,
                         void* v_out, int32_t out_dtype, float out_scale, int32_t in_dtype) {
  int64_t kd = (int64_t)nope_dim + rope_dim;
  for (int32_t t = 0; t < num_tokens; ++t) {
    for (int32_t h = 0; h < num_heads; ++h) {
      int64_t krow = ((int64_t)t * num_heads + h) * kd;
      for (int32_t i = 0; i < nope_dim; ++i) {
        uint16_t e = k_nope[(int64_t)t * kn_token_stride + (int64_t)h * kn_head_stride + i];
        put_from_16(e, in_dtype, key_out, out_dtype, krow + i, out_scale);
      }
      for (int32_t j = 0; j < rope_dim; ++j) {
        int64_t si = (int64_t)t * kpe_token_stride + j;
        int64_t di = krow + nope_dim + j;
        if (is16(kpe_dtype)) {
          put_from_16(((const uint16_t*)k_pe)[si], in_dtype, key_out, out_dtype, di, out_scale);
        } else if (is16(out_dtype)) {
          copy_elt(k_pe, kpe_dtype, si, key_out, out_dtype, di);
        } else {
          ((uint8_t*)key_out)[di] = ((const uint8_t*)k_pe)[si];
        }
      }
      if (v_out) {
        int64_t vrow = ((int64_t)t * num_heads + h) * v_dim;
        for (int32_t i = 0; i < v_dim; ++i) {
          uint16_t e = v[(int64_t)t * v_token_stride + (int64_t)h * v_head_stride + i];
          put_from_16(e, in_dtype, v_out, out_dtype, vrow + i, out_scale);
        }
      }
    }
  }
}

/* ======================================================================== */
/* Next steps of the chunked-context path (the gather fused into the pack,  */
/* and a scaled dequantising gather).                                        */
/* ======================================================================== */

/*
 * fp8 -> bf16 with a dequantisation scale: the exact value of the fp8 code
 * times the scale as ONE fp32 multiplication (round to nearest even), then
 * rounded once to bf16.  A NaN code gives the quiet NaN with the code's sign
 * (as the unscaled widening does); any other NaN product (an infinity times a
 * zero scale, a NaN scale) gives the positive quiet NaN 0x7FC0.
 *
 * The pages cast the gathered fp8 latent to the kv_b_proj input dtype with a
 * plain, unscaled ".to()" ("PR #51772", Implementation items 2 and 5); a cache
 * written with k_scale != 1 ("PR #55356", Source snippets: scaled_convert
 * divides by the layer's k_scale) holds value / k_scale, and multiplying by the
 * same k_scale is the dequantisation a bf16 kv_b_proj then needs.  This is
 * that scaled form of the cast.
 */
uint16_t orc_bf16_from_fp8_scaled(uint8_t c, int fmt, float scale) {
  double v = orc_fp8_to_f64(c, fmt);
  if (isnan(v)) return (uint16_t)(((c & 0x80u) ? 0x8000u : 0u) | 0x7FC0u);
  float p = (float)v * scale; /* (float)v is exact; the product rounds once */
  if (isnan(p)) return 0x7FC0u;
  return orc_bf16_from_f32(p);
}

/* The gather of orc_context_gather with every element widened by
 * orc_bf16_from_fp8_scaled (fp8 cache, bf16 output). */
uint32_t orc_context_gather_scaled(const void* cache, int32_t cache_dtype, int64_t num_blocks,
                                   int32_t block_size, int64_t block_stride, int64_t entry_stride,
                                   int32_t entry_dim, const int32_t* block_table,
                                   int64_t block_table_stride, const int32_t* cu_chunk_lens,
                                   const int32_t* chunk_starts, int32_t num_seqs,
                                   int32_t num_tokens, uint16_t* out, int64_t out_row_stride,
                                   float dequant_scale) {
  uint32_t err = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    for (int64_t i = cu_chunk_lens[s]; i < cu_chunk_lens[s + 1]; ++i) {
      if (i < 0 || i >= num_tokens) continue;
      int64_t p = (int64_t)chunk_starts[s] + (i - cu_chunk_lens[s]);
      int64_t k = p >= 0 ? p / block_size : -1;
      if (k < 0 || k >= block_table_stride) {
        err |= ORC_ERR_BLOCK_OOB;
        continue;
      }
      int32_t blk = block_table[(int64_t)s * block_table_stride + k];
      if (blk < 0 || (int64_t)blk >= num_blocks) {
        err |= ORC_ERR_BLOCK_OOB;
        continue;
      }
      const uint8_t* row =
          (const uint8_t*)cache + (int64_t)blk * block_stride + (p % block_size) * entry_stride;
      for (int32_t e = 0; e < entry_dim; ++e)
        out[i * out_row_stride + e] = orc_bf16_from_fp8_scaled(row[e], cache_dtype, dequant_scale);
    }
  }
  return err;
}

/*
 * The pack with k_pe read straight from the paged cache: token i of the chunk
 * takes its k_pe from the cache row the gather would fetch for it (sequence
 * by cu_chunk_lens, position chunk_starts[s] + i - cu_chunk_lens[s], block by
 * the table), elements rope_offset .. rope_offset + rope_dim.  Everything else
 * -- k_nope, V and every element rule -- is orc_context_kv_pack with that row
 * as k_pe (of the cache's element type).  A token whose row cannot be found
 * still gets its k_nope and V, and the rope slice of its key is left
 * untouched: silently when no sequence owns it, with ORC_ERR_BLOCK_OOB when its
 * block index or block id is out of range.  ("PR #51772" Implementation item
 * 1 reads k_pe from the gathered workspace, still in the cache layout; reading
 * the same bytes from the cache itself drops the workspace's k_pe columns.)
 */
uint32_t orc_context_kv_pack_paged(
    const uint16_t* k_nope, int64_t kn_token_stride, int64_t kn_head_stride, const uint16_t* v,
    int64_t v_token_stride, int64_t v_head_stride, const void* cache, int32_t cache_dtype,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride,
    int32_t rope_offset, const int32_t* block_table, int64_t block_table_stride,
    const int32_t* cu_chunk_lens, const int32_t* chunk_starts, int32_t num_seqs,
    int32_t num_tokens, int32_t num_heads, int32_t nope_dim, int32_t rope_dim, int32_t v_dim,
    void* key_out, void* v_out, int32_t out_dtype, float out_scale, int32_t in_dtype) {
  uint32_t err = 0;
  const size_t ce = is16(cache_dtype) ? 2u : 1u, oe = is16(out_dtype) ? 2u : 1u;
  const int64_t kd = (int64_t)nope_dim + rope_dim;
  uint8_t* key_tmp = (uint8_t*)malloc((size_t)num_heads * kd * oe);
  uint8_t* v_tmp = (uint8_t*)malloc((size_t)num_heads * v_dim * oe + 1);
  if (!key_tmp || !v_tmp) {
    free(key_tmp);
    free(v_tmp);
    return 0xFFFFFFFFu;
  }
  for (int32_t t = 0; t < num_tokens; ++t) {
    /* the cache row of token t, if any */
    const uint8_t* row = NULL;
    for (int32_t s = 0; s < num_seqs && !row; ++s) {
      if (t < cu_chunk_lens[s] || t >= cu_chunk_lens[s + 1]) continue;
      int64_t p = (int64_t)chunk_starts[s] + (t - cu_chunk_lens[s]);
      int64_t k = p >= 0 ? p / block_size : -1;
      if (k < 0 || k >= block_table_stride) {
        err |= ORC_ERR_BLOCK_OOB;
        break;
      }
      int32_t blk = block_table[(int64_t)s * block_table_stride + k];
      if (blk < 0 || (int64_t)blk >= num_blocks) {
        err |= ORC_ERR_BLOCK_OOB;
        break;
      }
      row = (const uint8_t*)cache +
            ((int64_t)blk * block_stride + (p % block_size) * entry_stride + rope_offset) * ce;
    }
    /* pack this one token with its row as k_pe (a dummy row when there is none) */
    uint16_t zero_pe[256] = {0};
    orc_context_kv_pack(k_nope + (int64_t)t * kn_token_stride, kn_token_stride, kn_head_stride,
                        v ? v + (int64_t)t * v_token_stride : NULL, v_token_stride, v_head_stride,
                        row ? (const void*)row : (const void*)zero_pe, 0, cache_dtype, 1,
                        num_heads, nope_dim, rope_dim, v_dim, key_tmp, v_out ? v_tmp : NULL,
                        out_dtype, out_scale, in_dtype);
    uint8_t* kdst = (uint8_t*)key_out + (int64_t)t * num_heads * kd * oe;
    for (int32_t h = 0; h < num_heads; ++h) {
      memcpy(kdst + (int64_t)h * kd * oe, key_tmp + (int64_t)h * kd * oe, (size_t)nope_dim * oe);
      if (row)
        memcpy(kdst + ((int64_t)h * kd + nope_dim) * oe, key_tmp + ((int64_t)h * kd + nope_dim) * oe,
               (size_t)rope_dim * oe);
    }
    if (v_out)
      memcpy((uint8_t*)v_out + (int64_t)t * num_heads * v_dim * oe, v_tmp,
             (size_t)num_heads * v_dim * oe);
  }
  free(key_tmp);
  free(v_tmp);
  return err;
}
