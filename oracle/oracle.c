/*
 * CPU oracle for the MTP draft-layer tail — TEST INFRASTRUCTURE, not product.
 *
 * Plain, slow, single-threaded C.  It shares no code, header, table or helper
 * with the CUDA library; only tests, the smoke check and the benchmark's CPU
 * baseline call it.  Compile without fast-math and with -ffp-contract=off so
 * every fp32 operation below is one IEEE-754 operation in source order.
 *
 * What it computes (pages cited by title and section):
 *  - "[Quant][MTP] Reuse packed FP8 logits inputs", Purpose: the draft layer's
 *    final all-reduce and RMSNorm feed a packed FP8 quantisation for the shared
 *    LM head, and the layer returns two different values — the packed
 *    QuantizedActivation and the post-final-norm BF16 hidden state.
 *  - "[Spec Decode][Perf] Fuse the MTP trailing all-reduce; local-argmax draft
 *    tokens", intro: the trailing all-reduce is fused into the final RMSNorm;
 *    greedy draft tokens come from a vocab-parallel local argmax.  Accuracy:
 *    the fused kernel accumulates in fp32; local argmax changes how ties at
 *    vocab-shard boundaries are broken.
 * Readings adopted where the pages are silent: the k tensor-parallel partial
 * outputs are summed in fp32 in index order, then the residual is added; RMSNorm
 * is x * rsqrt(mean(x^2) + eps) * w with eps = 1e-6 (computed here in fp64 and
 * rounded once to BF16); the quantiser sees the BF16 hidden, uses one fp32
 * scale = amax / 448 per 1x128 group and e4m3fn codes rounded to nearest even
 * with saturation; the LM head is sum_k (qa*sa)*(qw*sw) accumulated in fp32 in
 * k order; the argmax takes the lowest global vocab index among exact ties.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- codecs -- */

/* BF16 is the upper half of an IEEE binary32 pattern: decoding is exact. */
float or_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a double to the nearest BF16 value, ties to even significand.
 * BF16 keeps 8 significant bits: in the binade [2^E, 2^(E+1)) the spacing is
 * 2^(E-7); below 2^-126 the spacing stays 2^-133 (subnormals).  Values that
 * round to 2^128 or above overflow to infinity. */
uint16_t or_f64_to_bf16(double d) {
  if (isnan(d)) return 0x7FC0;
  uint16_t sign = signbit(d) ? 0x8000 : 0;
  double a = fabs(d);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
  int E = e - 1;
  double q = ldexp(1.0, (E < -126 ? -126 : E) - 7);
  double r = rint(a / q) * q;   /* rint rounds half to even in the default mode */
  if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
  float rf = (float)r;          /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &rf, 4);
  return sign | (uint16_t)(u >> 16);
}

uint16_t or_f32_to_bf16(float f) { return or_f64_to_bf16((double)f); }

/* OCP FP8 e4m3fn: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8; subnormals m * 2^-9. */
float or_e4m3_to_f32(uint8_t c) {
  int s = c >> 7, ex = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (ex == 0xF && m == 7) return NAN;
  if (ex == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, ex - 7);
  return (float)(s ? -v : v);
}

/* Exact e4m3 encoding of a non-negative value that is representable. */
static uint8_t e4m3_encode_exact(double r) {
  if (r == 0.0) return 0;
  if (r < ldexp(1.0, -6)) return (uint8_t)(r / ldexp(1.0, -9));
  int e;
  frexp(r, &e);
  int E = e - 1;
  int m = (int)((r / ldexp(1.0, E) - 1.0) * 8.0);
  return (uint8_t)(((E + 7) << 3) | m);
}

/* f32 -> e4m3fn, round to nearest even, saturating to +-448 (NaN -> 0x7F).
 * In the binade [2^E, 2^(E+1)) the e4m3 spacing is 2^(E-3); below the smallest
 * normal 2^-6 it is 2^-9.  A negative value that rounds to zero keeps its sign
 * (0x80). */
uint8_t or_f32_to_e4m3(float f) {
  if (isnan(f)) return 0x7F;
  uint8_t sign = signbit(f) ? 0x80 : 0;
  double a = fabs((double)f);
  if (a >= 448.0) return sign | 0x7E;
  double q;
  if (a < ldexp(1.0, -6)) {
    q = ldexp(1.0, -9);
  } else {
    int e;
    frexp(a, &e);
    q = ldexp(1.0, (e - 1) - 3);
  }
  double r = rint(a / q) * q;
  if (r > 448.0) r = 448.0;
  return sign | e4m3_encode_exact(r);
}

/* ------------------------------------------- stage 1: reduce, norm, quant -- */

/*
 * For rows r = 0..R-1 (each H wide, H a multiple of 128):
 *   x[h]   = ((p_0[h] + p_1[h]) + ... + p_{k-1}[h]) + residual[h]      (fp32)
 *   ms     = (sum_h x[h]^2) / H,  rr = 1 / sqrt(ms + eps)              (fp64)
 *   hidden = bf16_rne(x[h] * rr * w[h])                                  (fp64 -> bf16)
 *   per group g of 128: amax = max |hidden|, scale = amax / 448          (fp32)
 *   code   = scale == 0 ? 0 : e4m3_rne_sat(hidden / scale)               (fp32 divide)
 * partials: k blocks of [R][H] BF16 patterns, block i at partials + i*R*H.
 * x_out (float [R][H]) and rr_out (double [R]) may be NULL.
 */
void or_reduce_norm_quant(const uint16_t *partials, int k, const uint16_t *residual,
                          const uint16_t *norm_w, double eps, int R, int H,
                          uint16_t *hidden, uint8_t *codes, float *scales,
                          float *x_out, double *rr_out) {
  float *x = (float *)malloc(sizeof(float) * (size_t)H);
  if (!x) return;
  const size_t plane = (size_t)R * (size_t)H;
  for (int r = 0; r < R; ++r) {
    const size_t row = (size_t)r * (size_t)H;
    for (int h = 0; h < H; ++h) {
      float s = or_bf16_to_f32(partials[row + h]);
      for (int i = 1; i < k; ++i) s = s + or_bf16_to_f32(partials[(size_t)i * plane + row + h]);
      s = s + or_bf16_to_f32(residual[row + h]);
      x[h] = s;
    }
    double ss = 0.0;
    for (int h = 0; h < H; ++h) ss += (double)x[h] * (double)x[h];
    double ms = ss / (double)H;
    double rr = 1.0 / sqrt(ms + eps);
    if (rr_out) rr_out[r] = rr;
    if (x_out) memcpy(x_out + row, x, sizeof(float) * (size_t)H);
    for (int h = 0; h < H; ++h)
      hidden[row + h] = or_f64_to_bf16(((double)x[h] * rr) * (double)or_bf16_to_f32(norm_w[h]));
    const int G = H / 128;
    for (int g = 0; g < G; ++g) {
      float amax = 0.0f;
      for (int j = 0; j < 128; ++j) {
        float v = fabsf(or_bf16_to_f32(hidden[row + (size_t)g * 128 + j]));
        if (v > amax) amax = v;
      }
      float scale = amax / 448.0f;
      scales[(size_t)r * G + g] = scale;
      for (int j = 0; j < 128; ++j) {
        size_t at = row + (size_t)g * 128 + j;
        codes[at] = (scale == 0.0f) ? 0 : or_f32_to_e4m3(or_bf16_to_f32(hidden[at]) / scale);
      }
    }
  }
  free(x);
}

/* ------------------------------------------------ stage 2: LM head, argmax -- */

/*
 * logits[i][v - v0] for the tokens listed in tok[0..n_tok) and vocab rows
 * v0 <= v < v1:
 *   L = sum_{k=0}^{H-1} (dec(qa[t][k]) * sa[t][k/128]) * (dec(qw[v][k]) * sw[v/128][k/128])
 * every product and every partial sum in fp32, k ascending.
 * qa [T][H] e4m3 codes, sa [T][H/128] fp32, qw [V][H] e4m3 codes,
 * sw [ceil(V/128)][H/128] fp32.
 */
void or_lm_head_logits(const uint8_t *qa, const float *sa, int H, const int32_t *tok,
                       int n_tok, const uint8_t *qw, const float *sw, int v0, int v1,
                       float *logits) {
  const int G = H / 128;
  float *ad = (float *)malloc(sizeof(float) * (size_t)n_tok * (size_t)H);
  float *wd = (float *)malloc(sizeof(float) * (size_t)H);
  if (!ad || !wd) { free(ad); free(wd); return; }
  for (int i = 0; i < n_tok; ++i) {
    const size_t t = (size_t)tok[i];
    for (int k = 0; k < H; ++k)
      ad[(size_t)i * H + k] = or_e4m3_to_f32(qa[t * H + k]) * sa[t * G + k / 128];
  }
  const size_t W = (size_t)(v1 - v0);
  for (int v = v0; v < v1; ++v) {
    const size_t row = (size_t)v * (size_t)H;
    for (int k = 0; k < H; ++k)
      wd[k] = or_e4m3_to_f32(qw[row + k]) * sw[(size_t)(v / 128) * G + k / 128];
    for (int i = 0; i < n_tok; ++i) {
      const float *a = ad + (size_t)i * H;
      float L = 0.0f;
      for (int k = 0; k < H; ++k) L = L + a[k] * wd[k];
      logits[(size_t)i * W + (size_t)(v - v0)] = L;
    }
  }
  free(ad);
  free(wd);
}

/*
 * Greedy draft tokens from full logit rows [n][V] split into S equal vocab
 * shards [s*V/S, (s+1)*V/S):
 *   shard_idx[i][s], shard_val[i][s]: largest logit in shard s and the lowest
 *       global index holding it (ascending scan, strict >; -0 == +0)
 *   tok[i], val[i]: the same over the whole row — equal to the best shard
 *       result with ties going to the lower shard
 *   gap[i]: (L1 - L2) / |L1| where L2 is the best logit at any other index
 *       (L1 - L2 when L1 == 0).
 * Output pointers other than tok may be NULL.
 */
void or_argmax(const float *logits, int n, int V, int S, int32_t *tok, float *val,
               int32_t *shard_idx, float *shard_val, double *gap) {
  const int width = V / S;
  for (int i = 0; i < n; ++i) {
    const float *L = logits + (size_t)i * (size_t)V;
    for (int s = 0; s < S; ++s) {
      int b = s * width;
      float best = L[b];
      int bi = b;
      for (int v = b + 1; v < b + width; ++v)
        if (L[v] > best) { best = L[v]; bi = v; }
      if (shard_idx) shard_idx[(size_t)i * S + s] = bi;
      if (shard_val) shard_val[(size_t)i * S + s] = best;
    }
    float best = L[0];
    int bi = 0;
    for (int v = 1; v < V; ++v)
      if (L[v] > best) { best = L[v]; bi = v; }
    tok[i] = bi;
    if (val) val[i] = best;
    if (gap) {
      double second = -INFINITY;
      for (int v = 0; v < V; ++v)
        if (v != bi && (double)L[v] > second) second = (double)L[v];
      double d = (double)best - second;
      gap[i] = (best == 0.0f) ? d : d / fabs((double)best);
    }
  }
}

/* ======================================================= NVFP4 variant == */
/*
 * The benchmark pages serve an NVFP4 checkpoint ("[Spec Decode][Perf] Fuse the
 * MTP trailing all-reduce; local-argmax draft tokens", Benchmarks) but define no
 * FP4 arithmetic.  The readings here follow the published NVFP4 format: values
 * are OCP FP4 e2m1 codes, each block of 16 consecutive elements along the hidden
 * dimension carries one unsigned e4m3 scale, and a row (token or tensor) carries
 * one fp32 scale chosen so that the largest block scale is 448:
 *   g      = amax_row / (448 * 6)                                      (fp32)
 *   sb     = e4m3_rne_sat(amax_block / (6 * g))                        (fp32, two roundings)
 *   eff    = dec(sb) * g                                               (fp32)
 *   code   = eff == 0 ? 0 : e2m1_rne_sat(x / eff)                      (fp32 divide)
 * Codes are packed two to a byte, element 2i in the low nibble of byte i.
 */

/* OCP FP4 e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
 * 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6; no infinities or NaN. */
float or_e2m1_to_f32(uint8_t c) {
  int s = (c >> 3) & 1, ex = (c >> 1) & 3, m = c & 1;
  double v = (ex == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, ex - 1);
  return (float)(s ? -v : v);
}

/* f32 -> e2m1, round to nearest even, saturating to +-6.  The spacing is 0.5
 * below 2, 1 in [2, 4) and 2 in [4, 8); an even multiple of the spacing has a
 * zero mantissa bit.  A negative value that rounds to zero keeps its sign (8). */
uint8_t or_f32_to_e2m1(float f) {
  uint8_t sign = signbit(f) ? 8 : 0;
  double a = fabs((double)f);
  if (isnan(f)) return sign | 7;
  if (a >= 6.0) return sign | 7;
  double q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
  double r = rint(a / q) * q;
  if (r > 6.0) r = 6.0;
  if (r == 0.0) return sign;
  if (r == 0.5) return sign | 1;
  int e;
  frexp(r, &e);                       /* r in [2^(e-1), 2^e) */
  int ex = e;                         /* biased exponent: r = (1 + m/2) * 2^(ex-1) */
  int m = (int)((r / ldexp(1.0, e - 1) - 1.0) * 2.0);
  return sign | (uint8_t)((ex << 1) | m);
}

/*
 * NVFP4 quantisation of BF16 rows [R][H] (H a multiple of 16): codes [R][H/2]
 * (packed), block scales [R][H/16] (unsigned e4m3 codes), row scales [R].
 */
void or_nvfp4_quant(const uint16_t *hidden, int R, int H, uint8_t *codes, uint8_t *bscales,
                    float *gscales) {
  const int B = H / 16;
  for (int r = 0; r < R; ++r) {
    const uint16_t *y = hidden + (size_t)r * (size_t)H;
    float amax = 0.0f;
    for (int h = 0; h < H; ++h) {
      float v = fabsf(or_bf16_to_f32(y[h]));
      if (v > amax) amax = v;
    }
    const float g = amax / 2688.0f;
    gscales[r] = g;
    for (int b = 0; b < B; ++b) {
      float ab = 0.0f;
      for (int j = 0; j < 16; ++j) {
        float v = fabsf(or_bf16_to_f32(y[b * 16 + j]));
        if (v > ab) ab = v;
      }
      uint8_t sb = 0;
      if (g != 0.0f) {
        const float d = 6.0f * g;
        sb = or_f32_to_e4m3(ab / d);
      }
      bscales[(size_t)r * B + b] = sb;
      const float eff = or_e4m3_to_f32(sb) * g;
      for (int j = 0; j < 16; j += 2) {
        uint8_t lo = 0, hi = 0;
        if (eff != 0.0f) {
          lo = or_f32_to_e2m1(or_bf16_to_f32(y[b * 16 + j]) / eff);
          hi = or_f32_to_e2m1(or_bf16_to_f32(y[b * 16 + j + 1]) / eff);
        }
        codes[(size_t)r * (H / 2) + (size_t)(b * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

/*
 * NVFP4 LM head logits for the tokens tok[0..n_tok) and rows v0 <= v < v1:
 *   c_b = (dec(sa[t][b]) * dec(sw[v][b])) * sum_{j<16} e2m1(qa[t][16b+j]) * e2m1(qw[v][16b+j])
 *   L   = (sum_b c_b, b ascending, fp32) * (ga[t] * gw)
 * Each c_b is exact in fp32 (products of 4-bit significands); only the sum over
 * blocks and the two final multiplications round.
 * qa [T][H/2], sa [T][H/16], ga [T]; qw [V][H/2], sw [V][H/16]; gw a scalar.
 */
void or_lm_head_logits_nvfp4(const uint8_t *qa, const uint8_t *sa, const float *ga, int H,
                             const int32_t *tok, int n_tok, const uint8_t *qw,
                             const uint8_t *sw, float gw, int v0, int v1, float *logits) {
  const int B = H / 16;
  float *ad = (float *)malloc(sizeof(float) * (size_t)n_tok * (size_t)H);
  float *wd = (float *)malloc(sizeof(float) * (size_t)H);
  if (!ad || !wd) { free(ad); free(wd); return; }
  for (int i = 0; i < n_tok; ++i) {
    const size_t t = (size_t)tok[i];
    for (int k = 0; k < H; ++k) {
      uint8_t byte = qa[t * (size_t)(H / 2) + (size_t)k / 2];
      ad[(size_t)i * H + k] = or_e2m1_to_f32((k & 1) ? (byte >> 4) : (byte & 15));
    }
  }
  const size_t W = (size_t)(v1 - v0);
  for (int v = v0; v < v1; ++v) {
    for (int k = 0; k < H; ++k) {
      uint8_t byte = qw[(size_t)v * (size_t)(H / 2) + (size_t)k / 2];
      wd[k] = or_e2m1_to_f32((k & 1) ? (byte >> 4) : (byte & 15));
    }
    for (int i = 0; i < n_tok; ++i) {
      const size_t t = (size_t)tok[i];
      const float *a = ad + (size_t)i * H;
      float acc = 0.0f;
      for (int b = 0; b < B; ++b) {
        float bs = 0.0f;
        for (int j = 0; j < 16; ++j) bs = bs + a[b * 16 + j] * wd[b * 16 + j];
        const float s = or_e4m3_to_f32(sa[t * (size_t)B + b]) * or_e4m3_to_f32(sw[(size_t)v * B + b]);
        acc = acc + s * bs;
      }
      logits[(size_t)i * W + (size_t)(v - v0)] = acc * (ga[t] * gw);
    }
  }
  free(ad);
  free(wd);
}

/* ================================================= unfused reference arm == */
/*
 * The path without the fusions ("[Spec Decode][Perf] Fuse the MTP trailing
 * all-reduce; local-argmax draft tokens", intro and Accuracy: the trailing
 * all-reduce is a separate BF16 collective before the final RMSNorm, and the
 * draft tokens come from the argmax of the gathered full-vocab logits):
 *   s      = bf16_rne((p_0 + p_1) + ... + p_{k-1})               fp32 sum, one rounding
 *   hidden = bf16_rne((s + residual) * rsqrt(mean(.^2) + eps) * w)   as stage 1 (fp64 norm)
 *   codes/scales from hidden exactly as stage 1
 *   logits = bf16_rne(fp32 LM-head logits) [T][V]; token = lowest index of the maximum
 */
void or_unfused_reduce_bf16(const uint16_t *partials, int k, int R, int H, uint16_t *out) {
  const size_t plane = (size_t)R * (size_t)H;
  for (size_t i = 0; i < plane; ++i) {
    float s = or_bf16_to_f32(partials[i]);
    for (int j = 1; j < k; ++j) s = s + or_bf16_to_f32(partials[(size_t)j * plane + i]);
    out[i] = or_f32_to_bf16(s);
  }
}

/* RMSNorm of (x + residual), both BF16 rows [R][H]: the hidden only. */
void or_unfused_add_rmsnorm(const uint16_t *x, const uint16_t *residual, const uint16_t *norm_w,
                            double eps, int R, int H, uint16_t *hidden) {
  float *v = (float *)malloc(sizeof(float) * (size_t)H);
  if (!v) return;
  for (int r = 0; r < R; ++r) {
    const size_t row = (size_t)r * (size_t)H;
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
      v[h] = or_bf16_to_f32(x[row + h]) + or_bf16_to_f32(residual[row + h]);
      ss += (double)v[h] * (double)v[h];
    }
    const double rr = 1.0 / sqrt(ss / (double)H + eps);
    for (int h = 0; h < H; ++h)
      hidden[row + h] = or_f64_to_bf16(((double)v[h] * rr) * (double)or_bf16_to_f32(norm_w[h]));
  }
  free(v);
}

/* Packed FP8 quantisation of BF16 rows [R][H], exactly stage 1's rule. */
void or_quant_fp8_rows(const uint16_t *hidden, int R, int H, uint8_t *codes, float *scales) {
  const int G = H / 128;
  for (int r = 0; r < R; ++r) {
    for (int g = 0; g < G; ++g) {
      const size_t base = (size_t)r * (size_t)H + (size_t)g * 128;
      float amax = 0.0f;
      for (int j = 0; j < 128; ++j) {
        float a = fabsf(or_bf16_to_f32(hidden[base + j]));
        if (a > amax) amax = a;
      }
      const float scale = amax / 448.0f;
      scales[(size_t)r * G + g] = scale;
      for (int j = 0; j < 128; ++j)
        codes[base + j] = (scale == 0.0f) ? 0 : or_f32_to_e4m3(or_bf16_to_f32(hidden[base + j]) / scale);
    }
  }
}

/* Greedy token per row of BF16 logits [n][V]: the lowest index of the maximum
 * (-0 == +0).  The BF16 rounding makes exact ties common. */
void or_argmax_bf16(const uint16_t *logits, int n, int V, int32_t *tok) {
  for (int i = 0; i < n; ++i) {
    const uint16_t *L = logits + (size_t)i * (size_t)V;
    float best = or_bf16_to_f32(L[0]);
    int bi = 0;
    for (int v = 1; v < V; ++v) {
      const float x = or_bf16_to_f32(L[v]);
      if (x > best) { best = x; bi = v; }
    }
    tok[i] = bi;
  }
}

/* Element-wise or_f32_to_bf16 over an array (one call for many values). */
void or_f32_to_bf16_array(const float *x, size_t n, uint16_t *out) {
  for (size_t i = 0; i < n; ++i) out[i] = or_f32_to_bf16(x[i]);
}
