/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for NVFP4 quantization with per-token (or per-tensor)
 * FP32 scaling and Four-Over-Six (4/6) block-scale selection.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the executable statement of what the CUDA library must
 * compute, bit for bit.  Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or constant generator with the CUDA library, and the
 * library never calls it.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math).  Every float operation
 * below is one IEEE-754 binary32 operation with round-to-nearest-even; fmaf() is the one correctly
 * rounded fused multiply-add, used exactly where the spec says "fma".
 *
 * Sources (web pages, cited by title and section):
 *   [RL-blog]  "NVFP4 RL" blog post, jianyuh.github.io/nvfp4/2026/07/11/NVFP4-RL
 *              Sec. 2 "Baseline: Per-Token Scales & Targeted MoE Quantization" -- per-token FP32 scale
 *              over the hidden dimension, FP8 E4M3 block scales.
 *              Sec. 3 "Gradient Stability" -- dequantized backward y = x . DQ(Q(w)).
 *              Sec. 4 "The Four-Over-Six (4/6) Optimization" -- map the block max to +-6 or +-4,
 *              whichever lowers the block error; the candidate formula
 *              fp4_value * fp8_scale * amax / (E2M1_MAXVAL * E4M3_4OVER6_MAXVAL); error measured in
 *              FP32; "scale the target down by its inverse".
 *   [news]     "humans& Open-Sources the First Stable 4-Bit RL Training Recipe at 1.73x Speedup",
 *              section "Three instabilities, three fixes" (fixes 1 and 3).
 *   [TRACE]    "TRACE FP4 RL -- Rollout-guided FP4 rounding", Jargon entries "FP4 (E2M1) and NVFP4"
 *              and "Round-to-nearest (RTN)", and the "Worked example".
 *
 * Readings taken where the pages are silent (each one is listed in the design notes):
 *   - block size 16 along the row; E4M3 per the OCP FP8 definition (bias 7, max 448, subnormals);
 *   - E4M3_4OVER6_MAXVAL = 256 (M); plain mode "six" uses the ordinary E4M3 maximum, 448;
 *   - amax in the candidate formula is the per-token (or per-tensor) amax a;
 *   - S_enc = 6M/a, c6 = M/a, c4 = 1.5M/a (each clamped to FLT_MAX), S_dec = a/(6M), all FP32;
 *     a == 0 gives all four equal to 0;
 *   - s_T = E4M3(RNE, saturating)(fp32(m * c_T)), m the block amax, T in {6, 4};
 *   - target z = fp32(x * S_enc); scaled-down target t = fp32(z * fp32(1/s_T)) (0 when s_T == 0);
 *   - E2M1 rounding is RTN with ties to the even mantissa bit, saturating at 6, sign of t kept;
 *   - block error e_T = sum of (z - r*s_T)^2 in FP32: d_i = fma(-r_i, s_T, z_i), then
 *     e = 0; e = fma(d_i, d_i, e) for i = 0, 1, ..., 15 (one chain, ascending element order);
 *   - T = 4 iff mode is four_over_six and e_4 < e_6 (ties go to 6);
 *   - dequant y = bf16_RNE(fp32(fp32(r * s) * S_dec));
 *   - codes: row-major [rows][cols/2], element 2j in the low nibble of byte j;
 *     scales: row-major [rows][cols/16] E4M3 bytes; scale_out: S_dec per row (or one per tensor).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MODE_SIX 0
#define ORACLE_MODE_FOUR_OVER_SIX 1
#define ORACLE_MODE_FOUR_OVER_SIX_FP16 2
#define ORACLE_SCALE_ROW 0
#define ORACLE_SCALE_TENSOR 1
#define ORACLE_BLOCK 16

/* ------------------------------------------------------------------------------------------------
 * Number formats.
 * ---------------------------------------------------------------------------------------------- */

static float f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static uint32_t bits_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

/* BF16 is the upper half of an FP32 bit pattern, so widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* E2M1 (FP4): 1 sign, 2 exponent, 1 mantissa bit, exponent bias 1.  The eight magnitudes are
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 ([TRACE], Jargon "FP4 (E2M1) and NVFP4"). */
double oracle_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* Round-to-nearest onto the E2M1 grid ([TRACE], Jargon "Round-to-nearest (RTN)"): the codeword
 * closest to |t|, ties to the even mantissa bit, |t| beyond 6 giving 6; the sign of t is kept. */
int oracle_e2m1_encode(float t) {
  double mag = fabs((double)t);
  if (mag > 6.0) mag = 6.0; /* saturate first: for huge |t| the distances below would all round */
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double err = fabs(mag - oracle_e2m1_value(c));
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best = c;
      best_err = err;
    }
  }
  return (signbit(t) ? 8 : 0) | best;
}

/* FP8 E4M3 (OCP definition): bias 7, subnormal step 2^-9, no infinities, 0x7F/0xFF are NaN. */
double oracle_e4m3_value(int byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Nearest finite E4M3 value, ties to the even mantissa bit; values beyond the largest finite
 * value (448) give 448 (saturating).  The sign of v is kept. */
int oracle_e4m3_encode(float v) {
  double mag = fabs((double)v);
  if (mag > 448.0) mag = 448.0; /* saturate first, as for E2M1 */
  int best = 0;
  double best_err = INFINITY;
  for (int b = 0; b < 127; ++b) { /* 127 = 0x7F is NaN */
    double err = fabs(mag - oracle_e4m3_value(b));
    if (err < best_err || (err == best_err && (b & 1) == 0)) {
      best = b;
      best_err = err;
    }
  }
  return (signbit(v) ? 0x80 : 0) | best;
}

/* FP32 -> BF16 with round-to-nearest-even: pick the nearer of the two BF16 neighbours of v
 * (the truncation and the next value away from zero), ties to the even one.  A value at or past
 * the midpoint above the largest finite BF16 becomes infinity, as IEEE rounding requires. */
uint16_t oracle_bf16_encode(float v) {
  if (isnan(v)) return 0x7FC0;
  uint32_t u = bits_from_f32(v);
  uint32_t lo = u & 0xFFFF0000u;
  double dv = v, dlo = f32_from_bits(lo);
  if (dv == dlo) return (uint16_t)(lo >> 16);
  uint32_t hi = lo + 0x10000u;
  double dhi = ((hi & 0x7FFFFFFFu) == 0x7F800000u) ? copysign(ldexp(1.0, 128), dv)
                                                   : (double)f32_from_bits(hi);
  double elo = fabs(dv - dlo), ehi = fabs(dhi - dv);
  if (elo < ehi) return (uint16_t)(lo >> 16);
  if (ehi < elo) return (uint16_t)(hi >> 16);
  return (uint16_t)((((lo >> 16) & 1u) != 0) ? (hi >> 16) : (lo >> 16));
}

/* IEEE binary16 round-to-nearest-even of a double: 11 significant bits, subnormal quantum 2^-24,
 * magnitudes at or past 65520 (the midpoint above the largest finite, 65504) become infinity. */
double oracle_f16_round(double v) {
  if (isnan(v)) return v;
  double a = fabs(v);
  if (a >= 65520.0) return copysign(INFINITY, v);
  if (a == 0.0) return v;
  int e;
  frexp(a, &e);                            /* a = f * 2^e, f in [0.5, 1) */
  int q = (e - 1 < -14) ? -24 : (e - 1) - 10; /* quantum exponent */
  double r = ldexp(rint(ldexp(a, -q)), q);  /* rint: ties to even in the default rounding mode */
  return copysign(r, v);
}

/* ------------------------------------------------------------------------------------------------
 * The method.
 * ---------------------------------------------------------------------------------------------- */

/* E4M3_4OVER6_MAXVAL of the 4/6 candidate formula ([RL-blog] Sec. 4); the page names it without a
 * value.  256 keeps 1.5*M <= 448, so the scale-to-4 candidate never saturates. */
static float oracle_mode_max(int mode) { return mode == ORACLE_MODE_SIX ? 448.0f : 256.0f; }

static float clamp_to_finite(float v) { return v > FLT_MAX ? FLT_MAX : v; }

/* Per-token (or per-tensor) FP32 factors from the amax a ([RL-blog] Sec. 2 and Sec. 4):
 * S_enc = 6M/a maps a to E2M1_MAXVAL * M; c6 = M/a and c4 = 1.5M/a turn a block amax into the
 * scale-to-6 and scale-to-4 block scales; S_dec = a/(6M) is the stored dequant multiplier. */
void oracle_factors(float a, int mode, float out[4]) {
  float M = oracle_mode_max(mode);
  if (a == 0.0f) {
    out[0] = out[1] = out[2] = out[3] = 0.0f;
    return;
  }
  out[0] = clamp_to_finite((6.0f * M) / a); /* S_enc */
  out[1] = clamp_to_finite(M / a);          /* c6    */
  out[2] = clamp_to_finite((1.5f * M) / a); /* c4    */
  out[3] = a / (6.0f * M);                  /* S_dec */
}

/* Quantize one 16-element block with scale-to-T for T = 6 (c = c6) or T = 4 (c = c4):
 * returns the E4M3 scale byte, writes the 16 E2M1 codes and the block error e_T. */
static int quantize_candidate(const float x[ORACLE_BLOCK], float m, float S_enc, float c,
                              uint8_t code_out[ORACLE_BLOCK], float* err_out) {
  float u = m * c;
  int sbyte = oracle_e4m3_encode(u);
  float s = (float)oracle_e4m3_value(sbyte);
  float inv = (s == 0.0f) ? 0.0f : 1.0f / s;
  float d[ORACLE_BLOCK];
  for (int i = 0; i < ORACLE_BLOCK; ++i) {
    float z = x[i] * S_enc;   /* target in the S_enc-scaled domain            */
    float t = z * inv;        /* scaled down by the inverse of the block scale */
    int code = oracle_e2m1_encode(t);
    float r = (float)oracle_e2m1_value(code);
    code_out[i] = (uint8_t)code;
    d[i] = fmaf(-r, s, z);    /* r*s is exact in FP32 */
  }
  /* The block squared error, summed from +0 over the elements in ascending order, one fma each. */
  float e = 0.0f;
  for (int i = 0; i < ORACLE_BLOCK; ++i) e = fmaf(d[i], d[i], e);
  *err_out = e;
  return sbyte;
}

/* The FP16 reading of the 4/6 fast path ([RL-blog] Sec. 4, "The optimization": do the casting
 * losslessly in FP16 and, rather than multiplying the candidate up by the fractional scales,
 * scale the target down by their inverse).  The candidate value q*s is exact in FP16 (an E2M1
 * value times an E4M3 value has at most 6 significant bits and magnitude at most 2688); the
 * target is x scaled down by the inverse of the per-token scale, z = fp32(x * S_enc), cast to
 * FP16; the residual is one FP16 rounding of the exact z_h - q*s; its square is exact in FP32 and
 * the squares are summed in FP32 from +0 in ascending element order, e = fma(d_i, d_i, e). */
static float candidate_error_fp16(const float x[ORACLE_BLOCK], float S_enc, float s,
                                  const uint8_t code[ORACLE_BLOCK]) {
  float e = 0.0f;
  for (int i = 0; i < ORACLE_BLOCK; ++i) {
    float z = x[i] * S_enc;
    double zh = oracle_f16_round((double)z);
    double qs = oracle_e2m1_value(code[i]) * (double)s; /* exact */
    float d = (float)oracle_f16_round(zh - qs);
    e = fmaf(d, d, e);
  }
  return e;
}

/* One block: both candidates (only scale-to-6 in mode six), then the 4/6 choice ([RL-blog] Sec. 4).
 * Writes 8 packed code bytes and the scale byte; returns 1 when scale-to-4 was chosen. */
static int quantize_block(const float x[ORACLE_BLOCK], const float f[4], int mode,
                          uint8_t packed[ORACLE_BLOCK / 2], uint8_t* scale_byte, float* e6_out,
                          float* e4_out) {
  float m = 0.0f;
  for (int i = 0; i < ORACLE_BLOCK; ++i) m = fmaxf(m, fabsf(x[i]));
  uint8_t c6[ORACLE_BLOCK], c4[ORACLE_BLOCK];
  float e6 = 0.0f, e4 = 0.0f;
  int s6 = quantize_candidate(x, m, f[0], f[1], c6, &e6);
  int pick4 = 0, s4 = 0;
  if (mode == ORACLE_MODE_FOUR_OVER_SIX) {
    s4 = quantize_candidate(x, m, f[0], f[2], c4, &e4);
    pick4 = e4 < e6; /* ties go to 6 */
  } else if (mode == ORACLE_MODE_FOUR_OVER_SIX_FP16) {
    s4 = quantize_candidate(x, m, f[0], f[2], c4, &e4);
    e6 = candidate_error_fp16(x, f[0], (float)oracle_e4m3_value(s6), c6);
    e4 = candidate_error_fp16(x, f[0], (float)oracle_e4m3_value(s4), c4);
    pick4 = e4 < e6;
  }
  const uint8_t* c = pick4 ? c4 : c6;
  for (int j = 0; j < ORACLE_BLOCK / 2; ++j) packed[j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
  *scale_byte = (uint8_t)(pick4 ? s4 : s6);
  if (e6_out) *e6_out = e6;
  if (e4_out) *e4_out = e4;
  return pick4;
}

float oracle_amax(const uint16_t* x, int64_t n) {
  float a = 0.0f;
  for (int64_t i = 0; i < n; ++i) a = fmaxf(a, fabsf(oracle_bf16_to_f32(x[i])));
  return a;
}

static int check_shape(int64_t rows, int64_t cols, int mode) {
  if (rows < 0 || cols <= 0 || cols % ORACLE_BLOCK != 0) return 1;
  if (mode != ORACLE_MODE_SIX && mode != ORACLE_MODE_FOUR_OVER_SIX &&
      mode != ORACLE_MODE_FOUR_OVER_SIX_FP16)
    return 1;
  return 0;
}

/* Quantize rows [0, rows) of x given one amax per row (amax_per_row != 0) or one amax for all
 * rows.  choice (nullable) gets 1 per block where scale-to-4 won; errs (nullable) gets e6, e4. */
static void quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int mode, int per_row,
                          float tensor_amax, uint8_t* codes, uint8_t* scales, float* scale_out,
                          uint8_t* choice, float* errs) {
  int64_t nb = cols / ORACLE_BLOCK;
  float f[4];
  if (!per_row) {
    oracle_factors(tensor_amax, mode, f);
    scale_out[0] = f[3];
  }
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * cols;
    if (per_row) {
      oracle_factors(oracle_amax(xr, cols), mode, f);
      scale_out[r] = f[3];
    }
    for (int64_t b = 0; b < nb; ++b) {
      float xb[ORACLE_BLOCK];
      for (int i = 0; i < ORACLE_BLOCK; ++i) xb[i] = oracle_bf16_to_f32(xr[b * ORACLE_BLOCK + i]);
      float e6, e4;
      int pick4 = quantize_block(xb, f, mode, codes + r * (cols / 2) + b * (ORACLE_BLOCK / 2),
                                 scales + r * nb + b, &e6, &e4);
      if (choice) choice[r * nb + b] = (uint8_t)pick4;
      if (errs) {
        errs[2 * (r * nb + b)] = e6;
        errs[2 * (r * nb + b) + 1] = e4;
      }
    }
  }
}

/* Per-token ([RL-blog] Sec. 2) or per-tensor quantization.  scale_out holds S_dec: rows floats for
 * the row scale, one float for the tensor scale.  Returns 0, or 1 on a bad shape or mode. */
int oracle_quantize(const uint16_t* x, int64_t rows, int64_t cols, int mode, int scale_kind,
                    uint8_t* codes, uint8_t* scales, float* scale_out, uint8_t* choice,
                    float* errs) {
  if (check_shape(rows, cols, mode)) return 1;
  if (scale_kind == ORACLE_SCALE_ROW) {
    quantize_rows(x, rows, cols, mode, 1, 0.0f, codes, scales, scale_out, choice, errs);
  } else if (scale_kind == ORACLE_SCALE_TENSOR) {
    quantize_rows(x, rows, cols, mode, 0, oracle_amax(x, rows * cols), codes, scales, scale_out,
                  choice, errs);
  } else {
    return 1;
  }
  return 0;
}

/* Per-tensor quantization with the amax supplied by the caller (e.g. a max over shards). */
int oracle_quantize_given_amax(const uint16_t* x, int64_t rows, int64_t cols, int mode, float amax,
                               uint8_t* codes, uint8_t* scales, float* scale_out) {
  if (check_shape(rows, cols, mode)) return 1;
  quantize_rows(x, rows, cols, mode, 0, amax, codes, scales, scale_out, 0, 0);
  return 0;
}

/* Dequantize ([RL-blog] Sec. 3 and Sec. 4): y = bf16(fp32(fp32(r * s) * S_dec)), the exact value
 * the quantizer encoded, rounded once to FP32 and once to BF16. */
int oracle_dequantize(const uint8_t* codes, const uint8_t* scales, const float* scale,
                      int scale_kind, int64_t rows, int64_t cols, uint16_t* y) {
  if (rows < 0 || cols <= 0 || cols % ORACLE_BLOCK != 0) return 1;
  if (scale_kind != ORACLE_SCALE_ROW && scale_kind != ORACLE_SCALE_TENSOR) return 1;
  int64_t nb = cols / ORACLE_BLOCK;
  for (int64_t r = 0; r < rows; ++r) {
    float S_dec = scale[scale_kind == ORACLE_SCALE_ROW ? r : 0];
    for (int64_t k = 0; k < cols; ++k) {
      uint8_t byte = codes[r * (cols / 2) + k / 2];
      int code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      float rv = (float)oracle_e2m1_value(code);
      float s = (float)oracle_e4m3_value(scales[r * nb + k / ORACLE_BLOCK]);
      float qs = rv * s; /* exact */
      y[r * cols + k] = oracle_bf16_encode(qs * S_dec);
    }
  }
  return 0;
}

/* Residual quantization after Rollout-ResQ ("HiFloat4 Format for End-To-End Reinforcement
 * Learning Post-Training of Large Language Models", Rollout-ResQ section: dX = X - Q(X), then
 * Q(X) and Q(dX) are both used), with per-token NVFP4 4/6 for both terms.  Per row: Q(x);
 * y = DQ(Q(x)); the residual dx = bf16(fp32(x) - fp32(y)); Q(dx) with dx's own row scale. */
int oracle_quantize_residual(const uint16_t* x, int64_t rows, int64_t cols, int mode,
                             uint8_t* codes, uint8_t* scales, float* scale_out, uint8_t* res_codes,
                             uint8_t* res_scales, float* res_scale_out) {
  if (check_shape(rows, cols, mode)) return 1;
  uint16_t* y = (uint16_t*)malloc((size_t)cols * sizeof(uint16_t));
  uint16_t* dx = (uint16_t*)malloc((size_t)cols * sizeof(uint16_t));
  if (!y || !dx) {
    free(y);
    free(dx);
    return 1;
  }
  int64_t nb = cols / ORACLE_BLOCK;
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * cols;
    quantize_rows(xr, 1, cols, mode, 1, 0.0f, codes + r * (cols / 2), scales + r * nb,
                  scale_out + r, 0, 0);
    oracle_dequantize(codes + r * (cols / 2), scales + r * nb, scale_out + r, ORACLE_SCALE_ROW, 1,
                      cols, y);
    for (int64_t k = 0; k < cols; ++k)
      dx[k] = oracle_bf16_encode(oracle_bf16_to_f32(xr[k]) - oracle_bf16_to_f32(y[k]));
    quantize_rows(dx, 1, cols, mode, 1, 0.0f, res_codes + r * (cols / 2), res_scales + r * nb,
                  res_scale_out + r, 0, 0);
  }
  free(y);
  free(dx);
  return 0;
}

/* TRACE rollout-guided rounding ("TRACE FP4 RL -- Rollout-guided FP4 rounding": between the two
 * neighbouring codewords of its own scaled value, the trainer picks the one closest to the
 * codeword the rollout recorded, using the rollout-side scale).  The scale comes from the
 * rollout: its per-token amax (row_amax, one float per row) gives S_enc as in the quantizer, and
 * its E4M3 block scale bytes give s.  t is formed exactly as the quantizer forms it.  The
 * neighbours are lo = the largest signed grid value <= t and hi = the smallest >= t, with t
 * beyond +-6 saturating to +-6; the output is whichever of lo, hi lies closer to the rollout's
 * value (they coincide when t is on the grid).  A zero output keeps the sign of t. */
int oracle_quantize_guided(const uint16_t* x, int64_t rows, int64_t cols, int mode,
                           const float* row_amax, const uint8_t* ref_codes,
                           const uint8_t* ref_scales, uint8_t* codes_out) {
  if (check_shape(rows, cols, mode)) return 1;
  static const double grid[15] = {-6, -4, -3, -2, -1.5, -1, -0.5, 0, 0.5, 1, 1.5, 2, 3, 4, 6};
  int64_t nb = cols / ORACLE_BLOCK;
  for (int64_t r = 0; r < rows; ++r) {
    float f[4];
    oracle_factors(row_amax[r], mode, f);
    for (int64_t k = 0; k < cols; ++k) {
      float s = (float)oracle_e4m3_value(ref_scales[r * nb + k / ORACLE_BLOCK]);
      float inv = (s == 0.0f) ? 0.0f : 1.0f / s;
      float z = oracle_bf16_to_f32(x[r * cols + k]) * f[0];
      float t = z * inv;
      double tc = t > 6.0f ? 6.0 : (t < -6.0f ? -6.0 : (double)t);
      double lo = grid[0], hi = grid[14];
      for (int g = 0; g < 15; ++g) {
        if (grid[g] <= tc) lo = grid[g];
        if (grid[14 - g] >= tc) hi = grid[14 - g];
      }
      uint8_t byte = ref_codes[r * (cols / 2) + k / 2];
      int ref = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      double rv = oracle_e2m1_value(ref);
      double v = (fabs(hi - rv) < fabs(lo - rv)) ? hi : lo;
      int code = oracle_e2m1_encode((float)v);
      if (v == 0.0) code = signbit(t) ? 8 : 0;
      uint8_t* out = &codes_out[r * (cols / 2) + k / 2];
      *out = (k % 2 == 0) ? (uint8_t)((*out & 0xF0) | code) : (uint8_t)((*out & 0x0F) | (code << 4));
    }
  }
  return 0;
}

/* Array forms of the format conversions, for the format tests. */
void oracle_e2m1_encode_array(const float* t, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e2m1_encode(t[i]);
}

void oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e4m3_encode(v[i]);
}

void oracle_f16_round_array(const double* v, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_round(v[i]);
}

void oracle_bf16_encode_array(const float* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_encode(v[i]);
}
