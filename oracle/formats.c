/*
 * oracle/formats.c -- the CPU oracle's format arithmetic (TEST INFRASTRUCTURE).
 *
 * This file is part of the oracle: a plain, slow, obviously correct CPU
 * restatement of what the fused grouped-MLP forward and the group quantisers
 * compute.  Only the tests, __graft_entry__.smoke() and bench.py's CPU-baseline
 * leg may load it.  It shares no code, header or table with the CUDA path.
 *
 * Sources (TransformerEngine pull-request pages):
 *   - PR #3837 "Reduce NVFP4 quantization work for the fused GroupedMLP fc2
 *     input with activation recompute", Description and commits: NVFP4 with a
 *     randomized Hadamard transform (RHT) and a per-quantizer sign mask; the
 *     per-group (pre-RHT, post-RHT) amax pair; quantize-with-amax.
 *   - PR #2769 "GEMM + Swiglu fused Grouped MLP for MXFP8", Greptile summary and
 *     sequence diagram: MXFP8 operands with block scales.
 * The pages give no rounding rules.  The format facts used here are those the
 * method statement fixes: E2M1 values {0,0.5,1,1.5,2,3,4,6}; E4M3 max 448 (no
 * infinity, S.1111.111 is NaN); MXFP8 block scale 2^(floor(log2 amax) - 8) in
 * E8M0; H16 * H16^T = 16 I.  Every reading beyond those is stated at the
 * function that takes it (round-to-nearest-even, saturation, the NVFP4 scale
 * chain and its FLT_MAX caps).
 *
 * Arithmetic: exact values are carried in double; wherever the method fixes an
 * FP32 operation (the NVFP4 scale chain, the RHT butterfly) it is done in
 * float, one IEEE round-to-nearest-even operation per C operator.  The file is
 * compiled with -ffp-contract=off so no multiply-add is fused.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, fp32 exponent range,
 * subnormal quantum 2^-133), ties to even, overflow to infinity. */
uint16_t orc_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int E;
  frexp(a, &E);
  int x = E - 1; /* floor(log2 a) */
  int q = (x < -126) ? -133 : x - 7;
  double r = ldexp(rint(ldexp(a, -q)), q);
  if (r > ldexp(2.0 - ldexp(1.0, -7), 127)) return sign | 0x7F80;
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

void orc_bf16_from_double_array(const double* v, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_double(v[i]);
}

void orc_bf16_to_double_array(const uint16_t* b, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_double(b[i]);
}

/* ------------------------------------------------------------------ E4M3 */

/* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent field 0 is
 * subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity. */
double orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
  return s ? -v : v;
}

/* Nearest E4M3 value, ties to the even mantissa, |v| >= 448 saturates to 448
 * (the "satfinite" reading of "E4M3 max 448").  The sign is copied, so -0 and
 * negative values that round to zero give 0x80. */
uint8_t orc_e4m3_encode(double v) {
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs(v);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal grid k * 2^-9; k = 8 is the smallest normal, code 0x08 */
    return sign | (uint8_t)rint(ldexp(a, 9));
  }
  int E;
  frexp(a, &E);
  int x = E - 1; /* floor(log2 a), in [-6, 8] */
  double mant = rint((ldexp(a, -x) - 1.0) * 8.0);
  if (mant == 8.0) {
    x += 1;
    mant = 0.0;
  }
  return sign | (uint8_t)(((x + 7) << 3) | (int)mant);
}

/* ------------------------------------------------------------------ E2M1 */

/* 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit: magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}. */
double orc_e2m1_decode(uint8_t c) {
  int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* Nearest E2M1 value, ties to the even mantissa, |v| >= 6 saturates to 6,
 * sign copied (negative values rounding to zero give 0x8). */
uint8_t orc_e2m1_encode(double v) {
  uint8_t sign = signbit(v) ? 8 : 0;
  double a = fabs(v);
  if (a >= 6.0) return sign | 7;
  if (a < 1.0) return sign | (uint8_t)rint(a * 2.0); /* 0, 0.5, or 1.0 (code 2) */
  int E;
  frexp(a, &E);
  int x = E - 1; /* 0, 1 or 2 */
  double mant = rint((ldexp(a, -x) - 1.0) * 2.0);
  if (mant == 2.0) {
    x += 1;
    mant = 0.0;
  }
  return sign | (uint8_t)(((x + 1) << 1) | (int)mant);
}

/* ------------------------------------------------------------------ MXFP8 */

/* E8M0 scale exponent of one 1x32 block: floor(log2 amax) - 8, clamped to
 * [-127, 127]; an all-zero block takes -127 (byte 0). */
int orc_mxfp8_scale_exponent(double amax) {
  if (amax == 0.0) return -127;
  int E;
  frexp(amax, &E);
  int e = (E - 1) - 8;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* Rowwise MXFP8 of a row-major bf16 [rows, K] matrix: for every run of 32
 * consecutive elements of a row, one E8M0 scale byte (e + 127) and 32 E4M3
 * codes of x * 2^-e.  scales is compact: [rows, K/32]. */
void orc_mxfp8_quantize_rows(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes,
                             uint8_t* scales) {
  int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint16_t* blk = x + r * K + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(orc_bf16_to_double(blk[i])));
      int e = orc_mxfp8_scale_exponent(amax);
      scales[r * nb + b] = (uint8_t)(e + 127);
      for (int i = 0; i < 32; ++i)
        codes[r * K + b * 32 + i] = orc_e4m3_encode(ldexp(orc_bf16_to_double(blk[i]), -e));
    }
  }
}

void orc_mxfp8_dequant_rows(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K,
                            double* out) {
  int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k)
      out[r * K + k] = ldexp(orc_e4m3_decode(codes[r * K + k]), (int)scales[r * nb + k / 32] - 127);
}

/* ------------------------------------------------------------------ NVFP4 */

/* FP32 per-group (or per-tensor) encode scale S = 448 * 6 / amax.  amax = 0
 * gives 1; an FP32 overflow gives FLT_MAX. */
float orc_nvfp4_global_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  float S = 2688.0f / amax;
  if (isinf(S)) S = FLT_MAX;
  return S;
}

/* One 1x16 NVFP4 block of FP32 values v under global scale S:
 *   b   = max |v_i|
 *   t   = fp32(fp32(b / 6) * S),  sf = E4M3(t)            (block scale byte)
 *   enc = sf == 0 ? 0 : min(fp32(S / sf), FLT_MAX)
 *   q_i = E2M1(fp32(v_i * enc))                           (codes)
 * Codes are packed two per byte, the even element in the low nibble.  The
 * encode factor saturates at FLT_MAX as S does (reading: the format has no
 * infinities, so a zero element stays zero when S / sf overflows; this only
 * happens when the group amax is below ~1e-35). */
void orc_nvfp4_quantize_block(const float* v, float S, uint8_t* codes8, uint8_t* sf_out) {
  float b = 0.0f;
  for (int i = 0; i < 16; ++i) b = fmaxf(b, fabsf(v[i]));
  float q = b / 6.0f;
  float t = q * S;
  uint8_t sf = orc_e4m3_encode((double)t);
  float sfv = (float)orc_e4m3_decode(sf);
  float enc = (sfv == 0.0f) ? 0.0f : S / sfv;
  if (isinf(enc)) enc = FLT_MAX;
  for (int i = 0; i < 16; i += 2) {
    float p0 = v[i] * enc;
    float p1 = v[i + 1] * enc;
    codes8[i / 2] = (uint8_t)(orc_e2m1_encode((double)p0) | (orc_e2m1_encode((double)p1) << 4));
  }
  *sf_out = sf;
}

/* Rowwise NVFP4 of a row-major bf16 [rows, K] matrix under one global scale S:
 * codes [rows, K/2], compact scales [rows, K/16]. */
void orc_nvfp4_quantize_rows(const uint16_t* x, int64_t rows, int64_t K, float S, uint8_t* codes,
                             uint8_t* scales) {
  int64_t nb = K / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      float v[16];
      for (int i = 0; i < 16; ++i) v[i] = (float)orc_bf16_to_double(x[r * K + b * 16 + i]);
      orc_nvfp4_quantize_block(v, S, codes + r * (K / 2) + b * 8, scales + r * nb + b);
    }
  }
}

/* dequant = E2M1(q) * E4M3(sf) / S, in double */
void orc_nvfp4_dequant_rows(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K,
                            float S, double* out) {
  int64_t nb = K / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t q = (k & 1) ? (byte >> 4) : (byte & 15);
      out[r * K + k] = orc_e2m1_decode(q) * orc_e4m3_decode(scales[r * nb + k / 16]) / (double)S;
    }
}

/* ------------------------------------------------------------------ RHT */

/* 16-point randomized Hadamard transform y = 1/4 * H16 * diag(s) * v, where
 * s_i = -1 when bit i of mask is set and H16 is the Sylvester Hadamard matrix.
 * Evaluated in FP32 as the four butterfly stages h = 1, 2, 4, 8, each mapping
 * the pair (v[i], v[i+h]) with (i & h) == 0 to (v[i] + v[i+h], v[i] - v[i+h]),
 * then the exact scaling by 1/4. */
void orc_rht16(const float* in, uint32_t mask, float* out) {
  float w[16];
  for (int i = 0; i < 16; ++i) w[i] = ((mask >> i) & 1u) ? -in[i] : in[i];
  for (int h = 1; h < 16; h <<= 1)
    for (int i = 0; i < 16; ++i)
      if (!(i & h)) {
        float a = w[i], b = w[i + h];
        w[i] = a + b;
        w[i + h] = a - b;
      }
  for (int i = 0; i < 16; ++i) out[i] = w[i] * 0.25f;
}

/* Load the column-c chunk j of one group: rows off + 16j .. off + 16j + 15,
 * zero past the group's m rows. */
static void load_col_chunk(const uint16_t* x, int64_t K, int64_t off, int64_t m, int64_t j,
                           int64_t c, float* v) {
  for (int i = 0; i < 16; ++i) {
    int64_t r = 16 * j + i;
    v[i] = (r < m) ? (float)orc_bf16_to_double(x[(off + r) * K + c]) : 0.0f;
  }
}

/* Per-group amax of a token-sorted bf16 [M, K] tensor split into G groups:
 *   amax_pre[g]  = max |x| over the group's rows;
 *   amax_post[g] = max |RHT16(chunk)| over every column and every 16-row
 *                  column chunk of the group (chunks start at the group's
 *                  first row; a short last chunk is zero-padded). */
void orc_group_hadamard_amax(const uint16_t* x, int64_t M, int64_t K, const int64_t* splits,
                             int G, uint32_t mask, float* amax_pre, float* amax_post) {
  (void)M;
  int64_t off = 0;
  for (int g = 0; g < G; ++g) {
    int64_t m = splits[g];
    float pre = 0.0f, post = 0.0f;
#pragma omp parallel for reduction(max : pre) schedule(static)
    for (int64_t r = 0; r < m; ++r)
      for (int64_t c = 0; c < K; ++c) pre = fmaxf(pre, fabsf((float)orc_bf16_to_double(x[(off + r) * K + c])));
    int64_t nchunks = (m + 15) / 16;
#pragma omp parallel for reduction(max : post) schedule(static)
    for (int64_t j = 0; j < nchunks; ++j)
      for (int64_t c = 0; c < K; ++c) {
        float v[16], y[16];
        load_col_chunk(x, K, off, m, j, c, v);
        orc_rht16(v, mask, y);
        for (int i = 0; i < 16; ++i) post = fmaxf(post, fabsf(y[i]));
      }
    amax_pre[g] = pre;
    amax_post[g] = post;
    off += m;
  }
}

/* Columnwise NVFP4 of each group: for every column c and 16-row chunk j of
 * group g, the 16 values (RHT-transformed when use_rht) form one block under
 * S_g = global_scale(amax_col[g]).  Per group, codes are [K, Mpad_g/2] and
 * compact scales [K, Mpad_g/16] with Mpad_g = 16 * ceil(m_g / 16); groups
 * follow one another in both buffers. */
void orc_group_quantize_col(const uint16_t* x, int64_t M, int64_t K, const int64_t* splits, int G,
                            int use_rht, uint32_t mask, const float* amax_col, uint8_t* col_codes,
                            uint8_t* col_scales) {
  (void)M;
  int64_t off = 0, code_base = 0, sf_base = 0;
  for (int g = 0; g < G; ++g) {
    int64_t m = splits[g];
    int64_t mpad = (m + 15) / 16 * 16;
    float S = orc_nvfp4_global_scale(amax_col[g]);
    int64_t nchunks = mpad / 16;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < K; ++c)
      for (int64_t j = 0; j < nchunks; ++j) {
        float v[16], y[16];
        load_col_chunk(x, K, off, m, j, c, v);
        if (use_rht)
          orc_rht16(v, mask, y);
        else
          memcpy(y, v, sizeof(y));
        orc_nvfp4_quantize_block(y, S, col_codes + code_base + c * (mpad / 2) + 8 * j,
                                 col_scales + sf_base + c * (mpad / 16) + j);
      }
    off += m;
    code_base += K * mpad / 2;
    sf_base += K * mpad / 16;
  }
}

/* max |x| over a bf16 array (used for per-expert weight amax) */
float orc_amax_bf16(const uint16_t* x, int64_t n) {
  float a = 0.0f;
#pragma omp parallel for reduction(max : a) schedule(static)
  for (int64_t i = 0; i < n; ++i) a = fmaxf(a, fabsf((float)orc_bf16_to_double(x[i])));
  return a;
}
