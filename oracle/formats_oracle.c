/*
 * formats_oracle.c — the oracle for the other weight formats of the skinny product: a 5-bit
 * k-quant (Q5K), NVFP4 (W4A16) and 4-bit integers with one scale per 128 columns (INT4).
 * TEST INFRASTRUCTURE ONLY, like q4k_oracle.c: plain, slow, decoded from the written layouts
 * below, sharing nothing with the GPU library.
 *
 * Where the formats come from.  The pages run Q4_K_M files, which mix k-quant widths ("sixi-asi
 * 0.9", section "Numbers"); they weigh NVFP4 W4A16 weights (FlashRT issue #153: the NVFP4 W4A16
 * GEMM is most of the decode time; "sixi-asi 0.9", section "What I got wrong in 0.8": block-scaled
 * FP4 reached through tcgen05) and plain 4-bit integer weights with one scale per 128 columns
 * ("sixi-asi 0.11", section "What did not work").  None prints a byte layout; the layouts here are
 * the library's, and every weight value below is a single IEEE rounding of an exact number.
 *
 * Format codes: 1 Q5K, 2 NVFP4, 3 INT4, 4 Q6K (0 is Q4K, in q4k_oracle.c).
 *
 * Q5K: 176 bytes per super-block of 256 weights of one row (rows one after another, blocks in
 * order of k):
 *   bytes 0-1    d, binary16;  bytes 2-3  dmin, binary16
 *   bytes 4-15   96-bit integer F: sub-block j (0..7, weights 32j..32j+31): sc_j = F bits
 *                [12j, 12j+6), m_j = F bits [12j+6, 12j+12)
 *   bytes 16-47  eight 32-bit little-endian words; word j holds the high bits of sub-block j:
 *                weight t = 32j + 8c + i (c = 0..3, i = 0..7) has its high bit at bit 4i + c
 *   bytes 48-175 1024-bit integer L: the low 4 bits of weight t are L bits [4t, 4t+4)
 *   q_t = low + 16 * high (0..31); weight = RN32(d*sc_j*q_t - dmin*m_j).
 *
 * NVFP4: 144 bytes per 256 weights, then one 16-byte trailer after all N rows:
 *   bytes 0-15   s_0..s_15, E4M3 (sign, 4 exponent bits with bias 7, 3 fraction bits; no
 *                infinities; exponent 15 with fraction 7 is NaN), s_b scales weights 16b..16b+15
 *   bytes 16-143 1024-bit integer Q: weight t has the E2M1 code Q bits [4t, 4t+4) (sign bit 3,
 *                2 exponent bits with bias 1, 1 fraction bit)
 *   trailer      g, binary32 (the tensor scale), then 12 zero bytes
 *   weight = RN32(g * s_b * v_t); s_b * v_t is exact in binary32, so this is one rounding.
 *
 * Q6K: 208 bytes per super-block of 256 weights of one row (rows one after another), then a
 * plane of N x K/256 binary16 super-block scales d (row-major) at byte N*(K/256)*208:
 *   bytes 0-15    u_j, sub-block j = weights 16j..16j+15: sc_j = (u_j & 127) - 64 (-64..63;
 *                 bit 7 is not used)
 *   bytes 16-143  1024-bit integer L: the low 4 bits of weight t are L bits [4t, 4t+4)
 *   bytes 144-207 sixteen 32-bit little-endian words; word m holds the 2-bit high parts of
 *                 weights 16m..16m+15: weight t = 16m + 8a + i (a = 0..1, i = 0..7) at bits
 *                 8a + 16*(i >= 4) + 2*(i % 4)
 *   q_t = low + 16 * high (0..63); weight = RN32(d*sc_j*(q_t - 32)), exact in binary32 (at most
 *   11 + 6 + 6 significant bits).
 *
 * INT4: a quant plane, then a scale plane:
 *   quant plane  N rows of K/2 bytes; weight k of a row: the two's-complement 4-bit integer
 *                q (-8..7) at bits [4k, 4k+4) of the row's little-endian integer
 *   scale plane  N x K/128 binary16, row-major, at byte N*K/2: s_{n,g} scales weights
 *                128g..128g+127 of row n
 *   weight = s * q, exact in binary32.
 *
 * Packers (the pages give none; plain rules, binary32 arithmetic, one rounding per operation):
 *   Q5K  the Q4K rule of q4k_oracle.c with 31 quant levels instead of 15.
 *   NVFP4 amax = max |w| over the tensor, g = amax / 2688 (2688 = 6 * 448; g = 1 when that is
 *        not positive); per 16 weights a = max |w|, s = E4M3(a / 6 / g) rounded to nearest even
 *        and clamped to 448; S = value(s) * g; v_t = E2M1(w_t / S) rounded to nearest even and
 *        clamped to 6 (S = 0: v_t = 0); the sign of w_t is kept, also when v_t rounds to 0.
 *   INT4 per 128 weights a = max |w|, s = binary16(a / 7) (error 6 on overflow), S = value(s),
 *        q = S > 0 ? clamp(rint(w / S), -8, 7) : 0.
 *   Q6K  per 16 weights a_j = max |w|, scale_j = a_j / 31; d = binary16(max_j scale_j / 63)
 *        (error 6 on overflow), D = value(d); sc_j = D > 0 ? clamp(rint(scale_j / D), 0, 63) : 0;
 *        q_t = D*sc_j > 0 ? clamp(rint(w_t / (D*sc_j)), -32, 31) + 32 : 32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double oracle_half_value(uint16_t h);
double oracle_bf16_value(uint16_t b);
int oracle_half_from_float(float f, uint16_t* out);

enum { FMT_Q5K = 1, FMT_NVFP4 = 2, FMT_INT4 = 3, FMT_Q6K = 4 };

static unsigned bits_of(const uint8_t* p, int64_t pos, int n) {
  unsigned v = 0;
  for (int i = 0; i < n; i++) {
    int64_t b = pos + i;
    v |= (unsigned)((p[b / 8] >> (b % 8)) & 1) << i;
  }
  return v;
}

static void put_bits(uint8_t* p, int64_t pos, int n, unsigned v) {
  for (int i = 0; i < n; i++) {
    int64_t b = pos + i;
    if ((v >> i) & 1) p[b / 8] |= (uint8_t)(1u << (b % 8));
    else p[b / 8] &= (uint8_t)~(1u << (b % 8));
  }
}

/* ---- the number formats, from their definitions ----------------------------------------- */

/* E4M3: 1 sign, 4 exponent (bias 7), 3 fraction bits; exponent 0 subnormal (f * 2^-9);
 * 0x7F / 0xFF NaN; no infinities. */
double oracle_e4m3_value(uint8_t c) {
  int sign = (c >> 7) & 1, e = (c >> 3) & 15, f = c & 7;
  double v;
  if (e == 15 && f == 7) v = NAN;
  else if (e == 0) v = ldexp((double)f, -9);
  else v = ldexp((double)(8 + f), e - 10);   /* (1 + f/8) * 2^(e-7) */
  return sign ? -v : v;
}

/* E2M1: 1 sign, 2 exponent (bias 1), 1 fraction bit; exponent 0 subnormal (f * 0.5). */
double oracle_e2m1_value(uint8_t c) {
  int sign = (c >> 3) & 1, e = (c >> 1) & 3, f = c & 1;
  double v = (e == 0) ? 0.5 * f : ldexp((double)(2 + f), e - 2);   /* (1 + f/2) * 2^(e-1) */
  return sign ? -v : v;
}

/* Nearest code of a non-negative finite value among the first `ncodes` non-negative codes of a
 * format whose values increase with the code, ties to the even code, values past the last
 * code clamped to it. */
static unsigned nearest_code(double a, unsigned ncodes, double (*value)(uint8_t)) {
  unsigned best = 0;
  for (unsigned c = 1; c < ncodes; c++) {
    double lo = value((uint8_t)(c - 1)), hi = value((uint8_t)c);
    if (a >= hi) { best = c; continue; }
    double mid = 0.5 * (lo + hi);                 /* exact: both have few significant bits */
    if (a > mid || (a == mid && (c % 2) == 0)) best = c;
    break;
  }
  return best;
}

/* E4M3 code of a non-negative finite float: nearest even, clamped to 448 (code 0x7E). */
uint8_t oracle_e4m3_from_float(float x) { return (uint8_t)nearest_code((double)x, 127, oracle_e4m3_value); }

/* E2M1 code of a finite float: nearest even magnitude, clamped to 6, sign kept. */
uint8_t oracle_e2m1_from_float(float x) {
  unsigned c = nearest_code(fabs((double)x), 8, oracle_e2m1_value);
  return (uint8_t)(c | (signbit(x) ? 8u : 0u));
}

/* ---- sizes ------------------------------------------------------------------------------ */

int64_t oracle_fmt_packed_bytes(int fmt, int64_t N, int64_t K) {
  switch (fmt) {
    case FMT_Q5K: return N * (K / 256) * 176;
    case FMT_NVFP4: return N * (K / 256) * 144 + 16;
    case FMT_INT4: return N * (K / 2) + N * (K / 128) * 2;
    case FMT_Q6K: return N * (K / 256) * 208 + N * (K / 256) * 2;
    default: return -1;
  }
}

/* ---- dequantization: row n into w[0..K) ------------------------------------------------- */

static void dequant_row(int fmt, const uint8_t* Wq, int64_t N, int64_t K, int64_t n, float* w) {
  int64_t nb = K / 256;
  if (fmt == FMT_Q5K) {
    for (int64_t b = 0; b < nb; b++) {
      const uint8_t* blk = Wq + (n * nb + b) * 176;
      double d = oracle_half_value((uint16_t)(blk[0] | (blk[1] << 8)));
      double dmin = oracle_half_value((uint16_t)(blk[2] | (blk[3] << 8)));
      for (int t = 0; t < 256; t++) {
        int j = t / 32, c = (t % 32) / 8, i = t % 8;
        unsigned sc = bits_of(blk + 4, 12 * j, 6), m = bits_of(blk + 4, 12 * j + 6, 6);
        unsigned hi = bits_of(blk + 16, 32 * j + 4 * i + c, 1);
        unsigned q = bits_of(blk + 48, 4 * t, 4) + 16 * hi;
        /* both products are multiples of 2^-24 below 2^27: the difference is exact in fp64 */
        w[b * 256 + t] = (float)(d * (double)sc * (double)q - dmin * (double)m);
      }
    }
  } else if (fmt == FMT_NVFP4) {
    const uint8_t* tr = Wq + N * nb * 144;
    uint32_t gb = (uint32_t)tr[0] | ((uint32_t)tr[1] << 8) | ((uint32_t)tr[2] << 16) | ((uint32_t)tr[3] << 24);
    float gf;
    memcpy(&gf, &gb, 4);
    double g = (double)gf;
    for (int64_t b = 0; b < nb; b++) {
      const uint8_t* blk = Wq + (n * nb + b) * 144;
      for (int t = 0; t < 256; t++) {
        double s = oracle_e4m3_value(blk[t / 16]);
        double v = oracle_e2m1_value((uint8_t)bits_of(blk + 16, 4 * t, 4));
        /* s*v has <= 6 significant bits, g 24: the product is exact in fp64 */
        w[b * 256 + t] = (float)(g * (s * v));
      }
    }
  } else if (fmt == FMT_Q6K) {
    const uint8_t* dp = Wq + N * nb * 208 + n * nb * 2;
    for (int64_t b = 0; b < nb; b++) {
      const uint8_t* blk = Wq + (n * nb + b) * 208;
      double d = oracle_half_value((uint16_t)(dp[2 * b] | (dp[2 * b + 1] << 8)));
      for (int t = 0; t < 256; t++) {
        int j = t / 16, m = t / 16, a = (t % 16) / 8, i = t % 8;
        int sc = (int)(blk[j] & 127) - 64;
        unsigned hi = bits_of(blk + 144, 32 * m + 8 * a + 16 * (i >= 4) + 2 * (i % 4), 2);
        int q = (int)(bits_of(blk + 16, 4 * t, 4) + 16 * hi);
        w[b * 256 + t] = (float)(d * (double)sc * (double)(q - 32));
      }
    }
  } else {  /* FMT_INT4 */
    const uint8_t* row = Wq + n * (K / 2);
    const uint8_t* sc = Wq + N * (K / 2) + n * (K / 128) * 2;
    for (int64_t k = 0; k < K; k++) {
      unsigned u = bits_of(row, 4 * k, 4);
      int q = (u >= 8) ? (int)u - 16 : (int)u;
      double s = oracle_half_value((uint16_t)(sc[2 * (k / 128)] | (sc[2 * (k / 128) + 1] << 8)));
      w[k] = (float)(s * (double)q);
    }
  }
}

/* out[r*K .. r*K+K) = row rows[r] (rows == NULL: row r) of the dequantized matrix. */
void oracle_fmt_dequant(int fmt, const uint8_t* Wq, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                        float* out) {
  for (int64_t r = 0; r < nrows; r++) dequant_row(fmt, Wq, N, K, rows ? rows[r] : r, out + r * K);
}

/* Y[i*nrows + r] = sum_k w[n][k] * x[i][k] and S[...] = sum_k |w[n][k] * x[i][k]| in binary64,
 * in increasing k, for n = rows[r] (rows == NULL: n = r); x: M x K bf16 bit patterns. */
void oracle_fmt_matmul(int fmt, const uint8_t* Wq, int64_t N, int64_t K, const uint16_t* X, int M,
                       const int64_t* rows, int64_t nrows, double* Y, double* S, int threads) {
  double* xv = (double*)malloc(sizeof(double) * (size_t)M * (size_t)K);
  for (int64_t e = 0; e < (int64_t)M * K; e++) xv[e] = oracle_bf16_value(X[e]);
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
#pragma omp parallel
  {
    float* w = (float*)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; r++) {
      dequant_row(fmt, Wq, N, K, rows ? rows[r] : r, w);
      for (int i = 0; i < M; i++) {
        const double* x = xv + (int64_t)i * K;
        double y = 0.0, s = 0.0;
        for (int64_t k = 0; k < K; k++) {
          double p = (double)w[k] * x[k];
          y += p;
          s += fabs(p);
        }
        Y[(int64_t)i * nrows + r] = y;
        S[(int64_t)i * nrows + r] = s;
      }
    }
    free(w);
  }
  free(xv);
}

/* ---- packers ---------------------------------------------------------------------------- */

static float clampf_(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

static int pack_q5k_block(const float* w, uint8_t* blk) {
  float scale[8], off[8];
  for (int j = 0; j < 8; j++) {
    const float* s = w + 32 * j;
    float lo = 0.0f, hi = s[0];
    for (int t = 0; t < 32; t++) {
      if (s[t] < lo) lo = s[t];
      if (s[t] > hi) hi = s[t];
    }
    scale[j] = (hi - lo) / 31.0f;
    off[j] = 0.0f - lo;
  }
  float smax = 0.0f, omax = 0.0f;
  for (int j = 0; j < 8; j++) {
    if (scale[j] > smax) smax = scale[j];
    if (off[j] > omax) omax = off[j];
  }
  uint16_t dh, mh;
  if (oracle_half_from_float(smax / 63.0f, &dh)) return 6;
  if (oracle_half_from_float(omax / 63.0f, &mh)) return 6;
  float D = (float)oracle_half_value(dh), Dm = (float)oracle_half_value(mh);
  memset(blk, 0, 176);
  blk[0] = (uint8_t)(dh & 0xff); blk[1] = (uint8_t)(dh >> 8);
  blk[2] = (uint8_t)(mh & 0xff); blk[3] = (uint8_t)(mh >> 8);
  for (int j = 0; j < 8; j++) {
    unsigned sc = (D > 0.0f) ? (unsigned)clampf_(rintf(scale[j] / D), 0.0f, 63.0f) : 0u;
    unsigned m = (Dm > 0.0f) ? (unsigned)clampf_(rintf(off[j] / Dm), 0.0f, 63.0f) : 0u;
    put_bits(blk + 4, 12 * j, 6, sc);
    put_bits(blk + 4, 12 * j + 6, 6, m);
    float step = D * (float)sc, dmm = Dm * (float)m;
    for (int u = 0; u < 32; u++) {
      int t = 32 * j + u;
      unsigned q = 0;
      if (step > 0.0f) q = (unsigned)clampf_(rintf((w[t] + dmm) / step), 0.0f, 31.0f);
      put_bits(blk + 48, 4 * t, 4, q & 15u);
      put_bits(blk + 16, 32 * j + 4 * (u % 8) + u / 8, 1, q >> 4);
    }
  }
  return 0;
}

static void pack_nvfp4_block(const float* w, float g, uint8_t* blk) {
  memset(blk, 0, 144);
  for (int b = 0; b < 16; b++) {
    float a = 0.0f;
    for (int t = 16 * b; t < 16 * b + 16; t++)
      if (fabsf(w[t]) > a) a = fabsf(w[t]);
    float r = a / 6.0f;
    r = r / g;
    uint8_t s = oracle_e4m3_from_float(r);
    blk[b] = s;
    float S = (float)oracle_e4m3_value(s) * g;
    for (int t = 16 * b; t < 16 * b + 16; t++) {
      uint8_t c = (S > 0.0f) ? oracle_e2m1_from_float(w[t] / S) : 0;
      put_bits(blk + 16, 4 * t, 4, c);
    }
  }
}

static int pack_q6k_block(const float* w, uint8_t* blk, uint8_t* dbits) {
  float scale[16];
  for (int j = 0; j < 16; j++) {
    float a = 0.0f;
    for (int t = 16 * j; t < 16 * j + 16; t++)
      if (fabsf(w[t]) > a) a = fabsf(w[t]);
    scale[j] = a / 31.0f;
  }
  float smax = 0.0f;
  for (int j = 0; j < 16; j++)
    if (scale[j] > smax) smax = scale[j];
  uint16_t dh;
  if (oracle_half_from_float(smax / 63.0f, &dh)) return 6;
  float D = (float)oracle_half_value(dh);
  dbits[0] = (uint8_t)(dh & 0xff);
  dbits[1] = (uint8_t)(dh >> 8);
  memset(blk, 0, 208);
  for (int j = 0; j < 16; j++) {
    unsigned sc = (D > 0.0f) ? (unsigned)clampf_(rintf(scale[j] / D), 0.0f, 63.0f) : 0u;
    blk[j] = (uint8_t)(sc + 64);
    float step = D * (float)sc;
    for (int t = 16 * j; t < 16 * j + 16; t++) {
      int q = 32;
      if (step > 0.0f) q = (int)clampf_(rintf(w[t] / step), -32.0f, 31.0f) + 32;
      int m = t / 16, a = (t % 16) / 8, i = t % 8;
      put_bits(blk + 16, 4 * t, 4, (unsigned)q & 15u);
      put_bits(blk + 144, 32 * m + 8 * a + 16 * (i >= 4) + 2 * (i % 4), 2, (unsigned)q >> 4);
    }
  }
  return 0;
}

/* W: N x K row-major binary32.  Returns 0, 6 on a non-finite weight or a binary16 overflow,
 * 2 on an unknown format. */
int oracle_fmt_pack(int fmt, const float* W, int64_t N, int64_t K, uint8_t* out) {
  for (int64_t e = 0; e < N * K; e++)
    if (!isfinite(W[e])) return 6;
  int64_t nb = K / 256;
  if (fmt == FMT_Q5K) {
    for (int64_t n = 0; n < N; n++)
      for (int64_t b = 0; b < nb; b++) {
        int rc = pack_q5k_block(W + n * K + b * 256, out + (n * nb + b) * 176);
        if (rc) return rc;
      }
    return 0;
  }
  if (fmt == FMT_NVFP4) {
    float amax = 0.0f;
    for (int64_t e = 0; e < N * K; e++)
      if (fabsf(W[e]) > amax) amax = fabsf(W[e]);
    float g = amax / 2688.0f;
    if (!(g > 0.0f)) g = 1.0f;
    for (int64_t n = 0; n < N; n++)
      for (int64_t b = 0; b < nb; b++) pack_nvfp4_block(W + n * K + b * 256, g, out + (n * nb + b) * 144);
    uint8_t* tr = out + N * nb * 144;
    memset(tr, 0, 16);
    memcpy(tr, &g, 4);   /* little-endian hosts */
    return 0;
  }
  if (fmt == FMT_Q6K) {
    uint8_t* dplane = out + N * nb * 208;
    for (int64_t n = 0; n < N; n++)
      for (int64_t b = 0; b < nb; b++) {
        int rc = pack_q6k_block(W + n * K + b * 256, out + (n * nb + b) * 208, dplane + (n * nb + b) * 2);
        if (rc) return rc;
      }
    return 0;
  }
  if (fmt == FMT_INT4) {
    uint8_t* scales = out + N * (K / 2);
    memset(out, 0, (size_t)(N * (K / 2)));
    for (int64_t n = 0; n < N; n++)
      for (int64_t gi = 0; gi < K / 128; gi++) {
        const float* s = W + n * K + gi * 128;
        float a = 0.0f;
        for (int t = 0; t < 128; t++)
          if (fabsf(s[t]) > a) a = fabsf(s[t]);
        uint16_t h;
        if (oracle_half_from_float(a / 7.0f, &h)) return 6;
        uint8_t* sp = scales + (n * (K / 128) + gi) * 2;
        sp[0] = (uint8_t)(h & 0xff);
        sp[1] = (uint8_t)(h >> 8);
        float S = (float)oracle_half_value(h);
        for (int t = 0; t < 128; t++) {
          int q = (S > 0.0f) ? (int)clampf_(rintf(s[t] / S), -8.0f, 7.0f) : 0;
          put_bits(out + n * (K / 2), 4 * (gi * 128 + t), 4, (unsigned)q & 15u);
        }
      }
    return 0;
  }
  return 2;
}
