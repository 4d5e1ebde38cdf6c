/*
 * q4k_oracle.c — the oracle: a plain, slow, obviously correct CPU statement of what the
 * skinny Q4K x bf16 product computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg call it; the library never does.  It shares no code,
 * header or table with the GPU library and reads the byte format from its written
 * definition (super-block layout below).
 *
 * The computation ("sixi-asi 0.9", section "What I got wrong in 0.8": the quantized matrix
 * products of a verify pass over 4-bit k-quant weights):
 *     Y[i][n] = sum_k w[n][k] * x[i][k],   S[i][n] = sum_k |w[n][k] * x[i][k]|
 * in fp64, summed in increasing k.  The acceptance bound on a GPU result is
 * |Y_gpu - Y| <= 1e-4 * S per element.
 *
 * Super-block layout (144 bytes per 256 weights of one row; rows stored one after another):
 *   bytes 0-1   d, IEEE binary16 little-endian
 *   bytes 2-3   dmin, IEEE binary16 little-endian
 *   bytes 4-15  96-bit little-endian integer F; sub-block j (0..7): sc_j = F bits [12j,12j+6),
 *               m_j = F bits [12j+6, 12j+12)
 *   bytes 16-143 1024-bit little-endian integer Q; weight t (0..255): q_t = Q bits [4t, 4t+4);
 *               weight t is in sub-block t/32
 *   weight value: the fp32 round-to-nearest-even of the exact number d*sc_j*q_t - dmin*m_j.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math).  Floating point
 * here is IEEE binary32/binary64 with FLT_EVAL_METHOD == 0 (x86-64 SSE and AArch64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define SB_WEIGHTS 256
#define SB_BYTES 144

/* ---- number formats, from their IEEE-754 definitions ------------------------------------ */

/* Value of an IEEE binary16 bit pattern (1 sign, 5 exponent, 10 fraction bits, bias 15). */
double oracle_half_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int f = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
  } else if (e == 31) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* Value of a bf16 bit pattern (1 sign, 8 exponent, 7 fraction bits, bias 127). */
double oracle_bf16_value(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 255;
  int f = b & 127;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133);                /* subnormal: f * 2^-133 */
  } else if (e == 255) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(128 + f), e - 134);     /* (1 + f/128) * 2^(e-127) */
  }
  return sign ? -v : v;
}

/* Round a finite float to the nearest binary16 (ties to even).  Returns 0 and the pattern in
 * *out, or 1 when the rounded magnitude overflows binary16 (>= 65520 before rounding). */
int oracle_half_from_float(float f, uint16_t* out) {
  double v = (double)f;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (!isfinite(a)) return 1;
  if (a == 0.0) { *out = sign; return 0; }
  int e2;
  frexp(a, &e2);                               /* a = m * 2^e2, m in [0.5, 1) */
  int E = e2 - 1;                              /* floor(log2 a) */
  int qexp = (E < -14) ? -24 : E - 10;         /* spacing of binary16 numbers near a */
  double r = ldexp(nearbyint(ldexp(a, -qexp)), qexp);   /* exact scale, then round to even */
  if (r >= 65536.0) return 1;
  uint16_t bits;
  if (r < ldexp(1.0, -14)) {
    bits = (uint16_t)ldexp(r, 24);             /* subnormal fraction */
  } else {
    frexp(r, &e2);
    E = e2 - 1;
    int frac = (int)(ldexp(r, 10 - E) - 1024.0);
    bits = (uint16_t)(((E + 15) << 10) | frac);
  }
  *out = (uint16_t)(sign | bits);
  return 0;
}

/* ---- field access, from the layout definition ------------------------------------------- */

/* Bits [pos, pos+n) of the little-endian integer whose bytes start at p (n <= 16). */
static unsigned get_bits(const uint8_t* p, int pos, int n) {
  unsigned v = 0;
  for (int i = 0; i < n; i++) {
    int b = pos + i;
    v |= (unsigned)((p[b / 8] >> (b % 8)) & 1) << i;
  }
  return v;
}

static void set_bits(uint8_t* p, int pos, int n, unsigned v) {
  for (int i = 0; i < n; i++) {
    int b = pos + i;
    if ((v >> i) & 1) p[b / 8] |= (uint8_t)(1u << (b % 8));
    else p[b / 8] &= (uint8_t)~(1u << (b % 8));
  }
}

/* Dequantize one super-block into 256 floats.
 * The real value d*sc*q - dmin*m is computed exactly in binary64: d and dmin are binary16, so
 * both products are integer multiples of 2^-24 below 2^26 in magnitude, and so is their
 * difference; that needs at most 50 significant bits, which binary64 holds.  The cast to
 * float is then the single round-to-nearest-even of the exact value. */
static void dequant_block(const uint8_t* blk, float* out) {
  uint16_t dh = (uint16_t)(blk[0] | (blk[1] << 8));
  uint16_t mh = (uint16_t)(blk[2] | (blk[3] << 8));
  double d = oracle_half_value(dh);
  double dmin = oracle_half_value(mh);
  const uint8_t* F = blk + 4;
  const uint8_t* Q = blk + 16;
  for (int t = 0; t < SB_WEIGHTS; t++) {
    int j = t / 32;
    unsigned sc = get_bits(F, 12 * j, 6);
    unsigned m = get_bits(F, 12 * j + 6, 6);
    unsigned q = get_bits(Q, 4 * t, 4);
    double exact = d * (double)sc * (double)q - dmin * (double)m;
    out[t] = (float)exact;
  }
}

/* out[N*K] = dequantized weights, row-major. */
void oracle_dequant(const uint8_t* Wq, int64_t N, int64_t K, float* out) {
  int64_t nb = K / SB_WEIGHTS;
  for (int64_t n = 0; n < N; n++)
    for (int64_t b = 0; b < nb; b++)
      dequant_block(Wq + (n * nb + b) * SB_BYTES, out + n * K + b * SB_WEIGHTS);
}

/* ---- the product ------------------------------------------------------------------------ */

/* For each requested weight row n = rows[r] (rows == NULL: n = r for r < nrows) and each
 * activation row i < M:
 *   Y[i*nrows + r] = sum_{k=0}^{K-1} w[n][k] * x[i][k]      (binary64, in increasing k)
 *   S[i*nrows + r] = sum_{k=0}^{K-1} |w[n][k] * x[i][k]|
 * x is M x K bf16 bit patterns, row-major.  Each product of a binary32 weight and a bf16
 * activation is exact in binary64 (24 + 8 significant bits).  threads <= 0: OpenMP default. */
void oracle_matmul(const uint8_t* Wq, int64_t N, int64_t K, const uint16_t* X, int M,
                   const int64_t* rows, int64_t nrows, double* Y, double* S, int threads) {
  (void)N;
  double* xv = (double*)malloc(sizeof(double) * (size_t)M * (size_t)K);
  for (int64_t e = 0; e < (int64_t)M * K; e++) xv[e] = oracle_bf16_value(X[e]);
  int64_t nb = K / SB_WEIGHTS;
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
      int64_t n = rows ? rows[r] : r;
      for (int64_t b = 0; b < nb; b++) dequant_block(Wq + (n * nb + b) * SB_BYTES, w + b * SB_WEIGHTS);
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

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- the packer (asymmetric min/max rule; binary32 arithmetic, one rounding per op) ------ */

static float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Pack one super-block of 256 floats.  Returns 0, or 6 when a scale overflows binary16. */
static int pack_block(const float* w, uint8_t* blk) {
  float scale[8], off[8];
  for (int j = 0; j < 8; j++) {
    const float* s = w + 32 * j;
    float lo = 0.0f, hi = s[0];
    for (int t = 0; t < 32; t++) {
      if (s[t] < lo) lo = s[t];
      if (s[t] > hi) hi = s[t];
    }
    scale[j] = (hi - lo) / 15.0f;
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
  float D = (float)oracle_half_value(dh);
  float Dm = (float)oracle_half_value(mh);
  unsigned sc[8], m[8];
  for (int j = 0; j < 8; j++) {
    sc[j] = (D > 0.0f) ? (unsigned)clampf(rintf(scale[j] / D), 0.0f, 63.0f) : 0u;
    m[j] = (Dm > 0.0f) ? (unsigned)clampf(rintf(off[j] / Dm), 0.0f, 63.0f) : 0u;
  }
  memset(blk, 0, SB_BYTES);
  blk[0] = (uint8_t)(dh & 0xff); blk[1] = (uint8_t)(dh >> 8);
  blk[2] = (uint8_t)(mh & 0xff); blk[3] = (uint8_t)(mh >> 8);
  for (int j = 0; j < 8; j++) {
    set_bits(blk + 4, 12 * j, 6, sc[j]);
    set_bits(blk + 4, 12 * j + 6, 6, m[j]);
  }
  for (int t = 0; t < SB_WEIGHTS; t++) {
    int j = t / 32;
    float step = D * (float)sc[j];
    float dmm = Dm * (float)m[j];
    unsigned q = 0;
    if (step > 0.0f) q = (unsigned)clampf(rintf((w[t] + dmm) / step), 0.0f, 15.0f);
    set_bits(blk + 16, 4 * t, 4, q);
  }
  return 0;
}

/* W: N x K row-major binary32.  out: N*(K/256)*144 bytes.  Returns 0, or 6 on a non-finite
 * weight or an fp16 overflow of d or dmin. */
int oracle_pack(const float* W, int64_t N, int64_t K, uint8_t* out) {
  for (int64_t e = 0; e < N * K; e++)
    if (!isfinite(W[e])) return 6;
  int64_t nb = K / SB_WEIGHTS;
  for (int64_t n = 0; n < N; n++)
    for (int64_t b = 0; b < nb; b++) {
      int rc = pack_block(W + n * K + b * SB_WEIGHTS, out + (n * nb + b) * SB_BYTES);
      if (rc) return rc;
    }
  return 0;
}
