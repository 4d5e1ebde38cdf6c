// qmm_pack.cpp — host packer: fp32 weights -> Q4K super-blocks (the cold path).
//
// The pages run GGUF "Q4_K_M" files ("sixi-asi 0.9", section "Numbers") and never show how
// those weights were quantized; this packer uses the plain asymmetric min/max rule stated in
// qmm.h: per 32-weight sub-block the range [min(0, min w), max w] is split into 15 steps,
// the per-sub-block step and offset are quantized to 6 bits against fp16 super-block scales,
// and each weight goes to the nearest 4-bit level.  Every operation is one IEEE fp32
// operation rounded to nearest even (built with -ffp-contract=off).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

#include "q4k_internal.h"

namespace q4k {
namespace {

inline float to_half_and_back(float v, uint16_t* bits, bool* overflow) {
  const _Float16 h = static_cast<_Float16>(v);  // IEEE binary16, round to nearest even
  std::memcpy(bits, &h, sizeof(*bits));
  const float back = static_cast<float>(h);
  *overflow = std::isinf(back);
  return back;
}

inline uint32_t level(float v, float hi) {
  const float r = std::rint(v);  // round half to even in the default rounding mode
  return static_cast<uint32_t>(r < 0.0f ? 0.0f : (r > hi ? hi : r));
}

// Packs one super-block (256 weights at w) into 144 bytes at out.  Returns false on overflow.
bool pack_superblock(const float* w, uint8_t* out) {
  float step_raw[8], offset_raw[8];
  for (int j = 0; j < 8; ++j) {
    const float* s = w + 32 * j;
    float mn = 0.0f;
    float mx = s[0];
    for (int t = 0; t < 32; ++t) {
      mn = (s[t] < mn) ? s[t] : mn;
      mx = (s[t] > mx) ? s[t] : mx;
    }
    step_raw[j] = (mx - mn) / 15.0f;
    offset_raw[j] = 0.0f - mn;
  }
  float step_max = 0.0f, offset_max = 0.0f;
  for (int j = 0; j < 8; ++j) {
    step_max = std::max(step_max, step_raw[j]);
    offset_max = std::max(offset_max, offset_raw[j]);
  }
  uint16_t d_bits = 0, dmin_bits = 0;
  bool ovf_d = false, ovf_m = false;
  const float D = to_half_and_back(step_max / 63.0f, &d_bits, &ovf_d);
  const float Dm = to_half_and_back(offset_max / 63.0f, &dmin_bits, &ovf_m);
  if (ovf_d || ovf_m) return false;

  uint32_t sc[8], mn[8];
  for (int j = 0; j < 8; ++j) {
    sc[j] = (D > 0.0f) ? level(step_raw[j] / D, 63.0f) : 0u;
    mn[j] = (Dm > 0.0f) ? level(offset_raw[j] / Dm, 63.0f) : 0u;
  }

  // 96-bit field: 12-bit group j = sc_j | m_j << 6 at bit 12 j.
  uint64_t f_lo = 0, f_hi = 0;
  for (int j = 0; j < 8; ++j) {
    const uint64_t g = (uint64_t)(sc[j] | (mn[j] << 6));
    const int bit = 12 * j;
    if (bit + 12 <= 64) {
      f_lo |= g << bit;
    } else if (bit >= 64) {
      f_hi |= g << (bit - 64);
    } else {
      f_lo |= g << bit;
      f_hi |= g >> (64 - bit);
    }
  }
  out[0] = (uint8_t)(d_bits & 0xFF);
  out[1] = (uint8_t)(d_bits >> 8);
  out[2] = (uint8_t)(dmin_bits & 0xFF);
  out[3] = (uint8_t)(dmin_bits >> 8);
  for (int b = 0; b < 8; ++b) out[4 + b] = (uint8_t)(f_lo >> (8 * b));
  for (int b = 0; b < 4; ++b) out[12 + b] = (uint8_t)(f_hi >> (8 * b));

  // Quants: weight t in byte 16 + t/2, low nibble for even t.
  for (int j = 0; j < 8; ++j) {
    const float step = D * static_cast<float>(sc[j]);
    const float off = Dm * static_cast<float>(mn[j]);
    for (int t = 32 * j; t < 32 * j + 32; t += 2) {
      uint32_t q0 = 0, q1 = 0;
      if (step > 0.0f) {
        q0 = level((w[t] + off) / step, 15.0f);
        q1 = level((w[t + 1] + off) / step, 15.0f);
      }
      out[16 + t / 2] = (uint8_t)(q0 | (q1 << 4));
    }
  }
  return true;
}

// ---- the other formats -------------------------------------------------------------------

// Q5K super-block (176 bytes): the Q4K header and scale fields, 31 quant levels; the low nibble
// of weight t at bits 4t of bytes 48.., its high bit in the 32-bit word of its sub-block j at
// bit 4i + c (t = 32j + 8c + i).
bool pack_q5k_superblock(const float* w, uint8_t* out) {
  float step_raw[8], offset_raw[8];
  for (int j = 0; j < 8; ++j) {
    const float* s = w + 32 * j;
    float mn = 0.0f, mx = s[0];
    for (int t = 0; t < 32; ++t) {
      mn = (s[t] < mn) ? s[t] : mn;
      mx = (s[t] > mx) ? s[t] : mx;
    }
    step_raw[j] = (mx - mn) / 31.0f;
    offset_raw[j] = 0.0f - mn;
  }
  float step_max = 0.0f, offset_max = 0.0f;
  for (int j = 0; j < 8; ++j) {
    step_max = std::max(step_max, step_raw[j]);
    offset_max = std::max(offset_max, offset_raw[j]);
  }
  uint16_t d_bits = 0, dmin_bits = 0;
  bool ovf_d = false, ovf_m = false;
  const float D = to_half_and_back(step_max / 63.0f, &d_bits, &ovf_d);
  const float Dm = to_half_and_back(offset_max / 63.0f, &dmin_bits, &ovf_m);
  if (ovf_d || ovf_m) return false;
  std::memset(out, 0, 176);
  out[0] = (uint8_t)(d_bits & 0xFF);
  out[1] = (uint8_t)(d_bits >> 8);
  out[2] = (uint8_t)(dmin_bits & 0xFF);
  out[3] = (uint8_t)(dmin_bits >> 8);
  uint64_t f_lo = 0, f_hi = 0;
  for (int j = 0; j < 8; ++j) {
    const uint32_t sc = (D > 0.0f) ? level(step_raw[j] / D, 63.0f) : 0u;
    const uint32_t mn = (Dm > 0.0f) ? level(offset_raw[j] / Dm, 63.0f) : 0u;
    const uint64_t g = (uint64_t)(sc | (mn << 6));
    const int bit = 12 * j;
    if (bit + 12 <= 64) {
      f_lo |= g << bit;
    } else if (bit >= 64) {
      f_hi |= g << (bit - 64);
    } else {
      f_lo |= g << bit;
      f_hi |= g >> (64 - bit);
    }
    const float step = D * static_cast<float>(sc);
    const float off = Dm * static_cast<float>(mn);
    uint32_t hi_word = 0;
    for (int u = 0; u < 32; ++u) {
      const int t = 32 * j + u;
      const uint32_t q = step > 0.0f ? level((w[t] + off) / step, 31.0f) : 0u;
      out[48 + t / 2] |= (uint8_t)((q & 15u) << (4 * (t & 1)));
      hi_word |= (q >> 4) << (4 * (u & 7) + (u >> 3));
    }
    for (int b = 0; b < 4; ++b) out[16 + 4 * j + b] = (uint8_t)(hi_word >> (8 * b));
  }
  for (int b = 0; b < 8; ++b) out[4 + b] = (uint8_t)(f_lo >> (8 * b));
  for (int b = 0; b < 4; ++b) out[12 + b] = (uint8_t)(f_hi >> (8 * b));
  return true;
}

// E4M3 (bias 7, 3 fraction bits, largest finite 448) of a non-negative finite value: round to
// nearest even on the format's grid, clamped to 448.
uint8_t e4m3_code(float x) {
  if (!(x > 0.0f)) return 0;
  if (x >= 448.0f) return 0x7E;
  int e = 0;
  std::frexp(x, &e);                       // x = m 2^e, m in [0.5, 1)
  const int E = e - 1;                     // floor(log2 x)
  const int qe = E < -6 ? -9 : E - 3;      // grid spacing: 2^-9 below 2^-6, else 2^(E-3)
  const float r = std::ldexp(std::rint(std::ldexp(x, -qe)), qe);
  if (r >= 448.0f) return 0x7E;
  if (r < 0.015625f) return (uint8_t)std::ldexp(r, 9);   // subnormal: r / 2^-9
  int e2 = 0;
  std::frexp(r, &e2);
  const int E2 = e2 - 1;
  const int f = (int)(std::ldexp(r, 3 - E2)) - 8;
  return (uint8_t)(((E2 + 7) << 3) | f);
}

float e4m3_float(uint8_t c) {
  const int e = (c >> 3) & 15, f = c & 7;
  const float v = e == 0 ? std::ldexp((float)f, -9) : std::ldexp((float)(8 + f), e - 10);
  return (c & 0x80) ? -v : v;
}

// E2M1 (bias 1, 1 fraction bit, largest 6) of a finite value: nearest even magnitude, clamped
// to 6, the sign bit of x kept.
uint8_t e2m1_code(float x) {
  const float a = std::fabs(x);
  uint8_t c = 7;
  if (a < 6.0f) {
    int e = 0;
    std::frexp(a, &e);
    const int E = a > 0.0f ? e - 1 : -1;
    const int qe = E < 0 ? -1 : E - 1;     // spacing 0.5 below 1, else 2^(E-1)
    const float r = std::ldexp(std::rint(std::ldexp(a, -qe)), qe);
    if (r < 1.0f) {
      c = (uint8_t)(r * 2.0f);
    } else {
      int e2 = 0;
      std::frexp(r, &e2);
      const int E2 = e2 - 1;
      c = (uint8_t)(((E2 + 1) << 1) | ((int)std::ldexp(r, 1 - E2) - 2));
    }
  }
  return std::signbit(x) ? (uint8_t)(c | 8u) : c;
}

// NVFP4 block (144 bytes): 16 E4M3 scales, then the E2M1 codes of the 256 weights (low nibble
// first), against the tensor scale g.
void pack_nvfp4_superblock(const float* w, float g, uint8_t* out) {
  std::memset(out, 0, 144);
  for (int b = 0; b < 16; ++b) {
    float a = 0.0f;
    for (int t = 16 * b; t < 16 * b + 16; ++t) a = std::max(a, std::fabs(w[t]));
    const float r = (a / 6.0f) / g;
    const uint8_t s = e4m3_code(r);
    out[b] = s;
    const float S = e4m3_float(s) * g;
    for (int t = 16 * b; t < 16 * b + 16; ++t) {
      const uint8_t c = S > 0.0f ? e2m1_code(w[t] / S) : 0;
      out[16 + t / 2] |= (uint8_t)(c << (4 * (t & 1)));
    }
  }
}

// INT4 row: K/2 bytes of two's-complement quants (low nibble first) and K/128 binary16 scales.
bool pack_int4_row(const float* w, int64_t K, uint8_t* q, uint8_t* scales) {
  for (int64_t g = 0; g < K / 128; ++g) {
    const float* s = w + 128 * g;
    float a = 0.0f;
    for (int t = 0; t < 128; ++t) a = std::max(a, std::fabs(s[t]));
    uint16_t bits = 0;
    bool ovf = false;
    const float S = to_half_and_back(a / 7.0f, &bits, &ovf);
    if (ovf) return false;
    scales[2 * g] = (uint8_t)(bits & 0xFF);
    scales[2 * g + 1] = (uint8_t)(bits >> 8);
    for (int t = 0; t < 128; t += 2) {
      int v[2] = {0, 0};
      for (int u = 0; u < 2; ++u) {
        if (S > 0.0f) {
          const float r = std::rint(s[t + u] / S);
          v[u] = (int)(r < -8.0f ? -8.0f : (r > 7.0f ? 7.0f : r));
        }
      }
      q[64 * g + t / 2] = (uint8_t)((v[0] & 15) | ((v[1] & 15) << 4));
    }
  }
  return true;
}

// Q6K super-block (208 bytes, its binary16 d written to dbits): 16 scale bytes u = sc + 64, the
// low nibbles of the 256 quants, then per 16 weights one 32-bit word of their 2-bit high parts
// (weight 8a + i of the sub-block at bit 8a + 16 (i >= 4) + 2 (i % 4)).
bool pack_q6k_superblock(const float* w, uint8_t* out, uint8_t* dbits) {
  float scale[16];
  float smax = 0.0f;
  for (int j = 0; j < 16; ++j) {
    float a = 0.0f;
    for (int t = 16 * j; t < 16 * j + 16; ++t) a = std::max(a, std::fabs(w[t]));
    scale[j] = a / 31.0f;
    smax = std::max(smax, scale[j]);
  }
  uint16_t d_bits = 0;
  bool ovf = false;
  const float D = to_half_and_back(smax / 63.0f, &d_bits, &ovf);
  if (ovf) return false;
  dbits[0] = (uint8_t)(d_bits & 0xFF);
  dbits[1] = (uint8_t)(d_bits >> 8);
  std::memset(out, 0, 208);
  for (int j = 0; j < 16; ++j) {
    const uint32_t sc = D > 0.0f ? level(scale[j] / D, 63.0f) : 0u;
    out[j] = (uint8_t)(sc + 64);
    const float step = D * static_cast<float>(sc);
    uint32_t hw = 0;
    for (int u = 0; u < 16; ++u) {
      const int t = 16 * j + u;
      int q = 32;
      if (step > 0.0f) {
        const float r = std::rint(w[t] / step);
        q = (int)(r < -32.0f ? -32.0f : (r > 31.0f ? 31.0f : r)) + 32;
      }
      out[16 + t / 2] |= (uint8_t)((q & 15) << (4 * (t & 1)));
      const int a = u >> 3, i = u & 7;
      hw |= (uint32_t)(q >> 4) << (8 * a + 16 * (i >> 2) + 2 * (i & 3));
    }
    for (int b = 0; b < 4; ++b) out[144 + 4 * j + b] = (uint8_t)(hw >> (8 * b));
  }
  return true;
}

// Rows [0, N) split over up to `threads` threads; fn(n) packs row n and returns false on error.
template <class Fn>
int for_rows(int64_t N, int threads, Fn fn) {
  int nthr = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
  if (nthr < 1) nthr = 1;
  nthr = (int)std::min<int64_t>(nthr, N);
  std::vector<int> status(nthr, 0);
  auto work = [&](int tid) {
    const int64_t r0 = N * tid / nthr, r1 = N * (tid + 1) / nthr;
    for (int64_t n = r0; n < r1; ++n)
      if (!fn(n)) {
        status[tid] = 6;
        return;
      }
  };
  if (nthr == 1) {
    work(0);
  } else {
    std::vector<std::thread> pool;
    for (int t = 0; t < nthr; ++t) pool.emplace_back(work, t);
    for (auto& th : pool) th.join();
  }
  for (int st : status)
    if (st) return st;
  return 0;
}

}  // namespace

int pack_q4k(const float* W, int64_t N, int64_t K, uint8_t* out, int threads) {
  const int64_t nb = K / 256;
  const int64_t total = N * K;
  for (int64_t e = 0; e < total; ++e)
    if (!std::isfinite(W[e])) return 6;
  int nthr = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
  if (nthr < 1) nthr = 1;
  nthr = (int)std::min<int64_t>(nthr, N);
  std::vector<int> status(nthr, 0);
  auto work = [&](int tid) {
    const int64_t r0 = N * tid / nthr, r1 = N * (tid + 1) / nthr;
    for (int64_t n = r0; n < r1; ++n)
      for (int64_t b = 0; b < nb; ++b)
        if (!pack_superblock(W + n * K + b * 256, out + (n * nb + b) * 144)) {
          status[tid] = 6;
          return;
        }
  };
  if (nthr == 1) {
    work(0);
  } else {
    std::vector<std::thread> pool;
    for (int t = 0; t < nthr; ++t) pool.emplace_back(work, t);
    for (auto& th : pool) th.join();
  }
  for (int s : status)
    if (s) return s;
  return 0;
}

int64_t fmt_packed_bytes(int fmt, int64_t N, int64_t K) {
  switch (fmt) {
    case kFmtQ4K: return N * (K / 256) * 144;
    case kFmtQ5K: return N * (K / 256) * 176;
    case kFmtNVFP4: return N * (K / 256) * 144 + 16;
    case kFmtINT4: return N * (K / 2) + N * (K / 128) * 2;
    case kFmtQ6K: return N * (K / 256) * 208 + N * (K / 256) * 2;
    default: return -1;
  }
}

int64_t fmt_aux_offset(int fmt, int64_t N, int64_t K) {
  if (fmt == kFmtNVFP4) return N * (K / 256) * 144;
  if (fmt == kFmtINT4) return N * (K / 2);
  if (fmt == kFmtQ6K) return N * (K / 256) * 208;
  return 0;
}

int pack_fmt(int fmt, const float* W, int64_t N, int64_t K, uint8_t* out, int threads) {
  if (fmt == kFmtQ4K) return pack_q4k(W, N, K, out, threads);
  const int64_t nb = K / 256;
  for (int64_t e = 0; e < N * K; ++e)
    if (!std::isfinite(W[e])) return 6;
  if (fmt == kFmtQ5K)
    return for_rows(N, threads, [&](int64_t n) {
      for (int64_t b = 0; b < nb; ++b)
        if (!pack_q5k_superblock(W + n * K + b * 256, out + (n * nb + b) * 176)) return false;
      return true;
    });
  if (fmt == kFmtNVFP4) {
    float amax = 0.0f;
    for (int64_t e = 0; e < N * K; ++e) amax = std::max(amax, std::fabs(W[e]));
    float g = amax / 2688.0f;   // 6 x 448: the largest E2M1 value times the largest E4M3 value
    if (!(g > 0.0f)) g = 1.0f;
    const int rc = for_rows(N, threads, [&](int64_t n) {
      for (int64_t b = 0; b < nb; ++b) pack_nvfp4_superblock(W + n * K + b * 256, g, out + (n * nb + b) * 144);
      return true;
    });
    uint8_t* tr = out + fmt_aux_offset(fmt, N, K);
    std::memset(tr, 0, 16);
    uint32_t gb = 0;
    std::memcpy(&gb, &g, 4);
    for (int b = 0; b < 4; ++b) tr[b] = (uint8_t)(gb >> (8 * b));
    return rc;
  }
  if (fmt == kFmtQ6K) {
    uint8_t* dplane = out + fmt_aux_offset(fmt, N, K);
    return for_rows(N, threads, [&](int64_t n) {
      for (int64_t b = 0; b < nb; ++b)
        if (!pack_q6k_superblock(W + n * K + b * 256, out + (n * nb + b) * 208, dplane + (n * nb + b) * 2))
          return false;
      return true;
    });
  }
  if (fmt == kFmtINT4) {
    uint8_t* scales = out + fmt_aux_offset(fmt, N, K);
    return for_rows(N, threads, [&](int64_t n) {
      return pack_int4_row(W + n * K, K, out + n * (K / 2), scales + n * (K / 128) * 2);
    });
  }
  return 2;
}

}  // namespace q4k
