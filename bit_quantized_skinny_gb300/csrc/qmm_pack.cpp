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

}  // namespace q4k
