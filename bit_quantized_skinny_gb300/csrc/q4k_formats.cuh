// q4k_formats.cuh — decode steps of the weight formats other than Q4K, shared by the
// tensor-core product kernel and the device dequantization hook.
//
// Each step turns one 32-bit word of a row's packed quants (8 weights) into four fp16 pairs.
// The k-quant and integer formats use the magic-number trick of the Q4K decode: a 4-bit field
// OR-ed into the mantissa of 1024.0 (0x6400) is 1024 + field exactly, and a field at bits 4..7
// gives 1024 + 16 * field; a fused multiply-add then removes the offset and applies the scale.
// Pairs come out as (weight c, weight c + 4) of the word, c = 0..3 -- the order the activations
// of those formats are laid out in.  NVFP4 uses the hardware E2M1 conversion, whose pairs are
// (weight 2c, weight 2c + 1): the natural order.
#pragma once
#include <cstdint>

namespace q4k {

// Q5K: word w of sub-block quants (weights 8ww .. 8ww+7 of the sub-block) and the high-bit word
// H of the sub-block (bit 4i + ww is the high bit of weight i of word ww).  Returns
//   p[0] = (1024 + q0, 1024 + q4)          p[1] = (1024 + 16 q1, 1024 + 16 q5)
//   p[2] = (1024 + q2, 1024 + q6)          p[3] = (1024 + 16 q3, 1024 + 16 q7)
// with q the 5-bit quants (each at most 1024 + 496 < 2048: exact in fp16).  With MAGIC = 0 the
// exponent field stays 0 and the pairs are the fp16 subnormals (q 2^-24, 16 q 2^-24).
template <int WW, uint32_t MAGIC = 0x64006400u>
__device__ __forceinline__ void q5k_magic(uint32_t w, uint32_t H, uint32_t (&p)[4]) {
  const uint32_t hl = H << (4 - WW);   // high bits of weights 0, 4 at bits 4, 20; of 1, 5 at 8, 24
  const uint32_t hr = H >> (4 + WW);   // of weights 2, 6 at bits 4, 20; of 3, 7 at 8, 24
  const uint32_t b8 = w >> 8;
  uint32_t u0, u1, u2, u3;
  asm("lop3.b32 %0, %1, 0x00100010, %2, 0xEA;" : "=r"(u0) : "r"(hl), "n"(MAGIC));
  asm("lop3.b32 %0, %1, 0x01000100, %2, 0xEA;" : "=r"(u1) : "r"(hl), "n"(MAGIC));
  asm("lop3.b32 %0, %1, 0x00100010, %2, 0xEA;" : "=r"(u2) : "r"(hr), "n"(MAGIC));
  asm("lop3.b32 %0, %1, 0x01000100, %2, 0xEA;" : "=r"(u3) : "r"(hr), "n"(MAGIC));
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(p[0]) : "r"(w), "r"(u0));
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;" : "=r"(p[1]) : "r"(w), "r"(u1));
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(p[2]) : "r"(b8), "r"(u2));
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;" : "=r"(p[3]) : "r"(b8), "r"(u3));
}

// Q6K: word w of low nibbles (weights 8a .. 8a+7 of a 16-weight sub-block, A = a) and the
// sub-block's high-part word H (weight i of word a at bits 8a + 16 (i >= 4) + 2 (i % 4)).  The
// 6-bit quants go to mantissa bits 4..9 (nibble at 4..7, high part at 8..9), so
//   p[c] = (1024 + 16 q_c, 1024 + 16 q_{c+4}),  c = 0..3   (at most 1024 + 1008: exact).
template <int A>
__device__ __forceinline__ void q6k_magic(uint32_t w, uint32_t H, uint32_t (&p)[4]) {
  const uint32_t h = H >> (8 * A);
  uint32_t u0, u1, u2, u3;
  asm("lop3.b32 %0, %1, 0x03000300, 0x64006400, 0xEA;" : "=r"(u0) : "r"(h << 8));   // high parts of 0, 4
  asm("lop3.b32 %0, %1, 0x03000300, 0x64006400, 0xEA;" : "=r"(u1) : "r"(h << 6));   // of 1, 5
  asm("lop3.b32 %0, %1, 0x03000300, 0x64006400, 0xEA;" : "=r"(u2) : "r"(h << 4));   // of 2, 6
  asm("lop3.b32 %0, %1, 0x03000300, 0x64006400, 0xEA;" : "=r"(u3) : "r"(h << 2));   // of 3, 7
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;" : "=r"(p[0]) : "r"(w << 4), "r"(u0));
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;" : "=r"(p[1]) : "r"(w), "r"(u1));
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;" : "=r"(p[2]) : "r"(w >> 4), "r"(u2));
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;" : "=r"(p[3]) : "r"(w >> 8), "r"(u3));
}

// INT4: word w of two's-complement 4-bit quants.  Flipping bit 3 of a field gives q + 8; one
// 3-input logic op per pair takes the field, flips its top bit and ORs in the exponent of 1024
// (lookup table 0x6A: b ? a ^ c : c, with b the field mask and c the magic plus the flipped bit).
//   p[0] = (1024 + q0 + 8, 1024 + q4 + 8)           p[1] = (1024 + 16 (q1 + 8), ...)
//   p[2] = (1024 + q2 + 8, 1024 + q6 + 8)           p[3] = (1024 + 16 (q3 + 8), ...)
__device__ __forceinline__ void int4_magic(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t b8 = w >> 8;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64086408, 0x6A;" : "=r"(p[0]) : "r"(w));
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64806480, 0x6A;" : "=r"(p[1]) : "r"(w));
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64086408, 0x6A;" : "=r"(p[2]) : "r"(b8));
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64806480, 0x6A;" : "=r"(p[3]) : "r"(b8));
}

// NVFP4: the eight E2M1 codes of w (low nibble first) as fp16 pairs (v_2c, v_2c+1), exact.
__device__ __forceinline__ void e2m1x8_pairs(uint32_t w, uint32_t (&p)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3]) : "r"(w));
}

// Two E4M3 codes (bits 0..7 and 8..15 of v) as an fp16 pair, exact.
__device__ __forceinline__ uint32_t e4m3x2_pair(uint32_t v) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n}" : "=r"(r) : "r"(v));
  return r;
}

}  // namespace q4k
