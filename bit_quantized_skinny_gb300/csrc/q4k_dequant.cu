// q4k_dequant.cu — device dequantization of packed weights (test hooks behind qmm_dequant and
// qmm_fmt_dequant).
// One thread per 32-weight sub-block; it decodes the scale fields and the quants with the same
// routines as the product kernels and writes w_t = fma(D*sc_j, q_t, -(Dm*m_j)) in fp32: the
// exact product is rounded once together with the subtraction, which is the format's
// definition of a weight.
#include <cuda_fp16.h>

#include "q4k_device.cuh"
#include "q4k_formats.cuh"
#include "q4k_internal.h"

namespace q4k {
namespace {

__global__ void __launch_bounds__(256) q4k_dequant_kernel(const uint8_t* __restrict__ W, int64_t nsub,
                                                          float* __restrict__ out) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= nsub) return;
  const int64_t blk = s >> 3;
  const int j = (int)(s & 7);
  const uint8_t* b = W + blk * kBlockBytes;
  const uint4 h = ldg_nc_v4(b);
  const uint4 q = ldg_nc_v4(b + 16 + 16 * j);
  const SubScale sc = decode_scales(h, j);
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
  float4* o = reinterpret_cast<float4*>(out + s * 32);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float q8[8];
    nibbles_to_f32(words[w], q8);
    float v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) v[p] = fmaf(sc.dsc, q8[p], -sc.dmm);
    o[2 * w] = make_float4(v[0], v[1], v[2], v[3]);
    o[2 * w + 1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

__device__ __forceinline__ float lo_f(uint32_t h2) { return __low2float(*reinterpret_cast<const __half2*>(&h2)); }
__device__ __forceinline__ float hi_f(uint32_t h2) { return __high2float(*reinterpret_cast<const __half2*>(&h2)); }

// The other formats: one thread per 32 consecutive weights of a row, decoded with the product
// kernel's steps (q4k_formats.cuh) and written as the format's definition of a weight:
//   Q5K   fma(D*sc_j, q, -(Dm*m_j))   (the exact value, rounded once)
//   NVFP4 g * (s_b * v)               (s_b * v exact; one rounding)
//   INT4  s * q                       (exact)
//   Q6K   (d * sc_j) * (q - 32)       (d * sc_j exact; one rounding, here none: 23 bits)
template <int FMT>
__global__ void __launch_bounds__(256) fmt_dequant_kernel(const uint8_t* __restrict__ W, int64_t N, int64_t K,
                                                          float* __restrict__ out) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= N * (K / 32)) return;
  float v[32];
  if constexpr (FMT == kFmtQ5K) {
    const uint8_t* b = W + (s >> 3) * 176;
    const int j = (int)(s & 7);
    const SubScale sc = decode_scales(ldg_nc_v4(b), j);
    const uint32_t H = __ldg(reinterpret_cast<const uint32_t*>(b + 16) + j);
    const uint4 q = ldg_nc_v4(b + 48 + 16 * j);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
    uint32_t p[4][4];
    q5k_magic<0>(words[0], H, p[0]);
    q5k_magic<1>(words[1], H, p[1]);
    q5k_magic<2>(words[2], H, p[2]);
    q5k_magic<3>(words[3], H, p[3]);
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) {
      const float qv[8] = {lo_f(p[ww][0]) - 1024.f, (lo_f(p[ww][1]) - 1024.f) * 0.0625f,
                           lo_f(p[ww][2]) - 1024.f, (lo_f(p[ww][3]) - 1024.f) * 0.0625f,
                           hi_f(p[ww][0]) - 1024.f, (hi_f(p[ww][1]) - 1024.f) * 0.0625f,
                           hi_f(p[ww][2]) - 1024.f, (hi_f(p[ww][3]) - 1024.f) * 0.0625f};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[8 * ww + i] = fmaf(sc.dsc, qv[i], -sc.dmm);
    }
  } else if constexpr (FMT == kFmtQ6K) {
    // weights 32 part .. 32 part + 31 of a super-block: sub-blocks 2 part and 2 part + 1
    const int64_t blk = s >> 3;
    const int part = (int)(s & 7);
    const uint8_t* b = W + blk * 208;
    const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(W + N * (K / 256) * 208) + blk)));
    const uint4 q = ldg_nc_v4(b + 16 + 16 * part);
    const uint2 hh = __ldg(reinterpret_cast<const uint2*>(b + 144) + part);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
    const uint32_t hwords[2] = {hh.x, hh.y};
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) {
      const int sub = 2 * part + (ww >> 1);
      const float dsc = d * (float)((int)(b[sub] & 127) - 64);   // exact: 11 + 7 bits
      uint32_t p[4];
      if (ww & 1) q6k_magic<1>(words[ww], hwords[ww >> 1], p);
      else q6k_magic<0>(words[ww], hwords[ww >> 1], p);
      // (1024 + 16 q) / 16 - 96 = q - 32, exact
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        v[8 * ww + c] = dsc * (lo_f(p[c]) * 0.0625f - 96.f);
        v[8 * ww + c + 4] = dsc * (hi_f(p[c]) * 0.0625f - 96.f);
      }
    }
  } else if constexpr (FMT == kFmtNVFP4) {
    const float g = __ldg(reinterpret_cast<const float*>(W + N * (K / 256) * 144));
    const uint8_t* b = W + (s >> 3) * 144;
    const int part = (int)(s & 7);   // weights 32 part .. 32 part + 31: scale blocks 2 part, 2 part + 1
    const uint32_t sw = __ldg(reinterpret_cast<const uint32_t*>(b) + (part >> 1));
    const uint32_t sp = e4m3x2_pair(sw >> (16 * (part & 1)));
    const float sc[2] = {lo_f(sp), hi_f(sp)};
    const uint4 q = ldg_nc_v4(b + 16 + 16 * part);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) {
      uint32_t p[4];
      e2m1x8_pairs(words[ww], p);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        v[8 * ww + 2 * c] = g * (sc[ww >> 1] * lo_f(p[c]));
        v[8 * ww + 2 * c + 1] = g * (sc[ww >> 1] * hi_f(p[c]));
      }
    }
  } else {
    const int64_t per_row = K / 32;
    const int64_t n = s / per_row, part = s - n * per_row;
    const uint16_t sbits = __ldg(reinterpret_cast<const unsigned short*>(W + N * (K / 2)) + n * (K / 128) + part / 4);
    const float scale = __half2float(__ushort_as_half(sbits));
    const uint4 q = ldg_nc_v4(W + n * (K / 2) + 16 * part);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) {
      uint32_t p[4];
      int4_magic(words[ww], p);
      const float qv[8] = {lo_f(p[0]) - 1032.f, (lo_f(p[1]) - 1024.f) * 0.0625f - 8.f,
                           lo_f(p[2]) - 1032.f, (lo_f(p[3]) - 1024.f) * 0.0625f - 8.f,
                           hi_f(p[0]) - 1032.f, (hi_f(p[1]) - 1024.f) * 0.0625f - 8.f,
                           hi_f(p[2]) - 1032.f, (hi_f(p[3]) - 1024.f) * 0.0625f - 8.f};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[8 * ww + i] = scale * qv[i];
    }
  }
  float4* o = reinterpret_cast<float4*>(out + s * 32);
#pragma unroll
  for (int k = 0; k < 8; ++k) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

}  // namespace

cudaError_t launch_dequant_fmt(int fmt, const void* W, int64_t N, int64_t K, float* out, cudaStream_t stream) {
  if (fmt == kFmtQ4K) return launch_dequant(W, N, K, out, stream);
  const int64_t threads = N * (K / 32);
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const uint8_t* w = static_cast<const uint8_t*>(W);
  if (fmt == kFmtQ5K) fmt_dequant_kernel<kFmtQ5K><<<(unsigned)blocks, 256, 0, stream>>>(w, N, K, out);
  else if (fmt == kFmtNVFP4) fmt_dequant_kernel<kFmtNVFP4><<<(unsigned)blocks, 256, 0, stream>>>(w, N, K, out);
  else if (fmt == kFmtINT4) fmt_dequant_kernel<kFmtINT4><<<(unsigned)blocks, 256, 0, stream>>>(w, N, K, out);
  else if (fmt == kFmtQ6K) fmt_dequant_kernel<kFmtQ6K><<<(unsigned)blocks, 256, 0, stream>>>(w, N, K, out);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_dequant(const void* W, int64_t N, int64_t K, float* out, cudaStream_t stream) {
  const int64_t nsub = N * (K / 256) * 8;
  const int64_t blocks = (nsub + 255) / 256;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  q4k_dequant_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint8_t*>(W), nsub, out);
  return cudaGetLastError();
}

}  // namespace q4k
