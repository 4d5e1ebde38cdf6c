// q4k_dequant.cu — device dequantization of packed Q4K weights (test hook behind qmm_dequant).
// One thread per 32-weight sub-block; it decodes the scale fields and the quants with the same
// routines as the product kernels and writes w_t = fma(D*sc_j, q_t, -(Dm*m_j)) in fp32: the
// exact product is rounded once together with the subtraction, which is the format's
// definition of a weight.
#include "q4k_device.cuh"
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

}  // namespace

cudaError_t launch_dequant(const void* W, int64_t N, int64_t K, float* out, cudaStream_t stream) {
  const int64_t nsub = N * (K / 256) * 8;
  const int64_t blocks = (nsub + 255) / 256;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  q4k_dequant_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint8_t*>(W), nsub, out);
  return cudaGetLastError();
}

}  // namespace q4k
