// q4k_ffn.cu — the step between the two products of one feed-forward block of the verify pass
// (the fused gate/up matrix and the down matrix of the configurations; the pages time them as
// "gate+up" and lm_head in FlashRT issue #153, the tile-bench tables): from the gate/up product
// G[M x 2F] (fp32; columns 0..F-1 gate, F..2F-1 up) to the activations of the down product,
//     H[i][f] = bf16( silu(G[i][f]) * G[i][F + f] ),   silu(g) = g / (1 + e^-g),
// computed in fp32 and rounded once to bf16 (round to nearest even).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "q4k_internal.h"

namespace q4k {
namespace {

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}

// One thread per 4 consecutive columns f of one row i (F % 4 == 0).
__global__ void __launch_bounds__(256) swiglu_bf16_kernel(const float* __restrict__ G, int64_t F, int M,
                                                          uint16_t* __restrict__ H) {
  const int64_t per_row = F / 4;
  const int64_t total = per_row * M;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = v / per_row;
    const int64_t f = (v - i * per_row) * 4;
    const float4 g = *reinterpret_cast<const float4*>(G + i * 2 * F + f);
    const float4 u = *reinterpret_cast<const float4*>(G + i * 2 * F + F + f);
    const uint32_t h0 = bf16_bits(silu(g.x) * u.x), h1 = bf16_bits(silu(g.y) * u.y);
    const uint32_t h2 = bf16_bits(silu(g.z) * u.z), h3 = bf16_bits(silu(g.w) * u.w);
    *reinterpret_cast<uint2*>(H + i * F + f) = make_uint2(h0 | (h1 << 16), h2 | (h3 << 16));
  }
}

}  // namespace

cudaError_t launch_swiglu(const float* G, int64_t F, int M, uint16_t* H, cudaStream_t stream) {
  const int64_t total = F / 4 * M;
  const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  swiglu_bf16_kernel<<<blocks, 256, 0, stream>>>(G, F, M, H);
  return cudaGetLastError();
}

}  // namespace q4k
