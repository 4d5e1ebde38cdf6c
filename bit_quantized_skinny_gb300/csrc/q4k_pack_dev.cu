// q4k_pack_dev.cu — device-side packer: fp32 weights in device memory -> Q4K super-blocks in
// device memory, byte for byte what the host packer (qmm_pack) writes.
//
// The quantizer is the one include/qmm.h states (the pages give none): per 32-weight sub-block
// the range [min(0, min w), max w] in 15 steps, the per-sub-block step and offset quantized to
// 6 bits against fp16 super-block scales, each weight to the nearest of 16 levels.  Every step
// is the same IEEE fp32 operation as on the host (round to nearest even; divisions are IEEE
// divisions, no contraction: the library is built with --fmad=false), so the bytes agree.
//
// Work: 8 threads per super-block, thread j owning sub-block j (32 weights, 128 contiguous
// bytes of the row); the 8 threads of a super-block are 8 neighbouring lanes of a warp.  The
// super-block maxima and the 96-bit field of 12-bit (sc, m) groups are formed with shuffles.
// A super-block with a non-finite weight, or whose scales overflow binary16, is written as
// zeros and sets bit 1 of this file's status word (the host packer rejects the whole matrix).
#include <cuda_fp16.h>
#include <cstdint>

#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {
namespace {

__device__ unsigned g_status;   // this file's kernels' status word

constexpr int kPackThreads = 256;   // 32 super-blocks per CTA
constexpr unsigned kErrPackNonfinite = 2u;

// rint with the clamp of the host's level(): r < 0 -> 0, r > hi -> hi.
__device__ __forceinline__ uint32_t level(float v, float hi) {
  const float r = rintf(v);
  return (uint32_t)(r < 0.0f ? 0.0f : (r > hi ? hi : r));
}

__global__ void __launch_bounds__(kPackThreads) q4k_pack_kernel(const float* __restrict__ W, int64_t N, int64_t K,
                                                                 uint8_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int j = lane & 7;                       // sub-block of this thread
  const unsigned grp = 0xFFu << (lane & 24);    // the 8 lanes of this super-block
  const int64_t nb = K / 256;
  const int64_t blk = (int64_t)blockIdx.x * (kPackThreads / 8) + (threadIdx.x >> 3);
  const bool live = blk < N * nb;
  const int64_t n = live ? blk / nb : 0, b = live ? blk - n * nb : 0;

  float w[32];
  if (live) {
    const float4* src = reinterpret_cast<const float4*>(W + n * K + b * 256 + 32 * j);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 f = __ldg(src + v);
      w[4 * v] = f.x; w[4 * v + 1] = f.y; w[4 * v + 2] = f.z; w[4 * v + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t) w[t] = 0.0f;
  }
  bool bad = false;
  float mn = 0.0f, mx = w[0];
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    bad = bad || !isfinite(w[t]);
    mn = (w[t] < mn) ? w[t] : mn;
    mx = (w[t] > mx) ? w[t] : mx;
  }
  const float step_raw = (mx - mn) / 15.0f;
  const float offset_raw = 0.0f - mn;
  // super-block maxima, from +0 as on the host: every value here is +-0 or positive, so the
  // order does not matter, and a zero maximum is +0
  float step_max = step_raw, offset_max = offset_raw;
#pragma unroll
  for (int s = 1; s < 8; s <<= 1) {
    step_max = fmaxf(step_max, __shfl_xor_sync(0xffffffffu, step_max, s));
    offset_max = fmaxf(offset_max, __shfl_xor_sync(0xffffffffu, offset_max, s));
  }
  step_max = step_max > 0.0f ? step_max : 0.0f;
  offset_max = offset_max > 0.0f ? offset_max : 0.0f;
  const __half dh = __float2half_rn(step_max / 63.0f);
  const __half mh = __float2half_rn(offset_max / 63.0f);
  const float D = __half2float(dh), Dm = __half2float(mh);
  bad = bad || isinf(D) || isinf(Dm);
  bad = (__ballot_sync(0xffffffffu, bad) & grp) != 0u;   // the whole super-block

  const uint32_t sc = (D > 0.0f) ? level(step_raw / D, 63.0f) : 0u;
  const uint32_t m = (Dm > 0.0f) ? level(offset_raw / Dm, 63.0f) : 0u;
  const float step = D * (float)sc;
  const float off = Dm * (float)m;
  uint32_t q[4] = {0u, 0u, 0u, 0u};   // weight t of the sub-block at bits 4 (t % 8) of word t / 8
  if (step > 0.0f) {
#pragma unroll
    for (int t = 0; t < 32; ++t) q[t >> 3] |= level((w[t] + off) / step, 15.0f) << (4 * (t & 7));
  }
  // the 12-bit groups of the 8 sub-blocks at bit 12 j of the 96-bit field
  const uint32_t g = sc | (m << 6);
  uint32_t f[3] = {0u, 0u, 0u};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t gk = __shfl_sync(0xffffffffu, g, (lane & 24) | k);
    const int bit = 12 * k;
    f[bit >> 5] |= gk << (bit & 31);
    if ((bit & 31) > 20) f[(bit >> 5) + 1] |= gk >> (32 - (bit & 31));
  }
  if (!live) return;
  uint8_t* o = out + blk * 144;
  if (bad) {
    if (j == 0) atomicOr(&g_status, kErrPackNonfinite);
    *reinterpret_cast<uint4*>(o + 16 + 16 * j) = make_uint4(0u, 0u, 0u, 0u);
    if (j == 0) *reinterpret_cast<uint4*>(o) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  *reinterpret_cast<uint4*>(o + 16 + 16 * j) = make_uint4(q[0], q[1], q[2], q[3]);
  if (j == 0) {
    const uint32_t hd = (uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(mh) << 16);
    *reinterpret_cast<uint4*>(o) = make_uint4(hd, f[0], f[1], f[2]);
  }
}

}  // namespace

cudaError_t launch_pack_dev(const float* W, int64_t N, int64_t K, void* out, cudaStream_t stream) {
  const int64_t blocks = N * (K / 256);
  const int64_t grid = (blocks + kPackThreads / 8 - 1) / (kPackThreads / 8);
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  q4k_pack_kernel<<<(unsigned)grid, kPackThreads, 0, stream>>>(W, N, K, static_cast<uint8_t*>(out));
  return cudaGetLastError();
}

cudaError_t read_and_clear_pack_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  *out = v;
  return e;
}

}  // namespace q4k
