// qmm_probe.cu — the read-only streaming probe behind qmm_stream_read: the HBM read bandwidth a
// kernel of this GPU reaches when it only reads, the ceiling of the weight stream.  The pages
// check their kernels' GB/s against the memory system's own numbers (FlashRT issue #153, the
// device-to-device bandwidth check and the sustained-read microtest); this is that probe for
// the read side.
//
// Every byte of the buffer is read exactly once, as 16-byte loads that bypass L1 and are
// marked evict-first in L2, in a grid-stride loop over a grid of a few CTAs per SM; the loaded
// words are folded into one XOR per CTA, written to sink[blockIdx.x] so the loads cannot be
// dropped.
#include <cstdint>
#include <cuda_runtime_api.h>

#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {
namespace {

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads) stream_read_kernel(const uint4* __restrict__ src, size_t n16,
                                                                    uint32_t* __restrict__ sink) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  uint32_t acc = 0;
  const size_t stride = (size_t)gridDim.x * kProbeThreads;
  size_t i = (size_t)blockIdx.x * kProbeThreads + threadIdx.x;
  // four independent 16-byte loads in flight per thread and iteration
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                   : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                   : "l"(src + i + u * stride), "l"(pol));
#pragma unroll
    for (int u = 0; u < 4; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ldg_nc_v4(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  __shared__ uint32_t part[kProbeThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = 0;
    for (int w = 0; w < kProbeThreads / 32; ++w) a ^= part[w];
    sink[blockIdx.x] = a;
  }
}

}  // namespace

int stream_read_grid() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return 4 * sms;
}

cudaError_t launch_stream_read(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t stream) {
  const int grid = stream_read_grid();
  if (grid <= 0) return cudaErrorInvalidDevice;
  stream_read_kernel<<<grid, kProbeThreads, 0, stream>>>(static_cast<const uint4*>(buf), bytes / 16, sink);
  return cudaGetLastError();
}

}  // namespace q4k
