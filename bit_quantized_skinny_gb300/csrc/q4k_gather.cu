// q4k_gather.cu — row gather and scatter around the indexed-expert product (qmm_run_indexed):
// each activation row i of X is multiplied by the weight matrix of expert ids[i].  The rows of
// each expert are gathered into a contiguous block (the products then run as one batched
// launch over the experts in use) and the results are scattered back to their rows.
#include <cstdint>
#include <cuda_runtime.h>

#include "q4k_internal.h"

namespace q4k {
namespace {

// Row i of X (K bf16) -> row dst[i] of the gathered block.  One CTA per row.
__global__ void __launch_bounds__(256) gather_rows_kernel(const __grid_constant__ RowMap map, const uint16_t* __restrict__ X,
                                                          int64_t K, uint16_t* __restrict__ Xg) {
  const int i = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(X + (int64_t)i * K);
  uint4* dst = reinterpret_cast<uint4*>(Xg + (int64_t)map.row[i] * K);
  for (int64_t v = threadIdx.x; v < K / 8; v += blockDim.x) dst[v] = src[v];
}

// Row src[i] of the gathered results (N fp32) -> row i of Y.  One CTA per row.
__global__ void __launch_bounds__(256) scatter_rows_kernel(const __grid_constant__ RowMap map, const float* __restrict__ Yg,
                                                           int64_t N, float* __restrict__ Y) {
  const int i = blockIdx.x;
  const float* src = Yg + (int64_t)map.row[i] * N;
  float* dst = Y + (int64_t)i * N;
  for (int64_t v = threadIdx.x; v < N; v += blockDim.x) dst[v] = src[v];
}

}  // namespace

cudaError_t launch_gather_rows(const RowMap& map, int M, const uint16_t* X, int64_t K, uint16_t* Xg,
                               cudaStream_t stream) {
  gather_rows_kernel<<<M, 256, 0, stream>>>(map, X, K, Xg);
  return cudaGetLastError();
}

cudaError_t launch_scatter_rows(const RowMap& map, int M, const float* Yg, int64_t N, float* Y,
                                cudaStream_t stream) {
  scatter_rows_kernel<<<M, 256, 0, stream>>>(map, Yg, N, Y);
  return cudaGetLastError();
}

}  // namespace q4k
