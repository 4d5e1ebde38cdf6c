// q4k_internal.h — launch interface between the C-ABI layer (qmm_api.cpp) and the kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime_api.h>

namespace q4k {

// Weight formats (the qmm_format codes of the C ABI).
enum WeightFormat : int { kFmtQ4K = 0, kFmtQ5K = 1, kFmtNVFP4 = 2, kFmtINT4 = 3, kFmtQ6K = 4 };

// One product handed to a kernel: Y[M x N] = X[M x K] * dequant(W)^T.  fmt is the weight
// format; aux points into the packed buffer at what the format keeps outside its row blocks
// (NVFP4: the fp32 tensor scale; INT4: the scale plane; Q6K: the plane of super-block scales;
// otherwise unused).
struct Job {
  const void* W;
  const uint16_t* X;
  float* Y;
  int64_t N;
  int64_t K;
  int fmt = kFmtQ4K;
  const void* aux = nullptr;
  // gated: rows 2f and 2f+1 are the gate and up rows of output f; Y is then the bf16 matrix
  // H[M x N/2] = bf16(silu(gate) * up) instead of the fp32 product (tensor cores, no K split)
  bool gated = false;
};

// Launch the CUDA-core (fma) kernel over `count` jobs sharing M, in one launch.
// Returns a cudaError_t (cudaSuccess when enqueued).
cudaError_t launch_fma(const Job* jobs, int count, int M, cudaStream_t stream);

// Launch the tensor-core (tcgen05) kernel; cudaErrorNotSupported when it cannot run the shape.
cudaError_t launch_tc(const Job* jobs, int count, int M, cudaStream_t stream);
bool tc_supports(int M, int64_t N, int64_t K);
// Modelled duration (us) of a tensor-core launch over these jobs (the dispatcher's cost model).
double tc_estimate_us(const Job* jobs, int count, int M);

// Tensor-core product with the prepared activations in the library's fixed device buffer
// (no allocation).  noalloc_scratch_needed(M, K) must not exceed noalloc_scratch_bytes().
cudaError_t launch_tc_noalloc(const Job& job, int M, cudaStream_t stream);
size_t noalloc_scratch_bytes();
size_t noalloc_scratch_needed(int M, int64_t K);

// The feed-forward step between the gate/up product and the down product: H[M x F] bf16 from
// G[M x 2F] fp32 (gate columns 0..F-1, up columns F..2F-1), H = bf16(silu(gate) * up).
cudaError_t launch_swiglu(const float* G, int64_t F, int M, uint16_t* H, cudaStream_t stream);

// Row maps of the indexed-expert product: for each of the M activation rows, the row it goes to
// (gather) or comes from (scatter) in the gathered blocks.
struct RowMap {
  int row[32];
};
cudaError_t launch_gather_rows(const RowMap& map, int M, const uint16_t* X, int64_t K, uint16_t* Xg,
                               cudaStream_t stream);
cudaError_t launch_scatter_rows(const RowMap& map, int M, const float* Yg, int64_t N, float* Y,
                                cudaStream_t stream);

// Device dequantization test hooks (Q4K; the other formats).
cudaError_t launch_dequant(const void* W, int64_t N, int64_t K, float* out, cudaStream_t stream);
cudaError_t launch_dequant_fmt(int fmt, const void* W, int64_t N, int64_t K, float* out, cudaStream_t stream);

// The tensor-core kernel's per-(device, stream) workspaces: free them all; bytes held now.
cudaError_t release_workspaces();
size_t workspace_bytes_held();

// Failure-detection hook: bound the tensor-core kernel's pipeline waits to `polls` polls of at
// most suspend_ns each (0, 0: the kernel's own bound) in launches made from now on.
void set_wait_limit(uint32_t polls, uint32_t suspend_ns);

// The read-only streaming probe: read `bytes` (a multiple of 16) at buf once; sink holds
// stream_read_grid() words.
cudaError_t launch_stream_read(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t stream);
int stream_read_grid();

// Device status words of the kernel files: read and clear (synchronous; 0 = no error).
// Device-side packer: fp32 W (device) -> Q4K super-blocks (device), the host packer's bytes; a
// super-block with a non-finite weight or an fp16 scale overflow is written as zeros and sets
// bit 1 of the pack status word.
cudaError_t launch_pack_dev(const float* W, int64_t N, int64_t K, void* out, cudaStream_t stream);
cudaError_t read_and_clear_pack_status(unsigned* out);
cudaError_t read_and_clear_fma_status(unsigned* out);
cudaError_t read_and_clear_tc_status(unsigned* out);

// Host packers (qmm_pack.cpp).  Return 0, or 6 on non-finite input / fp16 overflow.
int pack_q4k(const float* W, int64_t N, int64_t K, uint8_t* out, int threads);
int pack_fmt(int fmt, const float* W, int64_t N, int64_t K, uint8_t* out, int threads);
// Bytes of a packed N x K matrix in format fmt, and the offset of its aux part (0: none).
int64_t fmt_packed_bytes(int fmt, int64_t N, int64_t K);
int64_t fmt_aux_offset(int fmt, int64_t N, int64_t K);

}  // namespace q4k
