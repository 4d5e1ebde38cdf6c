// qmm_api.cpp — the C ABI (include/qmm.h): argument validation, variant dispatch, launches.
//
// Dispatch follows the pages' "switch point" idea ("sixi-asi 0.9", section "The patch": the
// row count at which the skinny product moves from one kernel family to another, tuned per
// GPU).  Here the families are the CUDA-core kernel (q4k_fma.cu) and the tensor-core kernel;
// the switch point below is the measured one for GB300.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda_runtime_api.h>

#include "../../include/qmm.h"
#include "q4k_internal.h"

namespace {

thread_local char g_last_cuda_error[256] = "no error";

qmm_status cuda_fail(cudaError_t e) {
  const char* s = cudaGetErrorString(e);
  std::strncpy(g_last_cuda_error, s ? s : "unknown CUDA error", sizeof(g_last_cuda_error) - 1);
  g_last_cuda_error[sizeof(g_last_cuda_error) - 1] = 0;
  return QMM_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qmm_status check_shape(int64_t N, int64_t K) {
  if (N < 1 || N >= (int64_t(1) << 31)) return QMM_ERR_SHAPE;
  if (K < 256 || K > (int64_t(1) << 20) || K % 256 != 0) return QMM_ERR_SHAPE;
  return QMM_OK;
}

bool valid_format(int fmt) { return fmt >= QMM_FMT_Q4K && fmt <= QMM_FMT_Q6K; }

qmm_status check_job(const void* W, int64_t N, int64_t K, const uint16_t* X, const float* Y) {
  if (!W || !X || !Y) return QMM_ERR_NULL;
  qmm_status s = check_shape(N, K);
  if (s != QMM_OK) return s;
  if (!aligned(W, 16) || !aligned(X, 16) || !aligned(Y, 4)) return QMM_ERR_ALIGN;
  return QMM_OK;
}

// Switch point between the two kernel families, measured on GB300 (the pages tune the same
// kind of switch point per GPU: "sixi-asi 0.9", section "The patch").  Each family gets a
// small cost model fitted to its measured timings; the cheaper one runs.
//   CUDA cores: ceil(M / rows-per-pass) passes, each streaming all weights at ~2.4 TB/s
//               (1 activation row per pass) or ~1.8 TB/s (2 rows per pass) and taking at
//               least ~2.5 us, plus ~5 us.
//   tensor cores: q4k::tc_estimate_us (fixed cost, per-SM super-blocks, split tasks).
struct CostModel {
  double fma_us = 0, tc_us = 0;
};

CostModel model(const q4k::Job* jobs, int count, int M) {
  CostModel c;
  double bytes = 0;
  for (int k = 0; k < count; ++k) bytes += (double)jobs[k].N * (double)(jobs[k].K / 256) * 144.0;
  const double passes = (M == 1) ? 1.0 : std::ceil(M / 2.0);
  const double bw = (M == 1) ? 2.4e6 : 1.8e6;   // bytes per microsecond
  c.fma_us = 5.0 + passes * std::max(2.5, bytes / bw);
  c.tc_us = q4k::tc_estimate_us(jobs, count, M);
  return c;
}

// QMM_FORCE_VARIANT=fma|tc (read once): every automatic choice takes that family instead of
// the cost model's (for tests and benchmarks; any other value is ignored).
int forced_variant() {
  static const int v = [] {
    const char* e = std::getenv("QMM_FORCE_VARIANT");
    if (!e) return QMM_VARIANT_AUTO;
    if (std::strcmp(e, "fma") == 0) return QMM_VARIANT_FMA;
    if (std::strcmp(e, "tc") == 0) return QMM_VARIANT_TC;
    return QMM_VARIANT_AUTO;
  }();
  return v;
}

int select_variant_jobs(const q4k::Job* jobs, int count, int M) {
  for (int k = 0; k < count; ++k)
    if (!q4k::tc_supports(M, jobs[k].N, jobs[k].K)) return QMM_VARIANT_FMA;
  if (forced_variant() != QMM_VARIANT_AUTO) return forced_variant();
  const CostModel c = model(jobs, count, M);
  return (c.tc_us < c.fma_us) ? QMM_VARIANT_TC : QMM_VARIANT_FMA;
}

int select_variant(int M, int64_t N, int64_t K) {
  const q4k::Job job{nullptr, nullptr, nullptr, N, K};
  return select_variant_jobs(&job, 1, M);
}

qmm_status run_jobs(const q4k::Job* jobs, int count, int M, int variant, cudaStream_t stream) {
  if (variant == QMM_VARIANT_AUTO) variant = select_variant_jobs(jobs, count, M);
  cudaError_t e;
  if (variant == QMM_VARIANT_FMA) {
    e = q4k::launch_fma(jobs, count, M, stream);
  } else if (variant == QMM_VARIANT_TC) {
    for (int k = 0; k < count; ++k)
      if (!q4k::tc_supports(M, jobs[k].N, jobs[k].K)) return QMM_ERR_VARIANT;
    e = q4k::launch_tc(jobs, count, M, stream);
  } else {
    return QMM_ERR_VARIANT;
  }
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

size_t qmm_packed_bytes(int64_t N, int64_t K) {
  if (check_shape(N, K) != QMM_OK) return 0;
  return (size_t)N * (size_t)(K / 256) * QMM_BLOCK_BYTES;
}

qmm_status qmm_pack(const float* W_host, int64_t N, int64_t K, void* out_host, size_t out_bytes,
                    int threads) {
  if (!W_host || !out_host) return QMM_ERR_NULL;
  qmm_status s = check_shape(N, K);
  if (s != QMM_OK) return s;
  if (out_bytes < qmm_packed_bytes(N, K)) return QMM_ERR_BUFSIZE;
  const int rc = q4k::pack_q4k(W_host, N, K, static_cast<uint8_t*>(out_host), threads);
  return rc == 0 ? QMM_OK : QMM_ERR_NONFINITE;
}

qmm_status qmm_pack_dev(const float* W_dev, int64_t N, int64_t K, void* out_dev, size_t out_bytes,
                        cudaStream_t stream) {
  if (!W_dev || !out_dev) return QMM_ERR_NULL;
  qmm_status s = check_shape(N, K);
  if (s != QMM_OK) return s;
  if (out_bytes < qmm_packed_bytes(N, K)) return QMM_ERR_BUFSIZE;
  if (!aligned(W_dev, 16) || !aligned(out_dev, 16)) return QMM_ERR_ALIGN;
  const cudaError_t e = q4k::launch_pack_dev(W_dev, N, K, out_dev, stream);
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

qmm_status qmm_run_variant(const void* Wq_dev, int64_t N, int64_t K, const uint16_t* X_dev,
                           float* Y_dev, int M, int variant, cudaStream_t stream) {
  qmm_status s = check_job(Wq_dev, N, K, X_dev, Y_dev);
  if (s != QMM_OK) return s;
  if (M < 1 || M > QMM_MAX_M) return QMM_ERR_M_RANGE;
  const q4k::Job job{Wq_dev, X_dev, Y_dev, N, K};
  return run_jobs(&job, 1, M, variant, stream);
}

qmm_status qmm_run(const void* Wq_dev, int64_t N, int64_t K, const uint16_t* X_dev, float* Y_dev,
                   int M, cudaStream_t stream) {
  return qmm_run_variant(Wq_dev, N, K, X_dev, Y_dev, M, QMM_VARIANT_AUTO, stream);
}

qmm_status qmm_run_batched(const qmm_entry* entries_host, int count, int M, cudaStream_t stream) {
  if (!entries_host) return QMM_ERR_NULL;
  if (count < 1 || count > QMM_MAX_BATCH) return QMM_ERR_COUNT;
  if (M < 1 || M > QMM_MAX_M) return QMM_ERR_M_RANGE;
  q4k::Job jobs[QMM_MAX_BATCH];
  for (int k = 0; k < count; ++k) {
    const qmm_entry& e = entries_host[k];
    qmm_status s = check_job(e.Wq, e.N, e.K, e.X, e.Y);
    if (s != QMM_OK) return s;
    jobs[k] = q4k::Job{e.Wq, e.X, e.Y, e.N, e.K};
  }
  return run_jobs(jobs, count, M, QMM_VARIANT_AUTO, stream);
}

qmm_status qmm_run_noalloc(const void* Wq_dev, int64_t N, int64_t K, const uint16_t* X_dev, float* Y_dev,
                           int M, cudaStream_t stream) {
  qmm_status s = check_job(Wq_dev, N, K, X_dev, Y_dev);
  if (s != QMM_OK) return s;
  if (M < 1 || M > QMM_MAX_M) return QMM_ERR_M_RANGE;
  if (q4k::noalloc_scratch_needed(M, K) > q4k::noalloc_scratch_bytes()) return QMM_ERR_SCRATCH;
  const q4k::Job job{Wq_dev, X_dev, Y_dev, N, K};
  cudaError_t e = q4k::launch_tc_noalloc(job, M, stream);
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

size_t qmm_ffn_workspace_bytes(int M, int64_t F) {
  if (M < 1 || M > QMM_MAX_M || check_shape(1, F) != QMM_OK) return 0;
  const size_t g = ((size_t)M * 2 * (size_t)F * sizeof(float) + 15) & ~(size_t)15;
  return g + (size_t)M * (size_t)F * sizeof(uint16_t);
}

qmm_status qmm_run_ffn(const void* Wgu_dev, const void* Wdown_dev, int64_t F, int64_t K, const uint16_t* X_dev,
                       float* Y_dev, int M, void* workspace_dev, size_t workspace_bytes, cudaStream_t stream) {
  if (!workspace_dev) return QMM_ERR_NULL;
  qmm_status s = check_job(Wgu_dev, 2 * F, K, X_dev, Y_dev);
  if (s != QMM_OK) return s;
  s = check_job(Wdown_dev, K, F, X_dev, Y_dev);   // the down product: K outputs over F inputs
  if (s != QMM_OK) return s;
  if (M < 1 || M > QMM_MAX_M) return QMM_ERR_M_RANGE;
  if (!aligned(workspace_dev, 16)) return QMM_ERR_ALIGN;
  if (workspace_bytes < qmm_ffn_workspace_bytes(M, F)) return QMM_ERR_BUFSIZE;
  float* G = static_cast<float*>(workspace_dev);
  uint16_t* H = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace_dev) +
                                            (((size_t)M * 2 * (size_t)F * sizeof(float) + 15) & ~(size_t)15));
  const q4k::Job gate_up{Wgu_dev, X_dev, G, 2 * F, K};
  s = run_jobs(&gate_up, 1, M, QMM_VARIANT_AUTO, stream);
  if (s != QMM_OK) return s;
  cudaError_t e = q4k::launch_swiglu(G, F, M, H, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  const q4k::Job down{Wdown_dev, H, Y_dev, K, F};
  return run_jobs(&down, 1, M, QMM_VARIANT_AUTO, stream);
}

size_t qmm_ffn_fused_workspace_bytes(int M, int64_t F) {
  if (M < 1 || M > QMM_MAX_M || check_shape(1, F) != QMM_OK) return 0;
  return ((size_t)M * (size_t)F * sizeof(uint16_t) + 15) & ~(size_t)15;
}

qmm_status qmm_run_ffn_fused(const void* Wgu_dev, const void* Wdown_dev, int64_t F, int64_t K, const uint16_t* X_dev,
                             float* Y_dev, int M, void* workspace_dev, size_t workspace_bytes, cudaStream_t stream) {
  if (!workspace_dev) return QMM_ERR_NULL;
  qmm_status s = check_job(Wgu_dev, 2 * F, K, X_dev, Y_dev);
  if (s != QMM_OK) return s;
  s = check_job(Wdown_dev, K, F, X_dev, Y_dev);
  if (s != QMM_OK) return s;
  if (M < 1 || M > QMM_MAX_M) return QMM_ERR_M_RANGE;
  if (!aligned(workspace_dev, 16)) return QMM_ERR_ALIGN;
  if (workspace_bytes < qmm_ffn_fused_workspace_bytes(M, F)) return QMM_ERR_BUFSIZE;
  uint16_t* H = static_cast<uint16_t*>(workspace_dev);
  q4k::Job gate_up{Wgu_dev, X_dev, reinterpret_cast<float*>(H), 2 * F, K};
  gate_up.gated = true;
  cudaError_t e = q4k::launch_tc(&gate_up, 1, M, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  const q4k::Job down{Wdown_dev, H, Y_dev, K, F};
  return run_jobs(&down, 1, M, QMM_VARIANT_AUTO, stream);
}

// Indexed-expert product.  Workspace: the gathered activation rows (M rows, then M rows of
// zeros that the last expert's block may read past its own rows) and the gathered results
// (used experts x rows of the largest expert; at most (M+1)^2/4 blocks of rows).
size_t indexed_x_bytes(int M, int64_t K) { return ((size_t)2 * M * (size_t)K * sizeof(uint16_t) + 15) & ~(size_t)15; }
size_t indexed_y_rows(int M) { return (size_t)(M + 1) * (M + 1) / 4 + 1; }

size_t qmm_indexed_workspace_bytes(int M, int64_t N, int64_t K) {
  if (M < 1 || M > QMM_MAX_M || check_shape(N, K) != QMM_OK) return 0;
  return indexed_x_bytes(M, K) + indexed_y_rows(M) * (size_t)N * sizeof(float);
}

qmm_status qmm_run_indexed(const void* const* experts_host, int n_experts, int64_t N, int64_t K,
                           const int32_t* ids_host, const uint16_t* X_dev, float* Y_dev, int M,
                           void* workspace_dev, size_t workspace_bytes, cudaStream_t stream) {
  if (!experts_host || !ids_host || !workspace_dev) return QMM_ERR_NULL;
  if (n_experts < 1 || n_experts > QMM_MAX_BATCH) return QMM_ERR_COUNT;
  if (M < 1 || M > QMM_MAX_M) return QMM_ERR_M_RANGE;
  for (int e = 0; e < n_experts; ++e) {
    qmm_status s = check_job(experts_host[e], N, K, X_dev, Y_dev);
    if (s != QMM_OK) return s;
  }
  if (!aligned(workspace_dev, 16)) return QMM_ERR_ALIGN;
  if (workspace_bytes < qmm_indexed_workspace_bytes(M, N, K)) return QMM_ERR_BUFSIZE;
  int count[QMM_MAX_BATCH] = {};
  for (int i = 0; i < M; ++i) {
    if (ids_host[i] < 0 || ids_host[i] >= n_experts) return QMM_ERR_SHAPE;
    ++count[ids_host[i]];
  }
  // experts in use, in order of expert index; their rows gathered in order of i
  int slot[QMM_MAX_BATCH], first[QMM_MAX_BATCH];
  int used = 0, rows = 0, mmax = 0;
  for (int e = 0; e < n_experts; ++e) {
    if (!count[e]) continue;
    slot[e] = used++;
    first[e] = rows;
    rows += count[e];
    mmax = count[e] > mmax ? count[e] : mmax;
  }
  if (used == 1) {   // every row goes to the same expert: X and Y are already its gathered blocks
    const q4k::Job job{experts_host[ids_host[0]], X_dev, Y_dev, N, K};
    return run_jobs(&job, 1, M, QMM_VARIANT_AUTO, stream);
  }
  uint16_t* Xg = static_cast<uint16_t*>(workspace_dev);
  float* Yg = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace_dev) + indexed_x_bytes(M, K));
  q4k::RowMap gather{}, scatter{};
  int seen[QMM_MAX_BATCH] = {};
  for (int i = 0; i < M; ++i) {
    const int e = ids_host[i];
    gather.row[i] = first[e] + seen[e];
    scatter.row[i] = slot[e] * mmax + seen[e];
    ++seen[e];
  }
  q4k::Job jobs[QMM_MAX_BATCH];
  for (int e = 0; e < n_experts; ++e)
    if (count[e])
      jobs[slot[e]] = q4k::Job{experts_host[e], Xg + (size_t)first[e] * K, Yg + (size_t)slot[e] * mmax * N, N, K};
  cudaError_t err = cudaMemsetAsync(Xg + (size_t)rows * K, 0, (size_t)mmax * K * sizeof(uint16_t), stream);
  if (err == cudaSuccess) err = q4k::launch_gather_rows(gather, M, X_dev, K, Xg, stream);
  if (err != cudaSuccess) return cuda_fail(err);
  qmm_status s = run_jobs(jobs, used, mmax, QMM_VARIANT_AUTO, stream);
  if (s != QMM_OK) return s;
  err = q4k::launch_scatter_rows(scatter, M, Yg, N, Y_dev, stream);
  return err == cudaSuccess ? QMM_OK : cuda_fail(err);
}

qmm_status qmm_dequant(const void* Wq_dev, int64_t N, int64_t K, float* out_dev, cudaStream_t stream) {
  if (!Wq_dev || !out_dev) return QMM_ERR_NULL;
  qmm_status s = check_shape(N, K);
  if (s != QMM_OK) return s;
  if (!aligned(Wq_dev, 16) || !aligned(out_dev, 16)) return QMM_ERR_ALIGN;
  cudaError_t e = q4k::launch_dequant(Wq_dev, N, K, out_dev, stream);
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

size_t qmm_fmt_packed_bytes(int fmt, int64_t N, int64_t K) {
  if (check_shape(N, K) != QMM_OK) return 0;
  const int64_t b = q4k::fmt_packed_bytes(fmt, N, K);
  return b < 0 ? 0 : (size_t)b;
}

qmm_status qmm_fmt_pack(int fmt, const float* W_host, int64_t N, int64_t K, void* out_host, size_t out_bytes,
                        int threads) {
  if (!valid_format(fmt)) return QMM_ERR_FORMAT;
  if (!W_host || !out_host) return QMM_ERR_NULL;
  qmm_status s = check_shape(N, K);
  if (s != QMM_OK) return s;
  if (out_bytes < qmm_fmt_packed_bytes(fmt, N, K)) return QMM_ERR_BUFSIZE;
  const int rc = q4k::pack_fmt(fmt, W_host, N, K, static_cast<uint8_t*>(out_host), threads);
  return rc == 0 ? QMM_OK : QMM_ERR_NONFINITE;
}

qmm_status qmm_fmt_run(int fmt, const void* Wq_dev, int64_t N, int64_t K, const uint16_t* X_dev, float* Y_dev,
                       int M, cudaStream_t stream) {
  if (!valid_format(fmt)) return QMM_ERR_FORMAT;
  if (fmt == QMM_FMT_Q4K) return qmm_run(Wq_dev, N, K, X_dev, Y_dev, M, stream);
  qmm_status s = check_job(Wq_dev, N, K, X_dev, Y_dev);
  if (s != QMM_OK) return s;
  if (M < 1 || M > QMM_MAX_M) return QMM_ERR_M_RANGE;
  q4k::Job job{Wq_dev, X_dev, Y_dev, N, K};
  job.fmt = fmt;
  job.aux = static_cast<const uint8_t*>(Wq_dev) + q4k::fmt_aux_offset(fmt, N, K);
  cudaError_t e = q4k::launch_tc(&job, 1, M, stream);
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

qmm_status qmm_fmt_run_batched(const qmm_fmt_entry* entries_host, int count, int M, cudaStream_t stream) {
  if (!entries_host) return QMM_ERR_NULL;
  if (count < 1 || count > QMM_MAX_BATCH) return QMM_ERR_COUNT;
  if (M < 1 || M > QMM_MAX_M) return QMM_ERR_M_RANGE;
  for (int k = 0; k < count; ++k) {
    const qmm_fmt_entry& e = entries_host[k];
    if (!valid_format(e.fmt)) return QMM_ERR_FORMAT;
    qmm_status s = check_job(e.Wq, e.N, e.K, e.X, e.Y);
    if (s != QMM_OK) return s;
  }
  q4k::Job jobs[QMM_MAX_BATCH];
  for (int fmt = QMM_FMT_Q4K; fmt <= QMM_FMT_Q6K; ++fmt) {
    int n = 0;
    for (int k = 0; k < count; ++k) {
      const qmm_fmt_entry& e = entries_host[k];
      if (e.fmt != fmt) continue;
      jobs[n] = q4k::Job{e.Wq, e.X, e.Y, e.N, e.K};
      jobs[n].fmt = fmt;
      jobs[n].aux = static_cast<const uint8_t*>(e.Wq) + q4k::fmt_aux_offset(fmt, e.N, e.K);
      ++n;
    }
    if (n == 0) continue;
    if (fmt == QMM_FMT_Q4K) {
      qmm_status s = run_jobs(jobs, n, M, QMM_VARIANT_AUTO, stream);
      if (s != QMM_OK) return s;
    } else {
      cudaError_t e = q4k::launch_tc(jobs, n, M, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }
  return QMM_OK;
}

qmm_status qmm_fmt_dequant(int fmt, const void* Wq_dev, int64_t N, int64_t K, float* out_dev, cudaStream_t stream) {
  if (!valid_format(fmt)) return QMM_ERR_FORMAT;
  if (!Wq_dev || !out_dev) return QMM_ERR_NULL;
  qmm_status s = check_shape(N, K);
  if (s != QMM_OK) return s;
  if (!aligned(Wq_dev, 16) || !aligned(out_dev, 16)) return QMM_ERR_ALIGN;
  cudaError_t e = q4k::launch_dequant_fmt(fmt, Wq_dev, N, K, out_dev, stream);
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

int qmm_select_variant(int M, int64_t N, int64_t K) { return select_variant(M, N, K); }

int qmm_select_variant_batched(const qmm_entry* entries_host, int count, int M) {
  if (!entries_host || count < 1 || count > QMM_MAX_BATCH || M < 1 || M > QMM_MAX_M) return -1;
  q4k::Job jobs[QMM_MAX_BATCH];
  for (int k = 0; k < count; ++k) {
    const qmm_entry& e = entries_host[k];
    if (check_shape(e.N, e.K) != QMM_OK) return -1;
    jobs[k] = q4k::Job{e.Wq, e.X, e.Y, e.N, e.K};
  }
  return select_variant_jobs(jobs, count, M);
}

size_t qmm_stream_read_sink_words(void) {
  const int g = q4k::stream_read_grid();
  return g > 0 ? (size_t)g : 0;
}

qmm_status qmm_stream_read(const void* buf_dev, size_t bytes, uint32_t* sink_dev, cudaStream_t stream) {
  if (!buf_dev || !sink_dev) return QMM_ERR_NULL;
  if (bytes == 0 || bytes % 16 != 0) return QMM_ERR_SHAPE;
  if (!aligned(buf_dev, 16) || !aligned(sink_dev, 4)) return QMM_ERR_ALIGN;
  const cudaError_t e = q4k::launch_stream_read(buf_dev, bytes, sink_dev, stream);
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

void qmm_set_wait_limit(uint32_t polls, uint32_t suspend_ns) { q4k::set_wait_limit(polls, suspend_ns); }

qmm_status qmm_release(void) {
  const cudaError_t e = q4k::release_workspaces();
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

size_t qmm_workspace_bytes_held(void) { return q4k::workspace_bytes_held(); }

qmm_status qmm_device_status(unsigned* status_out) {
  if (!status_out) return QMM_ERR_NULL;
  unsigned a = 0, b = 0, c = 0;
  cudaError_t e = q4k::read_and_clear_fma_status(&a);
  if (e == cudaSuccess) e = q4k::read_and_clear_tc_status(&b);
  if (e == cudaSuccess) e = q4k::read_and_clear_pack_status(&c);
  *status_out = a | b | c;
  return e == cudaSuccess ? QMM_OK : cuda_fail(e);
}

const char* qmm_strerror(qmm_status status) {
  switch (status) {
    case QMM_OK: return "ok";
    case QMM_ERR_NULL: return "a required pointer is NULL";
    case QMM_ERR_SHAPE: return "invalid shape: need 1 <= N < 2^31, 256 <= K <= 2^20, K % 256 == 0";
    case QMM_ERR_M_RANGE: return "M must be in [1, 32]";
    case QMM_ERR_ALIGN: return "Wq and X must be 16-byte aligned, Y 4-byte aligned";
    case QMM_ERR_BUFSIZE: return "output buffer too small";
    case QMM_ERR_NONFINITE: return "non-finite weight or fp16 overflow of a super-block scale";
    case QMM_ERR_CUDA: return "CUDA error (see qmm_last_cuda_error)";
    case QMM_ERR_COUNT: return "batched entry count must be in [1, QMM_MAX_BATCH]";
    case QMM_ERR_VARIANT: return "the requested kernel variant cannot run this shape";
    case QMM_ERR_SCRATCH: return "qmm_run_noalloc: the problem needs more than QMM_NOALLOC_SCRATCH_BYTES of scratch";
    case QMM_ERR_FORMAT: return "unknown weight format code";
  }
  return "unknown status";
}

const char* qmm_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
