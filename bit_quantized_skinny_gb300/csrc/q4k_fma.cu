// q4k_fma.cu — the CUDA-core variant of the skinny Q4K x bf16 product (sm_103a).
//
// The pages' verify-pass profile ("sixi-asi 0.9", section "What I got wrong in 0.8") spends its
// time in a matrix-vector kernel that decodes the 4-bit weights again for every activation row,
// and in a matrix kernel that is latency-bound because too few bytes are in flight (section
// "The patch": one 256-thread block per SM, 29% of DRAM bandwidth).  This kernel reads and
// decodes every weight once for all rows of X and keeps tens of kilobytes per SM in flight:
//
//   * Work: a product is cut into row ranges (tasks); one CTA of 8 warps owns a task.  Within a
//     task the K axis is cut into chunks of 4 super-blocks (1024 weights, 576 bytes per row) and
//     the (chunk, 4-row box) units are dealt to the 8 warps in equal contiguous slices.
//   * Streaming: each warp has its own 4-stage ring in shared memory.  One bulk copy
//     (cp.async.bulk, completion on an mbarrier) per row brings a box of 4 rows x 576 bytes; the
//     copy for box u+4 is issued as soon as box u is consumed.
//   * Decode: lane l owns sub-block l%8 of super-block l/8 of the chunk: 32 weights, 16 bytes of
//     quants.  Its 32 activations per row of X live in registers as fp32 values, loaded once
//     per chunk.  Nibbles become exact fp32 values (exponent trick + one subtraction), each
//     weight is formed by its definition, w_t = fma(D*sc_j, q_t, -(Dm*m_j)) (one rounding of the
//     exact value: the weight the oracle and qmm_dequant compute), and the dot product runs on
//     fp32 FMAs: part = sum_t w_t x_t.  Forming the weight first keeps the error of a part
//     within a few units of fp32 rounding of sum_t |w_t x_t|, also where d*sc_j*q_t and
//     dmin*m_j nearly cancel (a factored form (D*sc_j) sum q x - (Dm*m_j) sum x would round two
//     large sums separately).
//   * K-reduction: a warp-shuffle butterfly sums the 32 lanes (one chunk) for the 4 rows x MT
//     activation rows of a box; chunk partials go to shared memory and are summed over the
//     chunks in increasing order at the end of the task.  The order of every addition depends
//     only on K, so an M-row product is bitwise equal to M one-row products.
#include <cmath>
#include <cstdio>
#include <algorithm>
#include <vector>
#include <mutex>

#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {
namespace {

__device__ unsigned g_status;   // this file's kernels' status word

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRB = 4;        // rows per box
constexpr int kStages = 4;    // ring depth per warp
constexpr int kBoxBytes = kRB * kChunkBytes;               // 2304
constexpr int kRingBytes = kWarps * kStages * kBoxBytes;   // 73728
constexpr int kBarBytes = kWarps * kStages * 8;            // 256
constexpr uint32_t kWaitLimit = 1u << 17;   // polls of up to 20 us each: ~2.6 s
constexpr int kMinBlocksPerSM = 2;

struct FmaEntry {
  const uint8_t* W;
  const uint16_t* X;
  float* Y;
  int N;
  int K;
  int ranges;          // row ranges of this product (per pass)
  int rows_per_range;  // ceil(N / ranges)
  int task_begin;      // first task index of this entry
  int pad_;
};

template <int MAXE>
struct FmaParams {
  int count;
  int M;
  int passes;
  int tasks_total;
  int partial_cap;  // max over entries of rows_per_range * chunks (partial-buffer floats / MT)
  int pad_[3];
  FmaEntry e[MAXE];
};

template <int MT, int MAXE>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSM)
q4k_fma_kernel(const __grid_constant__ FmaParams<MAXE> P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t ring = smem_addr(smem) + warp * kStages * kBoxBytes;
  const uint32_t bars = smem_addr(smem + kRingBytes) + warp * kStages * 8;
  float* partial = reinterpret_cast<float*>(smem + kRingBytes + kBarBytes);

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bars + 8 * s, 1);
    fence_barrier_init();
  }
  __syncwarp();
  // programmatic dependent launch: the next launch in the stream may be scheduled from now on
  // (it waits for this grid before it touches memory); this grid may have started before the
  // kernel ahead of it finished, so it reads and writes nothing before that one is complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const uint64_t pol = policy_evict_first();
  uint32_t boxes_done = 0;    // boxes consumed by this warp so far (ring position)
  uint32_t boxes_issued = 0;  // boxes issued by this warp so far
  bool failed = false;

  for (int t = blockIdx.x; t < P.tasks_total; t += gridDim.x) {
    // ---- locate the task: entry, pass, row range
    int e = 0;
    if (MAXE > 1) {
      int lo = 0, hi = P.count - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.e[mid].task_begin <= t) lo = mid; else hi = mid - 1;
      }
      e = lo;
    }
    const FmaEntry& E = P.e[e];
    const int local = t - E.task_begin;
    const int pass = local / E.ranges;
    const int range = local - pass * E.ranges;
    const int r0 = range * E.rows_per_range;
    const int r1 = min(E.N, r0 + E.rows_per_range);
    const int i0 = pass * MT;
    const int nb = E.K >> 8;
    const int nch = (nb + kChunkBlocks - 1) / kChunkBlocks;
    const int rows = r1 - r0;
    const int nrb = (rows + kRB - 1) / kRB;
    const int T = nch * nrb;
    const int u_begin = (int)((int64_t)warp * T / kWarps);
    const int u_end = (int)((int64_t)(warp + 1) * T / kWarps);
    const int64_t rowbytes = (int64_t)nb * kBlockBytes;
    const uint8_t* W = E.W;

    auto issue = [&](int u) {
      const int c = u / nrb;
      const int rb = u - c * nrb;
      const int row0 = r0 + rb * kRB;
      const int nval = min(kRB, r1 - row0);
      const uint32_t cb = (uint32_t)min(kChunkBlocks, nb - c * kChunkBlocks) * kBlockBytes;
      const uint32_t stage = boxes_issued % kStages;
      const uint32_t bar = bars + 8 * stage;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(bar, nval * cb);
      __syncwarp();
      if (lane < nval)
        bulk_g2s(ring + stage * kBoxBytes + lane * kChunkBytes,
                 W + (int64_t)(row0 + lane) * rowbytes + (int64_t)c * kChunkBytes, cb, bar, pol);
      ++boxes_issued;
    };

    if (!failed)
      for (int u = u_begin; u < min(u_end, u_begin + kStages); ++u) issue(u);

    float xf[MT][32];
    int cur_c = -1;
    bool lane_valid = false;

    for (int u = u_begin; u < u_end && !failed; ++u) {
      const int c = u / nrb;
      const int rb = u - c * nrb;
      if (c != cur_c) {
        // activations of this lane's sub-block for rows i0..i0+MT-1, as fp32 pairs
        cur_c = c;
        const int kb = c * kChunkBlocks + (lane >> 3);
        lane_valid = kb < nb;
        const int64_t k0 = (int64_t)c * kChunkWeights + lane * 32;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          uint4 v[4];
          if (lane_valid && i0 + i < P.M) {
            const uint16_t* xr = E.X + (int64_t)(i0 + i) * E.K + k0;
#pragma unroll
            for (int g = 0; g < 4; ++g) v[g] = ldg_nc_v4(xr + 8 * g);
          } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) v[g] = make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t w4[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              xf[i][8 * g + 2 * h] = __uint_as_float(w4[h] << 16);
              xf[i][8 * g + 2 * h + 1] = __uint_as_float(w4[h] & 0xFFFF0000u);
            }
          }
        }
      }

      const uint32_t stage = boxes_done % kStages;
      const uint32_t parity = (boxes_done / kStages) & 1u;
      if (!mbar_wait(bars + 8 * stage, parity, kWaitLimit)) {
        atomicOr(&g_status, kErrWaitTimeout);
        failed = true;
        break;
      }

      constexpr int V = kRB * (MT == 1 ? 1 : (MT == 2 ? 2 : 4));
      float vals[V];
#pragma unroll
      for (int k = 0; k < V; ++k) vals[k] = 0.f;

      const int row0 = r0 + rb * kRB;
      const uint32_t sb = ring + stage * kBoxBytes + (lane >> 3) * kBlockBytes;
#pragma unroll
      for (int s = 0; s < kRB; ++s) {
        if (row0 + s < r1) {
          const uint4 h = lds128(sb + s * kChunkBytes);
          const uint4 q = lds128(sb + s * kChunkBytes + 16 + 16 * (lane & 7));
          const SubScale sc = decode_scales(h, lane & 7);
          float qf[32];
          nibbles_to_f32(q.x, *reinterpret_cast<float(*)[8]>(&qf[0]));
          nibbles_to_f32(q.y, *reinterpret_cast<float(*)[8]>(&qf[8]));
          nibbles_to_f32(q.z, *reinterpret_cast<float(*)[8]>(&qf[16]));
          nibbles_to_f32(q.w, *reinterpret_cast<float(*)[8]>(&qf[24]));
          const float ndmm = -sc.dmm;
#pragma unroll
          for (int t = 0; t < 32; ++t) qf[t] = fmaf(sc.dsc, qf[t], ndmm);   // the weight w_t
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            // four accumulators (weights t = 4k, 4k+1, 4k+2, 4k+3), summed in a fixed order
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int t = 0; t < 32; t += 4) {
              a0 = fmaf(qf[t], xf[i][t], a0);
              a1 = fmaf(qf[t + 1], xf[i][t + 1], a1);
              a2 = fmaf(qf[t + 2], xf[i][t + 2], a2);
              a3 = fmaf(qf[t + 3], xf[i][t + 3], a3);
            }
            const float dot = (a0 + a1) + (a2 + a3);
            vals[s * (V / kRB) + i] = lane_valid ? dot : 0.f;
          }
        }
      }
      __syncwarp();
      ++boxes_done;
      if (u + kStages < u_end) issue(u + kStages);

      butterfly_reduce<V>(vals, lane);
      constexpr int span = 32 / V;
      if ((lane & (span - 1)) == 0) {
        const int idx = lane / span;
        const int s = idx / (V / kRB);
        const int i = idx - s * (V / kRB);
        if (i < MT && row0 + s < r1)
          partial[((row0 - r0 + s) * nch + c) * MT + i] = vals[0];
      }
    }
    __syncthreads();

    // ---- sum the chunk partials in increasing chunk order and write Y
    for (int idx = threadIdx.x; idx < rows * MT; idx += kThreads) {
      const int i = idx / rows;
      const int rl = idx - i * rows;
      if (i0 + i < P.M) {
        float y = 0.f;
        for (int c = 0; c < nch; ++c) y += partial[(rl * nch + c) * MT + i];
        E.Y[(int64_t)(i0 + i) * E.N + r0 + rl] = y;
      }
    }
    __syncthreads();
  }

  // After a timed-out wait, give the copies still in flight a bounded time to land.
  if (failed) {
    while (boxes_done < boxes_issued) {
      const uint32_t stage = boxes_done % kStages;
      const uint32_t parity = (boxes_done / kStages) & 1u;
      if (!mbar_wait(bars + 8 * stage, parity, kWaitLimit)) break;
      ++boxes_done;
    }
  }
}

// ------------------------------------------------------------------------------------------
// Host side: task planning and launch.

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

DeviceInfo device_info() {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DeviceInfo{};
  std::lock_guard<std::mutex> g(mu);
  if (!cache[dev].ok) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DeviceInfo{};
    cache[dev].sms = sms;
    cache[dev].ok = true;
  }
  return cache[dev];
}

constexpr int kMaxSmem = 113 * 1024;  // two CTAs per SM

template <int MT, int MAXE>
cudaError_t launch_fma_t(const Job* jobs, int count, int M, cudaStream_t stream) {
  static_assert(sizeof(FmaParams<MAXE>) < 32000, "kernel parameters too large");
  const DeviceInfo dev = device_info();
  if (!dev.ok) return cudaErrorInvalidDevice;
  const int passes = (M + MT - 1) / MT;
  const int slots = dev.sms * kMinBlocksPerSM;

  FmaParams<MAXE> P;
  P.count = count;
  P.M = M;
  P.passes = passes;
  double total_bytes = 0;
  for (int k = 0; k < count; ++k) total_bytes += (double)jobs[k].N * (double)(jobs[k].K / 256) * 144.0;
  const double per_slot = total_bytes / slots;

  // Rows per range: a fair share of the weight bytes, at least one 4-row box, and a partial
  // buffer that keeps two CTAs per SM.
  int tasks = 0, partial_cap = 1;
  for (int k = 0; k < count; ++k) {
    const int64_t N = jobs[k].N, K = jobs[k].K;
    const int nb = (int)(K / 256);
    const int nch = (nb + kChunkBlocks - 1) / kChunkBlocks;
    const double bytes = (double)N * nb * 144.0;
    int64_t ranges = (int64_t)std::max(1.0, std::floor(bytes / per_slot + 0.5));
    ranges = std::min<int64_t>(ranges, (N + kRB - 1) / kRB);
    int64_t rpr = (N + ranges - 1) / ranges;
    const int64_t max_rows = (kMaxSmem - kRingBytes - kBarBytes) / ((int64_t)nch * MT * 4);
    if (rpr > max_rows) rpr = std::max<int64_t>(kRB, (max_rows / kRB) * kRB);
    ranges = (N + rpr - 1) / rpr;
    FmaEntry& E = P.e[k];
    E.W = static_cast<const uint8_t*>(jobs[k].W);
    E.X = jobs[k].X;
    E.Y = jobs[k].Y;
    E.N = (int)N;
    E.K = (int)K;
    E.ranges = (int)ranges;
    E.rows_per_range = (int)rpr;
    E.task_begin = tasks;
    E.pad_ = 0;
    tasks += (int)ranges * passes;
    partial_cap = std::max<int>(partial_cap, (int)(rpr * nch));
  }
  P.tasks_total = tasks;
  P.partial_cap = partial_cap;
  const size_t smem = kRingBytes + kBarBytes + (size_t)partial_cap * MT * sizeof(float);
  if (smem > (size_t)kMaxSmem) return cudaErrorInvalidConfiguration;

  auto kern = q4k_fma_kernel<MT, MAXE>;
  static std::mutex attr_mu;
  static bool attr_set[64] = {};
  int devno = 0;
  cudaError_t err = cudaGetDevice(&devno);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> g(attr_mu);
    if (devno >= 64 || !attr_set[devno]) {
      err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
      if (err != cudaSuccess) return err;
      if (devno < 64) attr_set[devno] = true;
    }
  }
  const int grid = std::min(tasks, slots);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace

cudaError_t launch_fma(const Job* jobs, int count, int M, cudaStream_t stream) {
  if (count == 1) {
    return (M == 1) ? launch_fma_t<1, 1>(jobs, count, M, stream)
                    : launch_fma_t<2, 1>(jobs, count, M, stream);
  }
  return (M == 1) ? launch_fma_t<1, 512>(jobs, count, M, stream)
                  : launch_fma_t<2, 512>(jobs, count, M, stream);
}

cudaError_t read_and_clear_fma_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  *out = v;
  return e;
}

}  // namespace q4k
