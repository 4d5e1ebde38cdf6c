// q4k_tc.cu — tensor-core (tcgen05) variant of the skinny Q4K x bf16 product (sm_103a).
//
// The skinny product of the pages' verify pass ("sixi-asi 0.9", section "What I got wrong in
// 0.8") is a weight stream: every weight is read once and used by M <= 32 activation rows.  On
// CUDA cores each weight costs one logic op, one subtraction and M fused multiply-adds; here the
// M multiplies go to the tensor cores and the per-weight CUDA-core work drops to about one
// instruction per pair of weights, the same for every M.  That is the M-dependent tiling of the
// pages (a matrix kernel from a few rows on, section "The patch") done with GB300's units.
//
// Operands ("swap AB": the 128-row MMA dimension runs over weight rows):
//   A[128 rows x 16 k] fp16 in tensor memory (TMEM): A = sc_j * q_t, an integer <= 945, exact.
//     Written by the dequant warps with tcgen05.st, one thread per weight row (lane).
//   B[16 k x Mpad] fp16 in shared memory: the activations of one super-block, x * 2^-s with one
//     power-of-two s per super-block so that every bf16 value is exact in fp16 (see below).
//   D[128 x Mpad] fp32 in TMEM, one accumulator per 256-weight super-block.
//   One more K=16 MMA per super-block multiplies A_ext = (m_0..m_7, m_0..m_7) with
//   B_ext = (hi_0..hi_7, lo_0..lo_7), the fp16 halves of the sub-block sums of x, so the
//   dmin term also comes from the tensor cores.  The epilogue forms, per super-block,
//     y += (D*2^s) * acc - (Dm*2^s*64) * acc_ext
//   in fp32 registers.  Products in the MMAs are exact; only fp32 accumulation rounds.
//
// K order inside a super-block: the nibble trick below yields the quants of one 32-bit word as
// fp16 pairs (q0,q4) (q1,q5) (q2,q6) (q3,q7); TMEM column 4w+c holds k = 8w+c (low half) and
// 8w+c+4 (high half), and the activations are laid out in B with the same permutation.
//
// Pipeline (one CTA per SM, persistent over 128-row tiles of every product in the launch):
//   warp 8        weights: one 2D TMA tile copy per super-block (128 rows x 144 bytes, rows
//                 dense at 144 bytes: 16-byte reads of 8 consecutive rows hit 32 distinct banks)
//                 into a 10-deep ring, evict-first in L2
//   warp 9        one bulk copy per super-block of the prepared activation block into a ring
//   warps 0..7    dequant: warp w owns TMEM lanes 32*(w%4).. and K half w/4 of each super-block,
//                 writes A units into its half's ring of TMEM slots
//   warps 10..12  MMA issue, super-blocks round robin (one issuing thread spends ~90 cycles per
//                 MMA, so the issue rate grows with the issuers); warp 10 owns TMEM
//   warps 13..16  epilogue: per super-block, read the accumulators and (d, dmin) of each row
// Every wait is bounded; on timeout the kernel records an error in the status word and drains.
//
// Activation preparation (q4k_xprep_kernel, one CTA per super-block of each distinct X): picks
// s so that the largest |x| of the super-block lands in [2^14, 2^15); a bf16 value is then exact
// in fp16 unless it is below 2^-32 of that largest value (such values are rounded to fp16's
// 2^-24 step of the scaled range), and writes B, B_ext and 2^s into a per-stream workspace.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "q4k_device.cuh"
#include "q4k_internal.h"
#include "q4k_tcgen05.cuh"

namespace q4k {


namespace {

__device__ unsigned g_status;   // this file's kernels' status word

constexpr int kTileRows = 128;
constexpr int kDqWarps = 8;        // warps 0..7: dequant (0..3 even K halves, 4..7 odd K halves)
constexpr int kWProdWarp = 8;      // TMA tiles of the weights
constexpr int kBProdWarp = 9;      // bulk copies of the prepared activations
constexpr int kMmaWarp = 10;       // warps 10..12: MMA issue; 10 owns TMEM
constexpr int kMmaWarps = 3;
constexpr int kEpiWarp0 = 13;      // warps 13..16: epilogue
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);   // 544
constexpr int kWStageBytes = kTileRows * kBlockBytes;    // 18432: one super-block of a tile
constexpr int kWStages = 10;
constexpr int kMaxASlots = 6;      // A slots of both K halves together (upper bound)
constexpr int kMaxAccSlots = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 17;
constexpr int kMaxEBatch = 160;    // products per batched launch (their tensor maps ride in the parameters)
constexpr int kMaxPrep = 512;      // distinct activations per preparation launch

__host__ __device__ constexpr int bblock_bytes(int mpad) { return mpad * 544 + 16; }
// activation-block ring depth; at least the number of MMA issuers (see the MMA warps)
__host__ __device__ constexpr int b_slots(int mpad) { return mpad <= 16 ? 4 : 2; }
// TMEM columns.  An even-half A unit: 64 columns of sc*q pairs (128 k); an odd-half unit adds 8
// columns of (m_j) pairs for the dmin MMA.  Accumulator slot: Mpad columns of the product, Mpad
// columns of the dmin term.  Each K half has its own ring of A slots, as deep as there are MMA
// issuers, so super-block su uses slot su % issuers of each ring and accumulator slot
// su % issuers, all owned by issuer su % issuers:
//   Mpad 16: 3 issuers; even 3 x 64 (0..191), odd 3 x 72 (192..407), accumulators 416..511
//   Mpad 32: 2 issuers; even 2 x 64 (0..127), odd 2 x 72 (128..271), accumulators 384..511
// Every slot thus has one waiting issuer, which sees its phases in order.
__host__ __device__ constexpr int acc_slots(int mpad) { return mpad <= 16 ? 3 : 2; }
__host__ __device__ constexpr int ar0(int mpad) { return acc_slots(mpad); }
__host__ __device__ constexpr int ar1(int mpad) { return acc_slots(mpad); }
__host__ __device__ constexpr uint32_t a0_col(int slot) { return 64u * slot; }
__host__ __device__ constexpr uint32_t a1_col(int mpad, int slot) { return 64u * ar0(mpad) + 72u * slot; }
__host__ __device__ constexpr uint32_t acc1_col(int mpad, int slot) {
  return 512u - 2u * mpad * acc_slots(mpad) + 2u * mpad * slot;
}
__host__ __device__ constexpr uint32_t acc2_col(int mpad, int slot) { return acc1_col(mpad, slot) + mpad; }
static_assert(a1_col(16, ar1(16)) <= acc1_col(16, 0) && a1_col(32, ar1(32)) <= acc1_col(32, 0),
              "TMEM column plan overlaps");
static_assert(ar0(16) + ar1(16) <= kMaxASlots && ar0(32) + ar1(32) <= kMaxASlots, "A slot count");
static_assert(acc_slots(16) <= kMmaWarps && acc_slots(32) <= kMmaWarps, "one MMA warp per accumulator slot");
static_assert(b_slots(16) >= acc_slots(16) && b_slots(32) >= acc_slots(32), "B ring shallower than the issuers");

// barrier indices inside the barrier block
constexpr int kMaxBSlots = 4;
enum : int {
  kBarWFull = 0, kBarWEmpty = kBarWFull + kWStages,
  kBarBFull = kBarWEmpty + kWStages, kBarBEmpty = kBarBFull + kMaxBSlots,
  kBarAFull = kBarBEmpty + kMaxBSlots, kBarAEmpty = kBarAFull + kMaxASlots,
  kBarAccFull = kBarAEmpty + kMaxASlots, kBarAccEmpty = kBarAccFull + kMaxAccSlots,
  kNumBars = kBarAccEmpty + kMaxAccSlots
};

template <int MPAD>
struct TcSmem {
  static constexpr int kW = 0;
  static constexpr int kB = kW + kWStages * kWStageBytes;
  static constexpr int kBars = kB + b_slots(MPAD) * bblock_bytes(MPAD);
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kTotal = kMisc + 16;   // TMEM address, abort flag
};
static_assert(TcSmem<16>::kTotal <= 232448 && TcSmem<32>::kTotal <= 232448, "shared memory");

struct TcEntry {
  float* Y;
  const uint8_t* B;    // prepared activation blocks of this entry's X
  int N;
  int K;
  int tiles;
  int task_begin;
};

// Launch parameters: the weights of entry e are reached through maps[e], a 2D tensor map over
// the packed rows (inner dimension: the row's bytes, outer: the N rows).
template <int MAXE>
struct TcParams {
  CUtensorMap maps[MAXE];
  TcEntry e[MAXE];
  int count;
  int M;
  int tasks_total;
  int pad_;
};

struct PrepEntry {
  const uint16_t* X;
  uint8_t* out;
  int K;
  int block_begin;   // first CTA index of this X
};

struct PrepParams {
  int count;
  int M;
  int blocks_total;
  int pad_;
  PrepEntry e[kMaxPrep];
};

__device__ __forceinline__ uint32_t h2bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 bits2h(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// ------------------------------------------------------------------------------------------
// Activation preparation.  Block = 8*MPAD threads; thread (i = t/8, j = t%8) handles token i,
// sub-block j (32 activations) of one super-block.
template <int MPAD>
__global__ void __launch_bounds__(8 * MPAD) q4k_xprep_kernel(const __grid_constant__ PrepParams P) {
  __shared__ unsigned s_max[8];
  const int b = blockIdx.x;
  int e = 0;
  {
    int lo = 0, hi = P.count - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (P.e[mid].block_begin <= b) lo = mid; else hi = mid - 1;
    }
    e = lo;
  }
  const PrepEntry& E = P.e[e];
  const int sb = b - E.block_begin;
  const int t = threadIdx.x;
  const int i = t >> 3, j = t & 7;
  const bool valid = i < P.M;
  uint4 v[4];
  if (valid) {
    const uint16_t* xr = E.X + (int64_t)i * E.K + (int64_t)sb * 256 + 32 * j;
#pragma unroll
    for (int g = 0; g < 4; ++g) v[g] = ldg_nc_v4(xr + 8 * g);
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g) v[g] = make_uint4(0, 0, 0, 0);
  }
  unsigned mx = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t w4[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      mx = max(mx, w4[h] & 0x7FFFu);
      mx = max(mx, (w4[h] >> 16) & 0x7FFFu);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((t & 31) == 0) s_max[t >> 5] = mx;
  __syncthreads();
  mx = 0;
#pragma unroll
  for (int w = 0; w < (8 * MPAD) / 32; ++w) mx = max(mx, s_max[w]);
  // largest |x| in [2^(e-127), 2^(e-126)); scale it into [2^14, 2^15)
  int s = 0;
  if (mx != 0) s = min(120, max(-120, (int)(mx >> 7) - 141));
  const float f = __uint_as_float((uint32_t)(127 - s) << 23);   // 2^-s

  uint8_t* out = E.out + (int64_t)sb * bblock_bytes(MPAD);
  float xsum = 0.f;
#pragma unroll
  for (int ww = 0; ww < 4; ++ww) {
    const int w = 4 * j + ww;  // word (8 activations) index within the super-block
    const uint32_t w4[4] = {v[ww].x, v[ww].y, v[ww].z, v[ww].w};
    float xv[8];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      xv[2 * h] = __uint_as_float(w4[h] << 16) * f;
      xv[2 * h + 1] = __uint_as_float(w4[h] & 0xFFFF0000u) * f;
    }
    uint32_t packed[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) packed[c] = h2bits(__floats2half2_rn(xv[c], xv[c + 4]));
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const __half2 hh = bits2h(packed[p & 3]);
      xsum += (p < 4) ? __low2float(hh) : __high2float(hh);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + ((i >> 3) * 32 + w) * 128 + (i & 7) * 16);
    *dst = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
  const float xs = xsum * 0.015625f;  // 2^-6: a sum of 32 values below 2^15 stays below 2^14
  const __half hi = __float2half_rn(xs);
  const __half lo = __float2half_rn(xs - __half2float(hi));
  __half* ext = reinterpret_cast<__half*>(out + MPAD * 512);
  ext[(((i >> 3) * 2 + 0) * 128 + (i & 7) * 16) / 2 + j] = hi;
  ext[(((i >> 3) * 2 + 1) * 128 + (i & 7) * 16) / 2 + j] = lo;
  if (t == 0) {
    float* sig = reinterpret_cast<float*>(out + MPAD * 544);
    sig[0] = __uint_as_float((uint32_t)(127 + s) << 23);  // 2^s
    sig[1] = 0.f;
    sig[2] = 0.f;
    sig[3] = 0.f;
  }
}

// ------------------------------------------------------------------------------------------
// 2D TMA tile copy global -> shared (this CTA), completing on the mbarrier; x is the byte offset
// in the row (a multiple of 16), y the first row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy) : "memory");
}

template <int MPAD, int MAXE>
__global__ void __launch_bounds__(kThreads, 1) q4k_tc_kernel(const __grid_constant__ TcParams<MAXE> P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using L = TcSmem<MPAD>;
  constexpr int kBB = bblock_bytes(MPAD);
  constexpr int kBSlots = b_slots(MPAD);
  constexpr int kAccSlots = acc_slots(MPAD);   // also the number of MMA warps that issue
  constexpr int kAR0 = ar0(MPAD), kAR1 = ar1(MPAD);   // A ring depths of the two K halves
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sW = smem_addr(smem + L::kW);
  const uint32_t sB = smem_addr(smem + L::kB);
  const uint32_t bars = smem_addr(smem + L::kBars);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  auto bar = [&](int k) { return bars + 8u * k; };

  if (threadIdx.x == 0) {
    for (int k = 0; k < kWStages; ++k) {
      mbar_init(bar(kBarWFull + k), 1);
      mbar_init(bar(kBarWEmpty + k), kDqWarps + kEpiWarps);   // dequant reads quants, epilogue (d, dmin)
    }
    for (int k = 0; k < kBSlots; ++k) { mbar_init(bar(kBarBFull + k), 1); mbar_init(bar(kBarBEmpty + k), 1); }
    for (int k = 0; k < kMaxASlots; ++k) { mbar_init(bar(kBarAFull + k), 4); mbar_init(bar(kBarAEmpty + k), 1); }
    for (int k = 0; k < kAccSlots; ++k) { mbar_init(bar(kBarAccFull + k), 1); mbar_init(bar(kBarAccEmpty + k), kEpiWarps); }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_addr(tmem_holder), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  auto wait = [&](int k, uint32_t parity) -> bool {
    if (mbar_try(bar(k), parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait(bar(k), parity, kWaitLimit)) return true;
    atomicOr(&g_status, kErrWaitTimeout);
    *abort_flag = 1;
    return false;
  };
  auto locate = [&](int t) {
    int lo = 0, hi = P.count - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (P.e[mid].task_begin <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
  };

  if (warp == kWProdWarp) {
    // ------------------------------------------------------------------ weight tiles
    // One TMA copy per super-block: rows row0 .. row0+127 (rows past N read as zeros), bytes
    // 144 sb .. 144 sb + 143 of each row.  The ring runs kWStages - 1 super-blocks ahead.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t su = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < P.tasks_total && ok; t += gridDim.x) {
        const int e = locate(t);
        const TcEntry& E = P.e[e];
        const int nb = E.K >> 8;
        const int row0 = (t - E.task_begin) * kTileRows;
        for (int sb = 0; sb < nb; ++sb, ++su) {
          const uint32_t ws = su % kWStages;
          if (!wait(kBarWEmpty + ws, ((su / kWStages) & 1u) ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(kBarWFull + ws), kWStageBytes);
          tma_load_2d(sW + ws * kWStageBytes, &P.maps[e], sb * kBlockBytes, row0, bar(kBarWFull + ws), pol);
        }
      }
    }
  } else if (warp == kBProdWarp) {
    // ------------------------------------------------------------------ activation blocks
    if (lane == 0) {
      uint32_t su = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < P.tasks_total && ok; t += gridDim.x) {
        const TcEntry& E = P.e[locate(t)];
        const int nb = E.K >> 8;
        for (int sb = 0; sb < nb; ++sb, ++su) {
          const uint32_t bs = su % kBSlots;
          if (!wait(kBarBEmpty + bs, ((su / kBSlots) & 1u) ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(kBarBFull + bs), kBB);
          bulk_g2s(sB + bs * kBB, E.B + (int64_t)sb * kBB, kBB, bar(kBarBFull + bs), 0ull);
        }
      }
    }
  } else if (warp >= kMmaWarp && warp < kMmaWarp + kMmaWarps) {
    // ------------------------------------------------------------------ MMA issue
    // Super-block su goes to warp su % kAccSlots (three issuers at Mpad 16, two at 32), which
    // owns accumulator slot su % kAccSlots and A slot su % kAccSlots of each K half's ring.  The
    // B ring is at least kAccSlots deep, so an issuer that saw super-block su - kAccSlots's block
    // arrive waits on the right phase of su's slot.
    const uint32_t mine = warp - kMmaWarp;
    if (lane == 0 && mine < (uint32_t)kAccSlots) {
      constexpr uint32_t idesc = tc::idesc_f16_f32(128, MPAD);
      uint32_t su = 0;   // super-blocks of this CTA so far
      uint32_t last = 0; // 1 + the last super-block this warp issued
      bool ok = true;
      for (int t = blockIdx.x; t < P.tasks_total && ok; t += gridDim.x) {
        const int nb = P.e[locate(t)].K >> 8;
        for (int sb = 0; sb < nb; ++sb, ++su) {
          if (su % kAccSlots != mine) continue;
          const uint32_t a0 = mine, a1 = kAR0 + mine;
          const uint32_t bs = su % kBSlots, es = mine;
          const uint32_t use = (su / kAccSlots) & 1u;   // phase parity of this warp's slots
          if (!wait(kBarAccEmpty + es, use ^ 1u) ||
              !wait(kBarBFull + bs, (su / kBSlots) & 1u) ||
              !wait(kBarAFull + a0, use)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t d1 = tmem + acc1_col(MPAD, es);
          const uint32_t d2 = tmem + acc2_col(MPAD, es);
          const uint32_t bslot = sB + bs * kBB;
          const uint64_t bdesc = tc::smem_desc_kmajor(bslot, 128, 4096);   // + 16 per MMA: 256 bytes
          tc::mma_f16_ts_x8(d1, tmem + a0_col(a0), bdesc, 16, idesc, 0);
          tc::commit(bar(kBarAEmpty + a0));
          if (!wait(kBarAFull + a1, use)) { ok = false; break; }
          tc::fence_after_sync();
          tc::mma_f16_ts_x8(d1, tmem + a1_col(MPAD, a1 - kAR0), bdesc + 8 * 16, 16, idesc, 1);
          tc::mma_f16_ts(d2, tmem + a1_col(MPAD, a1 - kAR0) + 64, tc::smem_desc_kmajor(bslot + MPAD * 512, 128, 256), idesc, 0);
          tc::commit(bar(kBarAccFull + es));
          tc::commit(bar(kBarAEmpty + a1));
          tc::commit(bar(kBarBEmpty + bs));
          last = su + 1;
        }
      }
      if (!ok && last > 0)   // let issued MMAs finish before TMEM is released
        mbar_wait(bar(kBarAccFull + (last - 1) % kAccSlots), ((last - 1) / kAccSlots) & 1u, kWaitLimit);
    }
  } else if (warp < kDqWarps) {
    // ------------------------------------------------------------------ dequant
    const int q = warp & 3;          // TMEM lane quarter / row quarter of the tile
    const int h = warp >> 2;         // K half of each super-block
    const int r = 32 * q + lane;     // row inside the tile
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    const __half2 k1024 = bits2h(0x64006400u);
    const __half2 kn1024 = __float2half2_rn(-1024.f);
    const __half2 k1o16 = __float2half2_rn(0.0625f);
    const __half2 kn64 = __float2half2_rn(-64.f);
    uint32_t su = 0;
    bool ok = true;
    bool pending = false;      // a unit whose TMEM stores are issued but not yet published
    uint32_t pending_as = 0;   // and its A slot
    for (int t = blockIdx.x; t < P.tasks_total && ok; t += gridDim.x) {
      const TcEntry& E = P.e[locate(t)];
      const int nb = E.K >> 8;
      for (int sb = 0; sb < nb && ok; ++sb, ++su) {
        const uint32_t ws = su % kWStages;
        if (!wait(kBarWFull + ws, (su / kWStages) & 1u)) { ok = false; break; }
        // this half's A ring: slot and how many times it was used before
        const uint32_t as = h ? kAR0 + su % kAR1 : su % kAR0;
        const uint32_t use = h ? su / kAR1 : su / kAR0;

        // ---- this row's half super-block from shared memory; the stage is then released
        const uint32_t rb = sW + ws * kWStageBytes + r * kBlockBytes;
        const uint4 hd = lds128(rb);
        uint4 qv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) qv[k] = lds128(rb + 16 + 64 * h + 16 * k);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarWEmpty + ws));

        // ---- the previous unit's TMEM stores have had the loads above to land: publish it
        if (pending) {
          tc::wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarAFull + pending_as));
          pending = false;
        }
        if (!wait(kBarAEmpty + as, (use & 1u) ^ 1u)) { ok = false; break; }
        tc::fence_after_sync();

        // ---- the 12-bit (sc, m) groups of this half's sub-blocks 4h .. 4h+3
        const uint64_t F = h ? ((uint64_t)hd.w << 32 | hd.z) : ((uint64_t)hd.z << 32 | hd.y);
        const int fbase = h ? 16 : 0;
        __half2 sc2[4], scm[4], sc16[4], sc64[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t g = (uint32_t)(F >> (fbase + 12 * jj)) & 0xFFFu;
          const uint32_t scb = ((g & 63u) | 0x6400u) * 0x10001u;       // (1024+sc, 1024+sc)
          sc2[jj] = __hsub2(bits2h(scb), k1024);                       // (sc, sc) exact
          scm[jj] = __hmul2(sc2[jj], kn1024);                           // -1024 sc
          sc16[jj] = __hmul2(sc2[jj], k1o16);                           // sc / 16
          sc64[jj] = __hmul2(sc2[jj], kn64);                            // -64 sc
        }

        // ---- A = sc*q as fp16 pairs, 16 columns per sub-block, into TMEM
        const uint32_t aaddr = tl + (h ? a1_col(MPAD, as - kAR0) : a0_col(as));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t words[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
          uint32_t cols[16];
#pragma unroll
          for (int ww = 0; ww < 4; ++ww) {
            const uint32_t wv = words[ww];
            const uint32_t b8 = wv >> 8;
            uint32_t p0, p1, p2, p3;
            asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(p0) : "r"(wv));
            asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(p1) : "r"(wv));
            asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(p2) : "r"(b8));
            asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(p3) : "r"(b8));
            cols[4 * ww + 0] = h2bits(__hfma2(bits2h(p0), sc2[k], scm[k]));   // (q0, q4) * sc
            cols[4 * ww + 1] = h2bits(__hfma2(bits2h(p1), sc16[k], sc64[k]));  // (q1, q5) * sc
            cols[4 * ww + 2] = h2bits(__hfma2(bits2h(p2), sc2[k], scm[k]));   // (q2, q6) * sc
            cols[4 * ww + 3] = h2bits(__hfma2(bits2h(p3), sc16[k], sc64[k]));  // (q3, q7) * sc
          }
          tc::st_x16(aaddr + 16 * k, cols);
        }
        if (h == 1) {
          // A_ext (odd unit): (m_0..m_7) at k = 0..7 and again at k = 8..15
          const uint64_t G = (uint64_t)hd.z << 32 | hd.y;   // groups 0..3 (bits 0..47)
          const uint64_t H = (uint64_t)hd.w << 32 | hd.z;   // groups 4..7 (bits 16..63)
          uint32_t mm[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            mm[jj] = (uint32_t)((jj < 4 ? (G >> (12 * jj)) : (H >> (16 + 12 * (jj - 4)))) >> 6) & 63u;
          uint32_t ext[8];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            ext[c] = ext[c + 4] =
                h2bits(__hsub2(bits2h((mm[2 * c] | 0x6400u) | ((mm[2 * c + 1] | 0x6400u) << 16)), k1024));
          tc::st_x8(aaddr + 64, ext);
        }
        // published (wait::st + arrive) after the next unit's loads, or below
        pending = true;
        pending_as = as;
      }
      if (ok && pending) {   // last unit of the task
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarAFull + pending_as));
        pending = false;
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    uint32_t ec = 0;   // super-blocks consumed
    bool ok = true;
    float y[MPAD];
    for (int t = blockIdx.x; t < P.tasks_total && ok; t += gridDim.x) {
      const TcEntry& E = P.e[locate(t)];
      const int nb = E.K >> 8;
      const int row0 = (t - E.task_begin) * kTileRows;
#pragma unroll
      for (int c = 0; c < MPAD; ++c) y[c] = 0.f;
      for (int sb = 0; sb < nb; ++sb) {
        const uint32_t es = ec % kAccSlots, ws = ec % kWStages;
        // 2^s of this super-block's activations (written by the preparation kernel)
        const float sigma = __ldg(reinterpret_cast<const float*>(E.B + (int64_t)sb * kBB + MPAD * 544));
        if (!wait(kBarWFull + ws, (ec / kWStages) & 1u)) { ok = false; break; }
        const uint32_t dpair = *reinterpret_cast<const uint32_t*>(smem + L::kW + ws * kWStageBytes + r * kBlockBytes);
        if (!wait(kBarAccFull + es, (ec / kAccSlots) & 1u)) { ok = false; break; }
        tc::fence_after_sync();
        const float2 dd = __half22float2(bits2h(dpair));
        const float2 sc = make_float2(dd.x * sigma, dd.y * sigma * 64.f);
        // read the accumulators 16 tokens at a time (keeps the register footprint small); the
        // slots are handed back as soon as the last read has landed, before the arithmetic
#pragma unroll
        for (int c0 = 0; c0 < MPAD; c0 += 16) {
          float a1[16], a2[16];
          tc::ld_x16(tl + acc1_col(MPAD, es) + c0, a1);
          tc::ld_x16(tl + acc2_col(MPAD, es) + c0, a2);
          tc::wait_ld();
          if (c0 + 16 == MPAD) {
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(bar(kBarAccEmpty + es));
              mbar_arrive(bar(kBarWEmpty + ws));
            }
          }
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            y[c0 + c] = fmaf(sc.x, a1[c], y[c0 + c]);
            y[c0 + c] = fmaf(-sc.y, a2[c], y[c0 + c]);
          }
        }
        ++ec;
      }
      if (!ok) break;
      if (row0 + r < E.N) {
#pragma unroll
        for (int c = 0; c < MPAD; ++c)
          if (c < P.M) E.Y[(int64_t)c * E.N + row0 + r] = y[c];
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------------------
// Per-(device, stream) workspace for the prepared activations.  Grown on demand with
// cudaMalloc (the first call on a stream, or a call needing more room, allocates; cudaFree of a
// smaller old buffer synchronizes the device, so no launch can still be using it).
class Workspace {
 public:
  static cudaError_t get(cudaStream_t stream, size_t bytes, void** out) {
    static std::mutex mu;
    static std::map<std::pair<int, uintptr_t>, std::pair<void*, size_t>> pool;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> g(mu);
    auto& slot = pool[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (slot.second < bytes) {
      if (slot.first) {
        err = cudaFree(slot.first);
        if (err != cudaSuccess) return err;
        slot = {nullptr, 0};
      }
      const size_t want = std::max(bytes, (size_t)1 << 20);
      void* p = nullptr;
      err = cudaMalloc(&p, want);
      if (err != cudaSuccess) return err;
      slot = {p, want};
    }
    *out = slot.first;
    return cudaSuccess;
  }
};

int num_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// ------------------------------------------------------------------------------------------
// Tensor maps.  cuTensorMapEncodeTiled is a driver entry point, looked up through the runtime
// (no link against the driver library).  A map depends only on (W, N, K), so encoded maps are
// kept in a small cache.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Map of a packed Q4K matrix as a 2D byte array: inner dimension the K/256*144 bytes of a row,
// outer dimension the N rows; the box is one super-block (144 bytes) of 128 rows.
cudaError_t weight_map(const void* W, int64_t N, int64_t K, CUtensorMap* out) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int64_t, int64_t>, CUtensorMap> cache;
  std::lock_guard<std::mutex> g(mu);
  const auto key = std::make_tuple(W, N, K);
  auto it = cache.find(key);
  if (it != cache.end()) { *out = it->second; return cudaSuccess; }
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t rowbytes = (cuuint64_t)(K / 256) * kBlockBytes;
  const cuuint64_t dims[2] = {rowbytes, (cuuint64_t)N};
  const cuuint64_t strides[1] = {rowbytes};
  const cuuint32_t box[2] = {(cuuint32_t)kBlockBytes, (cuuint32_t)kTileRows};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  const CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if (cache.size() >= 4096) cache.clear();
  cache.emplace(key, m);
  *out = m;
  return cudaSuccess;
}

template <int MPAD, int MAXE>
cudaError_t set_smem_attr() {
  static bool done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  err = cudaFuncSetAttribute(q4k_tc_kernel<MPAD, MAXE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem<MPAD>::kTotal);
  if (err == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return err;
}

// The main kernel over jobs[0 .. count) (count <= MAXE), whose prepared activations start at
// bsrc[k].  Parameters are built in a static block under the caller's lock.
template <int MPAD, int MAXE>
cudaError_t launch_main(const Job* jobs, const uint8_t* const* bsrc, int count, int M, cudaStream_t stream) {
  static TcParams<MAXE> par;
  par.count = count;
  par.M = M;
  int tasks = 0;
  for (int k = 0; k < count; ++k) {
    cudaError_t err = weight_map(jobs[k].W, jobs[k].N, jobs[k].K, &par.maps[k]);
    if (err != cudaSuccess) return err;
    const int tiles = (int)((jobs[k].N + kTileRows - 1) / kTileRows);
    par.e[k] = TcEntry{jobs[k].Y, bsrc[k], (int)jobs[k].N, (int)jobs[k].K, tiles, tasks};
    tasks += tiles;
  }
  par.tasks_total = tasks;
  cudaError_t err = set_smem_attr<MPAD, MAXE>();
  if (err != cudaSuccess) return err;
  const int grid = std::min(tasks, num_sms());
  q4k_tc_kernel<MPAD, MAXE><<<grid, kThreads, TcSmem<MPAD>::kTotal, stream>>>(par);
  return cudaGetLastError();
}

template <int MPAD>
cudaError_t launch_prep(const std::vector<std::pair<const uint16_t*, int64_t>>& xs, const std::vector<uint8_t*>& outs,
                        int M, cudaStream_t stream) {
  static PrepParams prep;   // large: built on the host, passed by value at launch
  prep.count = (int)xs.size();
  prep.M = M;
  int blocks = 0;
  for (size_t u = 0; u < xs.size(); ++u) {
    prep.e[u] = PrepEntry{xs[u].first, outs[u], (int)xs[u].second, blocks};
    blocks += (int)(xs[u].second / 256);
  }
  prep.blocks_total = blocks;
  q4k_xprep_kernel<MPAD><<<blocks, 8 * MPAD, 0, stream>>>(prep);
  return cudaGetLastError();
}

template <int MPAD>
cudaError_t launch_tc_t(const Job* jobs, int count, int M, cudaStream_t stream) {
  static_assert(sizeof(TcParams<kMaxEBatch>) < 32000 && sizeof(PrepParams) < 32000, "kernel parameters too large");
  constexpr int kBB = bblock_bytes(MPAD);
  // distinct activations (an X pointer with its K) get one prepared block run each
  std::vector<std::pair<const uint16_t*, int64_t>> xs;
  std::vector<int> xidx(count);
  for (int k = 0; k < count; ++k) {
    int found = -1;
    for (size_t u = 0; u < xs.size(); ++u)
      if (xs[u].first == jobs[k].X && xs[u].second == jobs[k].K) { found = (int)u; break; }
    if (found < 0) { found = (int)xs.size(); xs.push_back({jobs[k].X, jobs[k].K}); }
    xidx[k] = found;
  }
  size_t bytes = 0;
  std::vector<size_t> xoff(xs.size());
  for (size_t u = 0; u < xs.size(); ++u) {
    xoff[u] = bytes;
    bytes += (size_t)(xs[u].second / 256) * kBB;
  }
  void* wsp = nullptr;
  cudaError_t err = Workspace::get(stream, bytes, &wsp);
  if (err != cudaSuccess) return err;
  uint8_t* ws = static_cast<uint8_t*>(wsp);
  std::vector<uint8_t*> outs(xs.size());
  for (size_t u = 0; u < xs.size(); ++u) outs[u] = ws + xoff[u];
  std::vector<const uint8_t*> bsrc(count);
  for (int k = 0; k < count; ++k) bsrc[k] = outs[xidx[k]];

  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  err = launch_prep<MPAD>(xs, outs, M, stream);
  if (err != cudaSuccess) return err;
  if (count == 1) return launch_main<MPAD, 1>(jobs, bsrc.data(), 1, M, stream);
  for (int k0 = 0; k0 < count; k0 += kMaxEBatch) {
    err = launch_main<MPAD, kMaxEBatch>(jobs + k0, bsrc.data() + k0, std::min(kMaxEBatch, count - k0), M, stream);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

// ------------------------------------------------------------------------------------------
// Allocation-free entry (qmm_run_noalloc): the same two kernels, with the prepared activations
// in a fixed buffer that is part of this library's device image instead of the per-stream
// workspace.  Every GPU that loads the library holds the buffer until the process exits.
constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

template <int MPAD>
cudaError_t launch_tc_noalloc_t(const Job& job, int M, cudaStream_t stream, uint8_t* scratch) {
  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  const std::vector<std::pair<const uint16_t*, int64_t>> xs{{job.X, job.K}};
  const std::vector<uint8_t*> outs{scratch};
  cudaError_t err = launch_prep<MPAD>(xs, outs, M, stream);
  if (err != cudaSuccess) return err;
  const uint8_t* bsrc = scratch;
  return launch_main<MPAD, 1>(&job, &bsrc, 1, M, stream);
}

}  // namespace

cudaError_t read_and_clear_tc_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  *out = v;
  return e;
}

bool tc_supports(int M, int64_t N, int64_t K) {
  return M >= 1 && M <= 32 && N >= 1 && K >= 256 && K % 256 == 0;
}

size_t noalloc_scratch_bytes() { return kNoallocScratchBytes; }

size_t noalloc_scratch_needed(int M, int64_t K) {
  return (size_t)(K / 256) * (size_t)bblock_bytes(M <= 16 ? 16 : 32);
}

cudaError_t launch_tc_noalloc(const Job& job, int M, cudaStream_t stream) {
  // The host only knows a stand-in for the device array; its device address is looked up once
  // per device, with that device current.
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
      void* p = nullptr;
      err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (err != cudaSuccess) return err;
      addr[dev] = p;
    }
    scratch = addr[dev];
  }
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  return (M <= 16) ? launch_tc_noalloc_t<16>(job, M, stream, ws) : launch_tc_noalloc_t<32>(job, M, stream, ws);
}

cudaError_t launch_tc(const Job* jobs, int count, int M, cudaStream_t stream) {
  if (count < 1 || count > kMaxPrep) return cudaErrorInvalidValue;
  return (M <= 16) ? launch_tc_t<16>(jobs, count, M, stream) : launch_tc_t<32>(jobs, count, M, stream);
}

}  // namespace q4k
