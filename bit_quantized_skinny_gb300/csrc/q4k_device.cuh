// q4k_device.cuh — device-side building blocks shared by the Q4K kernels (sm_103a).
//
// * decode of one super-block's scale fields (d, dmin, sc_j, m_j) into fp32 factors,
// * exact nibble -> fp32 conversion with the exponent-field trick,
// * packed fp32x2 arithmetic (fma.rn.f32x2 / add.rn.f32x2, Blackwell),
// * mbarrier and bulk-copy (cp.async.bulk) wrappers with bounded waits,
// * a warp-shuffle butterfly that reduces V values per lane across the 32 lanes.
//
// Byte layout of a super-block (256 weights, 144 bytes): d (fp16) | dmin (fp16) | 96-bit F with
// sub-block j's 6-bit scale at bits 12j and 6-bit min at 12j+6 | 128 bytes of 4-bit quants,
// weight t at bits 4t.  Weight = one fp32 rounding of d*sc_j*q_t - dmin*m_j.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace q4k {

constexpr int kBlockBytes = 144;
constexpr int kChunkBlocks = 4;                        // super-blocks per K-chunk
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes; // 576
constexpr int kChunkWeights = kChunkBlocks * 256;       // 1024: one 32-weight sub-block per lane

// Error codes written to the device status word.
constexpr unsigned kErrWaitTimeout = 1u;

// ---------------------------------------------------------------- packed fp32x2 ----------
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Bit pattern of an fp32x2 pair of constants (element 0 in the low word).
__host__ __device__ constexpr uint64_t pair_bits(uint32_t lo, uint32_t hi) { return (uint64_t(hi) << 32) | lo; }

// ---------------------------------------------------------------- scale decode -----------
// fp32 factors of sub-block j of a super-block whose first 16 bytes are `h`:
// dsc = D*sc_j and dmm = Dm*m_j, both exact (D and Dm are binary16 values).
struct SubScale {
  float dsc;
  float dmm;
};

__device__ __forceinline__ SubScale decode_scales(uint4 h, int j) {
  const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&h.x));  // (D, Dm)
  // The 12-bit group of sub-block j starts at bit 12j of the 96-bit field (words h.y, h.z, h.w).
  const uint32_t lo = (j < 3) ? h.y : ((j < 6) ? h.z : h.w);
  const uint32_t hi = (j < 3) ? h.z : h.w;
  const uint32_t v = __funnelshift_r(lo, hi, (12 * j) & 31);
  // Small integers to fp32 exactly: OR the value into the mantissa of 2^23, subtract 2^23.
  const float sc = __uint_as_float((v & 63u) | 0x4B000000u) - 8388608.0f;
  const float m64 = __uint_as_float((v & 0xFC0u) | 0x4B000000u) - 8388608.0f;  // 64 * m_j
  SubScale r;
  r.dsc = dd.x * sc;
  r.dmm = (dd.y * 0.015625f) * m64;  // Dm * 2^-6 * 64 m = Dm * m, exact
  return r;
}

// ---------------------------------------------------------------- nibble -> fp32 ---------
// The 8 quants of one 32-bit word (nibble p = weight 8w+p) as exact fp32 values.  A nibble at
// bits [4p, 4p+4) with p <= 4 is ORed into a float whose exponent makes one unit of the nibble
// worth 1.0: the float is 2^(23-4p) + q; nibbles 5..7 are first shifted down by 12 bits.  One
// fp32 subtraction per weight removes the offset (exact).  Written as scalar code so that the
// compiler can pair the subtractions into packed fp32x2 instructions itself.
// (a & mask) | magic in one 3-input logic instruction.
__device__ __forceinline__ float and_or_f32(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));
  return __uint_as_float(r);
}

__device__ __forceinline__ void nibbles_to_f32(uint32_t a, float (&q)[8]) {
  const uint32_t b = a >> 12;
  q[0] = and_or_f32(a, 0x0000Fu, 0x4B000000u) - 8388608.0f;  // 2^23 + q0
  q[1] = and_or_f32(a, 0x000F0u, 0x49000000u) - 524288.0f;   // 2^19 + q1
  q[2] = and_or_f32(a, 0x00F00u, 0x47000000u) - 32768.0f;    // 2^15 + q2
  q[3] = and_or_f32(a, 0x0F000u, 0x45000000u) - 2048.0f;     // 2^11 + q3
  q[4] = and_or_f32(a, 0xF0000u, 0x43000000u) - 128.0f;      // 2^7  + q4
  q[5] = and_or_f32(b, 0x00F00u, 0x47000000u) - 32768.0f;
  q[6] = and_or_f32(b, 0x0F000u, 0x45000000u) - 2048.0f;
  q[7] = and_or_f32(b, 0xF0000u, 0x43000000u) - 128.0f;
}

// ---------------------------------------------------------------- single-thread issue ----
// One lane of a converged warp.  Code that issues tensor-core or bulk-copy instructions from one
// thread runs under this test rather than a lane-index test: the compiler then keeps the
// operands of that code in uniform registers, and a tcgen05.mma issue loop runs several times
// faster (measured on GB300: ~14 cycles per MMA against ~50 under `threadIdx.x == 0`).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(pred));
  return pred != 0;
}

// ---------------------------------------------------------------- shared memory / TMA ----
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Release/acquire fence at GPU scope: with an atomic between two of them it orders the writes
// before the first one ahead of the reads after the second one (cheaper than a sequentially
// consistent fence).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (bulk copy) writes to the same shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

// One bounded wait for phase `parity` of the mbarrier.  Each poll parks the thread until the
// phase completes or `kSuspendNs` pass (so a waiting warp takes no issue slots from the warps
// that compute); after `limit` polls the wait gives up and returns false.
constexpr uint32_t kSuspendNs = 20000;

// One non-blocking test: the cheap check for a phase that has most likely completed.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit,
                                          uint32_t suspend_ns = kSuspendNs) {
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done) : "r"(bar), "r"(parity), "r"(suspend_ns) : "memory");
    if (done) return true;
  }
  return false;
}

// Bulk copy global -> shared (this CTA), completing `bytes` on the mbarrier.  Both addresses
// 16-byte aligned, bytes a multiple of 16.  The weights are read once: evict-first in L2.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte read-only global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// ---------------------------------------------------------------- warp butterfly ---------
// v[0..V) per lane (V a power of two <= 32).  Afterwards lane l holds, in v[0], the sum over
// all 32 lanes of value index l / (32/V).  The additions form the same tree for every index
// (pairs of lanes at xor distance 16, then 8, ...), so the result does not depend on where a
// value sits in the array.
template <int V>
__device__ __forceinline__ void butterfly_reduce(float (&v)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
  int n = V;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      const bool upper = (lane & off) != 0;
      const int h = n >> 1;
#pragma unroll
      for (int k = 0; k < V / 2; ++k) {
        if (k < h) {
          const float send = upper ? v[k] : v[k + h];
          const float keep = upper ? v[k + h] : v[k];
          v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
}

}  // namespace q4k
