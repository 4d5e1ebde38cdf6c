// q4k_tcgen05.cuh — thin wrappers over the sm_100-family tensor-core instructions (tcgen05),
// tensor memory (TMEM) management and the shared-memory matrix descriptor.
//
// Tensor memory: 128 lanes x 512 columns of 32-bit cells per SM.  A warp of a CTA reaches the
// 32 lanes 32*(warp % 4) .. 32*(warp % 4) + 31 with the 32x32b access shape (thread t <-> lane).
// Addresses: bits [31:16] lane, bits [15:0] column.
#pragma once
#include <cstdint>

namespace q4k {
namespace tc {

// ---- allocation (one full warp executes these) -------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem_addr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem_addr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// ---- ordering between tensor-core operations and thread synchronization ------------------
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on an mbarrier when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}

// D[128 x N] (fp32, TMEM) (+)= A[128 x 16] (fp16, TMEM) * B[16 x N] (fp16, shared memory).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
      :: "r"(d_taddr), "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Eight chained MMAs D (+)= A[:, 16k..16k+15] * B[16k..16k+15, :], k = 0..7, in one statement:
// the A column address advances by 8 (16 fp16 per lane) and the B descriptor's start address by
// b_step_16 (in 16-byte units) per MMA.  accumulate_first selects whether the first one adds.
__device__ __forceinline__ void mma_f16_ts_x8(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc,
                                              uint32_t b_step_16, uint32_t idesc, uint32_t accumulate_first) {
  const uint64_t s = b_step_16;
  asm volatile(
      "{\n .reg .pred p0, p1;\n setp.ne.b32 p0, %4, 0;\n setp.eq.b32 p1, %4, %4;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %3, p1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %3, p1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %3, p1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%11], %12, %3, p1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%13], %14, %3, p1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%15], %16, %3, p1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%17], %18, %3, p1;\n}"
      :: "r"(d_taddr), "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate_first),
         "r"(a_taddr + 8), "l"(b_desc + s), "r"(a_taddr + 16), "l"(b_desc + 2 * s),
         "r"(a_taddr + 24), "l"(b_desc + 3 * s), "r"(a_taddr + 32), "l"(b_desc + 4 * s),
         "r"(a_taddr + 40), "l"(b_desc + 5 * s), "r"(a_taddr + 48), "l"(b_desc + 6 * s),
         "r"(a_taddr + 56), "l"(b_desc + 7 * s)
      : "memory");
}

// Instruction descriptor of kind::f16: fp32 accumulator, fp16 A and B, both K-major,
// M = 128 rows, N columns (N % 16 == 0, 16 <= N <= 256).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                       // D format: fp32
         | (0u << 7) | (0u << 10)        // A, B format: fp16
         | (0u << 15) | (0u << 16)       // A, B K-major
         | (uint32_t(N >> 3) << 17)      // N / 8
         | (uint32_t(M >> 4) << 24);     // M / 16
}

// Shared-memory descriptor of a K-major operand without swizzle.  The operand is stored as
// 8-row x 16-byte "core matrices" (128 contiguous bytes each); `lbo` is the byte distance
// between core matrices adjacent along K, `sbo` between core matrices adjacent along the
// other (row) dimension.
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo & 0x3FFFFu) >> 4) << 16;
  d |= uint64_t((sbo & 0x3FFFFu) >> 4) << 32;
  d |= uint64_t(1) << 46;                // descriptor version for the sm_100 family
  // base offset 0, absolute LBO mode 0, layout type 0 (no swizzle)
  return d;
}

// ---- register <-> TMEM copies (32x32b shape: thread t of the warp <-> its lane) -----------
__device__ __forceinline__ void st_x2(uint32_t taddr, uint32_t a, uint32_t b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" :: "r"(taddr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                  "r"(v[7]) : "memory");
}

__device__ __forceinline__ void st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
         "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Columns 2j and 2j+1 both take v[j] (j = 0..7).
__device__ __forceinline__ void st_x16_pairs(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %1, %2, %2, %3, %3, %4, %4, %5, %5, %6, %6, %7, %7, %8, %8};"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void ld_x8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr) : "memory");
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(r[k]);
}

__device__ __forceinline__ void ld_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(r[k]);
}

__device__ __forceinline__ void ld_x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
}

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace q4k
