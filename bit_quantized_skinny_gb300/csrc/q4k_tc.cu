// q4k_tc.cu — tensor-core (tcgen05) variant of the skinny product of packed weights x bf16
// activations (sm_103a): Q4K, and through the FMT template the other weight formats (Q5K, Q6K,
// NVFP4, INT4 with one scale per 128 columns; their decode steps are in q4k_formats.cuh).
//
// The skinny product of the pages' verify pass ("sixi-asi 0.9", section "What I got wrong in
// 0.8") is a weight stream: every weight is read once and used by M <= 32 activation rows.  On
// CUDA cores each weight costs one logic op, one subtraction and M fused multiply-adds; here the
// M multiplies go to the tensor cores and the per-weight CUDA-core work drops to about one
// instruction per pair of weights, the same for every M.  That is the M-dependent tiling of the
// pages (a matrix kernel from a few rows on, section "The patch") done with GB300's units.
//
// Operands ("swap AB": the 128-row MMA dimension runs over weight rows), described for Q4K:
//   A[128 rows x 16 k] fp16 in tensor memory (TMEM): A = (sc_j q_t - k_j) 2^-14 with the min
//     term folded in (k_j = rint(m_j Dm / D), see Fold below): an integer times 2^-14, exact,
//     and exactly zero for a weight that is exactly zero.  Written by the dequant warps with
//     tcgen05.st, one thread per weight row (lane).
//   B[16 k x Mpad] fp16 in shared memory: the activations of one super-block, x * 2^-s_i with one
//     power of two per token i so that its bf16 values are exact in fp16 (see the preparation).
//   D[128 x Mpad] fp32 in TMEM, one accumulator per 256-weight super-block.
//   Two more K=16 MMAs per super-block multiply A_ext (the fp16 pair (hi, lo) of the residual
//   rho_j T of each sub-block, twice) with B_ext (the fp16 pair of the sub-block sums of x as
//   rows (hi, hi, lo, lo)): the residual of the min term also comes from the tensor cores.  The
//   epilogue forms, per super-block and token i,
//     y_i += sigma_i (D acc_i + f_e acc_ext_i),   sigma_i = 2^(s_i + 14), f_e = -2^(e - 16)
//   in fp32 registers.  Products in the MMAs are exact; only fp32 accumulation rounds.
//   The other formats keep A exact in fp16 too (Q5K sc*q - k <= 1953; Q6K sc*(q-32) <= 2048 with
//   7-bit scales; NVFP4 s*v, at most 6 significant bits; INT4 q itself) and differ in the
//   epilogue: NVFP4 and Q6K have one accumulator (factor g 2^-14 or d 2^-14), INT4 one per K half
//   (its two scale groups), Q5K the Q4K pair.
//
// K order inside a super-block: the nibble masks below yield the quants of one 32-bit word as
// fp16 pairs (q0,q4) (q1,q5) (q2,q6) (q3,q7); TMEM column 4w+c holds k = 8w+c (low half) and
// 8w+c+4 (high half), and the activations are laid out in B with the same permutation.
//
// Work: a task is one 128-row tile of one product over a range of its super-blocks (a K split).
// A launch's tasks are dealt to its (dequant group, CTA) slots in back-and-forth rounds.
// Summation order: a row's super-blocks are summed in chunks of 4 (each chunk from zero, in order
// of k) and the chunk sums are added in chunk order; splits cut only at chunk boundaries, so a
// product's bits depend neither on M nor on how its work is split or batched.  One CTA per SM.
//
// Roles (512 threads; 352 for INT4 at 32 token columns):
//   dequant groups (3; 2 for INT4 at 32 token columns, whose groups own two accumulator blocks
//                next to the slot; 4 warps each, warp q <-> TMEM lanes
//                32q..32q+31, the rows of the tile).  Each group owns one A slot and its
//                accumulators in TMEM and walks its tasks' super-blocks, software-pipelined:
//                while the MMAs of super-block i run it waits for the stage of i+1 and takes its
//                header, per-token scales and hard-token mask; then it reads i's accumulator and
//                decodes i+1 one K half at a time, each half handed to its MMA warp as soon as it
//                is written; hard tokens (see the preparation) are summed on CUDA cores just
//                before the stage is released.
//   copy warp    per super-block one 2D TMA tile copy of the weights (128 rows x the format's
//                bytes per 256 weights) and one bulk copy of the prepared activation block into
//                a stage of the ring (8 stages for 8 token columns, 7 for 16, 4 or 5 for 32; fewer
//                for the wider formats), in the CTA's super-block order (rounds over the groups).
//                The first ring's weights are requested before the preparation grid finishes.
//   MMA warps    one per group (the first owns TMEM); one elected lane issues its group's MMAs
//                (8 per K half, and two for the min term of the k-quants) and commits them to the
//                group's completion barrier and the stage's empty barrier.  Issuing from an
//                elect.sync branch keeps the operands in uniform registers (~14 cycles per MMA).
// Every barrier is waited on only by threads that see all of its phases in order (a parity wait
// is exact only then): full barriers per (group, stage), handoff and completion barriers per
// group.  Every wait is bounded; on timeout the kernel records an error in the status word, the
// other roles stop at their next wait, and in-flight copies and MMAs are waited for before the
// CTA ends.
//
// Split K (single products with few tiles): a split task stores its chunk sums to a per-call
// workspace; the last split of a (tile, lane quarter) slice to finish (an atomic counter per
// slice, zeroed by the preparation kernel of the same call) adds all chunk sums of the tile in
// chunk order and writes Y.
//
// Activation preparation (q4k_xprep_kernel, one CTA per super-block of each distinct X): per
// token a power of two s_i that puts its largest |x| in [2^14, 2^15); B, B_ext, sigma_i and a
// trailer (hard-token mask, K, the address of X) go to a per-stream workspace.  A token whose
// staging would not be exact (a value below fp16's range after scaling, or a sub-block sum too
// small for its (hi, lo) pair) is "hard": its B and B_ext rows are zero and the product kernel
// computes its part of that super-block from X on CUDA cores.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4k_device.cuh"
#include "q4k_formats.cuh"
#include "q4k_internal.h"
#include "q4k_tcgen05.cuh"

namespace q4k {


namespace {

__device__ unsigned g_status;   // this file's kernels' status word

constexpr int kTileRows = 128;
constexpr int kGroupWarps = 4;     // a dequant group: one warp per TMEM lane quarter (32 rows)
constexpr int kMaxGroups = 3;
// The formats with one accumulator block per group (no dmin term, one scale group per
// super-block).
__host__ __device__ constexpr bool single_acc(int f) { return f == kFmtNVFP4 || f == kFmtQ6K; }
__host__ __device__ constexpr bool has_min(int f) { return f == kFmtQ4K || f == kFmtQ5K; }
// Dequant groups (NG): three at Mpad 16 and for NVFP4 and Q6K at Mpad 32; two for INT4 at Mpad 32
// (what tensor memory holds, below); two or three for the k-quants at Mpad 32, chosen per launch
// (`wide`): three stream long task lists faster, two (with more stages: the running sums of
// fewer groups leave more shared memory) finish short, split products sooner.  With the copy
// warp and one MMA warp per group that is 16 warps (11 for two groups), four per SM
// sub-partition, which leaves each thread 128 registers (a sub-partition holds 16384; 168 with
// two groups).
__host__ __device__ constexpr int groups(int mpad, int f = kFmtQ4K, bool wide = true) {
  return (mpad <= 16 || single_acc(f)) ? 3 : ((has_min(f) && wide) ? 3 : 2);
}
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 17;
constexpr int kMaxEBatch = 160;    // products per batched launch (their tensor maps ride in the parameters)
constexpr int kMaxPrep = 512;      // distinct activations per preparation launch
constexpr int kSmemLimit = 232448; // shared memory per CTA (227 KB)

// Bytes of one row's 256 weights in the streamed weight plane (one TMA box column), per format:
// Q4K and NVFP4 144 (NVFP4: 16 E4M3 scales + 128 bytes of codes), Q5K 176, Q6K 208, INT4 128
// (INT4's scales and Q6K's super-block scales live in separate planes).  The min term (an extra
// MMA pair and a second accumulator column block) belongs to Q4K and Q5K only.
__host__ __device__ constexpr int blk_bytes(int f) {
  return f == kFmtQ5K ? 176 : (f == kFmtQ6K ? 208 : (f == kFmtINT4 ? 128 : 144));
}
__host__ __device__ constexpr int w_stage_bytes(int f) { return kTileRows * blk_bytes(f); }

// Prepared activation block of one super-block (bblock_bytes(TW) bytes, written by the
// preparation kernel, read by the product kernel from a stage of its ring).  TW, the token
// columns it stores, is MPAD, except for the 8-token kernels (M <= 8), whose MMAs (N = 16) take
// token columns 8..15 of B and 0..7 of B_ext from zero regions of shared memory: their blocks
// hold 8 columns (TW = 8, half the bytes of every copy).  With MPAD read as TW:
//   [0, MPAD*512)         B: the 256 activations of every token column i as fp16 x * 2^-s_i,
//                         K-major core matrices (8 tokens x 8 k, 128 bytes; 32 of them along k
//                         per group of 8 tokens: 4096 bytes)
//   [MPAD*512, MPAD*576)  B_ext: 32 rows per token, sub-block j's activation sum X_j * 2^(-s_i-6)
//                         as an fp16 pair (hi, lo): rows 4j .. 4j+3 = (hi, hi, lo, lo)
//                         (8 tokens x 4 core matrices: 512 bytes per group of 8 tokens)
//   [MPAD*576, MPAD*580)  sigma_i = 2^(s_i + 14) per token column, fp32
//   [MPAD*580, +16)       the mask of "hard" tokens (bit i), K, and the address of X (8 bytes)
// A hard token's staging would not be exact (see q4k_xprep_kernel); its B and B_ext rows are
// zero (its accumulator columns come out exactly 0) and the product kernel computes its part of
// the super-block from X itself.
__host__ __device__ constexpr int bext_off(int mpad) { return mpad * 512; }
__host__ __device__ constexpr int sig_off(int mpad) { return mpad * 576; }
__host__ __device__ constexpr int mask_off(int mpad) { return mpad * 580; }
__host__ __device__ constexpr int bblock_bytes(int mpad) { return mpad * 580 + 16; }
// A stage holds one super-block of a tile (the weight rows) and the prepared activation block
// of the same super-block: both arrive on one barrier, issued the same distance ahead.
// (rounded up to 128 bytes: a TMA tile copy writes to a 128-byte aligned address; INT4 tiles
// are copied with the 128-byte swizzle, whose destination is 1024-byte aligned)
__host__ __device__ constexpr int stage_bytes(int mpad, int f) {
  return f == kFmtINT4 ? (w_stage_bytes(f) + bblock_bytes(mpad) + 1023) / 1024 * 1024
                       : (w_stage_bytes(f) + bblock_bytes(mpad) + 127) / 128 * 128;
}
constexpr int kMaxStages = 9;
// TMEM columns.  Each group owns one A slot (one super-block: 64 columns of fp16 pairs per K
// half) and one accumulator block at the top of the 512 columns.
//   k-quants (Q4K, Q5K) have the min-term MMAs: A_ext, 16 columns (K = 32), after the slot's
//   128 columns.  With 8 token columns (M <= 8) the min-term MMAs accumulate into columns 8..15
//   of the product's own 16-column accumulator (their B_ext has the tokens in columns 8..15,
//   the product's B zeros there).  With 16 or 32 token columns the min term's accumulator lives
//   in the slot itself, in columns 16..15+Mpad: the min-term MMAs are issued only after the first
//   K half's MMAs (the slot's readers of those columns) have completed (their own commit), and
//   the group reads that accumulator before it writes the slot again.  With 32 token columns
//   A_ext too reuses the slot's first 16 columns, written by the group after that same commit.
//   Each group has its own MMA warp (with one MMA warp for all groups, a group waiting for its
//   first half's MMAs would hold up the other groups' MMAs, issued in order).
//   INT4: two accumulators (one per K half, its two scale groups); NVFP4, Q6K: one.
//     Q4K, Q5K   8 tokens: 3 x (144 + 16) = 480;  16 tokens: 3 x (144 + 16) = 480;  Mpad 32: 3 x (128 + 32)
//     INT4       3 x (128 + 32) = 480 at Mpad 16;  2 x (128 + 64) at Mpad 32
//     NVFP4, Q6K 3 x (128 + Mpad): 432 / 480
__host__ __device__ constexpr bool ext_in_a(int f, int mt, int ng) { return has_min(f) && mt == 32 && ng == 3; }
__host__ __device__ constexpr bool acc_in_a(int f, int mt, int ng) { return has_min(f) && (mt == 16 || (mt == 32 && ng == 3)); }
__host__ __device__ constexpr uint32_t acols(int f, int mt, int ng) { return (has_min(f) && !ext_in_a(f, mt, ng)) ? 144u : 128u; }
// MMA-issuing warps: one per group.  (With one MMA warp serving the groups in order, its wait
// for one group's handoff held up the MMAs of the others: measured on GB300 with clock stamps,
// the groups then advanced one at a time.)
// Threads of a CTA: the dequant groups, the copy warp and one MMA warp per group.
__host__ __device__ constexpr int cta_threads(int ng) { return 32 * (ng * kGroupWarps + 1 + ng); }
// Summation order of a product: the super-blocks of a row are summed in chunks of kChunkSb (each
// chunk from zero, in order of k), and the chunk sums are then added in chunk order.  A K split
// only ever cuts at chunk boundaries, so the bits of a product do not depend on the split.
constexpr int kChunkSb = 4;
__host__ __device__ constexpr uint32_t a_col(int g, int f, int mt, int ng) { return acols(f, mt, ng) * g; }
__host__ __device__ constexpr uint32_t acc_cols(int mpad, int f, int mt, int ng) {
  return single_acc(f) ? mpad : ((has_min(f) && (mt == 8 || acc_in_a(f, mt, ng))) ? mpad : 2u * mpad);
}
__host__ __device__ constexpr uint32_t acc1_col(int mpad, int g, int f, int mt, int ng) {
  return 512u - acc_cols(mpad, f, mt, ng) * ng + acc_cols(mpad, f, mt, ng) * g;
}
__host__ __device__ constexpr uint32_t acc2_col(int mpad, int g, int f, int mt, int ng) {
  return acc_in_a(f, mt, ng) ? a_col(g, f, mt, ng) + 16u : acc1_col(mpad, g, f, mt, ng) + mpad;
}
__host__ __device__ constexpr bool tmem_fits(int mpad, int f, int mt, int ng) {
  return a_col(ng, f, mt, ng) <= acc1_col(mpad, 0, f, mt, ng);
}
static_assert(tmem_fits(16, kFmtQ4K, 8, 3) && tmem_fits(16, kFmtQ4K, 16, 3) && tmem_fits(32, kFmtQ4K, 32, 3) &&
              tmem_fits(32, kFmtQ4K, 32, 2) && tmem_fits(16, kFmtINT4, 8, 3) && tmem_fits(16, kFmtINT4, 16, 3) &&
              tmem_fits(32, kFmtINT4, 32, 2) && tmem_fits(16, kFmtNVFP4, 16, 3) && tmem_fits(32, kFmtNVFP4, 32, 3) &&
              tmem_fits(32, kFmtQ6K, 32, 3), "TMEM column plan overlaps");

// Barrier indices inside the barrier block.  Every barrier is waited on by threads that see
// all of its phases in order (a parity wait is only exact then):
//   GFull[g][s]  stage s holds a super-block of group g (copies landed); group g, MMA lane
//   WEmpty[s]    stage s consumed (the group's 4 warps + the MMA commit); copy lane
//   AFull[g][h]  K half h of group g's A slot written; MMA lane
//   H0Done[g]    the first K half's MMAs of group g's latest super-block completed; group g
//                where A_ext reuses the first K half's columns (32 token columns), else the MMA
//                lane before the min-term MMAs that write into those columns (16)
//   GDone[g]     the MMAs of group g's latest super-block completed; group g
//   Drain        the last MMAs of the CTA completed; MMA lane
enum : int {
  kBarGFull = 0, kBarWEmpty = kBarGFull + kMaxGroups * kMaxStages,
  kBarAFull = kBarWEmpty + kMaxStages, kBarGDone = kBarAFull + 2 * kMaxGroups,
  kBarH0Done = kBarGDone + kMaxGroups, kBarDrain = kBarH0Done + kMaxGroups,
  kNumBars = kBarDrain + kMaxGroups
};

// The 8-token kernels keep two zero regions: 1024 bytes before the stages (token columns 0..7 of
// the min-term operand B_ext; 1024 keeps the stages 1024-byte aligned) and 4096 bytes after them
// (token columns 8..15 of B).  An MMA's B descriptor reaches the second group of 8 token columns
// at its start + SBO, so a stage's descriptor points there with SBO = zero region - stage
// (forwards for B) or starts in the zero region with SBO = stage - zero region (B_ext).
constexpr int kZeroExtBytes = 1024;
constexpr int kZeroMainBytes = 4096;
__host__ __device__ constexpr int token_width(int mpad, int mt) { return mt == 8 ? 8 : mpad; }
// With 16 or 32 token columns each group's running sum of chunk sums (MT tokens x 128 rows of
// fp32) lives in shared memory, not in registers (there it spilled); it is touched once per
// chunk of 4 super-blocks.
__host__ __device__ constexpr int ytot_bytes(int mt, int ng) { return mt >= 16 ? ng * mt * kTileRows * 4 : 0; }
// Each dequant warp keeps its own copy of the current super-block's per-token scales (the stage
// that brought them is released before the epilogue needs them): 32 floats for each of the
// two super-blocks in flight, per warp.
constexpr int kSigBytes = kMaxGroups * kGroupWarps * 64 * 4;
// Stages: 9 for 8 tokens, 8 at Mpad 16 and 5 at Mpad 32, or as many as fit beside the rest (7
// for 16 tokens, 4 for 32 with three groups' running sums in shared memory).
__host__ __device__ constexpr int zero_bytes(int mt) { return mt == 8 ? kZeroExtBytes + kZeroMainBytes : 0; }
__host__ __device__ constexpr int stages_fit(int mpad, int f, int mt, int ng) {
  return (kSmemLimit - zero_bytes(mt) - ytot_bytes(mt, ng) - kSigBytes - kNumBars * 8 - 32) /
         stage_bytes(token_width(mpad, mt), f);
}
__host__ __device__ constexpr int stage_cap(int mpad, int mt) { return mt == 8 ? 9 : (mpad <= 16 ? 8 : 5); }
__host__ __device__ constexpr int stages(int mpad, int f, int mt, int ng) {
  return stages_fit(mpad, f, mt, ng) < stage_cap(mpad, mt) ? stages_fit(mpad, f, mt, ng) : stage_cap(mpad, mt);
}

template <int MPAD, int FMT, int MT, int NG>
struct TcSmem {
  static constexpr int kZeroExt = 0;                                   // 8 tokens only
  static constexpr int kW = MT == 8 ? kZeroExtBytes : 0;
  static constexpr int kZeroMain = kW + stages(MPAD, FMT, MT, NG) * stage_bytes(token_width(MPAD, MT), FMT);
  static constexpr int kYtot = kZeroMain + (MT == 8 ? kZeroMainBytes : 0);
  static constexpr int kSig = kYtot + ytot_bytes(MT, NG);
  static constexpr int kBars = kSig + kSigBytes;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kTotal = kMisc + 32;   // TMEM address, abort flag, super-blocks per group (<= 4)
};
template <int FMT>
constexpr bool smem_fits() {
  return TcSmem<16, FMT, 8, 3>::kTotal <= kSmemLimit && TcSmem<16, FMT, 16, 3>::kTotal <= kSmemLimit &&
         TcSmem<32, FMT, 32, groups(32, FMT, false)>::kTotal <= kSmemLimit &&
         TcSmem<32, FMT, 32, groups(32, FMT, true)>::kTotal <= kSmemLimit;
}
static_assert(smem_fits<kFmtQ4K>() && smem_fits<kFmtQ5K>() && smem_fits<kFmtNVFP4>() && smem_fits<kFmtINT4>() &&
              smem_fits<kFmtQ6K>(), "shared memory");
static_assert(stages(16, kFmtQ4K, 8, 3) == 9 && stages(16, kFmtQ4K, 16, 3) == 7 && stages(32, kFmtQ4K, 32, 3) == 4 &&
              stages(32, kFmtQ4K, 32, 2) == 5 && stages(16, kFmtQ5K, 16, 3) >= 4 && stages(32, kFmtQ5K, 32, 3) >= 3 &&
              stages(32, kFmtINT4, 32, 2) >= 3 && stages(16, kFmtQ6K, 16, 3) >= 4 && stages(32, kFmtQ6K, 32, 3) >= 3,
              "stage counts");
static_assert(groups(16) <= kMaxGroups && groups(32) <= kMaxGroups, "group barriers");
static_assert(stage_bytes(16, kFmtQ4K) % 128 == 0 && stage_bytes(32, kFmtQ5K) % 128 == 0 &&
              stage_bytes(16, kFmtINT4) % 1024 == 0 && w_stage_bytes(kFmtQ5K) % 128 == 0 &&
              bblock_bytes(8) % 16 == 0 && bblock_bytes(16) % 16 == 0 && bblock_bytes(32) % 16 == 0 &&
              stage_bytes(8, kFmtQ4K) % 128 == 0 && stage_bytes(8, kFmtINT4) % 1024 == 0, "stage alignment");

struct TcEntry {
  float* Y;
  const uint8_t* B;    // prepared activation blocks of this entry's X
  float* partial;      // split > 1: tiles x chunks x Mpad x 128 chunk partial sums
  unsigned* counters;  // split > 1: tiles x 4 arrival counters (zeroed by the preparation)
  int N;
  int K;
  int tiles;
  int splits;          // K splits per tile
  int chunk;           // super-blocks per split, a multiple of kChunkSb (the last may have fewer)
  int chunks;          // summation chunks per row: ceil(K/256 / kChunkSb)
  int task_begin;
};

// Launch parameters: the weights of entry e are reached through maps[e], a 2D tensor map over
// the packed rows (inner dimension: the row's bytes, outer: the N rows).  aux[e]: what entry e
// keeps outside its row blocks (NVFP4: the fp32 tensor scale; INT4: the N x K/128 binary16 scale
// plane; Q6K: the N x K/256 binary16 d plane); Q4K has none (one unused slot).  Kept out of
// TcEntry: the Q4K kernel measured ~1.5 % slower with a different entry layout.
template <int MAXE, int NAUX>
struct TcParams {
  CUtensorMap maps[MAXE];
  TcEntry e[MAXE];
  int count;
  int M;
  int tasks_total;
  int gated;   // one product whose row pairs (2f, 2f+1) are (gate f, up f): Y holds bf16 H[M x N/2]
  uint32_t wait_polls;   // bound of the pipeline waits: polls (0: kWaitLimit) of at most
  uint32_t wait_ns;      // wait_ns each (0: kSuspendNs); set only by the failure-detection hook
  const void* aux[NAUX];
};
__host__ __device__ constexpr int naux(int f, int maxe) { return f == kFmtQ4K ? 1 : maxe; }

struct PrepEntry {
  const uint16_t* X;
  uint8_t* out;
  int K;
  int block_begin;   // first CTA index of this X
};

template <int NX>   // capacity: distinct activations of one preparation launch
struct PrepParams {
  int count;
  int M;
  int blocks_total;
  int zero_words;      // split counters of the main launches of this call, zeroed here
  unsigned* zero;
  PrepEntry e[NX];
};

__device__ __forceinline__ uint32_t h2bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 bits2h(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// ------------------------------------------------------------------------------------------
// Activation preparation.  Block = 8*MPAD threads; thread (i = t/8, j = t%8) handles token i,
// sub-block j (32 activations) of one super-block; the 8 threads of a token are 8 neighbouring
// lanes of one warp.
//
// Every token has its own power of two: s_i puts the largest |x| of its 256 activations in
// [2^14, 2^15) (s_i in [-112, 113]).  The token is staged exactly when
//   (a) every x * 2^-s_i is an fp16 value (true unless x is below about 2^-31 of that largest
//       value, or the largest value is a bf16 subnormal far below 2^-112), and
//   (b) every sub-block j with a nonzero activation has sum_t |x_t * 2^-s_i| >= 1/4: then the
//       fp16 pair (hi, lo) that carries X_j * 2^(-s_i-6) is within 2^-19 of sum_t |x_t|.
// Otherwise the token is "hard": its B and B_ext rows are zeros, and the product kernel computes
// its outputs for this super-block on CUDA cores in fp32 from X.
// B pairs are in the order of the weight decode: (x_c, x_c+4), c = 0..3, of each 8-activation
// word, or with NAT (NVFP4) the natural (x_2c, x_2c+1).
template <int MPAD, int NX, bool NAT>
__global__ void __launch_bounds__(8 * MPAD) q4k_xprep_kernel(const __grid_constant__ PrepParams<NX> P) {
  // the product kernel that follows may start its prologue now (programmatic dependent launch);
  // it waits for this grid's completion before it reads what this grid writes.  This grid itself
  // is launched in plain stream order: everything before it is complete, so the product's early
  // weight copies read finished data.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ unsigned s_hard[8 * MPAD / 32];
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
  const int lane = t & 31;
  for (int z = b * (8 * MPAD) + t; z < P.zero_words; z += P.blocks_total * (8 * MPAD)) P.zero[z] = 0u;
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
  // the token's largest |x| (bit pattern of |x|: larger patterns are larger values)
  unsigned mx = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t w4[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) mx = max(mx, max(w4[h] & 0x7FFFu, (w4[h] >> 16) & 0x7FFFu));
  }
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
  // largest |x| in [2^(E-127), 2^(E-126)), E = its biased exponent; scale it into [2^14, 2^15)
  int s = 0;
  if (mx != 0) s = min(113, max(-112, (int)(mx >> 7) - 141));
  const float f = __uint_as_float((uint32_t)(127 - s) << 23);    // 2^-s
  const float fs = __uint_as_float((uint32_t)(127 + s) << 23);   // 2^s

  uint32_t packed[4][4];
  float xsum = 0.f, asum = 0.f;
  bool exact = true;
#pragma unroll
  for (int ww = 0; ww < 4; ++ww) {
    const uint32_t w4[4] = {v[ww].x, v[ww].y, v[ww].z, v[ww].w};
    float xv[8];   // the word's 8 activations in order of k
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      xv[2 * h] = __uint_as_float(w4[h] << 16);
      xv[2 * h + 1] = __uint_as_float(w4[h] & 0xFFFF0000u);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float xa = NAT ? xv[2 * c] : xv[c];
      const float xb = NAT ? xv[2 * c + 1] : xv[c + 4];
      const __half2 hh = __floats2half2_rn(xa * f, xb * f);
      const float2 back = __half22float2(hh);
      exact = exact && (back.x * fs == xa) && (back.y * fs == xb);
      packed[ww][c] = h2bits(hh);
      xsum += back.x + back.y;
      asum += fabsf(xa * f) + fabsf(xb * f);
    }
  }
  const bool bad = !exact || (asum > 0.f && asum < 0.25f);
  const unsigned ballot = __ballot_sync(0xffffffffu, bad);
  const bool hard = valid && ((ballot >> (lane & 24)) & 0xFFu) != 0u;

  uint8_t* out = E.out + (int64_t)sb * bblock_bytes(MPAD);
#pragma unroll
  for (int ww = 0; ww < 4; ++ww) {
    const int w = 4 * j + ww;  // word (8 activations) index within the super-block
    uint4* dst = reinterpret_cast<uint4*>(out + ((i >> 3) * 32 + w) * 128 + (i & 7) * 16);
    *dst = hard ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(packed[ww][0], packed[ww][1], packed[ww][2], packed[ww][3]);
  }
  // B_ext: rows 4j .. 4j+3 of token column c = (hi, hi, lo, lo)
  const float xs = xsum * 0.015625f;  // 2^-6: a sum of 32 values below 2^15 stays below 2^14
  const __half hi = __float2half_rn(xs);
  const __half lo = __float2half_rn(xs - __half2float(hi));
  const uint32_t hb = __half_as_ushort(hi), lb = __half_as_ushort(lo);
  const uint2 ev = hard ? make_uint2(0u, 0u) : make_uint2(hb * 0x10001u, lb * 0x10001u);
  uint8_t* ext = out + bext_off(MPAD);
  auto ext_at = [&](int c) { return reinterpret_cast<uint2*>(ext + (c >> 3) * 512 + (j >> 1) * 128 + (c & 7) * 16 + (j & 1) * 8); };
  *ext_at(i) = ev;
  float* sig = reinterpret_cast<float*>(out + sig_off(MPAD));
  if (j == 0) sig[i] = __uint_as_float((uint32_t)(127 + 14 + s) << 23);   // 2^(s+14)
  const unsigned bits = __reduce_or_sync(0xffffffffu, (hard && j == 0) ? (1u << i) : 0u);
  if (lane == 0) s_hard[t >> 5] = bits;
  __syncthreads();
  if (t == 0) {
    unsigned m = 0;
#pragma unroll
    for (int w = 0; w < (8 * MPAD) / 32; ++w) m |= s_hard[w];
    const uint64_t xa = reinterpret_cast<uint64_t>(E.X);
    *reinterpret_cast<uint4*>(out + mask_off(MPAD)) = make_uint4(m, (uint32_t)E.K, (uint32_t)xa, (uint32_t)(xa >> 32));
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

// The last split of a (tile, lane quarter) slice: this thread's row of the tile, the sum of
// every chunk partial in chunk order, tokens below M, to y (nullptr: the row is past N).  Out of
// line: it runs once per split tile and would otherwise take registers from the hot loop.
template <int MPAD, int MT>
__device__ __noinline__ void reduce_chunks(const float* part, int chunks, int M, float* y, int N) {
  constexpr int kB = MT >= 32 ? 1 : (MT >= 16 ? 2 : 4);   // chunk partials loaded together (added in chunk order)
  float v[MT];
#pragma unroll
  for (int k = 0; k < MT; ++k) v[k] = (k < M) ? __ldcg(&part[k * kTileRows]) : 0.f;
  int ch = 1;
  for (; ch + kB <= chunks; ch += kB) {
    float t[kB][MT];
#pragma unroll
    for (int c = 0; c < kB; ++c)
#pragma unroll
      for (int k = 0; k < MT; ++k) t[c][k] = (k < M) ? __ldcg(&part[((size_t)(ch + c) * MPAD + k) * kTileRows]) : 0.f;
#pragma unroll
    for (int c = 0; c < kB; ++c)
#pragma unroll
      for (int k = 0; k < MT; ++k) v[k] = v[k] + t[c][k];
  }
  for (; ch < chunks; ++ch) {
#pragma unroll
    for (int k = 0; k < MT; ++k)
      if (k < M) v[k] = v[k] + __ldcg(&part[((size_t)ch * MPAD + k) * kTileRows]);
  }
  if (y) {
#pragma unroll
    for (int k = 0; k < MT; ++k)
      if (k < M) y[(int64_t)k * N] = v[k];
  }
}

// The feed-forward gating of a finished task whose running sums are in shared memory (token k
// of this thread's row at ysum[k * 128]): lanes r and r ^ 1 hold rows 2f (gate) and 2f+1 (up);
// the even lane stores bf16(silu(gate) * up) to H[k][f], silu(g) = g / (1 + e^-g), fp32 then
// one round to nearest even.  Out of line: it runs once per task and would otherwise take
// registers from the hot loop.
template <int MT>
__device__ __noinline__ void gate_store_smem(const float* ysum, int r, int row, int N, int M, uint16_t* H) {
  const int64_t F = N >> 1;
  for (int k = 0; k < MT; ++k) {
    const float mine = ysum[k * kTileRows];
    const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
    if (k < M && !(r & 1) && row < N) {
      const float h = mine / (1.0f + expf(-mine)) * other;
      const __nv_bfloat16 hb = __float2bfloat16_rn(h);
      H[(int64_t)k * F + (row >> 1)] = *reinterpret_cast<const uint16_t*>(&hb);
    }
  }
}

// Task t of the launch: its entry, tile and K split, and its super-block range.
template <class PT>
struct TaskView {
  int e, tile, split, sb0, sb1;
  __device__ __forceinline__ TaskView(const PT& P, int t) {
    int lo = 0, hi = P.count - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (P.e[mid].task_begin <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const TcEntry& E = P.e[e];
    const int u = t - E.task_begin;
    tile = u / E.splits;
    split = u - tile * E.splits;
    sb0 = split * E.chunk;
    sb1 = min(E.K >> 8, sb0 + E.chunk);
  }
};

// Walk over the tasks of one dequant group.  The launch's tasks are dealt to the NG x gridDim.x
// (group, CTA) slots in rounds, slot s = g * gridDim.x + blockIdx.x taking task r * S + s in even
// rounds r and r * S + (S - 1 - s) in odd ones (S slots; the host orders a launch's products by
// decreasing K, so the back-and-forth order evens out the slots' work); each super-block of each
// task in order.
template <class PT, int NG>
struct GroupCursor {
  int r, slot, t, e, tile, split, sb, end;
  __device__ __forceinline__ void load(const PT& P) {
    const int S = NG * (int)gridDim.x;
    t = r * S + ((r & 1) ? S - 1 - slot : slot);
    if (t >= P.tasks_total) { t = -1; return; }
    const TaskView<PT> T(P, t);
    e = T.e; tile = T.tile; split = T.split; sb = T.sb0; end = T.sb1;
  }
  __device__ __forceinline__ void start(const PT& P, int g) {
    r = 0;
    slot = g * (int)gridDim.x + (int)blockIdx.x;
    load(P);
  }
  // after the current super-block: true if it was the last of its task
  __device__ __forceinline__ bool advance(const PT& P) {
    if (++sb < end) return false;
    ++r;
    load(P);
    return true;
  }
};

// The CTA's super-block sequence su = 0, 1, ... runs in rounds: round i takes the i-th
// super-block of every group that has one, in group order.  With n_g super-blocks in group g,
// the i-th super-block of group g is
//   su = sum_h min(n_h, i) + #{h < g : n_h > i}.
template <int NG>
__device__ __forceinline__ uint32_t su_of(const int (&n)[NG], int g, int i, int nmin) {
  if (i < nmin) return (uint32_t)(NG * i + g);   // every group still has a super-block in round i
  uint32_t s = 0;
#pragma unroll
  for (int h = 0; h < NG; ++h) s += (uint32_t)min(n[h], i) + ((h < g && n[h] > i) ? 1u : 0u);
  return s;
}

// Weight decode of one K half (128 weights of a row) of each format into the A slot of TMEM.
// Inputs: the row's block in the stage at `rb`, its first 16 bytes `hd`, the half h; the A
// columns of the half at `aaddr`.  The quant words are read from shared memory before the
// caller releases the stage (the `in` structure), then decoded and stored with tcgen05.st.
template <int FMT>
struct HalfIn {
  uint4 qv[4];   // quants of the half: 16 bytes per 32 weights
  uint4 hb;      // Q5K: the high-bit words of the half's four sub-blocks
  uint4 hv[2];   // Q6K: the high-part words of the half's eight sub-blocks
};

// INT4 tiles are copied with the 128-byte swizzle: 16-byte chunk c of row r sits at chunk
// c ^ (r % 8) of the row (spreads the rows' reads over all shared-memory banks).  The stage is
// 1024-byte aligned and a row is 128 bytes, so r % 8 is bits 7..9 of the row's address rb:
// chunk c is at (rb ^ ((rb >> 3) & 0x70)) ^ 16c.
template <int FMT>
__device__ __forceinline__ void load_half(HalfIn<FMT>& in, uint32_t rb, int h) {
  if constexpr (FMT == kFmtINT4) {
    const uint32_t rbs = rb ^ ((rb >> 3) & 0x70u);
#pragma unroll
    for (int k = 0; k < 4; ++k) in.qv[k] = lds128(rbs ^ (uint32_t)(16 * (4 * h + k)));
  } else if constexpr (FMT == kFmtQ5K) {
#pragma unroll
    for (int k = 0; k < 4; ++k) in.qv[k] = lds128(rb + 48 + 64 * h + 16 * k);
    in.hb = lds128(rb + 16 + 16 * h);
  } else if constexpr (FMT == kFmtQ6K) {
#pragma unroll
    for (int k = 0; k < 4; ++k) in.qv[k] = lds128(rb + 16 + 64 * h + 16 * k);
    in.hv[0] = lds128(rb + 144 + 32 * h);
    in.hv[1] = lds128(rb + 144 + 32 * h + 16);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) in.qv[k] = lds128(rb + 16 + 64 * h + 16 * k);
  }
}

// fp16 constants of the decodes, made once per thread (outside the super-block loop)
struct DecodeConsts {
  __half2 k1024, kn1024, k64, k1o16, kn1032, kn72;
  __device__ __forceinline__ DecodeConsts()
      : k1024(bits2h(0x64006400u)), kn1024(bits2h(0xE400E400u)), k64(__float2half2_rn(64.f)),
        k1o16(__float2half2_rn(0.0625f)), kn1032(__float2half2_rn(-1032.f)), kn72(__float2half2_rn(-72.f)) {}
};

// The k-quants' min term, folded into the operands.  Weight t of sub-block j is
//   w_t = D sc_j q_t - Dm m_j = D (sc_j q_t - k_j) - rho_j,   rho_j = Dm m_j - D k_j,
// for any integer k_j.  With k_j = rint(m_j Dm / D) clamped to [0, 2047] (0 when Dm / D < 0):
//   * A_t = sc_j q_t - k_j is an integer in [-2047, 1953]: exact in fp16 (written as A_t 2^-14,
//     a normal fp16 number or 0), so a weight that is exactly zero contributes exactly zero;
//   * |rho_j| <= |w_t| for every t of the sub-block (unclamped: |rho_j| <= |D|/2 and
//     |D A_t| >= |D| when A_t != 0; clamped, or k_j = 0 with opposite signs: every w_t has the
//     sign of -rho_j and |w_t| >= |rho_j|), so the rho term only needs relative precision; and
//     |rho_j| <= 63 |Dm|, so rho_j T stays below 2^15;
//   * rho_j T (T = 2^(8-e), 2^e <= |Dm| < 2^(e+1)) is either >= 2^-3 in magnitude or a multiple
//     of 2^-24 below 2^-3 with at most 21 bits, and it is carried as an fp16 pair (hi, lo):
//     hi = rho_j T truncated to 11 significant bits, lo = the rest rounded to fp16, so
//     hi + lo is exact or within 2^-22 of rho_j T.
// The min-term MMAs take A_ext columns (hi_j, lo_j) twice per sub-block against the B_ext rows
// (X_hi, X_hi) and (X_lo, X_lo), so that the accumulator receives (hi + lo)(X_hi + X_lo).
// The sub-block's fields enter the fp32 steps as 64 m_j (exact), so the factors are kept divided
// by 64: (64 m) (R / 64) is m R exactly whenever R / 64 is a normal number, and below that
// m R < 2^-114 rounds to k = 0 either way; (64 m) (Dm T / 64) = m Dm T exactly.
struct Fold {
  float R64;     // Dm / D / 64 when >= 0, else 0 (+inf when D = 0: every k_j then clamps; D A_t vanishes)
  float DT;      // D * T
  float DmT64;   // Dm * T / 64, Dm T in [2^8, 2^9) (0 when Dm = 0, T = 1)
};
__device__ __forceinline__ Fold make_fold(float D, float Dm) {
  Fold f;
  float rD;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rD) : "f"(D));
  f.R64 = fmaxf(Dm * rD, 0.f) * 0.015625f;   // opposite signs (and D = 0 with Dm = 0): k = 0
  const uint32_t eb = __float_as_uint(Dm) & 0x7F800000u;
  const float T = eb ? __uint_as_float((262u << 23) - eb) : 1.0f;
  f.DT = D * T;
  f.DmT64 = Dm * T * 0.015625f;
  return f;
}
// The factor of the min-term accumulator: y += sigma (D acc + fe(Dm) acc_ext), fe = -2^(e-16)
// (acc_ext carries rho T X 2^(-s-6); sigma = 2^(s+14)).
__device__ __forceinline__ float fold_ext_factor(float Dm) {
  const uint32_t eb = __float_as_uint(Dm) & 0x7F800000u;
  return eb ? -__uint_as_float(eb - (16u << 23)) : 0.f;
}

// 32 bits of the 96-bit scale field (hd.y bits 0..31, hd.z 32..63, hd.w 64..95) from bit b on
// (the bits past 95 are not defined; callers mask them off).
__device__ __forceinline__ uint32_t field_at(const uint4& hd, int b) {
  const uint32_t lo = b < 32 ? hd.y : (b < 64 ? hd.z : hd.w);
  const uint32_t hi = b < 32 ? hd.z : hd.w;
  return __funnelshift_r(lo, hi, b & 31);
}

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));   // (a & mask) | bits
  return d;
}

// The decode constants of one sub-block: the fp16 pairs (-k 2^-14, -k 2^-14) (the addend),
// (sc 2^10, sc 2^10) and (sc 2^6, sc 2^6) (the multipliers of the two nibble positions), and
// the A_ext pair (hi, lo) of rho T.
struct SbConst {
  __half2 add, mlo, mhi;
  uint32_t ext;
};

// The constants of sub-blocks J and J + 1, whose 12-bit groups (sc | m << 6) start at bits 12J
// and 12J + 12 of the field; the fp32 steps of the two run as pairs (f32x2).
//   k = rint(m R) clamped to 2047: 1.5 2^23 + m R rounds to the integer in its low bits
//   rho T = (Dm m - D k) T = fma(-D T, k, m Dm T), exact or one rounding
template <int J>
__device__ __forceinline__ void fold_pair(const uint4& hd, const Fold& fd, const DecodeConsts& C, SbConst& c0,
                                          SbConst& c1) {
  constexpr float kMagic = 12582912.0f;                              // 1.5 2^23
  constexpr uint32_t kKK = 0u - 0x4B400000u * 0x10001u;              // bits(1.5 2^23 + k) * 0x10001 + kKK = k * 0x10001
  const uint32_t g0 = field_at(hd, 12 * J), g1 = field_at(hd, 12 * J + 12);
  // 64 m: 2^23 + 64 m has the bit pattern 0x4B000000 | (m << 6)
  const float2 m64 = __fadd2_rn(make_float2(__uint_as_float(lop_and_or(g0, 0xFC0u, 0x4B000000u)),
                                            __uint_as_float(lop_and_or(g1, 0xFC0u, 0x4B000000u))),
                                make_float2(-8388608.0f, -8388608.0f));
  const float2 tk = __ffma2_rn(m64, make_float2(fd.R64, fd.R64), make_float2(kMagic, kMagic));
  const float2 tc = make_float2(fminf(tk.x, kMagic + 2047.0f), fminf(tk.y, kMagic + 2047.0f));   // NaN (0 x inf) too
  const float2 kf = __fadd2_rn(tc, make_float2(-kMagic, -kMagic));
  const float2 rt = __ffma2_rn(make_float2(-fd.DT, -fd.DT), kf,
                               __fmul2_rn(m64, make_float2(fd.DmT64, fd.DmT64)));
  const float2 rhi = make_float2(__uint_as_float(__float_as_uint(rt.x) & 0xFFFFE000u),
                                 __uint_as_float(__float_as_uint(rt.y) & 0xFFFFE000u));   // 11 significant bits
  const float2 rlo = __ffma2_rn(rhi, make_float2(-1.0f, -1.0f), rt);
  c0.ext = h2bits(__floats2half2_rn(rhi.x, rlo.x));
  c1.ext = h2bits(__floats2half2_rn(rhi.y, rlo.y));
  // (k 2^-24, k 2^-24) has the bit pattern k * 0x10001; times -1024
  c0.add = __hmul2(bits2h(__float_as_uint(tc.x) * 0x10001u + kKK), C.kn1024);
  c1.add = __hmul2(bits2h(__float_as_uint(tc.y) * 0x10001u + kKK), C.kn1024);
  // (1024 + sc, 1024 + sc) has the bit pattern (0x6400 | sc) * 0x10001; minus 1024
  const __half2 sc0 = __hsub2(bits2h(lop_and_or(g0, 0x3Fu, 0x6400u) * 0x10001u), C.k1024);
  const __half2 sc1 = __hsub2(bits2h(lop_and_or(g1, 0x3Fu, 0x6400u) * 0x10001u), C.k1024);
  c0.mlo = __hmul2(sc0, C.k1024);
  c0.mhi = __hmul2(sc0, C.k64);
  c1.mlo = __hmul2(sc1, C.k1024);
  c1.mhi = __hmul2(sc1, C.k64);
}

template <int FMT>
__device__ __forceinline__ void decode_half(const HalfIn<FMT>& in, const uint4& hd, int h, uint32_t aaddr,
                                            const DecodeConsts& C, const Fold& fd, uint32_t* ext4) {
  if constexpr (FMT == kFmtQ4K || FMT == kFmtQ5K) {
    // the addend (-k 2^-14) and multipliers (sc 2^10, sc 2^6) of the two nibble positions of
    // sub-blocks 4h .. 4h+3, and their A_ext pairs
    SbConst sbc[4];
    if (h == 0) {
      fold_pair<0>(hd, fd, C, sbc[0], sbc[1]);
      fold_pair<2>(hd, fd, C, sbc[2], sbc[3]);
    } else {
      fold_pair<4>(hd, fd, C, sbc[0], sbc[1]);
      fold_pair<6>(hd, fd, C, sbc[2], sbc[3]);
    }
    __half2 mlo[4], mhi[4], add[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      add[jj] = sbc[jj].add;
      mlo[jj] = sbc[jj].mlo;
      mhi[jj] = sbc[jj].mhi;
      ext4[jj] = sbc[jj].ext;
    }
    // A = (sc q - k) 2^-14 as fp16 pairs, 16 columns per sub-block.  The quants enter as fp16
    // subnormals: q 2^-24 (bits 0..3 of a half) or 16 q 2^-24 (bits 4..7).
    const uint32_t hwords[4] = {in.hb.x, in.hb.y, in.hb.z, in.hb.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = in.qv[k];
      const uint32_t words[4] = {v.x, v.y, v.z, v.w};
      uint32_t cols[16];
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        const uint32_t wv = words[ww];
        uint32_t p[4];
        if constexpr (FMT == kFmtQ5K) {
          if (ww == 0) q5k_magic<0, 0u>(wv, hwords[k], p);
          if (ww == 1) q5k_magic<1, 0u>(wv, hwords[k], p);
          if (ww == 2) q5k_magic<2, 0u>(wv, hwords[k], p);
          if (ww == 3) q5k_magic<3, 0u>(wv, hwords[k], p);
        } else {
          const uint32_t b8 = wv >> 8;
          p[0] = wv & 0x000F000Fu;
          p[1] = wv & 0x00F000F0u;
          p[2] = b8 & 0x000F000Fu;
          p[3] = b8 & 0x00F000F0u;
        }
        cols[4 * ww + 0] = h2bits(__hfma2(bits2h(p[0]), mlo[k], add[k]));   // (q0, q4)
        cols[4 * ww + 1] = h2bits(__hfma2(bits2h(p[1]), mhi[k], add[k]));   // (q1, q5)
        cols[4 * ww + 2] = h2bits(__hfma2(bits2h(p[2]), mlo[k], add[k]));   // (q2, q6)
        cols[4 * ww + 3] = h2bits(__hfma2(bits2h(p[3]), mhi[k], add[k]));   // (q3, q7)
      }
      tc::st_x16(aaddr + 16 * k, cols);
    }
  } else if constexpr (FMT == kFmtQ6K) {
    // A = sc_j * (q - 32), |A| <= 64 * 32: exact in fp16.  The 6-bit quant is placed at mantissa
    // bits 4..9 (1024 + 16 q), then one HFMA2 with (sc/16, -96 sc) per pair.
    // scale bytes u of the half's sub-blocks 2k, 2k+1 (bytes 8h + 2k, 8h + 2k + 1 of the header)
    const uint32_t sw[2] = {h ? hd.z : hd.x, h ? hd.w : hd.y};
    const uint32_t hwords[8] = {in.hv[0].x, in.hv[0].y, in.hv[0].z, in.hv[0].w,
                                in.hv[1].x, in.hv[1].y, in.hv[1].z, in.hv[1].w};
    const __half2 k1o16 = C.k1o16;
    const __half2 kn68 = __float2half2_rn(-68.f), kn1536 = __float2half2_rn(-1536.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t ub;   // u of sub-block 2k in bits 0..7, of 2k+1 in bits 16..23
      asm("prmt.b32 %0, %1, 0, 0x4140;" : "=r"(ub) : "r"(sw[k >> 1] >> (16 * (k & 1))));
      uint32_t um;
      asm("lop3.b32 %0, %1, 0x007F007F, 0x64006400, 0xEA;" : "=r"(um) : "r"(ub));      // 1024 + (u & 127)
      const __half2 s16 = __hfma2(bits2h(um), k1o16, kn68);   // ((1024 + u)/16 - 68 = sc/16, exact)
      const __half2 c96 = __hmul2(s16, kn1536);               // -96 sc
      const __half2 s16_a = __low2half2(s16), s16_b = __high2half2(s16);
      const __half2 c96_a = __low2half2(c96), c96_b = __high2half2(c96);
      const uint4 v = in.qv[k];
      const uint32_t words[4] = {v.x, v.y, v.z, v.w};
      uint32_t cols[16];
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        uint32_t p[4];
        if (ww & 1) q6k_magic<1>(words[ww], hwords[2 * k + (ww >> 1)], p);
        else q6k_magic<0>(words[ww], hwords[2 * k + (ww >> 1)], p);
        const __half2 sa = ww < 2 ? s16_a : s16_b, ca = ww < 2 ? c96_a : c96_b;
#pragma unroll
        for (int c = 0; c < 4; ++c) cols[4 * ww + c] = h2bits(__hfma2(bits2h(p[c]), sa, ca));   // (q_c, q_c+4)
      }
      tc::st_x16(aaddr + 16 * k, cols);
    }
  } else if constexpr (FMT == kFmtINT4) {
    // A = q (the integer itself); the scale of each K half is applied in the epilogue
    const __half2 kn1032 = C.kn1032, k1o16 = C.k1o16, kn72 = C.kn72;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = in.qv[k];
      const uint32_t words[4] = {v.x, v.y, v.z, v.w};
      uint32_t cols[16];
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        uint32_t p[4];
        int4_magic(words[ww], p);
        cols[4 * ww + 0] = h2bits(__hadd2(bits2h(p[0]), kn1032));          // (q0, q4)
        cols[4 * ww + 1] = h2bits(__hfma2(bits2h(p[1]), k1o16, kn72));     // (q1, q5)
        cols[4 * ww + 2] = h2bits(__hadd2(bits2h(p[2]), kn1032));          // (q2, q6)
        cols[4 * ww + 3] = h2bits(__hfma2(bits2h(p[3]), k1o16, kn72));     // (q3, q7)
      }
      tc::st_x16(aaddr + 16 * k, cols);
    }
  } else {   // NVFP4: A = s_b * v, exact (at most 6 significant bits, at most 6 * 448)
    // the E4M3 scales of blocks 8h .. 8h+7 as fp16 pairs
    const uint32_t sw0 = h ? hd.z : hd.x, sw1 = h ? hd.w : hd.y;
    const uint32_t sp[4] = {e4m3x2_pair(sw0), e4m3x2_pair(sw0 >> 16), e4m3x2_pair(sw1), e4m3x2_pair(sw1 >> 16)};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = in.qv[k];
      const uint32_t words[4] = {v.x, v.y, v.z, v.w};
      // weights 32k .. 32k+15 use scale 2k of the half, 32k+16 .. 32k+31 scale 2k+1
      const __half2 s_lo = __low2half2(bits2h(sp[k])), s_hi = __high2half2(bits2h(sp[k]));
      uint32_t cols[16];
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        uint32_t p[4];
        e2m1x8_pairs(words[ww], p);
#pragma unroll
        for (int c = 0; c < 4; ++c) cols[4 * ww + c] = h2bits(__hmul2(bits2h(p[c]), ww < 2 ? s_lo : s_hi));
      }
      tc::st_x16(aaddr + 16 * k, cols);
    }
  }
}

// ------------------------------------------------------------------------------------------
// Hard tokens (q4k_xprep_kernel): their part of a super-block's outputs in fp32 on CUDA cores:
// this row's packed bytes from the stage at rb (the first 16 in hd), the activations from X
// (super-block sb of each token's row of K; X and K from the trailer of the prepared block at
// xblk).  Each weight is its format's definition (one rounding of the exact value, as the
// dequantization hook computes it); the 256 products are summed in order of k.  aux: what the
// format keeps outside its row blocks (Q6K's d plane, INT4's scale plane, NVFP4's tensor scale
// g), for row `row` of the product's N.
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

template <int FMT>
__device__ __forceinline__ float weight_at(uint32_t rb, const uint4& hd, int t, float aux0, float aux1) {
  if constexpr (FMT == kFmtQ4K || FMT == kFmtQ5K) {
    const int j = t >> 5;
    const uint64_t F = j < 5 ? ((uint64_t)hd.z << 32 | hd.y) : ((uint64_t)hd.w << 32 | hd.z);
    const uint32_t gr = (uint32_t)(F >> (j < 5 ? 12 * j : 12 * j - 32)) & 0xFFFu;
    const float2 dd = __half22float2(bits2h(hd.x));
    uint32_t q;
    if constexpr (FMT == kFmtQ4K) {
      q = (lds_u8(rb + 16 + (t >> 1)) >> (4 * (t & 1))) & 15u;
    } else {
      const int c = (t >> 3) & 3, i = t & 7;
      q = ((lds_u8(rb + 48 + (t >> 1)) >> (4 * (t & 1))) & 15u) + 16u * ((lds_u32(rb + 16 + 4 * j) >> (4 * i + c)) & 1u);
    }
    return fmaf(dd.x * (float)(gr & 63u), (float)q, -(dd.y * (float)(gr >> 6)));
  } else if constexpr (FMT == kFmtQ6K) {
    const int sc = (int)(lds_u8(rb + (t >> 4)) & 127u) - 64;
    const int tt = t & 15, a = tt >> 3, i = tt & 7;
    const uint32_t hi = (lds_u32(rb + 144 + 4 * (t >> 4)) >> (8 * a + 16 * (i >> 2) + 2 * (i & 3))) & 3u;
    const uint32_t q = ((lds_u8(rb + 16 + (t >> 1)) >> (4 * (t & 1))) & 15u) + 16u * hi;
    return (aux0 * (float)sc) * (float)((int)q - 32);
  } else if constexpr (FMT == kFmtNVFP4) {
    const float sb = __low2float(bits2h(e4m3x2_pair(lds_u8(rb + (t >> 4)))));
    uint32_t pr;
    const uint32_t code = lds_u8(rb + 16 + (t >> 1));
    asm("{\n .reg .b8 b0;\n cvt.u8.u32 b0, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}" : "=r"(pr) : "r"(code));
    const float v = (t & 1) ? __high2float(bits2h(pr)) : __low2float(bits2h(pr));
    return aux0 * (sb * v);
  } else {   // INT4: 128-byte rows copied with the 128-byte swizzle (chunk c at c ^ (row % 8))
    const uint32_t bi = (uint32_t)t >> 1;
    const uint32_t rbs = rb ^ ((rb >> 3) & 0x70u);
    const uint32_t byte = lds_u8((rbs ^ (16u * (bi >> 4))) + (bi & 15u));
    const int q = ((int)((byte >> (4 * (t & 1))) & 15u) ^ 8) - 8;
    return (t < 128 ? aux0 : aux1) * (float)q;
  }
}

template <int FMT, int MPAD, int MT>
__device__ __noinline__ void hard_dot(uint32_t rb, uint32_t xblk, const void* aux, int N, int row, int sb, uint4 hd,
                                      uint32_t mask, float* out) {
  const uint4 tr = lds128(xblk + mask_off(MPAD));   // (mask, K, address of X)
  const int K = (int)tr.y;
  const uint16_t* X = reinterpret_cast<const uint16_t*>((uint64_t)tr.z | ((uint64_t)tr.w << 32));
  float aux0 = 0.f, aux1 = 0.f;
  if constexpr (FMT == kFmtQ6K) {
    if (row < N)
      aux0 = __half2float(__ushort_as_half(__ldg(static_cast<const unsigned short*>(aux) + (int64_t)row * (K >> 8) + sb)));
  } else if constexpr (FMT == kFmtINT4) {
    if (row < N) {
      const uint32_t sc2 =
          __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(aux) + (int64_t)row * (K >> 7)) + sb);
      aux0 = __low2float(bits2h(sc2));
      aux1 = __high2float(bits2h(sc2));
    }
  } else if constexpr (FMT == kFmtNVFP4) {
    aux0 = __ldg(static_cast<const float*>(aux));
  }
  for (int k = 0; k < MT; ++k) out[k] = 0.f;
  for (int t = 0; t < 256; ++t) {
    const float w = weight_at<FMT>(rb, hd, t, aux0, aux1);
    for (int k = 0; k < MT; ++k) {
      if ((mask >> k) & 1u) {
        const uint32_t xbits = __ldg(X + (int64_t)k * K + (int64_t)sb * 256 + t);
        out[k] = fmaf(w, __uint_as_float(xbits << 16), out[k]);
      }
    }
  }
}

// FMT: weight format.  MPAD: MMA width (token columns of B and of the accumulators, 16 or 32).
// MT: the token columns the epilogue reads and sums (8 when M <= 8, else MPAD); columns past M
// hold zeros.  GATED: the feed-forward gating in the epilogue (a separate instance: its code in
// the regular kernels measured 2.5 % slower at M <= 8).
template <int FMT, int MPAD, int MT, int MAXE, bool GATED, int NG>
__global__ void __launch_bounds__(cta_threads(NG), 1)
    q4k_tc_kernel(const __grid_constant__ TcParams<MAXE, naux(FMT, MAXE)> P) {
  static_assert(MT == 8 || MT == MPAD, "token columns");
  extern __shared__ __align__(1024) uint8_t smem[];
  // programmatic dependent launch: the next launch in the stream may be scheduled from now on,
  // onto SMs this grid leaves.  That is another product launch of the same call (it issues
  // weight copies, which no launch of the call writes, then waits for this grid's completion)
  // or a CUDA-core product (it waits before it touches memory); the other kernels, the
  // preparation among them, start in plain stream order.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using L = TcSmem<MPAD, FMT, MT, NG>;
  constexpr int kProdWarp = NG * kGroupWarps;   // copies
  constexpr int kMmaWarp = kProdWarp + 1;       // (first) MMA issue warp; owns TMEM
  constexpr int kMmaWarps = NG;                 // one MMA warp per group
  constexpr int kTW = token_width(MPAD, MT);      // token columns of a prepared block
  constexpr int kBB = bblock_bytes(kTW);
  constexpr int kS = stages(MPAD, FMT, MT, NG);
  constexpr int kSB = stage_bytes(kTW, FMT);
  constexpr int kBlk = blk_bytes(FMT);
  constexpr int kWSB = w_stage_bytes(FMT);
  constexpr bool kExtInA = ext_in_a(FMT, MT, NG);
  constexpr bool kAccInA = acc_in_a(FMT, MT, NG);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sW = smem_addr(smem + L::kW);   // stage k: weights at sW + k*kSB, activations kWSB further
  const uint32_t bars = smem_addr(smem + L::kBars);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  int* group_sbs = reinterpret_cast<int*>(smem + L::kMisc + 16);   // n_g, g < NG
  auto bar = [&](int k) { return bars + 8u * k; };
  auto gfull = [&](int g, uint32_t s) { return bar(kBarGFull + g * kMaxStages + (int)s); };

  if (threadIdx.x == 0) {
    for (int g = 0; g < NG; ++g) {
      for (int k = 0; k < kS; ++k) mbar_init(gfull(g, k), 1);
      mbar_init(bar(kBarAFull + 2 * g), kGroupWarps);
      mbar_init(bar(kBarAFull + 2 * g + 1), kGroupWarps);
      mbar_init(bar(kBarGDone + g), 1);
      mbar_init(bar(kBarH0Done + g), 1);
    }
    // the consuming group's warps once they hold their bytes, and the MMA commit once the MMAs
    // have read the activations
    for (int k = 0; k < kS; ++k) mbar_init(bar(kBarWEmpty + k), kGroupWarps + 1);
    for (int m = 0; m < kMmaWarps; ++m) mbar_init(bar(kBarDrain + m), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if constexpr (MT == 8) {   // the zero regions the 8-token MMAs read as token columns
    uint4* z0 = reinterpret_cast<uint4*>(smem + L::kZeroExt);
    uint4* z1 = reinterpret_cast<uint4*>(smem + L::kZeroMain);
    for (int k = threadIdx.x; k < kZeroExtBytes / 16; k += blockDim.x) z0[k] = make_uint4(0u, 0u, 0u, 0u);
    for (int k = threadIdx.x; k < kZeroMainBytes / 16; k += blockDim.x) z1[k] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();   // visible to the tensor cores (async proxy) after the barrier below
  }
  if (warp == 0 && lane < NG) {   // super-blocks of each group
    GroupCursor<TcParams<MAXE, naux(FMT, MAXE)>, NG> cur;
    cur.start(P, lane);
    int cnt = 0;
    while (cur.t >= 0) { cnt += cur.end - cur.sb; ++cur.r; cur.load(P); }
    group_sbs[lane] = cnt;
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_addr(tmem_holder), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  int n[NG];
  int nmax = 0, nmin = 1 << 30;
#pragma unroll
  for (int g = 0; g < NG; ++g) { n[g] = group_sbs[g]; nmax = max(nmax, n[g]); nmin = min(nmin, n[g]); }

  auto wait = [&](uint32_t b, uint32_t parity) -> bool {
    if (mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait(b, parity, P.wait_polls ? P.wait_polls : kWaitLimit, P.wait_ns ? P.wait_ns : kSuspendNs))
      return true;
    atomicOr(&g_status, kErrWaitTimeout);
    *abort_flag = 1;
    return false;
  };

  if (warp == kProdWarp) {
    // ------------------------------------------------------------------ copies
    // Per super-block one TMA copy of the weights (rows row0 .. row0+127, rows past N read as
    // zeros; bytes 144 sb .. 144 sb + 143 of each row) and one bulk copy of the prepared
    // activation block, into the same stage, completing on that stage's barrier of the owning
    // group.  The ring runs kS - 1 super-blocks ahead, in the CTA's super-block order.  The
    // weights of the first kS super-blocks are requested before the preparation grid has finished
    // (they do not depend on it); their activation blocks once it has.
    if (elect_one()) {
      const uint64_t pol = policy_evict_first();
      GroupCursor<TcParams<MAXE, naux(FMT, MAXE)>, NG> cur[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) cur[g].start(P, g);
      uint32_t su = 0;
      uint32_t gbits = 0;    // parity of the next phase of each (group, stage) full barrier
      uint32_t owner = 0;    // group of the copies last issued into each stage, 2 bits a stage
      bool ok = true;
      // activation-block copies held back until the preparation grid is complete: those of the
      // super-blocks su < kS (in stage su), entry and super-block packed as e << 16 | sb
      uint32_t pend[kS];
      bool prepped = false;
      auto release_pending = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the prepared activations are written
        for (uint32_t k = 0; k < su && k < (uint32_t)kS; ++k) {
          const uint32_t g = (owner >> (2 * k)) & 3u;
          bulk_g2s(sW + k * kSB + kWSB, P.e[pend[k] >> 16].B + (int64_t)(pend[k] & 0xFFFFu) * kBB, kBB,
                   gfull((int)g, k), 0ull);
        }
        prepped = true;
      };
      for (int i = 0; i < nmax && ok; ++i) {
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          if (ok && i < n[g] && !prepped && su == (uint32_t)kS) release_pending();   // before a stage is reused
          if (ok && i < n[g]) ok = wait(bar(kBarWEmpty + su % kS), ((su / kS) & 1u) ^ 1u);
          if (ok && i < n[g]) {
            const uint32_t ws = su % kS;
            gbits ^= 1u << (g * kMaxStages + ws);
            owner = (owner & ~(3u << (2 * ws))) | ((uint32_t)g << (2 * ws));
            const uint32_t st = sW + ws * kSB;
            const int e = cur[g].e, sb = cur[g].sb;
            mbar_arrive_expect_tx(gfull(g, ws), kWSB + kBB);
            tma_load_2d(st, &P.maps[e], sb * kBlk, cur[g].tile * kTileRows, gfull(g, ws), pol);
            if (prepped) bulk_g2s(st + kWSB, P.e[e].B + (int64_t)sb * kBB, kBB, gfull(g, ws), 0ull);
            else pend[su] = (uint32_t)e << 16 | (uint32_t)sb;
            cur[g].advance(P);
            ++su;
          }
        }
      }
      if (!prepped) release_pending();
      // copies still in flight land before the CTA can end: wait for the last phase armed on
      // each stage's full barrier (complete already, or once its bytes have arrived)
      for (uint32_t k = (su > (uint32_t)kS ? su - kS : 0u); k < su; ++k) {
        const uint32_t ws = k % kS, g = (owner >> (2 * ws)) & 3u;
        mbar_wait(gfull((int)g, ws), ((gbits >> (g * kMaxStages + ws)) & 1u) ^ 1u, kWaitLimit);
      }
    }
  } else if (warp >= kMmaWarp) {
    // ------------------------------------------------------------------ MMA issue
    // Super-block su of group g: its A slot, handed over one K half at a time (each half full
    // once the group's 4 warps have arrived, so the first 8 MMAs run while the group still
    // dequantizes the second half), its activations in stage su % kS, its accumulator (read by
    // the group before it wrote the A slot again).  The k-quants add two min-term MMAs (A_ext
    // against B_ext) after the second half.  One elected lane waits, issues and commits, in
    // super-block order.
    // Warp kMmaWarp + g serves group g.
    const int g = warp - kMmaWarp;
    if (elect_one()) {
      constexpr uint32_t idesc = tc::idesc_f16_f32(128, MPAD);
      int ngl = 0;
#pragma unroll
      for (int h = 0; h < NG; ++h) if (h == g) ngl = n[h];
      const uint32_t abase = tmem + a_col(g, FMT, MT, NG);
      const uint32_t zext = smem_addr(smem + L::kZeroExt), zmain = smem_addr(smem + L::kZeroMain);
      const uint32_t d1 = tmem + acc1_col(MPAD, g, FMT, MT, NG);
      const uint32_t d2 = tmem + acc2_col(MPAD, g, FMT, MT, NG);
      uint32_t gbits = 0;   // parity of this group's full barrier of each stage
      for (int i = 0; i < ngl; ++i) {
        const uint32_t ws = su_of<NG>(n, g, i, nmin) % kS;
        if (!(wait(bar(kBarAFull + 2 * g), (uint32_t)i & 1u) && wait(gfull(g, ws), (gbits >> ws) & 1u))) break;
        gbits ^= 1u << ws;
        tc::fence_after_sync();
        const uint32_t bslot = sW + ws * kSB + kWSB;
        // token columns 8..15 (the second group of 8): 4096 bytes further, or the zero region
        const uint64_t bdesc = tc::smem_desc_kmajor(bslot, 128, MT == 8 ? zmain - bslot : 4096u);   // + 16 per MMA: 256 bytes
        tc::mma_f16_ts_x8(d1, abase, bdesc, 16, idesc, 0);
        if constexpr (kAccInA) tc::commit(bar(kBarH0Done + g));   // the group may reuse these A columns
        if (!wait(bar(kBarAFull + 2 * g + 1), (uint32_t)i & 1u)) break;
        tc::fence_after_sync();
        if constexpr (FMT == kFmtINT4) {
          // the second K half has its own scale: its own accumulator
          tc::mma_f16_ts_x8(d2, abase + 64, bdesc + 8 * 16, 16, idesc, 0);
        } else {
          tc::mma_f16_ts_x8(d1, abase + 64, bdesc + 8 * 16, 16, idesc, 1);
        }
        if constexpr (has_min(FMT)) {
          // the min term: A_ext (16 columns, K = 32) against B_ext, into the product's
          // accumulator (8 token columns: B_ext fills columns 8..15) or its own
          constexpr bool kShiftExt = MT == 8;   // the min term in columns 8..15 of d1
          // 8 tokens: columns 0..7 from the zero region, the tokens' rows as columns 8..15
          const uint64_t edesc = MT == 8 ? tc::smem_desc_kmajor(zext, 128, bslot + bext_off(kTW) - zext)
                                         : tc::smem_desc_kmajor(bslot + bext_off(kTW), 128, 512);
          const uint32_t ea = abase + (kExtInA ? 0u : 128u);
          if constexpr (kAccInA && !kExtInA) {
            if (!wait(bar(kBarH0Done + g), (uint32_t)i & 1u)) break;   // no MMA still reads d2's columns
            tc::fence_after_sync();
          }
          tc::mma_f16_ts(kShiftExt ? d1 : d2, ea, edesc, idesc, kShiftExt ? 1u : 0u);
          tc::mma_f16_ts(kShiftExt ? d1 : d2, ea + 8, edesc + 16, idesc, 1u);
        }
        tc::commit(bar(kBarGDone + g));
        tc::commit(bar(kBarWEmpty + ws));
      }
      // every MMA issued has finished before TMEM is released
      tc::commit(bar(kBarDrain + g));
      mbar_wait(bar(kBarDrain + g), 0u, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ dequant + epilogue
    // Software-pipelined over the group's super-blocks: once super-block i is handed to the
    // MMA warp, the group waits for the stage of super-block i+1 and takes what does not need
    // tensor memory (its header, per-token scales, the mask of hard tokens) while the MMAs of i
    // run; then it reads i's accumulator, and decodes i+1 (the hard tokens' part of i+1, if
    // any, just before the stage is released).
    const int grp = warp >> 2;       // dequant group: the CTA's local tasks j % NG == grp
    const int q = warp & 3;          // TMEM lane quarter / row quarter of the tile
    const int r = 32 * q + lane;     // row inside the tile
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    const DecodeConsts dc;
    auto wait_w = [&](uint32_t k, uint32_t parity) -> bool { return __all_sync(0xffffffffu, wait(k, parity)); };

    float y[MT];   // the current chunk's sum, tokens 0 .. MT-1 of this thread's row
#pragma unroll
    for (int k = 0; k < MT; ++k) y[k] = 0.f;
    // the task's running sum of chunk sums: registers, or shared memory (token k at [k * 128])
    // for 16 and 32 tokens
    constexpr bool kYtotSmem = MT >= 16;
    float ytot_r[kYtotSmem ? 1 : MT];
    float* ytot_s = reinterpret_cast<float*>(smem + L::kYtot) + (size_t)grp * MT * kTileRows + r;
#pragma unroll
    for (int k = 0; k < (kYtotSmem ? 1 : MT); ++k) ytot_r[k] = 0.f;
    auto ytot = [&](int k) -> float& { if constexpr (kYtotSmem) return ytot_s[k * kTileRows]; else return ytot_r[k]; };

    const uint32_t aslot = tl + a_col(grp, FMT, MT, NG);       // this group's A slot (this warp's lanes)
    const uint32_t aext = aslot + (kExtInA ? 0u : 128u);         // its min-term columns
    const uint32_t acc1 = tl + acc1_col(MPAD, grp, FMT, MT, NG);    // and accumulators
    const uint32_t acc2 = tl + acc2_col(MPAD, grp, FMT, MT, NG);
    // this warp's copies of the per-token scales of two super-blocks in flight (by parity)
    float* sigw = reinterpret_cast<float*>(smem + L::kSig) + warp * 64;
    float hard_sum[MT];   // the hard tokens' sums of the super-block being finished (rarely used)
    asm volatile("griddepcontrol.wait;" ::: "memory");   // split counters zeroed, activations written
    uint32_t sbits = 0;   // parity of this group's full barrier of each stage

    // What the look-ahead of a super-block yields.
    struct Ahead {
      uint32_t ws;        // its stage
      uint4 hd;           // this row's first 16 bytes
      uint32_t hmask;     // its hard tokens
      uint32_t ext[8];    // k-quants: the A_ext pairs of rho_j T (filled by the decode)
    };
    // Wait for the i-th super-block of the group and take its header, per-token scales and hard
    // tokens.
    auto ahead = [&](int i, Ahead& A) -> bool {
      A.ws = su_of<NG>(n, grp, i, nmin) % kS;
      if (!wait_w(gfull(grp, A.ws), (sbits >> A.ws) & 1u)) return false;
      sbits ^= 1u << A.ws;
      const uint32_t rb = sW + A.ws * kSB + r * kBlk;
      const uint32_t xblk = sW + A.ws * kSB + kWSB;
      A.hd = FMT == kFmtINT4 ? make_uint4(0, 0, 0, 0) : lds128(rb);
      float* sg = sigw + 32 * (i & 1);
      if (lane < MT / 4) *reinterpret_cast<uint4*>(sg + 4 * lane) = lds128(xblk + sig_off(kTW) + 16 * lane);
      A.hmask = lds_u32(xblk + mask_off(kTW)) & (MT == 32 ? 0xFFFFFFFFu : ((1u << MT) - 1u));
      return true;
    };

    using Cursor = GroupCursor<TcParams<MAXE, naux(FMT, MAXE)>, NG>;
    int ng = 0;   // super-blocks of this group
#pragma unroll
    for (int h = 0; h < NG; ++h) if (h == grp) ng = n[h];
    // Iteration i: look ahead to super-block i (the only call site of ahead), finish super-block
    // i - 1 (its accumulator, once its MMAs are done), then decode super-block i and hand it to
    // the MMA warp.
    Cursor cur;          // the super-block being finished (i - 1)
    Cursor nx;           // super-block i
    nx.start(P, grp);
    Ahead A;
    bool task_end = false;                 // super-block i - 1 ended its task
    float sx = 0.f, sy = 0.f;              // the accumulator factors of super-block i - 1
    uint32_t hm = 0;                       // its hard tokens
    for (int i = 0;; ++i) {
      if (i < ng && !ahead(i, A)) break;
      if (i >= 1) {
        // ---- the accumulator of super-block i - 1 into y (MT token columns)
        if (!wait_w(bar(kBarGDone + grp), (uint32_t)(i - 1) & 1u)) break;
        tc::fence_after_sync();
        constexpr bool kTwo = FMT != kFmtNVFP4 && FMT != kFmtQ6K;   // a second accumulator block to read
        constexpr bool kShift = has_min(FMT) && MT == 8;             // the min term in columns 8..15
        constexpr int kW = MT == 16 ? 16 : 8;   // token columns per TMEM read round
        const float* sg_i = sigw + 32 * ((i - 1) & 1);
#pragma unroll
        for (int c0 = 0; c0 < MT; c0 += kW) {
          float a1[kW], a2[kW];
          if constexpr (kShift) {
            float a[16];
            tc::ld_x16(acc1, a);
#pragma unroll
            for (int k = 0; k < 8; ++k) { a1[k] = a[k]; a2[k] = a[8 + k]; }
          } else if constexpr (kW == 8) {
            tc::ld_x8(acc1 + c0, a1);
            if constexpr (kTwo) tc::ld_x8(acc2 + c0, a2);
          } else {
            tc::ld_x16(acc1 + c0, a1);
            if constexpr (kTwo) tc::ld_x16(acc2 + c0, a2);
          }
          tc::wait_ld();
#pragma unroll
          for (int k = 0; k < kW; k += 4) {
            const float4 sg = *reinterpret_cast<const float4*>(sg_i + c0 + k);
            const float sgk[4] = {sg.x, sg.y, sg.z, sg.w};
            // two tokens per f32x2 operation: y += sigma (sx a1 + sy a2), each step rounded as
            // its scalar form
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              const float2 yy = make_float2(y[c0 + k + u], y[c0 + k + u + 1]);
              float2 r;
              if constexpr (kTwo) {
                const float2 t = __ffma2_rn(make_float2(sx, sx), make_float2(a1[k + u], a1[k + u + 1]),
                                            __fmul2_rn(make_float2(sy, sy), make_float2(a2[k + u], a2[k + u + 1])));
                r = __ffma2_rn(make_float2(sgk[u], sgk[u + 1]), t, yy);
              } else {
                r = __ffma2_rn(__fmul2_rn(make_float2(sx, sx), make_float2(sgk[u], sgk[u + 1])),
                               make_float2(a1[k + u], a1[k + u + 1]), yy);
              }
              y[c0 + k + u] = r.x;
              y[c0 + k + u + 1] = r.y;
            }
          }
        }
        // hard tokens: their accumulator columns are exactly 0; add their CUDA-core sums
        if (hm != 0u) {
#pragma unroll
          for (int k = 0; k < MT; ++k)
            if ((hm >> k) & 1u) y[k] += hard_sum[k];
        }

        // ---- end of a chunk: y (this chunk's sum) is added to the task's running sum, or, for a
        // split task, stored as the chunk's partial.  End of a task: the running
        // sum goes to Y; a split task counts itself in, and the last split of this (tile, lane
        // quarter) slice adds every chunk partial of the tile in chunk order.
        const int e = cur.e, tile = cur.tile, sb = cur.sb;
        const TcEntry& E = P.e[e];
        const int nb = E.K >> 8;
        if ((sb + 1) % kChunkSb == 0 || sb + 1 == nb) {
          if (E.splits == 1) {
            if (sb < kChunkSb) {
#pragma unroll
              for (int k = 0; k < MT; ++k) ytot(k) = y[k];
            } else {
#pragma unroll
              for (int k = 0; k < MT; ++k) ytot(k) = ytot(k) + y[k];
            }
          } else {
            float* part = E.partial + ((size_t)tile * E.chunks + sb / kChunkSb) * (MPAD * kTileRows) + r;
#pragma unroll
            for (int k = 0; k < MT; ++k)
              if (k < P.M) part[k * kTileRows] = y[k];
          }
#pragma unroll
          for (int k = 0; k < MT; ++k) y[k] = 0.f;
        }
        if (task_end) {
          const int row = tile * kTileRows + r;
          if constexpr (GATED) {
            // the feed-forward gating in the epilogue: lane r holds row 2f (gate) or 2f+1 (up) of
            // the same tile; the even lane forms silu(gate) * up in fp32 and stores its bf16
            // (round to nearest even), silu(g) = g / (1 + e^-g)
            uint16_t* H = reinterpret_cast<uint16_t*>(E.Y);
            if constexpr (kYtotSmem) {
              gate_store_smem<MT>(ytot_s, r, row, E.N, P.M, H);
            } else {
              const int64_t F = E.N >> 1;
#pragma unroll
              for (int k = 0; k < MT; ++k) {
                const float mine = ytot(k);
                const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
                if (k < P.M && !(r & 1) && row < E.N) {
                  const float h = mine / (1.0f + expf(-mine)) * other;
                  const __nv_bfloat16 hb = __float2bfloat16_rn(h);
                  H[(int64_t)k * F + (row >> 1)] = *reinterpret_cast<const uint16_t*>(&hb);
                }
              }
            }
          } else if (E.splits == 1) {
            if (row < E.N) {
#pragma unroll
              for (int k = 0; k < MT; ++k)
                if (k < P.M) E.Y[(int64_t)k * E.N + row] = ytot(k);
            }
          } else {
            // the warp's partial stores, then one release of them (the warp barrier orders the
            // other lanes' stores before lane 0's fence) and the arrival count of this slice
            __syncwarp();
            unsigned old = 0;
            if (lane == 0) {
              fence_acq_rel_gpu();   // release of the warp's partial sums
              old = atomicAdd(&E.counters[tile * kGroupWarps + q], 1u);
            }
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == (unsigned)(E.splits - 1)) {
              fence_acq_rel_gpu();   // acquire of the other splits' partial sums
              reduce_chunks<MPAD, MT>(E.partial + (size_t)tile * E.chunks * (MPAD * kTileRows) + r, E.chunks, P.M,
                                  row < E.N ? E.Y + row : nullptr, E.N);
            }
          }
        }
      }
      if (i >= ng) break;
      const uint32_t ws = A.ws;
      const uint4 hd = A.hd;
      const uint32_t rb = sW + ws * kSB + r * kBlk;   // this row's bytes of the super-block
      const uint32_t xblk = sW + ws * kSB + kWSB;      // its prepared activation block
      Fold fd{0.f, 0.f, 0.f};                          // k-quants: the row's fold factors
      if constexpr (has_min(FMT)) {
        const float2 dd = __half22float2(bits2h(hd.x));
        fd = make_fold(dd.x, dd.y);
      }
      // ---- decode: the row's super-block one K half at a time from the stage (this warp's part
      // of the stage is released once all is read), each half handed to the MMA warp
      // (the A slot is free: this group read its previous accumulator above)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        HalfIn<FMT> in;
        load_half<FMT>(in, rb, h);
        if (h == 1) {
          // hard tokens: this row's part of their outputs on CUDA cores (added after the
          // accumulator in the epilogue of this super-block)
          if (A.hmask != 0u)   // uniform over the CTA: the mask belongs to the super-block of X
            hard_dot<FMT, kTW, MT>(rb, xblk, P.aux[nx.e], P.e[nx.e].N, nx.tile * kTileRows + r, nx.sb, hd, A.hmask,
                                    hard_sum);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarWEmpty + ws));
        }
        decode_half<FMT>(in, hd, h, aslot + 64u * h, dc, fd, A.ext + 4 * h);
        if (h == 0) {   // the first K half goes to the MMA warp now
          tc::wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarAFull + 2 * grp));
        }
      }
      // INT4: the scales of this row's two K halves, from the scale plane; Q6K: the row's
      // super-block scale d, from its plane (read now, used by the epilogue)
      const int row0 = nx.tile * kTileRows + r;
      uint32_t int4_scales = 0;
      if constexpr (FMT == kFmtINT4) {
        const TcEntry& E0 = P.e[nx.e];
        if (row0 < E0.N)
          int4_scales = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(P.aux[nx.e]) +
                                                                (int64_t)row0 * (E0.K >> 7)) + nx.sb);
      } else if constexpr (FMT == kFmtQ6K) {
        const TcEntry& E0 = P.e[nx.e];
        if (row0 < E0.N)
          int4_scales = __ldg(static_cast<const unsigned short*>(P.aux[nx.e]) + (int64_t)row0 * (E0.K >> 8) + nx.sb);
      }
      if constexpr (has_min(FMT)) {
        // A_ext: the pair (hi_j, lo_j) of rho_j T twice per sub-block (against B_ext rows
        // (X_hi, X_hi) and (X_lo, X_lo)); where it reuses the first K half's columns, after
        // that half's MMAs have completed
        if constexpr (kExtInA) {
          if (!wait_w(bar(kBarH0Done + grp), (uint32_t)i & 1u)) break;
          tc::fence_after_sync();
        }
        tc::st_x16_pairs(aext, A.ext);   // column 2j and 2j+1: ext[j]
      }
      // ---- hand the second K half (and A_ext) to the MMA warp
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarAFull + 2 * grp + 1));

      // the factors of the accumulator blocks (sigma_k = 2^(s_k + 14) of token k applied last):
      //   k-quants  y += sigma (D acc + fe acc_ext)          (A = (sc q - k) 2^-14)
      //   NVFP4     y += sigma (g 2^-14) acc
      //   INT4      y += sigma 2^-14 (s_0 acc_half0 + s_1 acc_half1)
      //   Q6K       y += sigma (d 2^-14) acc
      if constexpr (has_min(FMT)) {
        const float2 dd = __half22float2(bits2h(hd.x));   // (D, Dm) of this row
        sx = dd.x;
        sy = fold_ext_factor(dd.y);
      } else if constexpr (FMT == kFmtNVFP4) {
        sx = __ldg(static_cast<const float*>(P.aux[nx.e])) * 0x1p-14f;
        sy = 0.f;
      } else if constexpr (FMT == kFmtQ6K) {
        sx = __half2float(__ushort_as_half((unsigned short)int4_scales)) * 0x1p-14f;
        sy = 0.f;
      } else {
        const float2 ss = __half22float2(bits2h(int4_scales));
        sx = ss.x * 0x1p-14f;
        sy = ss.y * 0x1p-14f;
      }
      hm = A.hmask;
      cur = nx;
      task_end = nx.advance(P);
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
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> g(mu());
    auto& slot = pool()[{dev, reinterpret_cast<uintptr_t>(stream)}];
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
  // Free every workspace (each with its device current; cudaFree waits for the work that may
  // still use it).  The calling thread's current device is restored.
  static cudaError_t release() {
    std::lock_guard<std::mutex> g(mu());
    if (pool().empty()) return cudaSuccess;
    int cur = 0;
    cudaError_t first = cudaGetDevice(&cur);
    for (auto& kv : pool()) {
      if (!kv.second.first) continue;
      cudaError_t err = cudaSetDevice(kv.first.first);
      if (err == cudaSuccess) err = cudaFree(kv.second.first);
      if (err != cudaSuccess && first == cudaSuccess) first = err;
    }
    pool().clear();
    const cudaError_t e2 = cudaSetDevice(cur);
    return first != cudaSuccess ? first : e2;
  }
  static size_t held_bytes() {
    std::lock_guard<std::mutex> g(mu());
    size_t b = 0;
    for (auto& kv : pool()) b += kv.second.second;
    return b;
  }

 private:
  static std::mutex& mu() { static std::mutex m; return m; }
  static std::map<std::pair<int, uintptr_t>, std::pair<void*, size_t>>& pool() {
    static std::map<std::pair<int, uintptr_t>, std::pair<void*, size_t>> p;
    return p;
  }
};

// The failure-detection hook's wait bound (0, 0: the kernels' own bound).
std::atomic<uint32_t> g_wait_polls{0}, g_wait_ns{0};

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

// Map of a packed matrix's weight plane as a 2D byte array: inner dimension the bytes of a row
// (K/256 blocks of blk_bytes(fmt)), outer dimension the N rows; the box is one 256-weight block
// of 128 rows.  INT4 boxes (128 bytes) are copied with the 128-byte swizzle.  L2 promotion to
// 128 bytes: with 256-byte promotion the evict-first rows of a 144-byte box pulled in bytes of
// the next super-block that were often gone again when it was copied (DRAM traffic 1.038x of
// lm_head's bytes against 1.017x, measured on GB300).
cudaError_t weight_map(const void* W, int64_t N, int64_t K, int fmt, CUtensorMap* out) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int64_t, int64_t, int>, CUtensorMap> cache;
  std::lock_guard<std::mutex> g(mu);
  const auto key = std::make_tuple(W, N, K, fmt);
  auto it = cache.find(key);
  if (it != cache.end()) { *out = it->second; return cudaSuccess; }
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t rowbytes = (cuuint64_t)(K / 256) * blk_bytes(fmt);
  const cuuint64_t dims[2] = {rowbytes, (cuuint64_t)N};
  const cuuint64_t strides[1] = {rowbytes};
  const cuuint32_t box[2] = {(cuuint32_t)blk_bytes(fmt), (cuuint32_t)kTileRows};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  const CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        fmt == kFmtINT4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if (cache.size() >= 4096) cache.clear();
  cache.emplace(key, m);
  *out = m;
  return cudaSuccess;
}

template <int FMT, int MPAD, int MT, int MAXE, bool GATED, int NG>
cudaError_t set_smem_attr() {
  static bool done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  err = cudaFuncSetAttribute(q4k_tc_kernel<FMT, MPAD, MT, MAXE, GATED, NG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcSmem<MPAD, FMT, MT, NG>::kTotal);
  if (err == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return err;
}

// One instance of the kernel: its shared memory attribute, block size and launch.
template <int FMT, int MPAD, int MT, int MAXE, bool GATED, int NG, class PT>
cudaError_t launch_instance(cudaLaunchConfig_t& cfg, const PT& par) {
  cudaError_t err = set_smem_attr<FMT, MPAD, MT, MAXE, GATED, NG>();
  if (err != cudaSuccess) return err;
  cfg.dynamicSmemBytes = TcSmem<MPAD, FMT, MT, NG>::kTotal;
  cfg.blockDim = dim3(cta_threads(NG));
  return cudaLaunchKernelEx(&cfg, q4k_tc_kernel<FMT, MPAD, MT, MAXE, GATED, NG>, par);
}

// Tensor-core launches over these products run the k-quants' three-group instance at 32 token
// columns when their tasks keep every group busy: a batched launch, or a product with at least
// three 128-row tiles per SM.
bool wide_launch(const Job* jobs, int count, int sms) {
  return count > 1 || (jobs[0].N + kTileRows - 1) / kTileRows >= 3 * (int64_t)sms;
}

// K split of a product: the number of splits of every 128-row tile and the super-blocks per
// split (a multiple of kChunkSb, so that the split does not change the summation order).  A
// batched launch has work enough for every SM and does not split; a single product picks the
// split with the least time on the busiest dequant group,
//   pace x (its tasks) x (super-blocks per task) + 2.5 x (its tasks, if split)
//     + 0.05 x (chunks summed by the last split)
// in units of one super-block of a tile at the pace of a CTA whose ng groups all work (the
// tasks are dealt to the SMs' (CTA, group) slots, GroupCursor).  An SM with fewer tasks than
// groups runs fewer groups, each faster: pace 0.65 for one group, 0.92 for two of three.  The
// constants are a least-squares fit to GB300 graph-replay timings of 5120 x 5120, 34816 x 5120
// and 5120 x 17408 products at 1 to 17 splits (a split task costs its partial-sum stores, a
// device-scope fence and an atomic on the busiest group).
struct Split {
  int splits;
  int chunk;
};

int chunks_of(int64_t K) { return (int)((K / 256 + kChunkSb - 1) / kChunkSb); }

struct SplitCost {
  Split split;
  double units;   // busiest group's time, in super-blocks of a tile at the full pace
};

SplitCost split_cost(int64_t N, int64_t K, int sms, int ng, bool batched) {
  const int64_t tiles = (N + kTileRows - 1) / kTileRows;
  const int nb = (int)(K / 256);
  const int nch = chunks_of(K);
  auto cost_of = [&](int splits, int chunk_sb) {
    const double per_cta = std::ceil((double)(tiles * splits) / (double)std::max(1, sms));
    const double per_group = std::ceil(per_cta / ng);
    const int active = (int)std::min<double>(ng, per_cta);
    const double pace = active >= ng ? 1.0 : (active == 1 ? (ng >= 3 ? 0.65 : 0.75) : 0.92);
    return pace * per_group * chunk_sb + (splits > 1 ? 2.5 * per_group + 0.05 * nch : 0.0);
  };
  SplitCost best{Split{1, nb}, cost_of(1, nb)};
  if (batched) return best;
  for (int cps = nch - 1; cps >= 1; --cps) {   // chunks per split
    const int splits = (nch + cps - 1) / cps;
    if ((nch + splits - 1) / splits != cps) continue;   // same splits, larger chunk seen
    const int chunk_sb = std::min(nb, cps * kChunkSb);
    const double c = cost_of(splits, chunk_sb);
    if (c < best.units - 1e-9) best = SplitCost{Split{splits, chunk_sb}, c};
  }
  return best;
}

Split split_for(int64_t N, int64_t K, int sms, int ng, bool batched) { return split_cost(N, K, sms, ng, batched).split; }

// Bytes of split workspace (partials, then counters) that a job needs.
struct SplitSpace {
  size_t partial_bytes = 0;
  size_t counter_words = 0;
};

template <int MPAD>
SplitSpace split_space(int64_t N, int64_t K, const Split& s) {
  SplitSpace r;
  if (s.splits > 1) {
    const size_t tiles = (size_t)((N + kTileRows - 1) / kTileRows);
    r.partial_bytes = tiles * (size_t)chunks_of(K) * MPAD * 128 * sizeof(float);
    r.counter_words = tiles * kGroupWarps;
  }
  return r;
}

// The main kernel over jobs[0 .. count) (count <= MAXE), whose prepared activations start at
// bsrc[k], with K splits sp[k] and split workspace part[k] / ctr[k].  Parameters are built in a
// static block under the caller's lock.
template <int FMT, int MPAD, int MAXE>
cudaError_t launch_main(const Job* jobs, const uint8_t* const* bsrc, const Split* sp, float* const* part,
                        unsigned* const* ctr, int count, int M, bool wide, cudaStream_t stream) {
  static TcParams<MAXE, naux(FMT, MAXE)> par;
  par.count = count;
  par.M = M;
  int tasks = 0;
  for (int k = 0; k < count; ++k) {
    cudaError_t err = weight_map(jobs[k].W, jobs[k].N, jobs[k].K, FMT, &par.maps[k]);
    if (err != cudaSuccess) return err;
    const int tiles = (int)((jobs[k].N + kTileRows - 1) / kTileRows);
    par.e[k] = TcEntry{jobs[k].Y, bsrc[k], part[k], ctr[k], (int)jobs[k].N, (int)jobs[k].K,
                       tiles, sp[k].splits, sp[k].chunk, chunks_of(jobs[k].K), tasks};
    tasks += tiles * sp[k].splits;
  }
  par.tasks_total = tasks;
  par.gated = (count == 1 && jobs[0].gated) ? 1 : 0;
  par.wait_polls = g_wait_polls.load(std::memory_order_relaxed);
  par.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  for (int k = 0; k < naux(FMT, MAXE) && k < count; ++k) par.aux[k] = jobs[k].aux;
  // Programmatic dependent launch: the kernel may start while the preparation kernel before it
  // in the stream still runs; it waits (griddepcontrol.wait) before it reads the prepared data.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)std::min(tasks, num_sms()));
  cfg.blockDim = dim3(0);   // set with the instance below
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (FMT == kFmtQ4K && MAXE == 1) {
    if (par.gated) {   // one product split into no tasks along K (split_for with whole rows)
      if constexpr (MPAD == 16) {
        if (M <= 8) return launch_instance<FMT, MPAD, 8, MAXE, true, 3>(cfg, par);
        return launch_instance<FMT, MPAD, 16, MAXE, true, 3>(cfg, par);
      } else {
        return launch_instance<FMT, MPAD, MPAD, MAXE, true, groups(MPAD, FMT, false)>(cfg, par);
      }
    }
  } else {
    if (par.gated) return cudaErrorNotSupported;   // the gated epilogue is Q4K's, single products
  }
  if constexpr (MPAD == 16) {
    if (M <= 8) return launch_instance<FMT, MPAD, 8, MAXE, false, 3>(cfg, par);
    return launch_instance<FMT, MPAD, 16, MAXE, false, 3>(cfg, par);
  } else if constexpr (MAXE > 1 || groups(MPAD, FMT, true) == groups(MPAD, FMT, false)) {
    return launch_instance<FMT, MPAD, MPAD, MAXE, false, groups(MPAD, FMT, true)>(cfg, par);   // batched: wide
  } else {
    if (wide) return launch_instance<FMT, MPAD, MPAD, MAXE, false, groups(MPAD, FMT, true)>(cfg, par);
    return launch_instance<FMT, MPAD, MPAD, MAXE, false, groups(MPAD, FMT, false)>(cfg, par);
  }
}

template <int MPAD, int NX, bool NAT>
cudaError_t launch_prep_n(const std::vector<std::pair<const uint16_t*, int64_t>>& xs, const std::vector<uint8_t*>& outs,
                          unsigned* zero, size_t zero_words, int M, cudaStream_t stream) {
  static PrepParams<NX> prep;   // built on the host, passed by value at launch
  prep.count = (int)xs.size();
  prep.M = M;
  prep.zero = zero;
  prep.zero_words = (int)zero_words;
  int blocks = 0;
  for (size_t u = 0; u < xs.size(); ++u) {
    prep.e[u] = PrepEntry{xs[u].first, outs[u], (int)xs[u].second, blocks};
    blocks += (int)(xs[u].second / 256);
  }
  prep.blocks_total = blocks;
  // plain stream order (launched early after a product kernel, this grid's CTAs waited on the
  // SMs that product left: single products at M >= 8 took 3-9 us longer on GB300)
  q4k_xprep_kernel<MPAD, NX, NAT><<<blocks, 8 * MPAD, 0, stream>>>(prep);
  return cudaGetLastError();
}

// The parameter block is copied at every launch: size it to the distinct activations.
template <int MPAD, bool NAT>
cudaError_t launch_prep(const std::vector<std::pair<const uint16_t*, int64_t>>& xs, const std::vector<uint8_t*>& outs,
                        unsigned* zero, size_t zero_words, int M, cudaStream_t stream) {
  if (xs.size() <= 1) return launch_prep_n<MPAD, 1, NAT>(xs, outs, zero, zero_words, M, stream);
  if (xs.size() <= 16) return launch_prep_n<MPAD, 16, NAT>(xs, outs, zero, zero_words, M, stream);
  return launch_prep_n<MPAD, kMaxPrep, NAT>(xs, outs, zero, zero_words, M, stream);
}

// Shared by the workspace and the no-allocation paths: prepare the distinct activations into
// `prep_base` (laid out by the caller), zero the split counters, and run the main kernel(s).
template <int FMT, int MPAD>
cudaError_t run_tc(const Job* jobs, int count, int M, cudaStream_t stream,
                   const std::vector<std::pair<const uint16_t*, int64_t>>& xs, const std::vector<uint8_t*>& outs,
                   const std::vector<int>& xidx, const std::vector<Split>& sp, uint8_t* split_base,
                   size_t zero_words) {
  std::vector<const uint8_t*> bsrc(count);
  std::vector<float*> part(count, nullptr);
  std::vector<unsigned*> ctr(count, nullptr);
  size_t off = 0, words = 0;
  for (int k = 0; k < count; ++k) {
    bsrc[k] = outs[xidx[k]];
    const SplitSpace s = split_space<MPAD>(jobs[k].N, jobs[k].K, sp[k]);
    if (s.partial_bytes) { part[k] = reinterpret_cast<float*>(split_base + off); off += s.partial_bytes; }
  }
  unsigned* counters = reinterpret_cast<unsigned*>(split_base + off);
  for (int k = 0; k < count; ++k) {
    const SplitSpace s = split_space<MPAD>(jobs[k].N, jobs[k].K, sp[k]);
    if (s.counter_words) { ctr[k] = counters + words; words += s.counter_words; }
  }
  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  // the blocks hold 8 token columns for the 8-token kernels (M <= 8), else MPAD
  cudaError_t err = (MPAD == 16 && M <= 8)
                        ? launch_prep<8, FMT == kFmtNVFP4>(xs, outs, counters, zero_words, M, stream)
                        : launch_prep<MPAD, FMT == kFmtNVFP4>(xs, outs, counters, zero_words, M, stream);
  if (err != cudaSuccess) return err;
  if (count == 1)
    return launch_main<FMT, MPAD, 1>(jobs, bsrc.data(), sp.data(), part.data(), ctr.data(), 1, M,
                                     wide_launch(jobs, 1, num_sms()), stream);
  // Launches of near-equal size, each with its products ordered by decreasing K (the kernel deals
  // tasks back and forth over its slots: large tasks first, then the small ones even them out).
  const int launches = (count + kMaxEBatch - 1) / kMaxEBatch;
  const int per = (count + launches - 1) / launches;
  std::vector<int> ord(count);
  for (int k = 0; k < count; ++k) ord[k] = k;
  std::vector<Job> pj(count);
  std::vector<const uint8_t*> pb(count);
  std::vector<Split> ps(count);
  std::vector<float*> pp(count);
  std::vector<unsigned*> pc(count);
  for (int k0 = 0; k0 < count; k0 += per) {
    const int n = std::min(per, count - k0);
    std::stable_sort(ord.begin() + k0, ord.begin() + k0 + n, [&](int a, int b) { return jobs[a].K > jobs[b].K; });
    for (int k = k0; k < k0 + n; ++k) {
      pj[k] = jobs[ord[k]];
      pb[k] = bsrc[ord[k]];
      ps[k] = sp[ord[k]];
      pp[k] = part[ord[k]];
      pc[k] = ctr[ord[k]];
    }
    err = launch_main<FMT, MPAD, kMaxEBatch>(pj.data() + k0, pb.data() + k0, ps.data() + k0, pp.data() + k0,
                                             pc.data() + k0, n, M, true, stream);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

template <int FMT, int MPAD>
cudaError_t launch_tc_t(const Job* jobs, int count, int M, cudaStream_t stream) {
  static_assert(sizeof(TcParams<kMaxEBatch, 1>) < 32000 && sizeof(PrepParams<kMaxPrep>) < 32000 &&
                sizeof(TcParams<kMaxEBatch, kMaxEBatch>) <= 32764, "kernel parameters too large");   // the launch limit
  const int kBB = bblock_bytes(MPAD == 16 && M <= 8 ? 8 : MPAD);   // one prepared block
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
  const int sms = num_sms();
  std::vector<Split> sp(count);
  size_t split_bytes = 0, zero_words = 0;
  for (int k = 0; k < count; ++k) {
    sp[k] = split_for(jobs[k].N, jobs[k].K, sms, groups(MPAD, FMT, wide_launch(jobs, count, sms) && !jobs[k].gated),
                      count > 1 || jobs[k].gated);   // gating needs whole rows
    const SplitSpace s = split_space<MPAD>(jobs[k].N, jobs[k].K, sp[k]);
    split_bytes += s.partial_bytes;
    zero_words += s.counter_words;
  }
  bytes = (bytes + 255) & ~(size_t)255;
  const size_t split_off = bytes;
  bytes += split_bytes + zero_words * sizeof(unsigned);
  void* wsp = nullptr;
  cudaError_t err = Workspace::get(stream, bytes, &wsp);
  if (err != cudaSuccess) return err;
  uint8_t* ws = static_cast<uint8_t*>(wsp);
  std::vector<uint8_t*> outs(xs.size());
  for (size_t u = 0; u < xs.size(); ++u) outs[u] = ws + xoff[u];
  return run_tc<FMT, MPAD>(jobs, count, M, stream, xs, outs, xidx, sp, ws + split_off, zero_words);
}

// ------------------------------------------------------------------------------------------
// Allocation-free entry (qmm_run_noalloc): the same two kernels, with the prepared activations
// in a fixed buffer that is part of this library's device image instead of the per-stream
// workspace, and no K split (a split needs workspace for its partial sums).  Every GPU that
// loads the library holds the buffer until the process exits.
constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

template <int MPAD>
cudaError_t launch_tc_noalloc_t(const Job& job, int M, cudaStream_t stream, uint8_t* scratch) {
  const std::vector<std::pair<const uint16_t*, int64_t>> xs{{job.X, job.K}};
  const std::vector<uint8_t*> outs{scratch};
  const std::vector<int> xidx{0};
  const std::vector<Split> sp{Split{1, (int)(job.K / 256)}};
  return run_tc<kFmtQ4K, MPAD>(&job, 1, M, stream, xs, outs, xidx, sp, scratch, 0);
}

}  // namespace

cudaError_t release_workspaces() { return Workspace::release(); }

void set_wait_limit(uint32_t polls, uint32_t suspend_ns) {
  g_wait_polls.store(polls, std::memory_order_relaxed);
  g_wait_ns.store(suspend_ns, std::memory_order_relaxed);
}
size_t workspace_bytes_held() { return Workspace::held_bytes(); }

cudaError_t read_and_clear_tc_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  *out = v;
  return e;
}

// Time model of a Q4K tensor-core launch over jobs[0 .. count), fitted to GB300 graph-replay
// timings: a fixed ~6 us (two launches, pipeline fill and drain) and the busiest dequant group's
// work (split_cost) at a full-CTA pace of 1.385 / 1.49 us per super-block of a tile for M <= 8 / 16
// (three groups) and 2.3 / 1.58 us for M <= 32 with three / two groups.  A batched launch (no
// splits) counts its tasks over all slots.
double tc_estimate_us(const Job* jobs, int count, int M) {
  const int sms = std::max(1, num_sms());
  const int ng = groups(M <= 16 ? 16 : 32, kFmtQ4K, wide_launch(jobs, count, sms));
  const double pace_us = M <= 8 ? 1.385 : (M <= 16 ? 1.49 : (ng == 3 ? 2.3 : 1.58));
  if (count == 1) return 6.0 + pace_us * split_cost(jobs[0].N, jobs[0].K, sms, ng, false).units;
  double tasks = 0, sbs = 0;
  for (int k = 0; k < count; ++k) {
    const double tiles = std::ceil((double)jobs[k].N / kTileRows);
    tasks += tiles;
    sbs += tiles * (double)(jobs[k].K / 256);
  }
  const double per_group_tasks = std::ceil(std::ceil(tasks / sms) / ng);
  return 6.0 + pace_us * per_group_tasks * (sbs / std::max(1.0, tasks));
}

bool tc_supports(int M, int64_t N, int64_t K) {
  return M >= 1 && M <= 32 && N >= 1 && K >= 256 && K % 256 == 0;
}

size_t noalloc_scratch_bytes() { return kNoallocScratchBytes; }

size_t noalloc_scratch_needed(int M, int64_t K) {
  return (size_t)(K / 256) * (size_t)bblock_bytes(M <= 8 ? 8 : (M <= 16 ? 16 : 32));
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
  const int fmt = jobs[0].fmt;
  for (int k = 1; k < count; ++k)
    if (jobs[k].fmt != fmt) return cudaErrorInvalidValue;   // one format per launch
  const bool narrow = M <= 16;
  switch (fmt) {
    case kFmtQ4K: return narrow ? launch_tc_t<kFmtQ4K, 16>(jobs, count, M, stream) : launch_tc_t<kFmtQ4K, 32>(jobs, count, M, stream);
    case kFmtQ5K: return narrow ? launch_tc_t<kFmtQ5K, 16>(jobs, count, M, stream) : launch_tc_t<kFmtQ5K, 32>(jobs, count, M, stream);
    case kFmtNVFP4: return narrow ? launch_tc_t<kFmtNVFP4, 16>(jobs, count, M, stream) : launch_tc_t<kFmtNVFP4, 32>(jobs, count, M, stream);
    case kFmtINT4: return narrow ? launch_tc_t<kFmtINT4, 16>(jobs, count, M, stream) : launch_tc_t<kFmtINT4, 32>(jobs, count, M, stream);
    case kFmtQ6K: return narrow ? launch_tc_t<kFmtQ6K, 16>(jobs, count, M, stream) : launch_tc_t<kFmtQ6K, 32>(jobs, count, M, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace q4k
