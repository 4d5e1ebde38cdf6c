/*
 * qmm.h — skinny-batch product of a 4-bit k-quant (Q4K) weight matrix with bf16 activations,
 * for one NVIDIA GB300 (sm_103a).
 *
 * What is computed.  The pages describe a speculative-decoding verify pass: anchor + k draft
 * rows go through the target model in one batch, and the quantized matrix products take
 * 83-92% of the GPU time ("sixi-asi 0.9", section "What I got wrong in 0.8").  Each such
 * product multiplies a weight matrix stored in 4-bit k-quant form with a skinny batch of
 * M = 1..32 activation rows.  This library computes exactly that product:
 *
 *     Y[i][n] = sum_k  w[n][k] * x[i][k]        0 <= i < M,  0 <= n < N,  0 <= k < K
 *
 * with x the bf16 activations, w the dequantized weights (below) and Y in fp32.  On the pages
 * the matrix-vector kernel decodes the 4-bit weights once per activation row ("sixi-asi 0.9",
 * same section); every kernel behind this header reads and decodes each weight byte once for
 * all M rows.
 *
 * ------------------------------------------------------------------------------------------
 * Q4K byte format.  The pages name the format (Q4_K_M GGUF weights, "sixi-asi 0.9" section
 * "Numbers") but print no byte layout; the fields are 256-weight super-blocks with fp16 d and
 * dmin, eight 32-weight sub-blocks with a 6-bit scale and a 6-bit min, and 4-bit quants, so
 * that w = d*sc*q - dmin*m.  This is the byte layout of this library:
 *
 *   A row of K weights (K a multiple of 256) is K/256 super-blocks of 256 consecutive weights,
 *   stored in order of k.  Rows are stored one after another, so super-block b of row n starts
 *   at byte  (n * (K/256) + b) * 144.  Every super-block is 144 bytes (4.5 bits per weight):
 *
 *     bytes [0, 2)    d     IEEE-754 binary16, little-endian   (scale of the scales)
 *     bytes [2, 4)    dmin  IEEE-754 binary16, little-endian   (scale of the mins)
 *     bytes [4, 16)   the 96-bit little-endian integer F.  Sub-block j (j = 0..7) owns
 *                     sc_j = bits [12j, 12j+6) of F and m_j = bits [12j+6, 12j+12) of F,
 *                     both unsigned 6-bit integers.
 *     bytes [16, 144) the 1024-bit little-endian integer Q.  Weight t of the super-block
 *                     (t = 0..255) has the unsigned 4-bit quant q_t = bits [4t, 4t+4) of Q:
 *                     byte 16 + t/2, low nibble for even t, high nibble for odd t.
 *                     Weight t belongs to sub-block j = t / 32.
 *
 *   Dequantization: with D = fp32(d) and Dm = fp32(dmin), weight t is the single
 *   round-to-nearest-even fp32 rounding of the exact real number D*sc_j*q_t - Dm*m_j.  (Both
 *   products are exact in fp32; the difference is rounded once.)  A zero weight is -0 exactly
 *   when D*sc_j*q_t is -0 and Dm*m_j is +0 (the IEEE-754 sign rule for a difference of
 *   zeros), otherwise +0.  qmm_dequant returns these values bit for bit.
 *
 * Quantizer used by qmm_pack (the pages give none; this is the plain asymmetric min/max rule):
 *   for each super-block and each sub-block j of 32 weights w_t:
 *     lo_j = min(0, min_t w_t),  hi_j = max_t w_t,  scale_j = (hi_j - lo_j)/15,  off_j = 0 - lo_j
 *   d = fp16(max(0, max_j scale_j) / 63), dmin = fp16(max(0, max_j off_j) / 63)
 *       (binary16 round to nearest even; the maxima start from +0, so no -0 is stored)
 *   sc_j = D > 0  ? clamp(rint(scale_j / D), 0, 63)  : 0
 *   m_j  = Dm > 0 ? clamp(rint(off_j / Dm), 0, 63)   : 0
 *   q_t  = D*sc_j > 0 ? clamp(rint((w_t + Dm*m_j) / (D*sc_j)), 0, 15) : 0
 *   All arithmetic is IEEE fp32, round to nearest even, each operation rounded separately.
 *
 * ------------------------------------------------------------------------------------------
 * Conventions for every call below.
 *   - Pointers named *_dev are CUDA device pointers, *_host are host pointers.  All buffers
 *     are owned by the caller; the library keeps no pointer after a call returns.
 *   - X is M x K row-major bf16 (raw bit patterns in uint16_t), Y is M x N row-major fp32.
 *     Wq and X must be 16-byte aligned; Y must be 4-byte aligned.  Y is overwritten, never
 *     accumulated, and must not overlap Wq or X.
 *   - 1 <= M <= 32, 1 <= N < 2^31, 256 <= K <= 2^20, K % 256 == 0.
 *   - GPU calls are asynchronous: they validate their arguments on the host, enqueue work on
 *     `stream` (0 = the legacy default stream) and return.  Argument errors are returned
 *     before anything is enqueued.  A launch failure returns QMM_ERR_CUDA (the CUDA error
 *     text is available from qmm_last_cuda_error).  Faults that happen while a kernel runs
 *     surface at the caller's next synchronization, as for any CUDA kernel.
 *   - Device memory: the tensor-core kernel keeps a workspace per (device, stream) for its
 *     prepared activations and K-split partial sums.  The first call on a stream that runs that
 *     kernel, and any later call that needs more room, allocates it with cudaMalloc (growing it
 *     frees the smaller one, which synchronizes the device); qmm_release frees every such
 *     workspace.  Every other buffer is the caller's.  qmm_run_noalloc allocates nothing.
 *   - Calls on different streams may run concurrently; the mutable global state (the workspace
 *     pool, a per-device cache of launch attributes and of tensor maps) is guarded by locks.
 *   - Stream order: the product kernels use programmatic dependent launch (each allows the next
 *     launch in the stream to be scheduled early; the library's own kernels wait for their
 *     predecessor before they depend on it).  A caller's kernel enqueued after a call sees
 *     every write of it as usual; one launched with programmatic stream serialization itself
 *     must wait for its prerequisite grid (cudaGridDependencySynchronize) before it reads Y.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMM_QK          256   /* weights per super-block                         */
#define QMM_BLOCK_BYTES 144   /* bytes per super-block                           */
#define QMM_MAX_M       32    /* largest activation batch (rows of X)            */
#define QMM_MAX_BATCH   512   /* largest entry count of one qmm_run_batched call */

typedef enum {
  QMM_OK = 0,
  QMM_ERR_NULL = 1,       /* a required pointer is NULL                                   */
  QMM_ERR_SHAPE = 2,      /* N or K out of range, or K % 256 != 0                          */
  QMM_ERR_M_RANGE = 3,    /* M outside [1, 32]                                             */
  QMM_ERR_ALIGN = 4,      /* Wq or X not 16-byte aligned, or Y not 4-byte aligned          */
  QMM_ERR_BUFSIZE = 5,    /* caller buffer smaller than required                          */
  QMM_ERR_NONFINITE = 6,  /* qmm_pack: a weight is Inf/NaN or a scale overflows fp16      */
  QMM_ERR_CUDA = 7,       /* a CUDA runtime call or kernel launch failed                   */
  QMM_ERR_COUNT = 8,      /* qmm_run_batched: count outside [1, QMM_MAX_BATCH]              */
  QMM_ERR_VARIANT = 9,    /* an explicitly requested kernel variant cannot run this shape  */
  QMM_ERR_SCRATCH = 10,   /* qmm_run_noalloc: problem larger than its fixed device buffer  */
  QMM_ERR_FORMAT = 11     /* qmm_fmt_*: unknown weight format code                         */
} qmm_status;

/* Bytes of the packed form of an N x K weight matrix: N * (K/256) * 144.
 * Returns 0 when the shape is invalid (see QMM_ERR_SHAPE). */
size_t qmm_packed_bytes(int64_t N, int64_t K);

/* Pack W_host (N x K row-major fp32, host memory) into the Q4K format above, written to the
 * caller's host buffer out_host of out_bytes >= qmm_packed_bytes(N, K) bytes.  Runs on the
 * host CPU (the cold path: weights are packed once), on up to `threads` threads (<= 0: all
 * hardware threads).  Errors: QMM_ERR_NULL, QMM_ERR_SHAPE, QMM_ERR_BUFSIZE,
 * QMM_ERR_NONFINITE; out_host is unspecified after an error. */
qmm_status qmm_pack(const float* W_host, int64_t N, int64_t K, void* out_host, size_t out_bytes,
                    int threads);

/* The same packing on the GPU: W_dev (N x K row-major fp32, device memory, 16-byte aligned)
 * into the caller's device buffer out_dev (16-byte aligned, out_bytes >= qmm_packed_bytes(N, K)),
 * enqueued on `stream`.  Every super-block is byte-identical to what qmm_pack writes (the
 * quantizer above, each step the same IEEE fp32 operation).  A super-block that holds a
 * non-finite weight, or whose d or dmin overflows binary16, is written as 144 zero bytes and
 * sets bit 1 of the device status word (qmm_device_status); qmm_pack instead rejects the whole
 * matrix with QMM_ERR_NONFINITE.  The weights are read once and not modified.  Errors (before
 * anything is enqueued): QMM_ERR_NULL, QMM_ERR_SHAPE, QMM_ERR_BUFSIZE, QMM_ERR_ALIGN;
 * QMM_ERR_CUDA if the launch fails. */
qmm_status qmm_pack_dev(const float* W_dev, int64_t N, int64_t K, void* out_dev, size_t out_bytes,
                        cudaStream_t stream);

/* Y_dev[M x N] = X_dev[M x K] * dequant(Wq_dev)^T, enqueued on `stream`.
 * Wq_dev: packed weights on the device (qmm_packed_bytes(N, K) bytes, 16-byte aligned).
 * X_dev: bf16 activations; Y_dev: fp32 result (overwritten).  The kernel variant is chosen
 * from (M, N, K) by the library's measured dispatch table (qmm_select_variant). */
qmm_status qmm_run(const void* Wq_dev, int64_t N, int64_t K, const uint16_t* X_dev,
                   float* Y_dev, int M, cudaStream_t stream);

/* One entry of a batched call: an independent product Y = X * dequant(Wq)^T. */
typedef struct {
  const void* Wq;      /* device, packed N x K */
  const uint16_t* X;   /* device, M x K bf16   */
  float* Y;            /* device, M x N fp32   */
  int64_t N;
  int64_t K;
} qmm_entry;

/* Run `count` independent products that share one M in one call on `stream`: one activation
 * preparation launch, then one product launch per 160 products (their tensor maps ride in the
 * launch parameters), equal in size, each allowed to start while the one before it finishes.
 * This is one pass over a model's layer matrices when every stream shares the pass
 * ("sixi-asi 0.11", section "Why sixteen streams were the ceiling"): many matrices, each
 * weight read once.  Entries may share X; the Y buffers must not overlap each other, any X
 * or any Wq.  entries_host is read during the call only (the work list travels in the
 * kernels' parameters; nothing is allocated besides the per-stream workspace).  Every entry is validated as in qmm_run; the
 * first invalid entry's error is returned and nothing is launched. */
qmm_status qmm_run_batched(const qmm_entry* entries_host, int count, int M, cudaStream_t stream);

/* Test hook: out_dev[N x K] (fp32, row-major) = the dequantized weights, computed on the
 * device with the same decode steps the product kernels use.  Bit-exact to the definition. */
qmm_status qmm_dequant(const void* Wq_dev, int64_t N, int64_t K, float* out_dev,
                       cudaStream_t stream);

/* Kernel variants.  qmm_run picks the one a cost model fitted to GB300 measurements predicts
 * faster (CUDA cores for one activation row and for small matrices, tensor cores otherwise);
 * qmm_run_variant forces one (tests and benchmarks use it to measure the switch point).
 * The tensor-core variant keeps a workspace for the prepared activations per (device, stream):
 * the first call on a stream, and any call that needs a larger one, allocates it with cudaMalloc
 * (make such a call before capturing the stream into a CUDA graph). */
typedef enum {
  QMM_VARIANT_AUTO = 0,
  QMM_VARIANT_FMA = 1,   /* CUDA cores: in-register dequant, fp32 FMA, warp-shuffle K reduce */
  QMM_VARIANT_TC = 2     /* tcgen05 tensor cores, fp32 accumulators in tensor memory        */
} qmm_variant;

/* As qmm_run with a forced variant; QMM_ERR_VARIANT if that variant cannot run the shape. */
qmm_status qmm_run_variant(const void* Wq_dev, int64_t N, int64_t K, const uint16_t* X_dev,
                           float* Y_dev, int M, int variant, cudaStream_t stream);

/* The variant qmm_run uses for this shape (never QMM_VARIANT_AUTO).  The environment variable
 * QMM_FORCE_VARIANT=fma or =tc, read once per process, makes every automatic choice take that
 * family (for tests and benchmarks). */
int qmm_select_variant(int M, int64_t N, int64_t K);

/* The variant qmm_run_batched uses for these entries (one family runs the whole batch);
 * -1 if the arguments are invalid. */
int qmm_select_variant_batched(const qmm_entry* entries_host, int count, int M);

/* Allocation-free variant of qmm_run (the pages have no counterpart; it exists for callers of
 * this library).  Some callers cannot allocate device memory when they call in: code that runs
 * while a stream is being captured into a CUDA graph (allocation is not a stream operation and
 * breaks or is barred from the capture), latency-critical decode loops that must never touch the
 * device allocator, and hosts that own a fixed device-memory budget or their own memory pool.
 * qmm_run may allocate on first use (the tensor-core kernel's per-stream workspace); this call
 * never does: it computes the same product with the tensor-core kernel and keeps the prepared
 * activations in a fixed buffer of QMM_NOALLOC_SCRATCH_BYTES (4 MiB) that is part of the
 * library's device image, held by every GPU that loads the library until the process exits.
 *   - Limit: (K/256) * (T*580 + 16) bytes must fit, T = 8 for M <= 8, 16 for M <= 16 and 32
 *     above: K <= 230400 for M <= 8, K <= 115456 for M <= 16, K <= 57600 for M > 16.  Larger
 *     problems return QMM_ERR_SCRATCH before anything is enqueued.
 *   - The first call on each device looks up the buffer's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream capture.
 *   - Every call shares the one buffer and leaves its contents behind; each call writes every
 *     byte it reads before reading it, so nothing has to start zeroed.  Calls that overlap on the
 *     GPU (concurrent streams, or host threads whose calls are not ordered) race on the buffer:
 *     order them on one stream or serialize them.
 * Arguments, layouts and the other errors are those of qmm_run. */
#define QMM_NOALLOC_SCRATCH_BYTES (4u << 20)
qmm_status qmm_run_noalloc(const void* Wq_dev, int64_t N, int64_t K, const uint16_t* X_dev,
                           float* Y_dev, int M, cudaStream_t stream);

/* One feed-forward block of the verify pass: the two matrices the configurations give per layer
 * ("Single FFN layer decode": the fused gate/up matrix and the down matrix; the pages time the
 * fused gate/up product as "gate+up", FlashRT issue #153, the tile-bench tables) run as one
 * dependent chain on `stream`:
 *     G[M x 2F] = X[M x K] * dequant(Wgu)^T          (fp32; columns 0..F-1 gate, F..2F-1 up)
 *     H[M x F]  = bf16( silu(G[:, f]) * G[:, F + f] ), silu(g) = g / (1 + e^-g), in fp32,
 *                 rounded once to bf16 (round to nearest even)
 *     Y[M x K]  = H * dequant(Wdown)^T               (fp32)
 * (the pages do not print the gating function between the two products; SiLU-gated is the
 * plainest reading for the model family they run).
 *   Wgu_dev: packed (2F) x K weights, gate rows 0..F-1 then up rows F..2F-1.
 *   Wdown_dev: packed K x F weights.  F and K are multiples of 256.
 *   X_dev: M x K bf16.  Y_dev: M x K fp32 (overwritten).
 *   workspace_dev: caller-owned device memory of at least qmm_ffn_workspace_bytes(M, F) bytes,
 *     16-byte aligned; it holds G and H (the library allocates nothing for the chain itself;
 *     the two products behave as qmm_run).  Both products are checked as in qmm_run; then
 *     QMM_ERR_ALIGN (workspace), QMM_ERR_BUFSIZE (workspace too small), QMM_ERR_NULL.
 * Each product picks its kernel variant as qmm_run does. */
size_t qmm_ffn_workspace_bytes(int M, int64_t F);
qmm_status qmm_run_ffn(const void* Wgu_dev, const void* Wdown_dev, int64_t F, int64_t K, const uint16_t* X_dev,
                       float* Y_dev, int M, void* workspace_dev, size_t workspace_bytes, cudaStream_t stream);

/* The same block with the gating fused into the gate/up product's epilogue (no G in memory, one
 * launch fewer): Wgu_dev holds the gate and up rows interleaved, row 2f = gate row f and row
 * 2f+1 = up row f, so that each pair sits in neighbouring lanes of the kernel; H is formed from
 * the fp32 results of the pair exactly as qmm_run_ffn forms it from G.  The gate/up product
 * always runs on the tensor cores and is never split along K; the down product is chosen as in
 * qmm_run.  workspace_dev (16-byte aligned) holds H: at least qmm_ffn_fused_workspace_bytes(M, F)
 * bytes.  Errors as qmm_run_ffn. */
size_t qmm_ffn_fused_workspace_bytes(int M, int64_t F);
qmm_status qmm_run_ffn_fused(const void* Wgu_interleaved_dev, const void* Wdown_dev, int64_t F, int64_t K,
                             const uint16_t* X_dev, float* Y_dev, int M, void* workspace_dev,
                             size_t workspace_bytes, cudaStream_t stream);

/* Indexed-expert product (the matrix-product-by-id case that the pages' backend op tests cover
 * next to the plain product: "sixi-asi 0.9", section "The patch", MUL_MAT and MUL_MAT_ID): row i
 * of X is multiplied by the weight matrix of expert ids_host[i],
 *     Y[i][n] = sum_k w_{ids[i]}[n][k] * x[i][k],   0 <= i < M,
 * with the same dequantization and rounding as qmm_run (each expert's rows are one product of
 * the batched launch; results as qmm_run_batched on those rows).  When every row has the same
 * expert, the call is that expert's qmm_run on X and Y directly (no gather, no scatter).
 *   experts_host: n_experts device pointers (host array), each a packed N x K matrix.
 *   ids_host: M expert indices (host array, read during the call), 0 <= ids[i] < n_experts.
 *   X_dev: M x K bf16; Y_dev: M x N fp32 (overwritten).
 *   workspace_dev: caller-owned device memory, >= qmm_indexed_workspace_bytes(M, N, K) bytes,
 *     16-byte aligned (gathered rows and results; the library allocates nothing else here).
 * Errors as qmm_run_batched, plus QMM_ERR_SHAPE (an id out of range), QMM_ERR_COUNT (n_experts
 * outside [1, QMM_MAX_BATCH]), QMM_ERR_ALIGN / QMM_ERR_BUFSIZE (workspace). */
size_t qmm_indexed_workspace_bytes(int M, int64_t N, int64_t K);
qmm_status qmm_run_indexed(const void* const* experts_host, int n_experts, int64_t N, int64_t K,
                           const int32_t* ids_host, const uint16_t* X_dev, float* Y_dev, int M,
                           void* workspace_dev, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Other weight formats.  The pages run Q4_K_M files, which mix k-quant widths ("sixi-asi 0.9",
 * section "Numbers"), and weigh two other 4-bit layouts: NVFP4 W4A16 weights on Blackwell
 * tensor cores (FlashRT issue #153: the NVFP4 W4A16 GEMM is most of the decode time; "sixi-asi
 * 0.9", section "What I got wrong in 0.8": block-scaled FP4 reached through tcgen05) and plain
 * 4-bit integers with one scale per 128 columns ("sixi-asi 0.11", section "What did not work").
 * None prints a byte layout; these are this library's.  Every weight below is one IEEE
 * rounding of an exact number, and qmm_fmt_dequant returns it bit for bit.
 *
 *   QMM_FMT_Q4K   the Q4K format above.
 *   QMM_FMT_Q5K   176 bytes per super-block of 256 weights of a row (rows one after another):
 *                 bytes [0, 16) as in Q4K (d, dmin, the 96-bit F of (sc_j, m_j));
 *                 bytes [16, 48) eight 32-bit little-endian words, word j the high bits of
 *                 sub-block j: weight t = 32j + 8c + i (c = 0..3, i = 0..7) has its high bit
 *                 at bit 4i + c (the layout the decode reads in one shift per pair);
 *                 bytes [48, 176) the low 4 bits of weight t at bits [4t, 4t+4), as Q4K.
 *                 q_t = low + 16 high (0..31); weight = RN32(d*sc_j*q_t - dmin*m_j).
 *   QMM_FMT_NVFP4 144 bytes per 256 weights: bytes [0, 16) sixteen E4M3 scales (sign, 4
 *                 exponent bits with bias 7, 3 fraction bits; largest 448), s_b for weights
 *                 16b .. 16b+15; bytes [16, 144) the E2M1 codes (sign, 2 exponent bits with
 *                 bias 1, 1 fraction bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6) of weight t at bits
 *                 [4t, 4t+4).  After all N rows: a 16-byte trailer, the binary32 tensor scale
 *                 g then 12 zero bytes.  weight = RN32(g * s_b * v_t).
 *   QMM_FMT_Q6K   208 bytes per super-block of 256 weights of a row (rows one after another),
 *                 then at byte N*(K/256)*208 a plane of N x K/256 binary16 super-block scales d:
 *                 bytes [0, 16) u_j for sub-blocks j of 16 weights, sc_j = (u_j & 127) - 64
 *                 (a 7-bit signed scale; bit 7 unused); bytes [16, 144) the low 4 bits of weight
 *                 t at bits [4t, 4t+4); bytes [144, 208) sixteen 32-bit little-endian words, word
 *                 m the 2-bit high parts of weights 16m .. 16m+15: weight 16m + 8a + i (a = 0..1,
 *                 i = 0..7) at bits 8a + 16 (i >= 4) + 2 (i % 4).  q_t = low + 16 high (0..63);
 *                 weight = RN32(d*sc_j*(q_t - 32)) (exact: at most 23 significant bits).  The
 *                 7-bit scales keep sc*(q - 32) within 2048, exact in fp16 on the tensor cores.
 *   QMM_FMT_INT4  a quant plane of N rows of K/2 bytes (weight k of a row: the two's-complement
 *                 4-bit integer at bits [4k, 4k+4) of the row), then at byte N*K/2 a scale
 *                 plane of N x K/128 binary16 scales, row-major; weight = s * q (exact).
 *
 * Packers (plain rules; binary32 arithmetic, one rounding per operation):
 *   Q5K   the Q4K rule with 31 levels: scale_j = (hi_j - lo_j)/31, q clamped to [0, 31].
 *   NVFP4 g = max|w| / 2688 (6 * 448; 1 if that is not positive); per 16 weights
 *         s = E4M3(max|w| / 6 / g), round to nearest even, clamped to 448; S = s * g;
 *         v = E2M1(w / S), nearest even, clamped to 6, sign kept (S = 0: v = +0).
 *   INT4  per 128 weights s = binary16(max|w| / 7); q = S > 0 ? clamp(rint(w / S), -8, 7) : 0
 *         (S = the value of s).
 *   Q6K   per 16 weights scale_j = max|w| / 31; d = binary16(max_j scale_j / 63); sc_j =
 *         D > 0 ? clamp(rint(scale_j / D), 0, 63) : 0; q = D*sc_j > 0 ? clamp(rint(w / (D*sc_j)),
 *         -32, 31) + 32 : 32 (D = the value of d).
 *
 * The products run on the tensor cores (the CUDA-core kernel is Q4K's); the other conventions
 * are those of qmm_run.  Shapes: as for Q4K (K % 256 == 0). */
typedef enum {
  QMM_FMT_Q4K = 0,
  QMM_FMT_Q5K = 1,
  QMM_FMT_NVFP4 = 2,
  QMM_FMT_INT4 = 3,
  QMM_FMT_Q6K = 4
} qmm_format;

/* Bytes of the packed form of an N x K matrix in format fmt (0 for an invalid shape or
 * format): Q4K N*(K/256)*144, Q5K N*(K/256)*176, NVFP4 N*(K/256)*144 + 16,
 * INT4 N*K/2 + N*(K/128)*2, Q6K N*(K/256)*210. */
size_t qmm_fmt_packed_bytes(int fmt, int64_t N, int64_t K);

/* Pack W_host (N x K row-major fp32, host) into format fmt, as qmm_pack does for Q4K.
 * Errors: QMM_ERR_FORMAT, QMM_ERR_NULL, QMM_ERR_SHAPE, QMM_ERR_BUFSIZE, QMM_ERR_NONFINITE. */
qmm_status qmm_fmt_pack(int fmt, const float* W_host, int64_t N, int64_t K, void* out_host,
                        size_t out_bytes, int threads);

/* Y_dev[M x N] = X_dev[M x K] * dequant(Wq_dev)^T for weights packed in format fmt
 * (qmm_fmt_packed_bytes(fmt, N, K) bytes on the device, 16-byte aligned).  QMM_FMT_Q4K is
 * qmm_run.  Errors as qmm_run, and QMM_ERR_FORMAT. */
qmm_status qmm_fmt_run(int fmt, const void* Wq_dev, int64_t N, int64_t K, const uint16_t* X_dev,
                       float* Y_dev, int M, cudaStream_t stream);

/* One entry of a batched call over weight formats: an independent product in format fmt. */
typedef struct {
  int fmt;             /* qmm_format code */
  const void* Wq;      /* device, packed N x K in format fmt */
  const uint16_t* X;   /* device, M x K bf16 */
  float* Y;            /* device, M x N fp32 */
  int64_t N;
  int64_t K;
} qmm_fmt_entry;

/* Run `count` independent products sharing one M whose weights may be in different formats (a
 * model file mixes k-quant widths, "sixi-asi 0.9", section "Numbers"): the entries are grouped
 * by format and each group runs as qmm_run_batched does (its own launches, the groups in
 * order of format code, on `stream`).  Entries are validated as in qmm_fmt_run; the first
 * invalid entry's error is returned and nothing is launched.  Each result equals the one of a
 * single qmm_fmt_run call bit for bit. */
qmm_status qmm_fmt_run_batched(const qmm_fmt_entry* entries_host, int count, int M, cudaStream_t stream);

/* Test hook: out_dev[N x K] = the dequantized weights of format fmt, computed on the device
 * with the decode steps of the product kernel.  Bit-exact to the definitions above. */
qmm_status qmm_fmt_dequant(int fmt, const void* Wq_dev, int64_t N, int64_t K, float* out_dev,
                           cudaStream_t stream);

/* Measurement probe: read bytes (a multiple of 16) of device memory at buf_dev exactly once,
 * with 16-byte loads that bypass L1 and are marked evict-first in L2, and write one word per CTA
 * (an XOR of what it read) to sink_dev, which holds qmm_stream_read_sink_words() words.  Timed
 * over a buffer much larger than L2, it gives the HBM read bandwidth this GPU reaches from a
 * kernel that only reads: the ceiling of the weight stream, against which the products' GB/s are
 * compared (the pages check their kernels' GB/s against the memory system's own numbers: FlashRT
 * issue #153, the device-to-device bandwidth check and the sustained-read microtest).
 * Enqueued on `stream`; errors: QMM_ERR_NULL, QMM_ERR_SHAPE, QMM_ERR_ALIGN, QMM_ERR_CUDA. */
size_t qmm_stream_read_sink_words(void);
qmm_status qmm_stream_read(const void* buf_dev, size_t bytes, uint32_t* sink_dev, cudaStream_t stream);

/* Free every tensor-core workspace the library holds (one per device and stream that ran the
 * tensor-core kernel; see "Device memory" above).  A synchronous call: cudaFree waits for the
 * work that may still use a workspace.  Later calls allocate again as needed.  Do not call it
 * while a stream that the library uses is being captured into a CUDA graph, or while a graph
 * that recorded a call of this library may still be launched (the graph refers to the freed
 * workspace).  Errors: QMM_ERR_CUDA. */
qmm_status qmm_release(void);

/* Bytes of device memory the tensor-core workspaces hold now (0 after qmm_release). */
size_t qmm_workspace_bytes_held(void);

/* Failure-detection hook.  Every wait inside the tensor-core kernel (for its weight copies, for
 * its tensor-core work, between its warps) is bounded: by default 2^17 polls of at most 20 us.
 * When a bound runs out the kernel sets bit 0 of the device status word (qmm_device_status),
 * stops its other warps at their next wait, waits for the copies and tensor-core operations it
 * has already issued (with the default bound), releases its tensor memory and returns; the
 * outputs of that call are invalid and the context stays usable.  This call sets the bound of
 * the launches made from now on to `polls` polls of at most `suspend_ns` nanoseconds each
 * (0, 0 restores the default), for every thread and stream of the process: a test hook, which
 * with a bound far below a memory access's latency makes the first wait run out. */
void qmm_set_wait_limit(uint32_t polls, uint32_t suspend_ns);

/* Read and clear the status word that the kernels of this library keep on the current device
 * (a synchronous call: it waits for the device).  0: no kernel reported a problem since the
 * last read.  Bit 0: a kernel stopped waiting for its own weight copies after a bounded number
 * of polls; the outputs of the calls since the last read are then invalid.  Bit 1: qmm_pack_dev
 * met a non-finite weight or an fp16 scale overflow and wrote zeros for that super-block. */
qmm_status qmm_device_status(unsigned* status_out);

/* Human-readable text of a status code (static storage). */
const char* qmm_strerror(qmm_status status);

/* Text of the CUDA error behind the last QMM_ERR_CUDA returned on this thread. */
const char* qmm_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
