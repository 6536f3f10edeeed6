/*
 * qmm.h -- C ABI of the GB300 verify matmul for speculative decoding.
 *
 * The operation.  One speculative-decoding step checks a whole drafted block
 * of M token positions with a single batched forward of the target model; in
 * that forward every weight matrix is read once and applied to all M rows, so
 * checking 16 positions costs about as much as checking one
 * ["Qwen3.8-27B on the AMD R9700: up to 227 tok/s", section "A block-diffusion
 * drafter, verified exactly"].  The hot part of that forward is the skinny
 * block-quantized matmul this library computes:
 *
 *     out[m][n] = sum_k act[m][k] * W[n][k]       1 <= M <= 16, fp32 accumulate
 *
 * with W stored compressed:
 *   QMM_FMT_Q4_0           32-element blocks, one fp16 scale d per block, 4-bit
 *                          codes q with an offset of 8: W = d * (q - 8)
 *                          ["Qwen3.8-27B at 45.7 tok/s: DFlash2 in 1bit serve,
 *                          and 4-bit activations with a Hadamard rotation",
 *                          section "Prompt processing: 4-bit activations,
 *                          rotated first"].
 *   QMM_FMT_FP8_E4M3_B128  E4M3 (OCP FN) codes with one fp32 scale per 128x128
 *                          tile: W = e4m3(c) * s[n/128][k/128]
 *                          ["r9k: a from-scratch inference engine for
 *                          Qwen3.8-27B on two Radeon AI PRO R9700", opening
 *                          section].

 *   QMM_FMT_Q8_0           32-element blocks, one fp16 scale d each, 8-bit
 *                          two's-complement codes: W = d * q (the 8-bit
 *                          reference format the pages name beside Q4_0,
 *                          ["Qwen3.8-27B on the AMD R9700: up to 227 tok/s",
 *                          TL;DR], read as the GGUF block layout of the same
 *                          family).  Its activations always take the f16
 *                          pre-pass, as FP8's do.
 * and optionally QMM_FLAG_HADAMARD32: every 32-block of each activation row is
 * rotated on the device by the unnormalised 32-point Walsh-Hadamard matrix H
 * (strides 1,2,4,8,16, each stage (x, y) -> (x + y, x - y), fp32), for weights
 * that were rotated the same way offline and divided by 32 (see
 * qmm_quantize_q4_0), so the product equals the unrotated one
 * ["Qwen3.8-27B at 45.7 tok/s ...", same section].  QMM_FLAG_HADAMARD64 and
 * QMM_FLAG_HADAMARD128 do the same with 64- and 128-point blocks, the larger
 * rotations that page lists as its next step ("What's next"), with the same
 * stride-ascending stage order (strides 1, 2, ..., B/2) and weights divided by
 * B; at most one of the three is set.
 *
 * qmm_prefill computes the same product for a prompt's worth of rows (any M)
 * on an FP8 handle, as a tensor-core GEMM (see its comment below).
 *
 * Conventions for every entry point:
 *   - Return value: QMM_OK (0) or one of the QMM_ERR_* codes below.  No call
 *     throws, aborts or prints.  qmm_strerror() names a code.
 *   - "device" pointers are CUDA global-memory pointers of the current device;
 *     "host" pointers are ordinary (pageable or pinned) host memory.
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls documented as asynchronous only enqueue work on it.
 *   - The caller owns every buffer it passes; the library never frees caller
 *     memory and keeps no pointer to it after the call returns (the one
 *     exception is the stamp buffer of the profiling hook qmm_debug_set_trace,
 *     kept until it is switched off or the handle is destroyed).
 *   - bf16 activations are passed as uint16_t bit patterns.
 */
#ifndef QMM_H_
#define QMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMM_ABI_VERSION 1

/* ---- status codes ------------------------------------------------------- */
enum {
  QMM_OK = 0,
  QMM_ERR_INVALID_ARG = 1, /* NULL pointer, bad enum, bad struct_size, bad flag */
  QMM_ERR_SHAPE = 2,       /* N or K not accepted by the format (see qmm_desc)   */
  QMM_ERR_M_RANGE = 3,     /* M outside [1, 16] (prefill: [1, QMM_PREFILL_MAX_M]) */
  QMM_ERR_ALIGN = 4,       /* pointer alignment or leading dimension rejected   */
  QMM_ERR_CUDA = 5,        /* a CUDA call failed; see qmm_last_cuda_error()     */
  QMM_ERR_TIMEOUT = 6,     /* a bounded device wait expired (qmm_sync_status)   */
  QMM_ERR_STATE = 7,       /* NULL, destroyed or otherwise unusable handle      */
  QMM_ERR_DEVICE = 8       /* no sm_103 device, or the handle's device is not current */
};

/* ---- formats and flags ---------------------------------------------------- */
typedef enum { QMM_FMT_Q4_0 = 0, QMM_FMT_FP8_E4M3_B128 = 1, QMM_FMT_Q8_0 = 2 } qmm_format;

enum {
  /* Rotate each 32-block of the activations on the device (weights must have
   * been rotated offline the same way and divided by 32). */
  QMM_FLAG_HADAMARD32 = 1u << 0,
  /* Use the CUDA-core (FP32 FMA) verify kernel instead of the tensor-core one.
   * Same results within the tolerance; kept as the measured baseline. */
  QMM_FLAG_SIMT = 1u << 1,
  /* Q4_0 without rotation: use the tcgen05 kernel (dequantized weights in
   * tensor memory, one MMA issuer per CTA) instead of the default warp-level
   * mma.sync kernel.  Same results within the tolerance; slower at M <= 16,
   * where a 128x16x16 tcgen05 MMA costs about as much as a 128x256x16 one. */
  QMM_FLAG_TCGEN05 = 1u << 2,
  /* As QMM_FLAG_HADAMARD32 with 64- or 128-point blocks (weights rotated the
   * same way offline and divided by 64 or 128); K must be a multiple of the
   * block.  At most one rotation flag. */
  QMM_FLAG_HADAMARD64 = 1u << 3,
  QMM_FLAG_HADAMARD128 = 1u << 4
};

/* Description of one weight matrix W[N][K]. */
typedef struct {
  uint32_t struct_size;      /* = sizeof(qmm_desc)                              */
  uint32_t format;           /* qmm_format                                      */
  int64_t N;                 /* output features (rows of W), N >= 1             */
  int64_t K;                 /* input features; Q4_0 and Q8_0: K % 32 == 0;
                                FP8: N % 128 == 0 and K % 128 == 0              */
  uint32_t flags;            /* QMM_FLAG_*                                      */
  int32_t weights_on_device; /* 1: weights/scales are device pointers; 0: host  */
  const void* weights;       /* Q4_0: N*(K/32) blocks of 18 bytes, row-major over
                                n then block: fp16 d (little endian), then 16 bytes
                                where byte j holds element j in its low nibble and
                                element j+16 in its high nibble.
                                FP8: uint8 E4M3 codes [N][K], row-major.
                                Q8_0: N*(K/32) blocks of 34 bytes, row-major over
                                n then block: fp16 d (little endian), then the
                                32 int8 codes in order.                          */
  const float* scales;       /* FP8: fp32 [N/128][K/128] row-major; Q4_0: NULL  */
  int32_t k_splits;          /* 0: the planner chooses; > 0: use this many K splits
                                (tuning and tests; clamped to the stage count
                                and to 16, the largest cluster)                 */
} qmm_desc;

/* Opaque handle: owns the device copy of W (repacked for the kernels) and the
 * per-handle scratch.  A handle may be used from one stream at a time. */
typedef struct qmm_handle* qmm_t;

/* What a handle holds and how it will launch (for benchmarks and tests). */
typedef struct {
  uint32_t struct_size;          /* = sizeof(qmm_info), set by the caller      */
  uint32_t format, flags;
  int64_t N, K;
  int64_t weight_bytes;          /* compressed bytes of W as the format defines
                                    them: Q4_0 N*K*18/32; Q8_0 N*K*34/32;
                                    FP8 N*K + 4*(N/128)*(K/128)                 */
  int64_t device_weight_bytes;   /* bytes of the repacked device copy (with padding) */
  int64_t scratch_bytes;         /* per-handle scratch                          */
  int32_t n_tiles;               /* row tiles of the verify grid                */
  int32_t k_splits;              /* K splits of the verify grid                 */
  int32_t ctas;                  /* CTAs per verify launch                      */
  int32_t stages_per_cta;        /* pipeline stages each CTA streams            */
  int32_t stage_bytes;           /* weight bytes of one stage                   */
  int32_t pipeline_depth;        /* stages in flight per CTA                    */
  int32_t device;                /* CUDA device ordinal the handle lives on     */
  int32_t sm_count;
} qmm_info;

/* ---- lifetime --------------------------------------------------------------- */

/* Create a handle for W.  Validates the description, allocates the device copy
 * and scratch, and repacks W on the device (from host memory if
 * weights_on_device == 0).  Returns after the repack finished on `stream`, so
 * the caller may free its weight buffers right away.
 * Errors: INVALID_ARG (NULL out/desc/weights, unknown format or flag, FP8
 * without scales), SHAPE (see qmm_desc), DEVICE, CUDA (allocation or copy
 * failure; nothing is leaked and *out is set to NULL). */
int qmm_create(qmm_t* out, const qmm_desc* desc, void* stream);

/* A handle over the rows [n_begin, n_end) of the matrix `desc` describes
 * (desc->N, desc->weights and desc->scales describe the whole W[N][K]): its
 * matrix is W[n_begin .. n_end - 1], N' = n_end - n_begin rows, so qmm_verify
 * on it writes out[m][0 .. N' - 1] = columns n_begin .. n_end - 1 of the full
 * product.  This is the unit of the multi-GPU split: the rows of W are
 * independent, so GPU g of G takes rows [g N / G, (g + 1) N / G) and computes
 * its columns with no reduction; an all-gather of the [M][N'] parts assembles
 * the result (r9k splits its model over two GPUs, "r9k: a from-scratch
 * inference engine for Qwen3.8-27B on two Radeon AI PRO R9700", opening
 * section; here the split needs no all-reduce).  Same ownership and
 * synchronisation as qmm_create.
 * Errors: as qmm_create, plus SHAPE when n_begin < 0, n_end > N, the range is
 * empty, or (FP8) n_begin or n_end is not a multiple of 128 (n_end == N
 * excepted, which is one already). */
int qmm_create_rows(qmm_t* out, const qmm_desc* desc, int64_t n_begin, int64_t n_end, void* stream);

/* Destroy a handle and free everything it owns (synchronises its device work
 * first).  NULL is accepted.  Using a handle after this returns QMM_ERR_STATE. */
int qmm_destroy(qmm_t h);

/* ---- the verify product ------------------------------------------------------ */

/* out[m][n] = sum_k act[m][k] * W[n][k] for 0 <= m < M, 0 <= n < N.
 *   act : device, bf16 bits, row m at act + m*lda; 16-byte aligned, lda >= K,
 *         lda % 8 == 0 (so every row starts on a 16-byte boundary).
 *   out : device, fp32, row m at out + m*ldo; 16-byte aligned, ldo >= N.  Fully
 *         overwritten (the caller does not clear it); rows >= M are untouched.
 * Asynchronous on `stream`: enqueues the activation pre-pass and the verify
 * kernel and returns; never synchronises.  Row m's result is bit-identical for
 * every M (the same kernel and summation order serves M = 1..16).
 * Errors: STATE, M_RANGE, INVALID_ARG (NULL act/out), ALIGN, CUDA (launch). */
int qmm_verify(qmm_t h, const uint16_t* act, int64_t lda, float* out, int64_t ldo,
               int M, void* stream);

/* The verify product followed by greedy acceptance of the drafted block, the
 * step that decides what is committed ["Qwen3.8-27B on the AMD R9700: up to
 * 227 tok/s", sections "A block-diffusion drafter, verified exactly" and
 * "What 'lossless' means here, precisely": every drafted token is checked
 * against the target's own greedy choice and the agreeing prefix is kept].
 * W is the output head (N = vocabulary size) and act the M block positions'
 * final hidden rows.  Computes out exactly as qmm_verify, and then
 *   argmax[m] = the first n with out[m][n] == max_n out[m][n] (a NaN counts
 *               as larger than every number; -0 and +0 are equal),
 *   accept[0] = k, the largest k <= M - 1 with argmax[m] == tokens[m + 1]
 *               for every m < k (the number of accepted drafts),
 *   accept[1] = argmax[k], the target's own token after them.
 *   tokens : device, int32 [M]: the block's input tokens; tokens[0] is the
 *            last committed token, tokens[1..M-1] the drafts.
 *   argmax : device, int32 [M], written.   accept : device, int32 [2], written.
 * The argmax is taken inside the verify kernel: every finished row tile folds
 * its best (score, row) pair into a per-handle maximum with one atomic, and
 * the last tile to finish writes argmax and accept, so the result needs no
 * second pass over the scores.  Because row results are bit-identical for every
 * M, so is argmax: a batched verify of M positions picks the same tokens as M
 * single-row calls.  Asynchronous on `stream`, like qmm_verify; the handle's
 * greedy state is per handle (one stream at a time).
 * Errors: as qmm_verify, plus INVALID_ARG (NULL tokens/argmax/accept, or a
 * handle created with QMM_FLAG_TCGEN05) and ALIGN (tokens/argmax/accept not
 * 4-byte aligned). */
int qmm_verify_greedy(qmm_t h, const uint16_t* act, int64_t lda, float* out, int64_t ldo, int M,
                      const int32_t* tokens, int32_t* argmax, int32_t* accept, void* stream);

/* The same product for callers that hold host buffers: copies act to the
 * handle's device staging buffer, runs qmm_verify, copies the result back into
 * out_host and waits for `stream` before returning (synchronous).  Pinned
 * host memory gives the fastest copies.  Same argument rules as qmm_verify
 * except that the 16-byte alignment rule does not apply to host pointers. */
int qmm_verify_host(qmm_t h, const uint16_t* act_host, int64_t lda, float* out_host,
                    int64_t ldo, int M, void* stream);

/* The same product as qmm_verify, for callers that cannot have device memory
 * allocated for them.  The pages have no counterpart of this call.  Some
 * callers may not allocate device memory when they run: code captured into a
 * CUDA graph under the global capture mode (cudaMalloc is refused there), or a
 * host runtime that owns every device allocation and hands the library only
 * the buffers it passes.  This call allocates nothing and does not use the
 * working memory of the handle: the rotated or f16 activation rows and their
 * per-(row, split) factors (the Hadamard and FP8 / Q8_0 paths), the split-K
 * partials and the per-tile arrival counts (plans with more than one K split)
 * live in one fixed array of QMM_NOALLOC_SCRATCH_BYTES bytes inside the
 * library, which every GPU that loads the library holds until the process
 * exits.  The handle (created earlier, which does allocate) supplies the
 * weights and the status word; act and out follow qmm_verify's rules.
 *   - The first call on a device looks up the array's device address (once,
 *     with that device current); make that first call before any stream
 *     capture.
 *   - All calls share the array and it keeps the last call's contents.  Every
 *     call rewrites the parts it reads before reading them, and clears the
 *     arrival counts (which must start at zero) with an asynchronous memset on
 *     `stream` first.  Calls that overlap on the GPU (other streams, other
 *     threads) race on the array and give wrong results; serialise them.
 *   - Asynchronous on `stream`.
 * Errors: as qmm_verify, plus QMM_ERR_SHAPE when the handle's plan needs more
 * than the array holds (f16 activations for K above about 127,000 columns, or
 * rows x splits beyond about 500 row tiles x K splits). */
#define QMM_NOALLOC_SCRATCH_BYTES (4u << 20)
int qmm_verify_noalloc(qmm_t h, const uint16_t* act, int64_t lda, float* out, int64_t ldo,
                       int M, void* stream);

/* ---- the prefill product --------------------------------------------------------- */

/* The same product for a prompt's worth of rows, on an FP8 handle:
 *     out[m][n] = sum_k act[m][k] * W[n][k]       1 <= M <= QMM_PREFILL_MAX_M
 * the block-scaled FP8 GEMM that processes the prompt ["r9k: a from-scratch
 * inference engine for Qwen3.8-27B on two Radeon AI PRO R9700", opening
 * section: prefill runs through a custom block-scaled FP8 GEMM over the
 * 128 x 128-scaled E4M3 weights].  It reads the handle's weights as they are
 * (no second copy) and runs on the tcgen05 tensor cores: each activation row
 * (rotated first for the Hadamard flags) is scaled by a power of two 2^e that
 * brings its largest magnitude into [2^14, 2^15), converted to f16 (exact for
 * unrotated bf16 rows down to 2^-17 after scaling; the page's prefill also
 * keeps 16-bit activations) and written to the workspace; the codes are converted to f16 exactly; every 128 x 128
 * tile product is accumulated in fp32, multiplied by its tile's scale and
 * added in fp32, and the row's sum is multiplied by 2^-e.  The result is held
 * to the same tolerance as qmm_verify.
 *   act : device, bf16 bits, row m at act + m*lda; 16-byte aligned, lda >= K,
 *         lda % 8 == 0.
 *   out : device, fp32, row m at out + m*ldo; 16-byte aligned, ldo >= N.  Rows
 *         0..M-1 fully overwritten.
 *   workspace : device, 256-byte aligned, at least the bytes
 *         qmm_prefill_workspace() gives for M; owned by the caller, used only
 *         while the call's kernels run on `stream` (the f16 rows, then their
 *         multipliers).
 * Asynchronous on `stream` (two kernels: the pre-pass and the GEMM).
 * Errors: STATE, INVALID_ARG (not an FP8 handle, NULL act/out/workspace,
 * workspace too small), M_RANGE, ALIGN, SHAPE (ceil(M/128) * N/128 * K/128,
 * the GEMM's stage count, above 2^31 - 1), DEVICE, CUDA (launch). */
#define QMM_PREFILL_MAX_M (1 << 22)
int qmm_prefill(qmm_t h, const uint16_t* act, int64_t lda, float* out, int64_t ldo, int64_t M,
                void* workspace, int64_t workspace_bytes, void* stream);

/* *bytes = the workspace qmm_prefill needs for M rows (M * K * 2 rounded up to
 * 256, plus M * 4).  Errors: INVALID_ARG (NULL bytes, not an FP8 handle),
 * STATE, M_RANGE. */
int qmm_prefill_workspace(qmm_t h, int64_t M, int64_t* bytes);

/* ---- status ------------------------------------------------------------------ */

/* Wait for `stream`, then read and clear the handle's device error word.
 * Returns QMM_OK, QMM_ERR_TIMEOUT (a kernel gave up on a bounded wait, or the
 * prefill GEMM found its shared memory misaligned; its output is undefined
 * and the handle's device state has been reset), or
 * QMM_ERR_CUDA (the stream reported an error). */
int qmm_sync_status(qmm_t h, void* stream);

/* The last cudaError_t recorded on the handle (0 if none); NULL handle gives
 * the last error recorded by a handle-less call. */
int qmm_last_cuda_error(qmm_t h);

/* Fill *info (info->struct_size must be set). */
int qmm_get_info(qmm_t h, qmm_info* info);

/* Static, NUL-terminated name of a status code. */
const char* qmm_strerror(int code);

/* ---- test and tool entry points ------------------------------------------------ */

/* Dequantize the handle's W into w_out (device, fp32 [N][K] row-major), exactly
 * (Q4_0: fp32(d) * (q - 8); FP8: fp32(e4m3) * s, one fp32 multiply).  Async. */
int qmm_dequantize(qmm_t h, float* w_out, void* stream);

/* Rotate every 32-block of M bf16 rows with the fp32 butterflies described at
 * the top of this file.  act: device [M][lda] bf16 (16-byte aligned, lda % 8 ==
 * 0, lda >= K); act_out: device fp32 [M][K].  K % 32 == 0, 1 <= M.  Async. */
int qmm_hadamard32(const uint16_t* act, int64_t lda, float* act_out, int M, int64_t K,
                   void* stream);

/* The same rotation with B-point blocks, B = block = 32, 64 or 128 (strides 1,
 * 2, ..., B/2, each stage (x, y) -> (x + y, x - y), fp32).  K % B == 0.
 * Errors: as qmm_hadamard32, plus INVALID_ARG for another block size.  Async. */
int qmm_hadamard(const uint16_t* act, int64_t lda, float* act_out, int M, int64_t K, int block,
                 void* stream);

/* Quantize fp32 weights w (device [N][K]) into Q4_0 blocks (device, N*(K/32)*18
 * bytes, layout as in qmm_desc).  Per block: d32 = (element of largest
 * magnitude, first on ties, with its sign) / -8; q = clamp(roundf(w / d32) + 8,
 * 0, 15) using w * (1/d32); stored d = fp16 round-to-nearest-even of d32.
 * With QMM_FLAG_HADAMARD32 (64, 128) in flags every 32-block (64-, 128-block)
 * is first rotated with the fp32 butterflies and divided by the block size
 * (the offline half of the Hadamard variants).  K % 32 == 0 (and K a multiple
 * of the rotation block).  The 64- and 128-point rotations go through a
 * temporary fp32 copy of w allocated and freed in stream order on `stream`.
 * Async. */
int qmm_quantize_q4_0(const float* w, int64_t N, int64_t K, uint32_t flags, uint8_t* blocks,
                      void* stream);

/* Quantize fp32 weights w (device [N][K]) into Q8_0 blocks (device, N*(K/32)*34
 * bytes, layout as in qmm_desc).  Per block: amax = largest |w|, d32 = amax /
 * 127, q = clamp(roundf(w * (1/d32)), -127, 127) (0 for an all-zero block),
 * stored d = fp16 round-to-nearest-even of d32.  The rotation flags rotate
 * first, as for qmm_quantize_q4_0 (through a stream-ordered temporary).
 * K % 32 == 0.  Async. */
int qmm_quantize_q8_0(const float* w, int64_t N, int64_t K, uint32_t flags, uint8_t* blocks,
                      void* stream);

/* Quantize fp32 weights w (device [N][K]) to E4M3 codes (device [N][K]) and
 * fp32 scales (device [N/128][K/128]): per 128x128 tile s = maxabs / 448 and
 * code = e4m3 round-to-nearest-even of w / s, saturated to +-448 (s == 0 gives
 * zero codes).  QMM_FLAG_HADAMARD32 (64, 128) rotates each 32-block (64-,
 * 128-block) first and divides by the block size, as qmm_quantize_q4_0.
 * N % 128 == 0, K % 128 == 0.  Async. */
int qmm_quantize_fp8(const float* w, int64_t N, int64_t K, uint32_t flags, uint8_t* codes,
                     float* scales, void* stream);

/* Test hook: limit, in nanoseconds, of every bounded device wait of this
 * handle's kernels (default 2e9).  0 makes every such wait give up at once,
 * which exercises the timeout path without hanging anything; the kernels
 * still drain their own copies in flight before returning. */
int qmm_debug_set_wait_limit(qmm_t h, int64_t ns);

/* Test hook: make the n-th device allocation made by qmm_create from now on
 * fail as if cudaMalloc had failed (n = 0 disables; the hook fires once). */
int qmm_debug_fail_allocs(int n);

/* Profiling hook: per-CTA timeline of the warp-level (mma.sync) verify
 * kernel.  A library built with QMM_TRACE defined has each CTA of each verify
 * call on h write, at the points below, the device's global timer (ns) into
 * buf (device, n_words 64-bit words): call c (counted from this call on)
 * writes slot c % (n_words / slot) of slot = ctas * QMM_TRACE_FIELDS words
 * (ctas from qmm_get_info), CTA b at words b * QMM_TRACE_FIELDS + field.
 * buf = NULL switches it off.  The caller owns buf and keeps it alive while
 * calls that write it may run.  Returns QMM_ERR_STATE if the library was
 * built without QMM_TRACE (the product build: the stamps are compiled out)
 * or h is not live, QMM_ERR_INVALID_ARG if buf holds no slot, and
 * QMM_ERR_SHAPE for a tcgen05 handle (which has no stamps). */
#define QMM_TRACE_FIELDS 16
enum {
  QMM_TR_ENTRY = 0,  /* the CTA's barriers are initialised                    */
  QMM_TR_SMID = 1,   /* (not a time) the SM the CTA runs on                   */
  QMM_TR_PDL = 2,    /* the previous kernel's writes are visible (thread 0)   */
  QMM_TR_DATA = 3,   /* warp 0's first chunk has landed                       */
  QMM_TR_LOOP = 4,   /* warp 0 has finished its last stage                    */
  QMM_TR_EPI = 5,    /* every warp has finished its stages                    */
  QMM_TR_RED = 6,    /* the chunk partials are in shared memory               */
  QMM_TR_PART = 7,   /* the CTA's result (S = 1) or split partial is written  */
  QMM_TR_ARRIVE = 8, /* S > 1: the split's arrival add has returned           */
  QMM_TR_LAST = 9,   /* (not a time) 1 if this split did the fix-up           */
  QMM_TR_EXIT = 10   /* thread 0 leaves the kernel                            */
};
int qmm_debug_set_trace(qmm_t h, uint64_t* buf, int64_t n_words);

#ifdef __cplusplus
}
#endif
#endif /* QMM_H_ */
