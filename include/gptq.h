/*
 * gptq.h -- C ABI of the GB300 (sm_103a) GPTQ per-layer quantization library.
 *
 * GPTQ quantizes a linear layer's weight W (m x d, out x in) column by column and,
 * after each column, moves the columns not yet quantized so that the layer output
 * on calibration inputs X stays close to the original ("GPTQ: fixing errors as you
 * go", sections "The algorithm, in words" and "going deeper / Objective").
 * The library runs the three stages of that method on one GPU:
 *
 *   1. gptq_hessian_accumulate  H += alpha * X^T X over token batches
 *   2. gptq_factor              damping, optional act-order, Hinv1 = upper
 *                               Cholesky factor of H_d^-1
 *   3. gptq_quantize_layer      blocked column loop: quantize, error feedback,
 *                               lazy block updates, packed b-bit codes
 *
 * Conventions shared by every call:
 *   - Pointers to matrices are DEVICE pointers owned by the caller. The library
 *     allocates no memory: scratch comes from a caller-provided device workspace
 *     whose size gptq_workspace_size() returns. The one exception is the
 *     host-buffer pipeline (gptq_pipeline_*), which takes HOST pointers and owns
 *     the device buffers it copies into.
 *   - Matrices are row-major with an explicit leading dimension in elements.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL means the legacy default
 *     stream) and runs asynchronously, except where a call documents a
 *     synchronization.
 *   - Every call returns a gptq_status. Argument errors are detected on the host
 *     and returned before anything is launched; no call aborts, traps or throws.
 *     gptq_last_error() gives a one-line description of the last failure on the
 *     calling thread.
 *   - Floating-point arithmetic is IEEE fp32 (bf16 inputs to the Hessian product).
 */
#ifndef GPTQ_GB300_H
#define GPTQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GPTQ_OK = 0,
  GPTQ_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or setting       */
  GPTQ_ERR_NOT_PD = 2,        /* Cholesky met a non-positive pivot (info = index) */
  GPTQ_ERR_NONFINITE = 3,     /* NaN or Inf met in H or W                      */
  GPTQ_ERR_UNSUPPORTED = 4,   /* valid request this build does not implement   */
  GPTQ_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed          */
  GPTQ_ERR_TIMEOUT = 6        /* a bounded on-device wait gave up              */
} gptq_status;

/* A cudaStream_t, passed as an opaque pointer so this header needs no CUDA header. */
typedef void* gptq_stream_t;

/* Static text for a status code ("GPTQ_OK", ...). Never NULL. */
const char* gptq_status_string(int status);

/* One-line description of the last failure on the calling thread ("" if none). */
const char* gptq_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int gptq_version(void);

/* Number of CUDA kernels this library has launched in the process so far. */
uint64_t gptq_launch_count(void);

/*
 * Synchronizes `stream`, then reads and clears the library's device error word,
 * which kernels raise when a bounded on-device wait gives up (GPTQ_ERR_TIMEOUT) or
 * when they meet a NaN or an Inf they cannot report otherwise (GPTQ_ERR_NONFINITE).
 * The word is shared by all calls on the current device.
 */
gptq_status gptq_device_check(gptq_stream_t stream);

/*
 * Stage 1 -- Hessian accumulation.
 *
 * Defined by "The GPTQ Algorithm" (procedure step 2, H = 2 X X^T), "GPTQ: fixing
 * errors as you go" (Objective: the squared error is a quadratic with Hessian
 * H = 2 X X^T, the same for every row) and "GPTQ-style round-to-nearest with Hessian
 * weighting" (section "Computing the Hessian": the layer's inputs reshaped to
 * tokens x features, H += x^T x per calibration batch).
 *
 * Computes, for i <= j,   H[i][j] = (zero_first ? 0 : H[i][j]) + alpha * sum_t X[t][i] * X[t][j]
 *
 *   X      device, bf16 bits (uint16), n x d row-major (token-major), leading
 *          dimension ldx >= d. The base must be 16-byte aligned and ldx a multiple
 *          of 8 (rows start on 16-byte boundaries).
 *   n      tokens in this batch (n >= 0; n == 0 only applies zero_first).
 *   d      channels, 8 <= d <= 65536, d a multiple of 8.
 *   H      device fp32, d x d row-major, leading dimension ldh >= d with ldh a
 *          multiple of 4 and the base 16-byte aligned. Only the
 *          upper triangle including the diagonal (i <= j) is written; the strictly
 *          lower triangle is never touched.
 *   alpha  scale of the product; 2 gives the pages' H = 2 X^T X. The caller keeps
 *          any token count (the codes do not depend on a positive scale of H).
 *   zero_first  non-zero: the upper triangle is overwritten instead of accumulated.
 *
 * Accumulation across calls in the same stream is exact in the sense of fp32
 * addition; the order of partial sums inside one call is not fixed, so results can
 * differ in the last bits from run to run.
 */
gptq_status gptq_hessian_accumulate(const uint16_t* X, int64_t n, int64_t d, int64_t ldx,
                                    float* H, int64_t ldh, float alpha, int zero_first,
                                    gptq_stream_t stream);

/* Workspace kinds for gptq_workspace_size(). */
enum { GPTQ_WS_FACTOR = 0, GPTQ_WS_QUANTIZE = 1, GPTQ_WS_DEQUANT_GEMM = 2 };

/*
 * Bytes of device workspace a call needs (0 for an invalid request). `which` is
 * GPTQ_WS_FACTOR (uses d only), GPTQ_WS_QUANTIZE (uses m, d, bits, group_size,
 * blocksize) or GPTQ_WS_DEQUANT_GEMM (uses m and d; d a multiple of 32). The workspace must be 256-byte aligned; its contents on entry do not
 * matter.
 */
size_t gptq_workspace_size(int which, int64_t m, int64_t d, int bits, int group_size,
                           int blocksize);

/*
 * Stage 2 -- damping, act-order and the inverse-Hessian factor.
 *
 * Defined by "GPTQ, Line by Line", questions "What does percdamp (dampening) do in
 * GPTQ?" (lambda = percdamp * mean of diag H added to every diagonal entry) and "Why
 * does GPTQ use Cholesky factorizations instead of inverting the Hessian directly?"
 * (Hinv1 = upper Cholesky factor of H^-1, whose row j gives the update direction
 * and whose diagonal gives the error denominator); act-order by "The GPTQ
 * Algorithm" (ActOrder) and "GPTQ: fixing errors as you go" (act-order / desc_act:
 * columns in order of decreasing H_qq).
 *
 *   H          device fp32, d x d, leading dimension d; only the upper triangle
 *              (i <= j) is read. Not modified.
 *   percdamp   damping fraction (the pages' default 0.01); must be >= 0.
 *   act_order  non-zero: perm_out receives the column order (stable sort of
 *              diag(H) descending, ties to the lower index) and Hinv1 is the
 *              factor of the permuted matrix H_d[perm][:, perm].
 *   perm_out   device int32[d]; required when act_order, ignored otherwise (may be
 *              NULL).
 *   Hinv1      device fp32, d x d, leading dimension d. Receives U with
 *              H_d^-1 = U^T U, U upper triangular with a positive diagonal; the
 *              strictly lower triangle is set to zero. Its previous contents are
 *              never read; after a failed factorization they are unspecified.
 *   ws         device workspace of gptq_workspace_size(GPTQ_WS_FACTOR, 0, d, ...)
 *              bytes.
 *   info       host pointer or NULL. When non-NULL the call synchronizes `stream`
 *              once and reports the outcome: *info = -1 on success, otherwise the
 *              column (0-based, in processing order, i.e. after act-order) whose
 *              pivot was not positive; the factorization runs from the last
 *              column to the first, so this is the highest such column. The
 *              return value is then GPTQ_ERR_NOT_PD, or
 *              GPTQ_ERR_NONFINITE when diag(H) holds a NaN or an Inf (*info = 0).
 *              When NULL nothing is synchronized and the outcome can be read later
 *              with gptq_factor_status().
 *
 * The returned Hinv1 equals the pages' three-step chain (Cholesky of H_d, inverse
 * by a Cholesky solve, upper Cholesky of the inverse) in exact arithmetic; the
 * library reaches it by one Cholesky factorization and one triangular inverse of
 * the index-reversed matrix: with J the reversal and J H_d J = L L^T (lower L),
 * Hinv1 = J L^-1 J.
 */
gptq_status gptq_factor(const float* H, int64_t d, float percdamp, int act_order,
                        int32_t* perm_out, float* Hinv1, void* ws, size_t ws_bytes,
                        int64_t* info, gptq_stream_t stream);

/*
 * Outcome of the last gptq_factor() that used this workspace: synchronizes
 * `stream`, sets *info as gptq_factor does and returns the same status.
 */
gptq_status gptq_factor_status(const void* ws, int64_t* info, gptq_stream_t stream);

/*
 * gptq_factor without a caller workspace, for callers that cannot allocate device
 * memory: code inside a runtime that owns the GPU's memory budget through its own
 * pool, or a pipeline that cannot take cudaMalloc's implicit device synchronization.
 * The pages have no counterpart of this call; it exists only for such callers.
 *
 * Same arguments, results and status codes as gptq_factor, minus ws / ws_bytes, with
 * one difference: `info` is required (NULL returns GPTQ_ERR_INVALID_ARG before
 * anything is launched), because the outcome lives in the library's shared scratch,
 * which no later call can read back and the next call overwrites; the call therefore
 * always synchronizes `stream` once. The scratch is a device array inside the
 * library sized for d <= 2048 (18 MiB + 256 bytes), held on every GPU that loads the
 * library until the process exits; d > 2048 returns GPTQ_ERR_INVALID_ARG before
 * anything is launched. The call allocates nothing.
 *
 * The first call on a device (with that device current) looks up the array's device
 * address and caches it; make that first call before any stream capture. All calls
 * on a device share the one array and it keeps the last call's contents (nothing in
 * it needs to start at zero): calls whose work overlaps on the GPU -- on different
 * streams, or from different threads -- race on it and must be serialized by the
 * caller.
 */
gptq_status gptq_factor_static(const float* H, int64_t d, float percdamp, int act_order,
                               int32_t* perm_out, float* Hinv1, int64_t* info,
                               gptq_stream_t stream);

/*
 * Stage 3 -- the blocked GPTQ column loop.
 *
 * Defined by "GPTQ, Line by Line", question "Why does GPTQ process the weight matrix
 * in blocks of 128 columns?" (inside a block each quantized column updates the
 * block's remaining columns by a rank-one product; after the block the block's
 * errors Err1 are applied to the columns right of it by one product
 * Err1 @ Hinv1[block, rest]) and by the listing of "GPTQ-style round-to-nearest with
 * Hessian weighting" (per-group min/max scale and zero, quantize, dequantize, error
 * divided by Hinv1[j][j], compensation along Hinv1[j][j+1:]).
 *
 *   W          device, m x d row-major, leading dimension ldw >= d; fp32
 *              (w_dtype 0) or bf16 bits (w_dtype 1). Not modified.
 *   Hinv1      device fp32 d x d (leading dimension d), the factor from
 *              gptq_factor for the same column order; only the upper triangle is
 *              read.
 *   perm       device int32[d] column order from gptq_factor(act_order), or NULL
 *              for the natural order. Outputs are always in the ORIGINAL column
 *              order.
 *   bits       2, 3, 4 or 8.
 *   group_size columns sharing one (scale, zero) per row; -1 means one per row
 *              (statistics from W before any update). Otherwise d % group_size == 0
 *              and group_size % blocksize == 0 or blocksize % group_size == 0, so
 *              that a group's statistics are read after all earlier compensation.
 *              With perm != NULL, groups are formed in processing order: group k
 *              holds the processed columns k*group_size ... (k+1)*group_size - 1,
 *              so original column j belongs to group g_idx[j] = p / group_size with
 *              perm[p] == j (scales and zeros are indexed by that group).
 *   blocksize  lazy-update block width in [1, 256]; this build runs 32, 64 and 128
 *              (the pages use 128) and returns GPTQ_ERR_UNSUPPORTED for others. It
 *              does not change the result in exact arithmetic. Group sizes must be
 *              multiples of 32 in this build (GPTQ_ERR_UNSUPPORTED otherwise).
 *   qweight    device uint32, m x ceil(d*bits/32): per row a little-endian
 *              bitstream, code of column j in bits [j*bits, j*bits + bits).
 *   scales, zeros  device fp32, m x G row-major, G = d / group_size (1 when -1);
 *              w_hat = (code - zero) * scale with the (scale, zero) of the column's
 *              group; zeros hold integers in [0, 2^bits-1].
 *   col_losses device fp32[d]: for every column, the sum over rows of Err1^2 / 2,
 *              the increase of 1/2 (w - w_hat) H_d (w - w_hat)^T caused by fixing that
 *              column; their total is 1/2 tr(dW H_d dW^T).
 *   ws         device workspace of gptq_workspace_size(GPTQ_WS_QUANTIZE, ...) bytes.
 *   info       host pointer or NULL. When non-NULL the call synchronizes `stream`
 *              and returns GPTQ_ERR_NONFINITE (with *info = 1) if W held a NaN or an
 *              Inf; *info = 0 otherwise. When NULL nothing is synchronized.
 */
gptq_status gptq_quantize_layer(const void* W, int w_dtype, int64_t m, int64_t d, int64_t ldw,
                                const float* Hinv1, const int32_t* perm, int bits,
                                int group_size, int blocksize, uint32_t* qweight,
                                float* scales, float* zeros, float* col_losses, void* ws,
                                size_t ws_bytes, int64_t* info, gptq_stream_t stream);

/*
 * Helper for checks: unpack codes written by gptq_quantize_layer into one byte per
 * code. qweight as above (m x ceil(d*bits/32) words, device); codes device uint8
 * m x d row-major. m <= 2^30, d <= 65536, m * d <= 2^36, else GPTQ_ERR_INVALID_ARG
 * before any launch.
 */
gptq_status gptq_unpack_codes(const uint32_t* qweight, int64_t m, int64_t d, int bits,
                              uint8_t* codes, gptq_stream_t stream);

/*
 * The quantized layer used again: Y = X W_hat^T computed straight from the packed
 * form, w_hat[r][j] = (code[r][j] - zero[r][g]) * scale[r][g] with g = g_idx[j], or
 * j / group_size when g_idx is NULL ("GPTQ: fixing errors as you go": once quantized,
 * the stored low-bit weights and per-group scales stand in for the layer's weights).
 * Every code is read once per 8 tokens. Codes in natural groups (g_idx NULL or one
 * group per row) are summed per group on the tensor cores (exact bf16 products of
 * code - zero and the token, fp32 accumulation), then scaled in fp32; act-order groups
 * and groups narrower than the kernel's column blocks take an fp32 FMA kernel. zeros
 * must hold integers (as gptq_quantize_layer writes them).
 *
 *   qweight, scales, zeros  as written by gptq_quantize_layer (device; m x
 *              ceil(d*bits/32) words, m x G floats each). qweight 16-byte aligned
 *              for 4 and 8 bits, 8-byte for 2.
 *   g_idx      device int32[d] group of every column (act-order groups), values in
 *              [0, G); or NULL.
 *   m, d       rows and columns of W; d a multiple of 32.
 *   bits       2, 3, 4 or 8.  group_size  -1 or a multiple of 32 dividing d.
 *   X          device bf16 bits, T x d token-major, row stride ldx (ldx >= d,
 *              ldx % 8 == 0, 16-byte aligned). 0 <= T < 2^31 tokens (8 per launch
 *              inside).
 *   Y          device fp32, T x m, row stride ldy >= m.
 * Asynchronous on `stream`; argument errors return GPTQ_ERR_INVALID_ARG before any
 * launch. This is the use of the stored layer that the pages describe, not a step of
 * the quantization itself.
 */
gptq_status gptq_dequant_gemv(const uint32_t* qweight, const float* scales, const float* zeros,
                              const int32_t* g_idx, int64_t m, int64_t d, int bits, int group_size,
                              const uint16_t* X, int64_t T, int64_t ldx, float* Y, int64_t ldy,
                              gptq_stream_t stream);

/*
 * The quantized layer applied to many tokens on the tensor cores: Y = X W_hat^T straight
 * from the packed form, with w_hat[r][j] = (code[r][j] - zero[r][g]) * scale[r][g] and
 * g = j / group_size ("GPTQ: fixing errors as you go": the stored low-bit weights and
 * per-group scales stand in for the layer's weights). This is also the propagation step
 * when layers are quantized one after another ("The GPTQ Algorithm", procedure steps
 * 1-4): with y_bf16 = 1 the outputs come out as bf16, ready to be the next layer's
 * calibration inputs for gptq_hessian_accumulate.
 *
 * code - zero is an integer of at most 8 bits, exact in bf16, so every product with a
 * bf16 token is exact; each group's partial sum is formed on the tensor cores with fp32
 * accumulation and added, times the group's scale, in fp32. Groups are the natural
 * consecutive column groups (act-order layers with several groups per row need the
 * dequant GEMV, which takes g_idx; per-channel layers, group_size -1, work in any column
 * order).
 *
 *   qweight, scales, zeros  as written by gptq_quantize_layer (device; m x
 *              ceil(d*bits/32) words, m x G floats each).
 *   m, d       rows and columns of W; d a multiple of 32, d <= 65536.
 *   bits       2, 3, 4 or 8.  group_size  -1 or a multiple of 32 dividing d.
 *   X          device bf16 bits, T x d token-major, row stride ldx (ldx >= d,
 *              ldx % 8 == 0, 16-byte aligned).
 *   T          tokens, 0 <= T < 2^31.
 *   Y          device, T x m with row stride ldy >= m: fp32 (y_bf16 = 0) or bf16 bits
 *              rounded to nearest even (y_bf16 = 1).
 *   ws         device workspace of gptq_workspace_size(GPTQ_WS_DEQUANT_GEMM, m, d, ...)
 *              bytes (the integer operand, m x d bf16), 256-byte aligned.
 * Asynchronous on `stream`; argument errors return GPTQ_ERR_INVALID_ARG before any
 * launch.
 */
gptq_status gptq_dequant_gemm(const uint32_t* qweight, const float* scales, const float* zeros,
                              int64_t m, int64_t d, int bits, int group_size, const uint16_t* X,
                              int64_t T, int64_t ldx, void* Y, int y_bf16, int64_t ldy, void* ws,
                              size_t ws_bytes, gptq_stream_t stream);

/*
 * One layer end to end from HOST memory ("The GPTQ Algorithm", procedure steps 2-4 for
 * one layer: the Hessian over the calibration batches, then the factor and the column
 * loop; "GPTQ-style round-to-nearest with Hessian weighting", section "Computing the
 * Hessian": H accumulated batch by batch). The tokens are copied to the GPU in chunks
 * on the pipeline's own copy stream while the Hessian of the previous chunk runs on
 * the caller's stream (two device chunk buffers in turn); W follows the last chunk;
 * then gptq_factor and gptq_quantize_layer run, and the outputs are copied back to
 * the caller's host buffers. Results equal those of the three device calls in a row
 * on the same data (H = 2 X^T X).
 *
 * Unlike the calls above, a pipeline OWNS device memory: gptq_pipeline_create makes,
 * on the current device, one allocation holding the two chunk buffers, W, H, Hinv1,
 * the permutation, both workspaces and the outputs, plus a copy stream and its
 * events. gptq_pipeline_run allocates nothing; gptq_pipeline_destroy frees all of it.
 *
 *   m, d, w_dtype, bits, group_size, blocksize, percdamp, act_order
 *                   as for gptq_factor and gptq_quantize_layer; d a multiple of 8.
 *   chunk_tokens    tokens per device chunk buffer, 1 <= chunk_tokens <= 2^24 (each
 *                   buffer holds chunk_tokens x d bf16 values).
 *   out             receives the pipeline; *out = NULL on failure.
 * Errors: GPTQ_ERR_INVALID_ARG / GPTQ_ERR_UNSUPPORTED for settings gptq_quantize_layer
 * would refuse, GPTQ_ERR_CUDA when the allocation or a stream or event fails (nothing
 * is kept then).
 */
typedef struct gptq_pipeline gptq_pipeline;

gptq_status gptq_pipeline_create(int64_t m, int64_t d, int w_dtype, int bits, int group_size,
                                 int blocksize, float percdamp, int act_order,
                                 int64_t chunk_tokens, gptq_pipeline** out);

/*
 * Enqueues one layer on `stream` (and the pipeline's copy stream) and returns without
 * waiting. All buffers here are HOST memory; page-locked buffers let the copies overlap
 * the Hessian (pageable ones work, with copies that do not overlap).
 *
 *   W            host, m x d row-major, row stride ldw >= d, type of w_dtype.
 *   X            host bf16 bits, n x d token-major, row stride ldx >= d; n >= 0.
 *   qweight, scales, zeros, col_losses
 *                host outputs laid out as gptq_quantize_layer's.
 *   perm         host int32[d] receiving the column order when the pipeline was made
 *                with act_order (may be NULL to skip it); ignored otherwise.
 * Every buffer must stay valid, and the outputs unread, until `stream` has been
 * synchronized. Runs on one pipeline are ordered: a run's copies wait for the previous
 * run's work, whatever streams they were given. The pipeline must be used on the
 * device it was made on (GPTQ_ERR_INVALID_ARG otherwise). The outcome of the factor
 * and of the column loop (not positive definite, non-finite W) is read afterwards with
 * gptq_pipeline_status; after a failed factor the outputs are unspecified.
 */
gptq_status gptq_pipeline_run(gptq_pipeline* p, const void* W, int64_t ldw, const uint16_t* X,
                              int64_t n, int64_t ldx, uint32_t* qweight, float* scales,
                              float* zeros, float* col_losses, int32_t* perm,
                              gptq_stream_t stream);

/*
 * Outcome of the last gptq_pipeline_run: synchronizes `stream`, then returns the
 * factor's status (with *info as gptq_factor sets it) or, when the factor succeeded,
 * the column loop's (GPTQ_ERR_NONFINITE with *info = 1 for a NaN or Inf in W); *info = -1
 * when both succeeded. info may be NULL.
 */
gptq_status gptq_pipeline_status(gptq_pipeline* p, int64_t* info, gptq_stream_t stream);

/* Waits for the pipeline's work, then frees its device memory, streams and events.
 * NULL is accepted. */
gptq_status gptq_pipeline_destroy(gptq_pipeline* p);

/*
 * Helper for checks: C = beta * C + alpha * A B (fp32, single batch) with the GEMM the
 * library uses for its block updates. engine 0: tensor cores, 3 x TF32 products with
 * fp32 accumulation of 32-deep partial products; engine 1: FFMA. a_kmajor != 0 means
 * A(i, k) = A[i * lda + k], else A[k * lda + i]; b_kmajor != 0 means
 * B(k, j) = B[j * ldb + k], else B[k * ldb + j]. lower_tiles != 0 (square C only)
 * skips 128 x 128 output tiles strictly above the diagonal. Device pointers; no
 * synchronization.
 */
gptq_status gptq_gemm_f32(int engine, int a_kmajor, int b_kmajor, int64_t M, int64_t N, int64_t K,
                          const float* A, int64_t lda, const float* B, int64_t ldb, float* C,
                          int64_t ldc, float alpha, float beta, int lower_tiles,
                          gptq_stream_t stream);

/*
 * Self-test of the bounded on-device waits (for tests; not a step of the method, and
 * the pages have no counterpart). Every spin-wait in the library gives up after a
 * wall-clock limit, raises the device error word and returns, so a stuck producer
 * cannot hang the GPU. This call runs one of those wait routines alone, on something nothing ever
 * completes, with a short limit: which = 0 the counter wait of the Cholesky panels
 * (acquire loads of a global counter that nothing publishes), which = 1 the mbarrier
 * wait used by every copy and tensor-core hand-over (a barrier nothing arrives on).
 * Nothing is in flight when the wait gives up.
 *
 *   limit_ns   the wait's limit in nanoseconds, 1e3 <= limit_ns <= 1e9.
 *
 * Synchronizes `stream`, then returns GPTQ_ERR_TIMEOUT (the expected outcome) when the
 * wait gave up; the device error word is raised as well, so the next
 * gptq_device_check() returns GPTQ_ERR_TIMEOUT once and clears it. Bad arguments
 * return GPTQ_ERR_INVALID_ARG before any launch.
 */
gptq_status gptq_wait_selftest(int which, int64_t limit_ns, gptq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GPTQ_GB300_H */
