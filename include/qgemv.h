/*
 * qgemv.h - C ABI of the GB300 small-M block-quantized GEMV library.
 *
 * Computes, for M = 1..17 activation rows (a width-6 speculative verifier uses
 * 6; the fused draft head uses rows 1..5), llama.cpp-family block-quantized
 * matrix-vector products against activations quantized on the fly to Q8_1,
 * and a fused LM-head that reduces each row to its greedy token id without
 * writing logits.  The pages this follows:
 *   [closure]  "Qwen3.6 27B Q4_0 DFlash/SYCL closure"
 *   [record]   "Q6_K M=6 fused DFlash top-1 production record"
 *   [q8cache]  "Qwen3.6 27B B70 follow-up: Q8 activation cache..."
 *   [handoff]  "Qwen3.6 27B AutoRound Handoff"
 *
 * Block formats (named on the pages, defined here as in llama.cpp):
 *   Q8_1  32 activations: fp16 d, fp16 s = d * sum(q), int8 q[32]      36 B
 *         d = max|x| / 127 (fp32), q = round(x / d) half away from zero,
 *         all-zero block -> d = s = 0, q = 0.
 *   Q4_0  32 weights: fp16 d, uint8 qs[16]; value i < 16 is the low nibble
 *         of qs[i], value i + 16 the high nibble; w = d * (q - 8)      18 B
 *   Q6_K  256 weights: uint8 ql[128], uint8 qh[64], int8 sc[16], fp16 d;
 *         low 4 bits of value i = nibble (i & 1) of ql[i >> 1], high 2 bits
 *         = bits 2 (i & 3) of qh[i >> 2]; w = d * sc[i >> 4] * (q - 32) 210 B
 *   Q8_0, Q4_K, Q5_K  the further formats, defined with their calls below.
 * All multi-byte fields are little endian.
 *
 * Conventions for every call:
 *   - Pointers named w_*, x, xq, y, ids, workspace are DEVICE pointers and
 *     must be 16-byte aligned; the caller allocates and owns all of them.
 *     The library allocates no memory and never synchronizes (it registers
 *     one page of its own host memory for the wait-timeout counter, below).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream); all work is enqueued on it, in order.
 *   - Arguments are validated on the host before anything is enqueued; on
 *     error nothing is enqueued and a negative status is returned.  Device
 *     faults surface at the caller's next synchronization.
 *   - Every wait inside the kernels is bounded (about a second).  A kernel
 *     whose wait runs out counts it and stops early, so that call's outputs
 *     are not valid; from then on every call that enqueues work returns
 *     QGEMV_WAIT_TIMEOUT before enqueueing anything, until
 *     qgemv_take_wait_timeouts has read the count (fail closed).  This needs
 *     the counter in mapped host memory (set up the first time a kernel needs
 *     it); where that cannot be set up, the count is still kept and read by
 *     qgemv_take_wait_timeouts, but calls are not refused.
 *   - Matrices are row-major: a weight is N rows of K values (K contiguous,
 *     the ggml [K, N] tensor); activations are M rows of K values with row
 *     stride ldx (in elements); outputs y are M rows of N values with row
 *     stride ldy, i.e. y[m * ldy + n] (the ggml [N, M] output).
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define QGEMV_OK 0
#define QGEMV_INVALID_ARG (-1)        /* null pointer, M/K/N/ld out of range  */
#define QGEMV_UNSUPPORTED_SHAPE (-2)  /* M > 17, K not a multiple of the block */
#define QGEMV_MISALIGNED (-3)         /* a pointer is not 16-byte aligned      */
#define QGEMV_WORKSPACE_TOO_SMALL (-4)
#define QGEMV_CUDA_ERROR (-5)         /* a CUDA call or launch failed          */
#define QGEMV_WAIT_TIMEOUT (-6)       /* an earlier call's kernel gave up      */

#define QGEMV_MAX_M 17
#define QGEMV_TOPK_MAX 8

/* Human-readable text for a status code (static storage). */
const char* qgemv_status_string(int status);

/* ---- sizes (host-only, no CUDA call) ---------------------------------- */

/* Bytes of the Q8_1 activation for M rows of K values: M * (K/32) * 36. */
size_t q8_1_bytes(int M, int K);
/* Bytes of a packed Q4_0 weight of N rows of K values.  Equal to the
 * canonical N * (K/32) * 18 when K % 256 == 0; otherwise each row's last
 * tile is padded to 16 bytes (at most 14 bytes per row). */
size_t q4_0_pack_bytes(int N, int K);
/* Bytes of a packed Q6_K weight: N * (K/256) * 210 (the canonical size). */
size_t q6_k_pack_bytes(int N, int K);
/* Bytes of a packed Q8_0 weight (qpack_q8_0): ceil(N/16) * (K/256) * 4352,
 * the canonical N * (K/32) * 34 when N % 16 == 0; 0 unless K % 256 == 0. */
size_t q8_0_pack_bytes(int N, int K);
/* Workspace bytes of lmhead_q6_k_top1 (256 + M * (K/32) * 36, rounded up to
 * 16) and argmax_f32_rows (256). */
size_t lmhead_q6_k_top1_workspace_bytes(int M, int K, int N);
size_t argmax_f32_rows_workspace_bytes(int M, int N);

/* ---- A1: activation quantizer ----------------------------------------- */

/* quantize_q8_1 - quantize M rows of K fp32 activations to Q8_1 blocks.
 * [q8cache] "Q8_1 activation cache prototype": the activation is quantized
 * once and the same Q8_1 copy feeds sibling matmuls (gate and up).
 *   x   fp32 [M][ldx] device, ldx >= K      (read)
 *   xq  uint8 [M][K/32][36] device           (written; q8_1_bytes(M, K))
 *   1 <= M <= 17, K % 32 == 0, K >= 32.
 * The output is caller-owned and may be passed to any number of qgemv_*
 * calls. */
int quantize_q8_1(const float* x, int64_t ldx, void* xq, int M, int K, void* stream);

/* rmsnorm_quantize_q8_1 - RMSNorm fused with the Q8_1 quantizer: the rows of
 * x normalized by their RMS and scaled by gamma, written as Q8_1 without an
 * fp32 copy.  [closure] "Qwen3.6 27B Q4_0 DFlash/SYCL closure", Closed or negative
 * paths: the down-to-next-RMSNorm/Q8 boundary (RMSNorm fused with
 * the Q8 quantization).  What is computed, per row: RMSNorm(x) * gamma,
 * xh_k = x_k * r * gamma_k with r = 1 / sqrt(sum_k x_k^2 / K + eps), then the
 * Q8_1 quantizer of quantize_q8_1 applied to xh.  xh is computed in fp32 in
 * a fixed order (all fp32, round to nearest, no fused multiply-add):
 *   s_t = sum over k = t, t + 512, ... < K, in increasing k, of x_k * x_k
 *         (t = 0..511, each added as s_t = s_t + (x_k * x_k));
 *   for h = 256, 128, ..., 1: s_t = s_t + s_{t+h} for t < h;   S = s_0;
 *   r = 1 / sqrt(S / K + eps);   xh_k = (x_k * r) * gamma_k;
 * so the output is deterministic (the same bytes on every call).  Against the
 * exact RMSNorm rounded to fp32 and quantized, with e = (K / 512 + 16) 2^-24,
 * the codes agree except where the exact xh_k / d lies within 508 e of a
 * half-integer (there the code may differ by one), and the fp16 scale agrees
 * except where d lies within a relative 4 e of a rounding midpoint between two
 * fp16 values (there it may be the neighbouring one): the fp32 sum of squares
 * is within a relative (K / 512 + 9) 2^-24 of the exact one, and a few more
 * roundings follow.
 *   x      fp32 [M][ldx] device, ldx >= K      (read)
 *   gamma  fp32 [K] device                      (read)
 *   eps    finite, >= 0
 *   xq     uint8 [M][K/32][36] device           (written)
 *   1 <= M <= 17, K % 32 == 0, 32 <= K < 2^24.
 * Errors: QGEMV_INVALID_ARG (null pointer, ldx < K, bad eps),
 * QGEMV_UNSUPPORTED_SHAPE (M, K), QGEMV_MISALIGNED. */
int rmsnorm_quantize_q8_1(const float* x, int64_t ldx, const float* gamma, float eps, void* xq, int M, int K,
                          void* stream);

/* ---- A2: weight repackers (offline) ------------------------------------ */

/* qpack_q4_0 - reorder canonical Q4_0 blocks into the kernel's tiles: each
 * row is cut into chunks of 32 blocks, and each (row, chunk) tile holds the
 * chunk's 16-byte code blocks followed by its fp16 scales (raw bits), padded
 * to 16 bytes; one tile is one aligned bulk copy.  [closure] "What materially worked" item 3
 * (offline-packed projections) and "Transfer" rule 7 (copy fp16 storage
 * bits, never convert them).
 *   w_canon  uint8 [N][K/32][18] device   (read)
 *   w_pack   q4_0_pack_bytes(N, K) device (written; must not alias w_canon)
 *   N >= 1, K % 32 == 0. */
int qpack_q4_0(const void* w_canon, void* w_pack, int N, int K, void* stream);

/* qpack_q6_k - reorder canonical Q6_K superblocks into the kernel's tiles:
 * per (row, 32-block chunk) 16 code bytes per block (the first 16 values'
 * six-bit codes, with the high two bits of the other 16 on top), 8 more per
 * block (the low four bits of those 16) and the subscales (2 B per block),
 * all rows' tiles back to back, then the fp16 superblock scales (raw bits);
 * same size.
 * [record] "Why this was slow" (the Q6_K output tensor is packed once).
 *   w_canon  uint8 [N][K/256][210] device (read)
 *   w_pack   q6_k_pack_bytes(N, K) device (written; must not alias w_canon)
 *   N >= 1, K % 256 == 0. */
int qpack_q6_k(const void* w_canon, void* w_pack, int N, int K, void* stream);

/* ---- A3 / A4: small-M MMVQ ---------------------------------------------- */

/* qgemv_q4_0 - y[m][n] = sum_b d_w[n,b] * d_a[m,b] * sum_i (q_w - 8) q_a,
 * integer block dots exact, fp32 accumulation.  Each weight byte is read
 * from HBM once and reused for all M rows.  [closure] "What materially
 * worked" item 2 (direct Q4_0 MMVQ for rows 1..17 removed repeated
 * full-weight reads).
 *   w_pack  packed Q4_0 (qpack_q4_0) of N rows of K values (read)
 *   xq      Q8_1 [M][K/32] from quantize_q8_1 (read)
 *   y       fp32, y[m * ldy + n] for n < N (written), ldy >= N
 *   1 <= M <= 17, K % 32 == 0, N >= 1. */
int qgemv_q4_0(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream);

/* qgemv_q6_k - y[m][n] = sum_b d6[n] * d_a[m,b] * sum_{half j of b} sc_j *
 * sum_i (q - 32) q_a.  [record] "Why this was slow" (the MMVQ part of the
 * fused head: each weight slice reused across all rows).
 *   w_pack  packed Q6_K (qpack_q6_k); xq, y, ldy as qgemv_q4_0;
 *   1 <= M <= 17, K % 256 == 0, N >= 1. */
int qgemv_q6_k(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream);

/* qgemv_q4_0_residual - qgemv_q4_0 with a residual epilogue:
 *   y[m][n] = (W x)[m][n] + residual[m * ldr + n],
 * the sum taken in fp32 when the output is stored (the MMVQ part exactly as
 * qgemv_q4_0 computes it, then one fp32 addition).  [closure] "Qwen3.6 27B
 * Q4_0 DFlash/SYCL closure", Closed or negative paths: an MMVQ with a
 * residual epilogue (the down projection writing its output plus the
 * residual stream in one pass).
 *   residual  DEVICE fp32, M rows of N values, row stride ldr >= N; it may be
 *             y itself (then ldr must equal ldy: an in-place residual add),
 *             otherwise it must not overlap y;
 *   other arguments as qgemv_q4_0.
 * Errors: QGEMV_INVALID_ARG for a null residual, ldr < N, or a residual that
 * partly overlaps y (or aliases it with ldr != ldy); QGEMV_MISALIGNED if it is
 * not 16-byte aligned; otherwise as qgemv_q4_0. */
int qgemv_q4_0_residual(const void* w_pack, const void* xq, const float* residual, int64_t ldr, float* y,
                        int64_t ldy, int M, int K, int N, void* stream);

/* qgemv_q4_0_pair - qgemv_q4_0 of two weights with the same K against one
 * Q8_1 activation in a single launch (the verifier MLP's gate and up):
 * y_a = W_a x, y_b = W_b x, each exactly as qgemv_q4_0 would compute it.
 * [record] "Strict run identity" (joint gate/up enabled) and [closure] "What
 * materially worked" item 3 (packed width-6 gate/up projections); one launch
 * pays the activation staging, the launch and the tail once for both.
 *   w_pack_a, w_pack_b  packed Q4_0 of N_a and N_b rows of K values (read)
 *   xq                  Q8_1 [M][K/32][36] (read)
 *   y_a, y_b            fp32 [M][ldy] (written), ldy >= max(N_a, N_b)
 *   1 <= M <= 17, K % 32 == 0, N_a >= 1, N_b >= 1. */
int qgemv_q4_0_pair(const void* w_pack_a, const void* w_pack_b, const void* xq, float* y_a, float* y_b, int64_t ldy,
                    int M, int K, int N_a, int N_b, void* stream);

/* ---- A5: fused LM-head top-1 -------------------------------------------- */

/* lmhead_q6_k_top1 - for each of M fp32 rows of x: quantize to Q8_1, project
 * through the Q6_K weight, and write the greedy token id (lowest id among
 * exactly equal maxima; -0 == +0; NaN never wins; a row of all NaN gives 0)
 * to ids[m].  No logits are written.  [record] "Outcome" and "Why this was
 * slow" (rows 1..5 only, reduced to five ids on device) and "Exactness and
 * safety contracts" item 3 (lowest-token-ID finite-tie contract).
 *   w_pack     packed Q6_K of N rows of K values (read)
 *   x          fp32 [M][ldx], ldx >= K (read); pass row 1 of a [6][K] block
 *              with M = 5 for the rows-1..5 view
 *   ids        int32 [M] (written)
 *   workspace  lmhead_q6_k_top1_workspace_bytes(M, K, N) bytes.  Its first
 *              256 bytes (the cross-CTA top-1 keys and counter) must be
 *              zero-filled before the first use, and every call leaves them
 *              zero-filled again; the rest receives the Q8_1 copy of x that
 *              a quantize_q8_1 pre-pass writes on `stream` before the MMVQ
 *              kernel reads it.  Calls that share a workspace must not
 *              overlap in time.
 *   1 <= M <= 17, K % 256 == 0, N >= 1. */
int lmhead_q6_k_top1(const void* w_pack, const float* x, int64_t ldx, int32_t* ids, void* workspace,
                     size_t ws_bytes, int M, int K, int N, void* stream);

/* lmhead_q6_k_candmax - the verifier's candidate-max over the same fused
 * LM-head: for each row m, the greedy id (ids[m], the lmhead_q6_k_top1
 * contract), its logit top_vals[m], and the logit of a given candidate id
 * cand[m] (a drafted token) in cand_vals[m].  No logits are written.
 * [handoff] "Current next-execution plan", the candidate-max precheck: a
 * target-verified speculation step needs each row's greedy id and value and
 * the score of the drafted candidate, not the logits.
 *   w_pack, x, ldx, workspace, ws_bytes, M, K, N  as lmhead_q6_k_top1
 *   cand       int32 [M] (read): the candidate id of each row; one outside
 *              0 .. N-1 gives cand_vals[m] = NaN
 *   ids        int32 [M] (written)
 *   top_vals   fp32 [M] (written): the greedy id's logit (NaN for a row of
 *              only NaN logits)
 *   cand_vals  fp32 [M] (written): the candidate's logit; equal, bit for
 *              bit, to top_vals[m] when cand[m] == ids[m]
 *   Both are the fused kernel's fp32 sums, within the library's fp32
 *   tolerance of the oracle's logits (and of qgemv_q6_k's, which may split K
 *   differently for small shapes). */
int lmhead_q6_k_candmax(const void* w_pack, const float* x, int64_t ldx, const int32_t* cand, int32_t* ids,
                        float* top_vals, float* cand_vals, void* workspace, size_t ws_bytes, int M, int K, int N,
                        void* stream);

/* lmhead_q6_k_topk_workspace_bytes - workspace bytes for lmhead_q6_k_topk:
 * the lmhead_q6_k_top1 workspace (its first 256 bytes under the same
 * zero-fill contract, then the Q8_1 copy of x), then, 256-byte aligned, one
 * list of k 64-bit keys per row for each CTA of the launch, at most
 * min(ceil(N / 4), 256) CTAs.  Host-only. */
size_t lmhead_q6_k_topk_workspace_bytes(int M, int K, int N, int k);

/* lmhead_q6_k_topk - the candidate-max's top-k form over the same fused
 * LM-head: for each row m, the k largest logits with their ids, in
 * descending order, plus (optionally) the logit of a given candidate id.
 * No logits are written.  [handoff] "Current next-execution plan", the
 * candidate-max precheck (the true top ids and values plus per-row candidate
 * scores).  Order: by value, larger first; exactly equal values by lower id
 * first; -0 == +0; NaN logits are never ranked; a row with fewer than k
 * non-NaN logits fills its last places with id -1 and value NaN.  Entry 0 is
 * lmhead_q6_k_top1's id except for a row of only NaN (there -1, not 0).
 * The result is deterministic: the logits are the fused kernel's fp32 sums
 * (each independent of where its row falls in the launch) and the ranking of
 * the (value, id) keys is a total order.
 *   w_pack, x, ldx, M, K, N  as lmhead_q6_k_top1
 *   k          1 <= k <= QGEMV_TOPK_MAX (8), k <= N
 *   cand       int32 [M] (read) or NULL: the candidate id of each row; one
 *              outside 0 .. N-1 gives cand_vals[m] = NaN
 *   ids        int32 [M][k] (written)
 *   vals       fp32 [M][k] (written) or NULL: the logits of ids
 *   cand_vals  fp32 [M] (written), NULL exactly when cand is NULL
 *   workspace  lmhead_q6_k_topk_workspace_bytes(M, K, N, k) bytes, first 256
 *              bytes zero-filled before the first use (every call leaves them
 *              so); calls that share a workspace must not overlap in time.
 *   Returns QGEMV_UNSUPPORTED_SHAPE where the activation does not fit next
 *   to the weight rings in shared memory (M * K beyond what the top-1 call
 *   serves with its ring kernel, e.g. M = 17 at K = 17408). */
int lmhead_q6_k_topk(const void* w_pack, const float* x, int64_t ldx, int k, const int32_t* cand, int32_t* ids,
                     float* vals, float* cand_vals, void* workspace, size_t ws_bytes, int M, int K, int N,
                     void* stream);

/* ---- A6: row argmax (the unfused control) -------------------------------- */

/* argmax_f32_rows - ids[m] = lowest n attaining max_n y[m * ldy + n], with the
 * same tie contract as lmhead_q6_k_top1.  [record] "Why this was slow" (the
 * separate argmax of the unfused path) and "Exactness and safety contracts"
 * item 3.
 *   y          fp32 [M][ldy] (read), ldy >= N
 *   ids        int32 [M] (written)
 *   workspace  argmax_f32_rows_workspace_bytes(M, N), same contract as above
 *   1 <= M <= 17, N >= 1. */
int argmax_f32_rows(const float* y, int64_t ldy, int32_t* ids, void* workspace, size_t ws_bytes, int M, int N,
                    void* stream);

/* ---- fused top-1 without a caller workspace -------------------------------- */

#define QGEMV_NOALLOC_MAX_M 17

/* lmhead_q6_k_top1_noalloc - lmhead_q6_k_top1 (same inputs, same ids) for
 * callers that cannot allocate device memory where they run it: a host whose
 * memory pool owns the whole device and forbids side allocations, a latency
 * path on which cudaMalloc could stall or synchronize the device, or a plugin
 * that is only handed input and output pointers.  It allocates nothing; the
 * cross-CTA scratch (one 64-bit key per row plus a counter) lives in a fixed
 * 256-byte array inside this library's device memory, which every GPU that
 * loads the library keeps until the process exits.
 * The pages have no counterpart: it exists for callers of this library.
 *   w_pack, x, ldx, ids, M, K, N, stream as lmhead_q6_k_top1.
 *   M > QGEMV_NOALLOC_MAX_M (17, the rows the fixed scratch holds) returns
 *   QGEMV_UNSUPPORTED_SHAPE before anything is enqueued.
 *   The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  The address is kept for the life of the
 *   process: after cudaDeviceReset (or any teardown of the device's primary
 *   context) it is stale, so do not call this entry point on that device
 *   again in the same process.  Each call clears the scratch on `stream`
 *   before its kernel.  All calls on a device share the one array: calls
 *   that overlap on the GPU (other streams, other host threads) race and may
 *   return wrong ids; serialize them. */
int lmhead_q6_k_top1_noalloc(const void* w_pack, const float* x, int64_t ldx, int32_t* ids, int M, int K, int N,
                             void* stream);

/* ---- checking aid --------------------------------------------------------- */

/* qgemv_block_dots_q4_0 / _q6_k - out[(m * N + n) * (K/32) + b] = the exact
 * int32 dot of weight block (n, b) with activation block (m, b), computed by
 * the same unpack and dot routines the MMVQ kernels use (Q4_0: sum (q-8) q_a;
 * Q6_K: sum over the two halves of sc * sum (q-32) q_a).  For checking the
 * integer part bit for bit; not a fast path.
 *   out  int32 [M][N][K/32] device (written). */
int qgemv_block_dots_q4_0(const void* w_pack, const void* xq, int32_t* out, int M, int K, int N, void* stream);
int qgemv_block_dots_q6_k(const void* w_pack, const void* xq, int32_t* out, int M, int K, int N, void* stream);

/* qgemv_set_q4_0_tensor_cores - choose the kernel family of qgemv_q4_0 and
 * qgemv_q4_0_pair, for shapes with N (and N_b) a multiple of 16 and K a
 * multiple of 1024 (other shapes always run on the SIMT dp4a kernels):
 *   1 (the default): the tensor cores (f16 mma.sync with exact integer block
 *     dots, the scales applied per block in fp32) from M = 5, and below 5
 *     rows on weights of at least 2^28 elements (N K, both weights of a
 *     pair); the small-M kernel up to M = 8, the general one above;
 *   2: the general tensor-core kernel for every M from 5;
 *   0: the SIMT dp4a kernels for every shape.
 * All compute the formula of qgemv_q4_0 within its fp32 rounding; the fp32
 * summation order differs, so they may differ in the last bits.
 * Process-wide; returns the previous setting.  (Not from the pages: a choice
 * of this implementation.) */
int qgemv_set_q4_0_tensor_cores(int enable);

/* qgemv_q4_0_plan - which kernel qgemv_q4_0 (N_b = 0) or qgemv_q4_0_pair
 * (N_b > 0) would launch for this shape under the current setting; writes
 * info[4] = {0 for the SIMT kernels, 1 for the general tensor-core kernel, 2
 * for the small-M one; CTAs per cluster (the K parts), grid size, ring
 * stages per warp}, zeros after the first for the SIMT kernels.  Enqueues
 * nothing; may query the current device.  (Not from the pages.) */
int qgemv_q4_0_plan(int M, int K, int N, int N_b, int* info);

/* lmhead_q6_k_top1_plan - the kernel lmhead_q6_k_top1 (and its candidate-max
 * and no-allocation forms) would launch for this shape: info[4] = {1 for the
 * ring kernel (the activation tile fits in shared memory), 0 for the
 * lock-step kernel (K is staged in chunks), grid size, warps per CTA, ring
 * stages per warp (0 for the lock-step kernel)}.  Enqueues nothing; may query
 * the current device.  (Not from the pages.) */
int lmhead_q6_k_top1_plan(int M, int K, int N, int* info);

/* qgemv_set_q6_k_tensor_cores - the kernel family of qgemv_q6_k.  The
 * tensor-core kernel takes shapes with M >= 7, N a multiple of 16 and K a
 * multiple of 1024 (per block two f16 mma.sync steps return the exact integer
 * dots of the two 16-value halves, combined with the int8 subscales exactly,
 * then d_a per block and d6 per superblock in fp32).  mode 1 (the default)
 * takes it only where it measured faster than the dp4a kernel: N below 16
 * row groups of 4 per SM and either M >= 12 or K >= 16384; mode 2 takes it
 * for every shape it accepts; mode 0 never.  The LM-head calls
 * (lmhead_q6_k_*) always run on the dp4a kernel.  Process-wide; returns the
 * previous mode.  (Not from the pages.)
 *
 * qgemv_q6_k_plan - which kernel qgemv_q6_k would launch for this shape;
 * writes info[4] as qgemv_q4_0_plan.  Enqueues nothing.  (Not from the
 * pages.) */
int qgemv_set_q6_k_tensor_cores(int mode);
int qgemv_q6_k_plan(int M, int K, int N, int* info);

/* ---- NEXT-4: a further format, Q8_0 ------------------------------------ */

/* Q8_0 (named on the pages among further quantization formats, defined as in
 * llama.cpp): 32 weights, fp16 d then int8 q[32]; value d * q.       34 B
 * [closure] "Qwen3.6 27B Q4_0 DFlash/SYCL closure" lists further K-quant
 * formats as the next coverage; this one runs on the tensor-core MMVQ.
 *
 * qpack_q8_0 - canonical [N][K/32] x 34 B -> the tensor-core pack: per
 * 16-row tile and job of 8 blocks one 4352-byte region (codes in MMA
 * fragment order as q + 128, then the 8 x 16 fp16 scales); rows padded to 16
 * with zeros.  K % 256 == 0; w_canon 2-byte aligned, w_pack 16-byte aligned
 * (q8_0_pack_bytes(N, K) bytes).
 *
 * qgemv_q8_0 - y[m][n] = sum_b d_w[n,b] * d_a[m,b] * sum_i q_w q_a (the block
 * dots exact, the scales in fp32), M = 1..17, K % 256 == 0, any N >= 1;
 * arguments as qgemv_q4_0.  QGEMV_UNSUPPORTED_SHAPE also when the activation
 * tile does not fit a plan (very large M * K). */
int qpack_q8_0(const void* w_canon, void* w_pack, int N, int K, void* stream);
int qgemv_q8_0(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream);

/* ---- NEXT-4: a further format, Q4_K ------------------------------------ */

/* Q4_K (named on the pages among the further K-quant formats; the Q4_K_M
 * draft models are built from it; defined as in llama.cpp): superblocks of
 * 256 weights = fp16 d, fp16 dmin, 12 bytes holding eight 6-bit scales sc_j
 * and eight 6-bit mins m_j (sub-block j < 4: sc = byte j & 63, m = byte j+4 &
 * 63; j >= 4: sc = (byte j+4 & 15) | (byte j-4 >> 6) << 4, m = (byte j+4 >> 4)
 * | (byte j >> 6) << 4), then 128 bytes of 4-bit codes (values 64c .. 64c+31
 * are the low nibbles of bytes 32c .. 32c+31, values 64c+32 .. 64c+63 their
 * high nibbles); value i = d * sc_{i/32} * q_i - dmin * m_{i/32}.      144 B
 * [closure] "Qwen3.6 27B Q4_0 DFlash/SYCL closure" lists further K-quant
 * formats as the next coverage; this one runs on the tensor-core MMVQ.
 *
 * qpack_q4_k - canonical [N][K/256] x 144 B -> the tensor-core pack: per
 * 16-row tile and superblock one 2368-byte region (codes in MMA fragment
 * order, per row and block 4 bytes per lane; the {scale, min} bytes, row by
 * row; the {d, dmin} bits); rows padded to 16 with zeros (148 B per row and
 * superblock).  K % 256 == 0; w_pack 16-byte aligned (q4_k_pack_bytes(N, K)
 * bytes, 0 when K % 256).
 *
 * qgemv_q4_k - y[m][n] = sum_b (d sc_b d_a[m,b] I - dmin m_b d_a[m,b] A), with
 * I = sum_i q_w q_a and A = sum_i q_a exact per 32-value block, the two terms
 * in fp32; M = 1..17, K % 256 == 0, any N >= 1; arguments as qgemv_q4_0.
 * QGEMV_UNSUPPORTED_SHAPE also when no launch plan fits (very large M * K).
 *
 * qgemv_q4_k_plan - as qgemv_q8_0_plan (blocks per job: 16, two adjacent
 * superblock regions in one copy, for M <= 8 where two stages of them fit
 * and K/32 is a multiple of 16; else 8).  (Not from the pages.) */
size_t q4_k_pack_bytes(int N, int K);
int qpack_q4_k(const void* w_canon, void* w_pack, int N, int K, void* stream);
int qgemv_q4_k(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream);
int qgemv_q4_k_plan(int M, int K, int N, int* info);

/* ---- NEXT-4: a further format, Q5_K ------------------------------------ */

/* Q5_K (named with Q4_K among the further K-quant formats; defined as in
 * llama.cpp): superblocks of 256 = fp16 d, fp16 dmin, the 12 scale/min bytes
 * of Q4_K, qh[32], then the 128 code bytes of Q4_K; the fifth bit of value i
 * is bit i/32 of qh[i % 32], so q_i = nibble + 16 * that bit (0..31) and
 * value i = d * sc_{i/32} * q_i - dmin * m_{i/32}.                     176 B
 *
 * qpack_q5_k - canonical [N][K/256] x 176 B -> the Q4_K pack layout with, after
 * the codes, a [block][row] 4-byte word of fifth bits (byte k, bit s = value
 * k + 4s of the block): 2880 B per 16-row tile and superblock (180 B per row
 * and superblock); q5_k_pack_bytes(N, K) bytes, 0 when K % 256.
 *
 * qgemv_q5_k / qgemv_q5_k_plan - as qgemv_q4_k / qgemv_q4_k_plan with 5-bit
 * codes.  (The plan query is not from the pages.) */
size_t q5_k_pack_bytes(int N, int K);
int qpack_q5_k(const void* w_canon, void* w_pack, int N, int K, void* stream);
int qgemv_q5_k(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream);
int qgemv_q5_k_plan(int M, int K, int N, int* info);

/* qgemv_q8_0_plan - the launch qgemv_q8_0 would make for this shape; writes
 * info[5] = {1, CTAs per cluster (the K parts), grid size, ring stages per
 * warp, blocks per job (8: a whole pack region; 4: half of one, taken where
 * 8-block stages do not fit shared memory)}.  QGEMV_UNSUPPORTED_SHAPE when no
 * plan fits.  Enqueues nothing; may query the current device.  (Not from
 * the pages.) */
int qgemv_q8_0_plan(int M, int K, int N, int* info);

/* qgemv_take_wait_timeouts - number of warps that, since the previous call,
 * waited about a second for their data (a weight copy, the activation) and
 * gave up (their launch's outputs are then invalid); reads and clears the
 * count, after which calls are accepted again.  Synchronize first, so that
 * every kernel launched before has finished.  0 in normal operation.  (Not
 * from the pages: a guard of this implementation's bounded waits.) */
int qgemv_take_wait_timeouts(unsigned int* count);

/* qgemv_debug_drop_next_copy - for tests of the timeout path only: the next
 * launch of the small-M tensor-core Q4_0 kernel (qgemv_q4_0 or
 * qgemv_q4_0_pair, 5 <= M <= 8, on its default path) issues no copy for the
 * first job of CTA 0, so the warp holding that job finds its bounded wait
 * running out (about a second); it counts the timeout and stops, with no copy
 * in flight for it, and the rest of the launch completes.  Process-wide; returns the previous
 * request (0 or 1).  (Not from the pages.) */
int qgemv_debug_drop_next_copy(void);

/* qgemv_debug_fail_fused - for tests of the fail-closed fallback only: the
 * next `count` calls of lmhead_q6_k_top1 that pass validation return
 * QGEMV_CUDA_ERROR without enqueueing anything, as a fused kernel that cannot
 * be launched would.  [record] Exactness and safety contracts: a fused call
 * that does not go through leaves the ordinary path to run.  Returns the
 * previous count.  The environment variable QGEMV_FAIL_FUSED=n adds n such
 * requests when the library first checks for one (a process started with
 * failing fused calls). */
int qgemv_debug_fail_fused(int count);

/* ---- the bounds-checking build ------------------------------------------ */

/* The library also builds with -DQGEMV_BOUNDS_CHECK (build.py --debug):
 * every kernel then checks the indexes it computes for its global and
 * shared-memory accesses (weight copies and tensor-map coordinates inside the
 * pack, activation and output offsets inside their [M][ld] extents, the
 * shared-memory layout inside the launch's size).  A failing check skips the
 * access (a skipped copy completes its pipeline stage with no bytes, so no
 * wait hangs) and is recorded; results are then wrong but the context stays
 * usable.  There is no counterpart on the pages: it stands in for a memory
 * checker where none can run.  The release build compiles every check away.
 *
 * qgemv_bounds_check_build - 1 for the bounds-checking build, 0 otherwise. */
int qgemv_bounds_check_build(void);

/* qgemv_take_bounds_errors - after a device synchronize, the number of failed
 * checks since the previous call and the site number of the first (0, 0 in
 * the release build), then clears both.  Returns QGEMV_INVALID_ARG for a null
 * pointer, QGEMV_CUDA_ERROR when the status page cannot be read. */
int qgemv_take_bounds_errors(unsigned int* count, unsigned int* first_site);

/* qgemv_debug_plant_bad_store - for tests of the bounds-checking build only:
 * the next MMVQ launch on the ring kernel (no top-1) moves the first stores
 * of its CTA 0, warp 0 one output row-length past their extent; its checks
 * skip them and record them.  Returns the previous request, or
 * QGEMV_UNSUPPORTED_SHAPE in the release build (where it does nothing). */
int qgemv_debug_plant_bad_store(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
