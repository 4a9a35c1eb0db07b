/*
 * fp8q.h -- fine-grained FP8 (E4M3) quantization and block-scaled FP8 GEMM
 * for NVIDIA B300 (sm_103a).  C ABI of libfp8q.so.
 *
 * The method (DeepSeek-V3 FP8 mixed-precision training, as retold by the
 * scraped pages this library follows):
 *  - activations are grouped and scaled per 1x128 tile (one token, 128
 *    channels), weights per 128x128 block (128 input x 128 output channels)
 *    -- dssusan.co.kr page, the Figure 7 (a) passage;
 *  - E4M3 on all tensors, for Fprop, Dgrad and Wgrad alike
 *    -- "Deepseek Ai News Expert Interview", the E4M3/E5M2 passage;
 *  - all three Linear GEMMs run in FP8, take FP8 inputs and produce BF16 or
 *    FP32 -- dssusan.co.kr page, the Figure 6 passage, and
 *    "Deepseek Ai News Expert Interview", the GEMM input/output passage;
 *  - tensor-core partial sums are promoted to FP32 on CUDA cores every 128
 *    K-elements, where full-precision FP32 accumulation happens and the
 *    dequantization scales are applied -- "Eliminate Deepseek Ai News For
 *    Good", the MMA-precision passage; inprokorea.com page, the
 *    accumulation-interval passage; "Is aI Hitting a Wall?", the
 *    dequantization passage;
 *  - activations are quantized before the MoE dispatch and the experts' FP8
 *    up-projection takes every routed row (no token dropping)
 *    -- "Eliminate Deepseek Ai News For Good", the dispatch passage;
 *    inprokorea.com page, the no-token-dropping sentence.
 *
 * Numeric definitions (where the pages are silent, their plainest reading):
 *  - E4M3 is E4M3FN: bias 7, no infinities, max finite 448.  Casts round to
 *    nearest even and saturate to +-448; the sign of zero is kept.
 *  - Each group: a = max(amax, 2^-100), s = a / 448 and inv = 448 / a (IEEE
 *    single divisions), code = E4M3(x * inv) with x * inv rounded to FP32.
 *    The stored scale s dequantizes: x ~ decode(code) * s.
 *  - GEMM: C[m][n] = sum over K-blocks kb (ascending) of
 *    sA(kb, m) * sB(kb, n) * P_kb[m][n], with P_kb the tensor-core sum over
 *    the 128 k of block kb, promoted to FP32 registers each block.
 *  Only finite inputs are defined; NaN/Inf propagate unspecified.
 *
 * Conventions common to every entry point:
 *  - Every pointer argument is DEVICE memory (cudaMalloc'd or equivalent),
 *    owned by the caller; the library never allocates or frees device
 *    memory and keeps no pointer after the call returns.
 *  - Every pointer must be 16-byte aligned.
 *  - Work is enqueued asynchronously on `stream` (0 = legacy default stream)
 *    of the current device; nothing blocks except fp8q_get_device_status.
 *  - Calls are stateless and may be made from several host threads.
 *  - Argument errors are reported synchronously (nothing is launched):
 *    FP8Q_ERR_NULL, FP8Q_ERR_SHAPE, FP8Q_ERR_ALIGN, FP8Q_ERR_DTYPE, and
 *    FP8Q_ERR_DEVICE when the current device is not sm_103.  A failed launch
 *    returns FP8Q_ERR_CUDA.  A kernel whose internal pipeline wait exceeds
 *    its time limit (a bug, never expected) records FP8Q_ERR_TIMEOUT in a
 *    device status word and exits early; fp8q_get_device_status reports it.
 *  - Code layouts are row-major uint8 with the contraction dimension K
 *    contiguous.  Scale arrays are FP32 and K-block-major: the scales one
 *    K-block of a tile needs are contiguous.
 *  - Sizes are int64_t element counts.  A zero-row problem is a no-op that
 *    returns FP8Q_OK once the sizes and codes are valid; its pointers are
 *    not inspected (empty buffers may be NULL).
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* the CUDA runtime's cudaStream_t */
struct CUstream_st;
typedef struct CUstream_st *fp8q_stream_t;

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_NULL = 1,     /* a required pointer is NULL                      */
    FP8Q_ERR_SHAPE = 2,    /* a size is negative or breaks a divisibility rule */
    FP8Q_ERR_ALIGN = 3,    /* a pointer is not 16-byte aligned                */
    FP8Q_ERR_DTYPE = 4,    /* unknown dtype / granularity code                */
    FP8Q_ERR_DEVICE = 5,   /* current device is not sm_103 (B300)             */
    FP8Q_ERR_CUDA = 6,     /* a CUDA call or launch failed                     */
    FP8Q_ERR_TIMEOUT = 7,  /* a kernel's pipeline wait timed out (device side) */
    FP8Q_ERR_WORKSPACE = 8 /* workspace smaller than fp8q_gemm_workspace_size() */
} fp8q_status;

typedef enum {
    FP8Q_BF16 = 0,
    FP8Q_FP32 = 1
} fp8q_dtype;

/*
 * fp8q_quantize_act -- activation quantization, 1x128 tiles plus the 128x1
 * transposed copy that Wgrad consumes.
 *   x       [M][K] row-major, BF16 or FP32 (in_dtype).  K % 128 == 0.
 *   q_row   [M][K] E4M3 codes of the 1x128 groups (one row, 128 channels).
 *   s_row   [K/128][M] their scales.
 *   q_colT  [K][M] E4M3 codes of the 128x1 groups (128 consecutive rows of
 *           one column of the ORIGINAL x), stored transposed: row k holds
 *           column k of x, token index contiguous.  Requires M % 128 == 0.
 *   s_col   [M/128][K] their scales.
 * Either output pair may be (NULL, NULL) to skip it, not both; a pair must
 * be both set or both NULL.  Codes and scales are bit-exact functions of x.
 * Groups: dssusan.co.kr page, the Figure 7 (a) passage; the transposed copy
 * serves FP8 Wgrad with activations cached in FP8 ("Is aI Hitting a Wall?",
 * the Wgrad/caching sentence).
 */
FP8Q_API int fp8q_quantize_act(const void *x, int in_dtype, int64_t M, int64_t K,
                      uint8_t *q_row, float *s_row, uint8_t *q_colT, float *s_col,
                      fp8q_stream_t stream);

/*
 * fp8q_quantize_act_gather -- 1x128 quantization fused with the MoE dispatch
 * permutation: output row r is the quantization of input row src_rows[r].
 *   x         [M][K] row-major, BF16 or FP32.  K % 128 == 0.
 *   src_rows  [R] int32 device array, each in [0, M).  Out-of-range indices
 *             are not checked on the device (the caller validates).
 *   q_row     [R][K] codes;  s_row [K/128][R] scales.
 * Equal, bit for bit, to quantize-then-gather, because 1x128 groups are
 * row-local.  Quantize before dispatch: "Eliminate Deepseek Ai News For
 * Good", the dispatch passage.
 */
FP8Q_API int fp8q_quantize_act_gather(const void *x, int in_dtype, int64_t M, int64_t K,
                             const int32_t *src_rows, int64_t R,
                             uint8_t *q_row, float *s_row, fp8q_stream_t stream);

/*
 * fp8q_quantize_weight -- 128x128 block quantization of a weight in PyTorch
 * Linear layout.
 *   w  [N][K] row-major (N output channels, K input channels), BF16 or FP32.
 *      N % 128 == 0, K % 128 == 0.
 *   q  [N][K] E4M3 codes;  s [N/128][K/128] block scales.
 * Blocks: dssusan.co.kr page, the Figure 7 (a) passage.
 */
FP8Q_API int fp8q_quantize_weight(const void *w, int in_dtype, int64_t N, int64_t K,
                         uint8_t *q, float *s, fp8q_stream_t stream);

/*
 * fp8q_quantize_weight_ex -- as fp8q_quantize_weight, and optionally also
 * writes the transposed codes and scales that Dgrad (dX = dY . W) uses as
 * its B operand:
 *   q_t [K][N] codes of w^T (same block scales: a 128x128 block's scale does
 *        not change under transposition);  s_t [K/128][N/128].
 * Any of the pairs (q, s), (q_t, s_t) may be (NULL, NULL), not both.
 * Dgrad in FP8: dssusan.co.kr page, the Figure 6 passage.
 */
FP8Q_API int fp8q_quantize_weight_ex(const void *w, int in_dtype, int64_t N, int64_t K,
                            uint8_t *q, float *s, uint8_t *q_t, float *s_t,
                            fp8q_stream_t stream);

/*
 * fp8q_gemm -- block-scaled FP8 GEMM with FP32 promotion every 128 K.
 * Passages: the tensor cores accumulate each 128-element K interval, the
 * partial is then copied to FP32 registers on the CUDA cores and added at
 * full precision ("Eliminate Deepseek Ai News For Good", the MMA-precision
 * passage; inprokorea.com page, the accumulation-interval passage); the
 * per-group scales are multiplied in at that promotion ("Is aI Hitting a
 * Wall?", the dequantization passage); FP8 inputs, BF16 or FP32 output
 * ("Deepseek Ai News Expert Interview", the GEMM input/output passage).
 *   Aq  [M][K] E4M3 codes, K contiguous (1x128-quantized rows).
 *   sA  [K/128][M] scales of A.
 *   Bq  [N][K] E4M3 codes, K contiguous (a weight in Linear layout).
 *   sB  [N/128][K/128] 128x128 block scales of B.
 *   C   [M][N] row-major output, BF16 (rounded to nearest even) or FP32
 *       (out_dtype).
 *   C[m][n] = sum_kb sA[kb][m] * sB[n/128][kb] * P_kb[m][n].
 * M >= 0 (any), N % 128 == 0, K % 128 == 0, K > 0.
 * Accuracy: |C - C*| <= 2e-3 * sum_k |a_dq * b_dq| per element against the
 * exact result C* (plus one BF16 rounding for BF16 output).
 */
FP8Q_API int fp8q_gemm(const uint8_t *Aq, const float *sA, const uint8_t *Bq, const float *sB,
              void *C, int64_t M, int64_t N, int64_t K, int out_dtype,
              fp8q_stream_t stream);

/*
 * fp8q_gemm_ex -- fp8q_gemm with a choice of B-scale granularity along N.
 * Passages: Wgrad runs in FP8 like Fprop and Dgrad (dssusan.co.kr page, the
 * Figure 6 passage; "Is aI Hitting a Wall?", the FP8 Wgrad sentence), whose
 * operands are grouped along the token dimension, so B's scale varies per
 * column; the promotion is fp8q_gemm's.
 *
 *   sb_gran_n == 128: sB is [N/128][K/128] (as fp8q_gemm);
 *   sb_gran_n == 1:   sB is [K/128][N], one scale per column n and K-block,
 *                     the layout of fp8q_quantize_act's s_col.  This is
 *                     Wgrad: dW = dY^T . X with both operands quantized in
 *                     128x1 groups along the token (K) dimension, i.e.
 *                     Aq = q_colT(dY), sA = s_col(dY), Bq = q_colT(X),
 *                     sB = s_col(X).
 */
FP8Q_API int fp8q_gemm_ex(const uint8_t *Aq, const float *sA, const uint8_t *Bq, const float *sB,
                 void *C, int64_t M, int64_t N, int64_t K, int out_dtype,
                 int sb_gran_n, fp8q_stream_t stream);

/*
 * fp8q_gemm_workspace_size -- bytes of device workspace fp8q_gemm_ws needs on
 * the current device (one flag word and one 128x256 FP32 partial tile per
 * SM, about 19 MB on a B300), or 0 if the current device is not sm_103.
 */
FP8Q_API size_t fp8q_gemm_workspace_size(void);

/*
 * fp8q_gemm_ws -- fp8q_gemm_ex with a caller-owned device workspace that lets
 * the persistent kernel balance its K loop across SMs ("stream-K").
 *   workspace        device memory of at least fp8q_gemm_workspace_size()
 *                    bytes, 16-byte aligned, ZERO-FILLED before its first use.
 *                    Every call that completes leaves it zeroed again, so one
 *                    allocation serves any number of calls on one stream.
 *                    After a call that reported FP8Q_ERR_TIMEOUT, zero it
 *                    again.  Calls sharing a workspace must not overlap on
 *                    the GPU (use one stream, or one workspace per stream).
 *   workspace_bytes  its size; smaller than required -> FP8Q_ERR_WORKSPACE.
 * workspace == NULL runs exactly as fp8q_gemm_ex.  Otherwise, when whole
 * 128x256 output tiles would leave the last wave of the one-CTA-per-SM grid
 * less than 95% busy, every SM takes an equal share of the tile-major
 * sequence of all tiles' 128-K blocks; a tile whose blocks are split between
 * SMs is finished by the SM holding its first blocks, which adds the other
 * SMs' FP32 partial tiles in SM order (deterministic).  The promotion every
 * 128 K is unchanged; only where the FP32 sum of a tile is formed moves.
 * Same layouts, accuracy and errors as fp8q_gemm_ex.
 */
FP8Q_API int fp8q_gemm_ws(const uint8_t *Aq, const float *sA, const uint8_t *Bq, const float *sB,
                 void *C, int64_t M, int64_t N, int64_t K, int out_dtype,
                 int sb_gran_n, void *workspace, size_t workspace_bytes,
                 fp8q_stream_t stream);

/*
 * fp8q_gemm_ws_static -- fp8q_gemm_ws that allocates nothing and takes no
 * workspace: the stream-K scratch is a fixed array inside the library.
 * (The pages have no counterpart to this; it exists for callers that cannot
 * allocate device memory -- e.g. a plugin or operator interface whose
 * enqueue step is handed only its input and output buffers, or a path that
 * must not take cudaMalloc's implicit device-wide synchronization.)
 *  - The array holds the workspace of a grid of up to 160 CTAs (one per SM;
 *    about 20 MB) and stays resident on every GPU that loads the library
 *    until the process exits.  A device with more SMs than that gets
 *    FP8Q_ERR_WORKSPACE.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.  The cached address belongs to the device's current
 *    primary context: do not call this entry point again after
 *    cudaDeviceReset() on that device in the same process.
 *  - Every call shares the one array and leaves its contents for the next;
 *    each call first clears the flag words on its stream (a small memset).
 *    Calls whose kernels overlap on the GPU race on the array: keep them on
 *    one stream, or use fp8q_gemm_ws with a workspace per stream.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 * Arguments, layouts, accuracy and errors as fp8q_gemm_ex.
 */
FP8Q_API int fp8q_gemm_ws_static(const uint8_t *Aq, const float *sA, const uint8_t *Bq, const float *sB,
                        void *C, int64_t M, int64_t N, int64_t K, int out_dtype,
                        int sb_gran_n, fp8q_stream_t stream);

/*
 * fp8q_grouped_gemm -- MoE grouped block-scaled FP8 GEMM over E experts with
 * ragged rows (no token dropping).
 * Passages: activations are quantized to FP8 before the dispatch and each
 * expert's up-projection consumes them in FP8 ("Eliminate Deepseek Ai News
 * For Good", the dispatch passage); no routed token is dropped
 * (inprokorea.com page, the no-token-dropping sentence); each expert's GEMM
 * promotes every 128 K as fp8q_gemm does.
 *   Aq           [total_rows][K] codes of the dispatched (expert-grouped) rows.
 *   sA           [K/128][total_rows] their scales.
 *   Bq           [E][N][K] expert weights' codes;  sB [E][N/128][K/128].
 *   C            [total_rows][N] output (BF16 or FP32).
 *   row_offsets  [E+1] int32 DEVICE array: rows [off[e], off[e+1]) belong to
 *                expert e; nondecreasing, off[0] == 0, off[E] == total_rows.
 *                Read on the device (no host synchronization); the library
 *                trusts it (it cannot check device contents without a sync).
 * Empty experts are allowed and write nothing.  Rows of expert e are
 * C[r] = (Aq[r], sA[:, r]) x (Bq[e], sB[e]) as in fp8q_gemm.
 * N % 128 == 0, K % 128 == 0, E >= 1, total_rows >= 0.
 */
FP8Q_API int fp8q_grouped_gemm(const uint8_t *Aq, const float *sA, const uint8_t *Bq, const float *sB,
                      void *C, const int32_t *row_offsets, int32_t E, int64_t total_rows,
                      int64_t N, int64_t K, int out_dtype, fp8q_stream_t stream);

/*
 * fp8q_gemm_unpromoted -- accumulation-precision diagnostic, not part of the
 * method: C = Aq . Bq^T over the decoded E4M3 codes with the WHOLE K
 * accumulated inside the tensor core (no promotion to FP32 registers, no
 * scales), FP32 out.  The pages report that limited tensor-core accumulation
 * precision reaches a maximum relative error near 2% for an inner dimension
 * of 4096 ("Eliminate Deepseek Ai News For Good", the accumulation-precision
 * sentence); comparing this against fp8q_gemm with unit scales measures that
 * effect on B300.  Aq [M][K], Bq [N][K] (K contiguous), C [M][N] FP32.
 * M >= 0, N % 128 == 0, K % 128 == 0.  Unoptimized (one tile per CTA).
 */
FP8Q_API int fp8q_gemm_unpromoted(const uint8_t *Aq, const uint8_t *Bq, float *C,
                         int64_t M, int64_t N, int64_t K, fp8q_stream_t stream);

/*
 * MX (microscaling) variant.  The pages state that the fine-grained strategy
 * follows the microscaling formats and that Blackwell tensor cores support
 * those formats with smaller groups ("Deepseek Ai News Expert Interview", the
 * DualPipe / microscaling paragraph).  Here: E4M3 codes in 1x32 groups along
 * K, one power-of-two scale per group stored as an E8M0 byte, and a GEMM
 * whose tensor cores apply those scales (no CUDA-core promotion).  Codes and
 * scales are NOT comparable with the FP32-scale path above.
 *
 * Conversion of one group of 32 (the MX formats' own definition):
 *   e = floor(log2(amax)) - 8, clamped to [-127, 127] (amax == 0: -127);
 *   scale byte = e + 127;  code = E4M3_rn_satfinite(x / 2^e)  (the largest
 *   elements of a group can saturate to +-448: x / 2^e < 512).
 *
 * Scale layout ("tiled"), for an operand of `rows` rows and K columns:
 *   s[K/128][ceil(rows/128)][512] bytes; in the 512-byte chunk of row tile rt
 *   and K-block kt, the scale of row 128*rt + r (r < 128) and 32-group
 *   4*kt + c (c < 4) sits at byte (r % 32) * 16 + (r / 32) * 4 + c.  This is
 *   the 32 x 16-byte matrix the tensor core's scale-factor copy consumes, so
 *   the GEMM moves each chunk into tensor memory as is.  Rows past `rows` in
 *   the last row tile hold byte 127 (scale 1).
 */

/* fp8q_mx_scale_bytes -- size in bytes of the tiled scale array of a
 * rows x K operand: (K/128) * ceil(rows/128) * 512.  0 if rows < 0, K <= 0 or
 * K % 128 != 0. */
FP8Q_API size_t fp8q_mx_scale_bytes(int64_t rows, int64_t K);

/*
 * fp8q_mx_quantize -- MX quantization of x[rows][K] (row-major, BF16 or FP32)
 * in 1x32 groups along K (activations and weights alike).
 *   q   [rows][K] E4M3 codes;  s  tiled scales, fp8q_mx_scale_bytes(rows, K).
 * rows >= 0 (any), K % 128 == 0.  x, q, s 16-byte aligned.  Codes and scale
 * bytes are exact functions of x (bit-exact with the oracle).
 */
FP8Q_API int fp8q_mx_quantize(const void *x, int in_dtype, int64_t rows, int64_t K,
                     uint8_t *q, uint8_t *s, fp8q_stream_t stream);

/*
 * fp8q_mx_gemm -- C[m][n] = sum_k (decode(Aq[m][k]) * 2^eA(m, k/32)) *
 * (decode(Bq[n][k]) * 2^eB(n, k/32)), the scales applied by the tensor core
 * (tcgen05.mma.kind::mxf8f6f4 with block scaling) and the whole K accumulated
 * in its FP32 accumulator.
 *   Aq [M][K], Bq [N][K] codes (K contiguous);  sA, sB tiled scales of each
 *   (as written by fp8q_mx_quantize);  C [M][N] BF16 (RNE) or FP32.
 * M >= 0 (any), N % 128 == 0, K % 128 == 0; pointers 16-byte aligned.
 * Accuracy: |C - C_exact| <= 2e-3 * sum_k |a_dq * b_dq| (+ one BF16 rounding).
 */
FP8Q_API int fp8q_mx_gemm(const uint8_t *Aq, const uint8_t *sA, const uint8_t *Bq, const uint8_t *sB,
                 void *C, int64_t M, int64_t N, int64_t K, int out_dtype, fp8q_stream_t stream);

/*
 * fp8q_selftest_wait_timeout -- failure-detection self-test, not part of the
 * method.  Launches one thread that waits on an mbarrier nothing arrives on,
 * through the same bounded wait the GEMM and quantizer pipelines use.  After
 * the wait limit (2 s) the kernel records FP8Q_ERR_TIMEOUT in the device
 * status word and ends normally (no trap, no fault, no hang); the next
 * fp8q_get_device_status(stream) returns FP8Q_ERR_TIMEOUT and clears it, and
 * the CUDA context stays usable.  Returns the launch status.
 */
FP8Q_API int fp8q_selftest_wait_timeout(fp8q_stream_t stream);

/*
 * fp8q_get_device_status -- synchronizes `stream`, then returns and clears
 * the current device's status word: FP8Q_OK, or FP8Q_ERR_TIMEOUT if a
 * kernel's bounded pipeline wait expired since the last call, or
 * FP8Q_ERR_CUDA if the synchronization itself failed.
 */
FP8Q_API int fp8q_get_device_status(fp8q_stream_t stream);

/* fp8q_status_string -- static human-readable text for a status code. */
FP8Q_API const char *fp8q_status_string(int status);

/* fp8q_version -- library version as 10000*major + 100*minor + patch. */
FP8Q_API int fp8q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
