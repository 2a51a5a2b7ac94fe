/*
 * fp8fg.h -- C ABI of the fine-grained FP8 Linear library for GB300 (sm_103a).
 *
 * The library quantizes BF16 tensors to FP8 with one FP32 scale per 1x128
 * activation/gradient tile or per 128x128 weight block, multiplies the FP8
 * operands on the tcgen05 tensor cores while applying the per-128-K-chunk
 * scales to FP32 partial sums, and provides the coarse per-tensor delayed-
 * scaling variant with its underflow/distortion monitors, the MoE grouped
 * variant over a 128-padded routing map, and the SwiGLU glue between the two
 * MLP GEMMs.
 *
 * Sources, cited by page title and section:
 *   [FP8-LM] "FP8-LM: Training FP8 Large Language Models" (paper review),
 *            "Core formulas": FP8 formats, tensor scaling x_fp8 = Cast(x / s).
 *   [Ling]   Ling 2.0 FP8 pretraining blog: "Where does the error come from?",
 *            "Fine-grained quantization (per-tile/block wise scaling)", the
 *            underflow/distortion monitor table, "FP8 on-demand transpose
 *            weight", "FP8 padding routing map".
 *   [FP8-RL] FP8-RL article, "Core breakthrough: dynamic weight sync"
 *            (128x128 weight blocks, E4M3 in [-448, 448], dynamic activations),
 *            and its MoE expert layers.
 *   [Infra]  "FP8 training infrastructure" guide, "Transformer Engine" and
 *            "Scaling strategies" (delayed scaling, amax history, HYBRID).
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates nothing.  Its only state is one device status word
 *     per GPU (see fp8_device_status).
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and returns a status code.  A non-OK
 *     return means nothing was launched; outputs are then unspecified.
 *   - Matrices are row-major.  BF16 inputs are given as raw 16-bit patterns.
 *   - FP8 tensors are byte arrays of E4M3 or E5M2 codes (fp8_format_t).
 *   - Scale layouts (FP32):
 *       1x128   tensor [R][C] quantized along C: S[C/128][R]  (chunk-major)
 *       128x1   the transposed copy [C][R] of a tensor [R][C], quantized
 *               along R: S[R/128][C]   (this IS the 1x128 layout of [C][R])
 *       128x128 tensor [R][C]: S[R/128][C/128]
 *       TENSOR  one FP32 value
 *   - Pointers to FP8/BF16 data and to scale arrays must be 16-byte aligned;
 *     leading dimensions are in elements and must keep rows 16-byte aligned.
 *   - Errors found on the device (non-finite amax, bounded-wait timeout, bad
 *     group offsets) are recorded in the device status word and read with
 *     fp8_device_status().
 */
#ifndef FP8FG_H
#define FP8FG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8FG_API __attribute__((visibility("default")))

#define FP8FG_ABI_VERSION 1

/* Status codes. */
enum {
    FP8_OK = 0,
    FP8_ERR_INVALID_ARG = 1, /* null pointer, bad enum, bad count, device: bad group offsets */
    FP8_ERR_SHAPE = 2,       /* a dimension is not a required multiple (128, 256) or < 0 */
    FP8_ERR_ALIGNMENT = 3,   /* pointer or leading dimension not 16-byte aligned */
    FP8_ERR_UNSUPPORTED = 4, /* format / granularity combination not provided */
    FP8_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch, attribute, query) */
    FP8_ERR_NONFINITE = 6,   /* device: a scaling group held Inf or NaN */
    FP8_ERR_TIMEOUT = 7,     /* device: a bounded pipeline wait gave up (about 1 s) */
    FP8_ERR_BOUNDS = 8       /* device, debug build only: a kernel's store fell outside its buffer
                                (the store was skipped) */
};

typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_format_t;

typedef enum {
    FP8_GRAN_1x128 = 0,
    FP8_GRAN_128x128 = 1,
    FP8_GRAN_TENSOR = 2,
    FP8_GRAN_128x1 = 3
} fp8_gran_t;

typedef enum { FP8_OUT_BF16 = 0, FP8_OUT_F32 = 1 } fp8_out_dtype_t;

typedef enum { FP8_AMAX_MAX = 0, FP8_AMAX_MOST_RECENT = 1 } fp8_amax_algo_t;

/* Monitors ([Ling] "Where does the error come from?" and its monitor table).
 * Device-resident, ACCUMULATED by every call that is given one: zero it first.
 *   nonzero      #(x != 0)
 *   underflow    #(x != 0 and q is +0 or -0)        (smaller is better)
 *   saturated    #(|fp32(x) / s| > fmax)
 *   distinct_in  sum over scaling groups of #distinct x values (+-0 as one)
 *   distinct_out sum over scaling groups of #distinct codes   (+-0 as one)
 * Underflow ratio = underflow / nonzero; distortion is reported as the
 * retention ratio distinct_out / distinct_in (larger is better). */
typedef struct {
    uint64_t nonzero;
    uint64_t underflow;
    uint64_t saturated;
    uint64_t distinct_in;
    uint64_t distinct_out;
} fp8_stats_t;

/* Delayed-scaling recipe ([Infra] "Transformer Engine": margin, fp8 format,
 * amax_history_len, amax_compute_algo).  HYBRID = E4M3 for forward tensors,
 * E5M2 for gradients: the caller picks `fmt` per tensor. */
typedef struct {
    int32_t fmt;         /* fp8_format_t */
    int32_t history_len; /* 1 .. 1024 */
    int32_t margin;      /* s = amax * 2^margin / fmax, -126 .. 126 */
    int32_t algo;        /* fp8_amax_algo_t */
} fp8_delayed_recipe_t;

/* ---------------------------------------------------------------- utility */

FP8FG_API int fp8_abi_version(void);

/* Human-readable name of a status code (static string). */
FP8FG_API const char *fp8_status_string(int status);

/* Synchronizes `stream`, copies the current device's status word to *out and
 * clears it.  Returns FP8_ERR_CUDA if the synchronize or copy fails. */
FP8FG_API int fp8_device_status(void *stream, int *out);

/* Self-test of the bounded wait used by every pipeline wait: launches one
 * block that waits on a barrier nothing arrives at, for `timeout_ms`
 * milliseconds (1 .. 2000), after which it records FP8_ERR_TIMEOUT in the
 * device status word and returns.  The CUDA context stays usable. */
FP8FG_API int fp8_selftest_wait_timeout(int timeout_ms, void *stream);

/* 1 when this library is the index-checked debug build (compiled with
 * FP8FG_DEBUG: every kernel store checks its index against the extent of the
 * buffer it writes, records FP8_ERR_BOUNDS and skips the store if outside),
 * 0 for the release build, in which the checks compile away. */
FP8FG_API int fp8_debug_build(void);

/* Self-test of the debug build's store check: writes 1.0f to buf[i] for
 * 0 <= i < n_write (device FP32 buffer of at least n_write elements, owned by
 * the caller) through the checked store, against a claimed extent of
 * n_claimed elements (0 <= n_claimed <= n_write, else FP8_ERR_INVALID_ARG).
 * The debug build writes only buf[0, n_claimed) and, when n_write > n_claimed,
 * records FP8_ERR_BOUNDS; the release build writes all n_write elements.
 * Every store stays inside the caller's buffer in both builds. */
FP8FG_API int fp8_selftest_bounds(float *buf, int64_t n_claimed, int64_t n_write, void *stream);

/* ----------------------------------------------------------- quantizers */

/* 1x128 quantization of activations / gradients ([Ling] "Fine-grained
 * quantization"; [FP8-RL]: activations are quantized dynamically each call;
 * [FP8-LM] "Tensor scaling").  For every row r and column chunk cb:
 *   amax = max_k |x[r][cb*128+k]|,  s = fp32(amax / fmax) (1 if amax == 0),
 *   q[r][c] = RNE_satfinite(fp32(x[r][c]) / s)   (IEEE binary32 division).
 * x:  BF16 [rows][ldx], rows >= 0, cols % 128 == 0, ldx >= cols, ldx % 8 == 0.
 * q:  [rows][cols] codes.   s: S[cols/128][rows].
 * qT, sT (both NULL or both set; then rows % 128 == 0): the wgrad operand
 *   ("grad (transpose)" in [Ling]'s monitor table) from the same read of x:
 *   qT[c][m] = RNE_satfinite(x[m][c] / sT[m/128][c]) with sT = the per-column
 *   amax over each 128 rows / fmax; qT is [cols][rows], sT is S[rows/128][cols].
 * A group holding Inf/NaN records FP8_ERR_NONFINITE (its outputs unspecified). */
FP8FG_API int fp8_quant_1x128(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                              void *q, float *s, void *qT, float *sT, void *stream);

/* 128x128 weight-block quantization ([FP8-RL] "dynamic weight sync": each
 * 128x128 block of a weight gets its own scale).
 * w: BF16 [rows][ldw], rows % 128 == 0, cols % 128 == 0.  q: [rows][cols],
 * s: S[rows/128][cols/128].  Optional qT ([cols][rows]) and sT
 * (S[cols/128][rows/128]) receive the transposed weight in the same pass:
 * block quantization commutes with transposition, so qT is exactly q^T. */
FP8FG_API int fp8_quant_128x128(const void *w, int64_t rows, int64_t cols, int64_t ldw, int fmt,
                                void *q, float *s, void *qT, float *sT, void *stream);

/* On-demand FP8 transpose of a 128x128-block-quantized weight ([Ling] "FP8
 * on-demand transpose weight": no cached W^T, a fast transpose when dgrad
 * needs it).  q [rows][cols] -> qT [cols][rows] byte-exact; s
 * S[rows/128][cols/128] -> sT S[cols/128][rows/128].  rows, cols % 128 == 0. */
FP8FG_API int fp8_transpose_128x128(const void *q, const float *s, int64_t rows, int64_t cols,
                                    void *qT, float *sT, void *stream);

/* The same for `batch` matrices stored back to back (e.g. the weights of the
 * MoE experts before their grouped dgrad): q [batch][rows][cols], s
 * [batch][rows/128][cols/128] -> qT [batch][cols][rows], sT
 * [batch][cols/128][rows/128].  0 <= batch <= 65535. */
FP8FG_API int fp8_transpose_128x128_batched(const void *q, const float *s, int batch, int64_t rows,
                                            int64_t cols, void *qT, float *sT, void *stream);

/* Bytes of the caller-owned workspace used by fp8_quant_pertensor_delayed and
 * by fp8_quant_stats(FP8_GRAN_TENSOR).  Zero it once (cudaMemset) before the
 * first use; every call that completes leaves it zeroed again. */
FP8FG_API size_t fp8_pertensor_workspace_bytes(void);

/* Per-tensor delayed scaling, one training step ([Infra] "Transformer
 * Engine" DelayedScaling and "Scaling strategies": the scale comes from the
 * amax seen in earlier iterations).  State is caller-owned device memory:
 *   amax_history[recipe->history_len], *step (starts at 0), *scale (s_t,
 *   start it at 1; any s_t >= 0 including +Inf is handled, the codes for a
 *   negative or NaN s_t are unspecified).
 * The call quantizes q = RNE_satfinite(x / s_t), writes this step's amax to
 * amax_history[step % L], sets *scale = s_{t+1} = m * 2^margin / fmax with
 * m = max(history) (or this step's amax for FP8_AMAX_MOST_RECENT; unchanged
 * if m == 0) and increments *step -- all on the device, no host round trip.
 * x: BF16 [rows][ldx], any rows, cols % 128 == 0.  q: [rows][cols].  qT
 * (optional, then rows % 128 == 0): [cols][rows] = q^T for the wgrad
 * operand.  stats (optional): monitors with the whole tensor as one group.
 * workspace: fp8_pertensor_workspace_bytes() bytes, see above.  Calls that
 * share one workspace must not overlap on the GPU. */
FP8FG_API int fp8_quant_pertensor_delayed(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                          const fp8_delayed_recipe_t *recipe, float *amax_history,
                                          int32_t *step, float *scale, void *q, void *qT,
                                          fp8_stats_t *stats, void *workspace, void *stream);

/* Per-tensor current scaling ([FP8-RL] "KV cache compression": after every
 * model update the FP8 KV cache's scaling factor is recomputed from the
 * current tensor, "inference-side calibration").  One group, the whole
 * tensor: *scale = s = fp32(amax / fmax) (1 if amax = 0), written on the
 * device, and q = RNE_satfinite(x / s).  x: BF16 [rows][ldx], cols % 8 == 0,
 * x 16-byte and q 8-byte aligned.  q: [rows][cols].  scale: DEVICE float.
 * workspace: fp8_pertensor_workspace_bytes() bytes, zeroed once and left
 * zeroed (calls sharing one workspace must not overlap on the GPU).  A tensor
 * holding Inf/NaN records FP8_ERR_NONFINITE (outputs unspecified). */
FP8FG_API int fp8_quant_pertensor_current(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                          int fmt, float *scale, void *q, void *workspace,
                                          void *stream);

/* MXFP8 quantization ([Infra] "Hardware requirements for FP8 training":
 * Blackwell adds MXFP8, micro-scaled FP8; "Scaling strategies and
 * stability": each block inside a tensor gets its own scale factor).  The
 * pages give neither the block size nor the scale encoding; here a block is
 * 32 consecutive elements of a row, and its scale is a power of two
 * X = 2^(e8 - 127) stored as an 8-bit exponent code: the smallest power of
 * two with amax / X <= fmax, so no element saturates (X = 1 for an all-zero
 * block).  q = RNE_satfinite(x / X), exact since X is a power of two.
 *   x: BF16 [rows][ldx], cols % 32 == 0, x 16-byte aligned, ldx % 8 == 0.
 *   q: [rows][cols] codes (fmt), 8-byte aligned.
 *   e8: [rows][cols/32] scale codes, any alignment.
 * A block holding Inf/NaN records FP8_ERR_NONFINITE (its outputs are
 * unspecified).  rows or cols == 0 is a no-op. */
FP8FG_API int fp8_quant_mx(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                           void *q, uint8_t *e8, void *stream);

/* fp8_quant_mx with the scale codes written in the layout fp8_mx_gemm_tiled
 * reads (the library's own layout; the pages fix none): for rows and cols
 * multiples of 128, the codes of rows 128 rb .. 128 rb + 127 and 32-blocks
 * 4 kc .. 4 kc + 3 form one 512-byte tile at byte (kc * rows/128 + rb) * 512;
 * inside it the code of row r, block b sits at byte
 * 16 (r % 32) + 4 ((r % 128) / 32) + (b % 4).  Same codes, values and
 * errors as fp8_quant_mx; only the position of each scale code differs.
 *   x, q: as fp8_quant_mx.  rows % 128 == 0, cols % 128 == 0.
 *   e8_tiled: rows * cols / 32 bytes (16-byte aligned if fp8_mx_gemm_tiled
 *   will read it).  rows or cols == 0 is a no-op. */
FP8FG_API int fp8_quant_mx_tiled(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, void *q,
                                 uint8_t *e8_tiled, void *stream);

/* MXFP8 GEMM ([Infra] "Scaling strategies and stability": per-block scaling,
 * each block of a tensor with its own scale factor; "Blackwell MXFP8 and
 * NVFP4: looking ahead"; block and scale encoding per the readings of
 * fp8_quant_mx): D = A . B^T with A [M][K] and B [N][K] FP8 codes (fmtA,
 * fmtB), K contiguous, and their scale exponents eA [M][K/32], eB [N][K/32]
 * as fp8_quant_mx writes them (X = 2^(e - 127)):
 *   D[m][n] = sum_b X_A(m, b) * X_B(n, b) * sum_{k in 32-block b} qA[m][k] * qB[n][k].
 * The tensor cores apply the two scales to every 32-block themselves
 * (tcgen05.mma kind::mxf8f6f4.block_scale, scale codes read as UE8M0) and
 * accumulate the whole K in FP32 in tensor memory; no promotion in
 * registers.  Scale codes are 0..254 (what fp8_quant_mx writes; the format
 * reads 255 as NaN).  D [M][ldD] BF16 (RN) or FP32.  M, N, K % 128 == 0; A,
 * B, D 16-byte aligned, eA, eB 4-byte aligned, ldD * element size a
 * multiple of 16 bytes.  K == 0 writes zeros; M or N == 0 is a no-op. */
FP8FG_API int fp8_mx_gemm(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const uint8_t *eA,
                          const void *B, int fmtB, const uint8_t *eB, void *D, int out_dtype, int64_t ldD,
                          void *stream);

/* fp8_mx_gemm with both operands' scale codes in the tiled layout of
 * fp8_quant_mx_tiled (eA_tiled for M rows, eB_tiled for N rows, K / 32 codes
 * per row).  The tiles are fetched by bulk copies beside the operand tiles, so
 * no thread of the GEMM reorders them; the result is bit-identical to
 * fp8_mx_gemm on the same codes.  eA_tiled and eB_tiled 16-byte aligned;
 * everything else as fp8_mx_gemm. */
FP8FG_API int fp8_mx_gemm_tiled(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const uint8_t *eA_tiled,
                                const void *B, int fmtB, const uint8_t *eB_tiled, void *D, int out_dtype,
                                int64_t ldD, void *stream);

/* The same delayed-scaling step for callers that cannot allocate device
 * memory -- for example code that runs inside another framework's fixed
 * memory plan or arena, or a plugin that is handed buffers but no allocator.
 * The pages have no counterpart: this is a library convenience.
 * Instead of a caller-owned workspace it uses a 16 KiB scratch block that the
 * library keeps in device memory for every GPU that loads it (until process
 * exit); the step needs fp8_pertensor_workspace_bytes() of it whatever the
 * tensor size, and a call returns FP8_ERR_UNSUPPORTED if that ever exceeded
 * the block.  The caller still passes x, the state and the outputs exactly as
 * for fp8_quant_pertensor_delayed, and results are identical.  The call
 * allocates nothing; it clears the scratch on `stream` before the kernel
 * (cudaMemsetAsync).  All calls share the one block, so calls that may run
 * at the same time on the GPU (different streams without ordering) race on
 * it.  The first call on each device looks up the block's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. */
FP8FG_API int fp8_quant_pertensor_delayed_noalloc(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                                  const fp8_delayed_recipe_t *recipe, float *amax_history,
                                                  int32_t *step, float *scale, void *q, void *qT,
                                                  fp8_stats_t *stats, void *stream);

/* Monitors of an existing quantization ([Ling] underflow / distortion
 * monitors), accumulated into *stats.  x: BF16 [rows][ldx]; q and s follow
 * `gran` (1x128, 128x128, TENSOR: q is [rows][cols]; 128x1: q is the
 * transposed copy [cols][rows] with S[rows/128][cols]).  `workspace` is
 * needed for FP8_GRAN_TENSOR only (same contract as above). */
FP8FG_API int fp8_quant_stats(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                              const void *q, const float *s, int gran, int fmt,
                              fp8_stats_t *stats, void *workspace, void *stream);

/* ---------------------------------------------------------------- GEMMs */

/* Block-scaled FP8 GEMM, D = A . B^T ([Ling]: FP8 GEMM with an FP32
 * accumulator; fine-grained tile/block scales):
 *   D[m][n] = sum_kb sA(m,kb) * sB(n,kb) * sum_{k in chunk kb} qA[m][k]*qB[n][k]
 * with each 128-deep chunk accumulated on the tensor cores and promoted to an
 * FP32 running sum with its two scales.  For granA == granB == TENSOR the
 * whole K is accumulated on the tensor cores and sA*sB applied once.
 *   A [M][K] codes (fmtA), B [N][K] codes (fmtB), K contiguous in both.
 *   granA in {1x128 (S[K/128][M]), 128x128 (S[M/128][K/128]), TENSOR};
 *   granB in {1x128 (S[K/128][N]), 128x128 (S[N/128][K/128]), TENSOR};
 *   TENSOR must be used on both sides or neither.
 *   fmtA/fmtB: E4M3 or E5M2, mixed allowed (HYBRID dgrad/wgrad).
 *   D [M][ldD], BF16 (round to nearest even) or FP32.
 * M % 128 == 0, N % 128 == 0, K % 128 == 0; M, N, K >= 0.  M == 0 or N == 0
 * is a no-op; K == 0 writes D[M][N] = 0 (the empty sum; A, B and the scales
 * may then be NULL). */
FP8FG_API int fp8_blockscaled_gemm(int64_t M, int64_t N, int64_t K,
                                   const void *A, int fmtA, const float *sA, int granA,
                                   const void *B, int fmtB, const float *sB, int granB,
                                   void *D, int out_dtype, int64_t ldD, void *stream);

/* Grouped MoE expert GEMM ([FP8-RL]: FP8 on the MoE expert layers; [Ling]
 * "FP8 padding routing map": every expert's row count is a multiple of 128).
 * Rows [off[g], off[g+1]) of A use expert g's weights:
 *   D[m][n] = the block-scaled GEMM of A's row m with B[g] (128x128 scales).
 * group_offsets: DEVICE int32[G+1], 0 = off[0] <= ... <= off[G] <= M_capacity,
 *   each a multiple of 128 (checked on the device: FP8_ERR_INVALID_ARG).
 * A [M_capacity][K] E4M3 with 1x128 scales S[K/128][M_capacity];
 * B [G][N][K] E4M3 with scales [G][N/128][K/128]; D [M_capacity][ldD]
 * (rows >= off[G] are not written).  N % 128 == 0, K % 128 == 0,
 * M_capacity % 128 == 0, 1 <= G <= 1024.  M_capacity, N or K == 0 is a
 * no-op: D is not written. */
FP8FG_API int fp8_grouped_gemm(int G, const int32_t *group_offsets, int64_t M_capacity,
                               int64_t N, int64_t K, const void *A, const float *sA,
                               const void *B, const float *sB, void *D, int out_dtype,
                               int64_t ldD, void *stream);

/* Grouped MoE weight gradient ([FP8-RL]: FP8 on the MoE expert layers; [Ling]
 * monitor table "grad (transpose)": the wgrad operands are the copies
 * quantized 128x1 along the token dimension).  Expert g's dispatch rows are
 * [off[g], off[g+1]) of two dispatch-ordered tensors; AT and BT are their
 * transposed copies (fp8_quant_1x128 with qT, sT), so
 *   D[g] = AT[:, off[g]:off[g+1]] . BT[:, off[g]:off[g+1]]^T, [N][K],
 * promoted per 128 rows with both operands' scales; an expert without rows
 * gets D[g] = 0.
 * group_offsets: DEVICE int32[G+1], 0 = off[0] <= ... <= off[G] <= M_capacity,
 *   multiples of 128 (checked on the device: FP8_ERR_INVALID_ARG).
 * AT [N][M_capacity] (fmtA) with scales S[M_capacity/128][N];
 * BT [K][M_capacity] (fmtB) with scales S[M_capacity/128][K];
 * D [G*N][ldD] (expert g at rows g*N ..), FP8_OUT_F32 or FP8_OUT_BF16.
 * N, K, M_capacity % 128 == 0, 1 <= G <= 1024. */
FP8FG_API int fp8_grouped_gemm_wgrad(int G, const int32_t *group_offsets, int64_t M_capacity,
                                     int64_t N, int64_t K, const void *AT, int fmtA, const float *sAT,
                                     const void *BT, int fmtB, const float *sBT, void *D,
                                     int out_dtype, int64_t ldD, void *stream);

/* ------------------------------------------------ high-precision dw monitor */

/* Error statistics of an FP8 wgrad D against its high-precision recompute R. */
typedef struct {
    double sum_sq_diff;   /* sum (D - R)^2 */
    double sum_sq_ref;    /* sum R^2 */
    float max_abs_diff;   /* max |D - R| */
    float max_abs_ref;    /* max |R| */
} fp8_wgrad_err_t;

/* High-precision dw recompute monitor ([Ling] "Where does the error come
 * from?": tensors flagged by the underflow / distortion monitors get their dw
 * recomputed in high precision and compared).  R = dY^T . X from the BF16
 * operands, token-major dY [M][N] and X [M][K] (row-major), products of BF16
 * values accumulated in FP32 over the M tokens on the tensor cores (this
 * library's kernel), written to ref_workspace [N][K] (caller-owned, N*K
 * floats, row stride K); then *err (DEVICE) = the statistics of D [N][ldD]
 * (FP32, e.g. fp8_blockscaled_gemm's wgrad output) against R: D - R in
 * FP32, its square and R's in FP64 (exact), summed in FP64.  err is cleared
 * by the call.  The relative Frobenius error is
 * sqrt(sum_sq_diff / sum_sq_ref).  N, K % 128 == 0 (FP8_ERR_SHAPE), any M
 * (0: R = 0); M, N, K < 2^31; dY, X, D, ref_workspace 16-byte aligned and
 * ldD % 4 == 0 (FP8_ERR_ALIGNMENT). */
FP8FG_API int fp8_wgrad_recompute_error(int64_t M, int64_t N, int64_t K, const void *dY, const void *X,
                                        const float *D, int64_t ldD, float *ref_workspace,
                                        fp8_wgrad_err_t *err, void *stream);

/* ------------------------------------------------------ FP8 optimizer states */

/* Hyper-parameters of one AdamW step, as binary32 numbers; the bias
 * corrections are the caller's roundings of 1 - beta^t for step t >= 1. */
typedef struct {
    float lr, beta1, beta2, one_minus_beta1, one_minus_beta2, eps, weight_decay;
    float bias_correction1, bias_correction2;
} fp8_adamw_hparams_t;

/* One AdamW step with the moments kept in FP8 ([Ling] "FP8 Optimizer": both
 * Adam moments in FP8 with fine-grained compression / decompression; [FP8-LM]
 * "Level 2: FP8 optimizer").  m: E4M3 codes [n] with scales m_scales[n/128],
 * v: E5M2 codes [n] with scales v_scales[n/128] (one scale per 128 consecutive
 * parameters, s = amax / fmax, 1 for an all-zero block; start from zero codes
 * and unit scales).  With g the BF16 gradient, every operation a correctly
 * rounded binary32 one in this order:
 *   m = dec(m) * sm;  m = beta1 * m + one_minus_beta1 * g
 *   v = dec(v) * sv;  v = beta2 * v + one_minus_beta2 * (g * g)
 *   u = (m / bias_correction1) / (sqrt(v / bias_correction2) + eps)
 *   param = param - lr * (u + weight_decay * param)
 * and m, v are re-quantized with their blocks' new scales -- all in place, one
 * pass.  param: FP32 master weights [n].  n % 128 == 0; param, grad, m, v
 * 16-byte aligned.  Gradients, parameters and moments are finite; the results
 * for a block holding Inf or NaN are unspecified. */
FP8FG_API int fp8_adamw_step_fp8_states(float *param, const void *grad, uint8_t *m, float *m_scales,
                                        uint8_t *v, float *v_scales, int64_t n,
                                        const fp8_adamw_hparams_t *hparams, void *stream);

/* -------------------------------------------------------------- MoE glue */

/* Router + padded routing map ([Ling] "FP8 padding routing map").
 * logits: FP32 [T][E] (E <= 256).  For each token: softmax in FP32 and the
 * top-k experts by logit (softmax is monotone), ties to the lower index:
 * topk_idx [T][topk], topk_prob [T][topk].  counts[E] = tokens routed to
 * each expert.  The routing map is then edited so that each expert's row
 * count is counts rounded up to a multiple of `align`: the added entries are
 * the lowest-index tokens not already routed to that expert, with router
 * probability 0 (so the result is unchanged).  Rows of expert e occupy
 * [group_offsets[e], group_offsets[e+1]) in ascending token order:
 * row_token[r] = token, row_prob[r] = its probability (0 for padding),
 * row_is_pad[r] (optional) = 1 for padding.  Rows from group_offsets[E] to
 * M_capacity get row_token = -1, row_prob = 0.  The total must fit
 * M_capacity and every padded count must be reachable with distinct tokens
 * (else FP8_ERR_INVALID_ARG on the device); T*topk + E*(align-1) always fits
 * M_capacity.  1 <= topk <= min(E, 8), align in {1..1024}.  The logits are
 * finite; the routing of a token with an Inf or NaN logit is unspecified. */
FP8FG_API int fp8_moe_route_pad(const float *logits, int64_t T, int E, int topk, int align,
                                int64_t M_capacity, int32_t *topk_idx, float *topk_prob,
                                int32_t *counts, int32_t *group_offsets, int32_t *row_token,
                                float *row_prob, uint8_t *row_is_pad, void *stream);

/* Dispatch: gather the FP8 rows and 1x128 scales of the routed tokens.
 * Quantizing once before the gather is exact: 1x128 scales are per row.
 * q [T][K], s S[K/128][T] -> qg [M_capacity][K], sg S[K/128][M_capacity] for
 * rows r < group_offsets[E] (read on the device); other rows untouched. */
FP8FG_API int fp8_moe_gather(const void *q, const float *s, int64_t T, int64_t K,
                             const int32_t *row_token, const int32_t *group_offsets, int E,
                             int64_t M_capacity, void *qg, float *sg, void *stream);

/* SwiGLU between the up and down projections (glue, FP32 math, BF16 out):
 * gu [rows][2F] holds gate in columns [0, F) and up in [F, 2F);
 * h[r][j] = silu(g) * u.   F % 8 == 0. */
FP8FG_API int fp8_swiglu_fwd(const void *gu, int64_t rows, int64_t F, void *h, void *stream);

/* Backward of the above: dgu[r][j] = dh*u*sig(g)*(1 + g*(1 - sig(g))),
 * dgu[r][F+j] = dh*silu(g). */
FP8FG_API int fp8_swiglu_bwd(const void *gu, const void *dh, int64_t rows, int64_t F, void *dgu,
                             void *stream);

/* SwiGLU fused into the 1x128 quantizer with its 128x1 transposed copy
 * ([Ling] "Fine-grained quantization": the activation that feeds the down
 * projection and the gradient that feeds the up projection's dgrad/wgrad are
 * quantized 1x128 per row, and 128x1 for the wgrad operand).  The BF16
 * values are those fp8_swiglu_fwd / fp8_swiglu_bwd would write, bit for bit,
 * but they are computed while loading and never stored; the outputs equal
 * fp8_quant_1x128(those values, qT, sT set) bit for bit.
 * Forward:  gu BF16 [rows][2F]  ->  H [rows][F] quantized:
 *   q [rows][F], s S[F/128][rows], qT [F][rows], sT S[rows/128][F].
 * Backward: gu, dh BF16 [rows][F]  ->  dGU [rows][2F] quantized:
 *   q [rows][2F], s S[2F/128][rows], qT [2F][rows], sT S[rows/128][2F].
 * rows % 128 == 0, F % 128 == 0, rows * (output cols / 128) < 2^31; all
 * pointers 16-byte aligned and owned by the caller.  A group holding Inf/NaN
 * records FP8_ERR_NONFINITE (its outputs unspecified). */
FP8FG_API int fp8_swiglu_quant_fwd(const void *gu, int64_t rows, int64_t F, int fmt, void *q, float *s,
                                   void *qT, float *sT, void *stream);
FP8FG_API int fp8_swiglu_bwd_quant(const void *gu, const void *dh, int64_t rows, int64_t F, int fmt,
                                   void *q, float *s, void *qT, float *sT, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8FG_H */
