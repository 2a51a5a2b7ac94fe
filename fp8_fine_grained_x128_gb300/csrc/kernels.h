// kernels.h -- host-side launchers of the sm_103a kernels.  Arguments are
// validated by the C ABI layer (api.cu) before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8fg.h"

namespace fp8fg {

// Number of SMs of the current device (cached per device).
int sm_count();

// Device address of the current device's status word (nullptr on failure).
int *status_word_ptr();

// quant.cu
int launch_quant_1x128(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, void *q, float *s,
                       void *qT, float *sT, int *status, cudaStream_t st);
// tiled: scale codes in the GEMM's 512-byte tile layout instead of row-major
int launch_quant_mx(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, void *q, uint8_t *e8,
                    bool tiled, int *status, cudaStream_t st);
int launch_quant_128x128(const void *w, int64_t rows, int64_t cols, int64_t ldw, int fmt, void *q, float *s,
                         void *qT, float *sT, int *status, cudaStream_t st);
// batch matrices of [rows][cols] stored back to back (scales likewise)
int launch_transpose_128x128(const void *q, const float *s, int64_t rows, int64_t cols, void *qT, float *sT,
                             cudaStream_t st, int batch = 1);

// api.cu: the argument contract of the delayed-scaling step (recipe bounds,
// shapes, required pointers, 16-byte alignment), shared by the entry point
// with a caller workspace and the one without (workspace_required = false)
int check_pertensor_delayed_args(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                 const fp8_delayed_recipe_t *recipe, const float *amax_history, const int32_t *step,
                                 const float *scale, const void *q, const void *qT, const fp8_stats_t *stats,
                                 const void *workspace, bool workspace_required);

// pertensor.cu
size_t pertensor_workspace_bytes();
int launch_pertensor_delayed(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, int hist_len,
                             int margin, int algo, float *hist, int32_t *step, float *scale, void *q, void *qT,
                             void *stats, void *ws, int *status, cudaStream_t st);
int launch_quant_stats(const void *x, int64_t rows, int64_t cols, int64_t ldx, const void *q, const float *s,
                       int gran, int fmt, void *stats, void *ws, int *status, cudaStream_t st);
int launch_pertensor_current(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, float *scale, void *q,
                             void *ws, int *status, cudaStream_t st);
int launch_selftest_wait(int timeout_ms, int *status, cudaStream_t st);
int launch_selftest_bounds(float *buf, int64_t n_claimed, int64_t n_write, int *status, cudaStream_t st);

// gemm.cu
int launch_gemm(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const float *sA, int granA,
                const void *B, int fmtB, const float *sB, int granB, void *D, int out_dtype, int64_t ldD,
                int *status, cudaStream_t st);
int launch_gemm_mx(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const uint8_t *eA, const void *B,
                   int fmtB, const uint8_t *eB, bool tiled, void *D, int out_dtype, int64_t ldD, int *status,
                   cudaStream_t st);
int launch_grouped_gemm(int G, const int32_t *offsets, int64_t Mcap, int64_t N, int64_t K, const void *A,
                        const float *sA, const void *B, const float *sB, void *D, int out_dtype, int64_t ldD,
                        int *status, cudaStream_t st);
int launch_grouped_wgrad(int G, const int32_t *offsets, int64_t Mcap, int64_t N, int64_t K, const void *AT, int fmtA,
                         const float *sAT, const void *BT, int fmtB, const float *sBT, void *D, int out_dtype,
                         int64_t ldD, int *status, cudaStream_t st);

// monitor_dw.cu
int launch_wgrad_recompute_error(int64_t M, int64_t N, int64_t K, const void *dY, const void *X, const float *D,
                                 int64_t ldD, float *R, fp8_wgrad_err_t *err, int *status, cudaStream_t st);

// optim.cu
int launch_adamw_fp8(float *p, const void *g, uint8_t *qm, float *sm, uint8_t *qv, float *sv, int64_t n,
                     const fp8_adamw_hparams_t &h, cudaStream_t st);

// moe.cu
int launch_moe_route_pad(const float *logits, int64_t T, int E, int topk, int align, int64_t Mcap,
                         int32_t *topk_idx, float *topk_prob, int32_t *counts, int32_t *offsets, int32_t *row_token,
                         float *row_prob, uint8_t *row_is_pad, int *status, cudaStream_t st);
int launch_moe_gather(const void *q, const float *s, int64_t T, int64_t K, const int32_t *row_token,
                      const int32_t *offsets, int E, int64_t Mcap, void *qg, float *sg, cudaStream_t st);
int launch_swiglu_fwd(const void *gu, int64_t rows, int64_t F, void *h, cudaStream_t st);
int launch_swiglu_bwd(const void *gu, const void *dh, int64_t rows, int64_t F, void *dgu, cudaStream_t st);
int launch_swiglu_quant(const void *gu, const void *dh, int64_t rows, int64_t F, int fmt, void *q, float *s,
                        void *qT, float *sT, int *status, cudaStream_t st);

}  // namespace fp8fg
