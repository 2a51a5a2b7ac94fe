// api.cu -- the C ABI declared in include/fp8fg.h: argument validation on the
// host (no launch on a bad argument), the per-device status word, and the
// dispatch to the kernel launchers.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

// The one piece of library state: a status word per device, written by
// kernels (first error wins) and read/cleared by fp8_device_status.
__device__ int g_status_word;

static std::mutex g_mu;
static int *g_status_ptr[64] = {};
static int g_sm_count[64] = {};

static int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

// Device address of this device's status word (looked up once per device).
static int *status_ptr()
{
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

int *status_word_ptr() { return status_ptr(); }

int sm_count()
{
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace fp8fg

using namespace fp8fg;

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool fmt_ok(int f) { return f == FP8_E4M3 || f == FP8_E5M2; }
inline cudaStream_t S(void *stream) { return static_cast<cudaStream_t>(stream); }

// Common prologue: resolve the status word (needs a working CUDA device).
#define FP8FG_STATUS_OR_RETURN(var) \
    int *var = status_ptr();        \
    if (!var) return FP8_ERR_CUDA

}  // namespace

namespace fp8fg {

int check_pertensor_delayed_args(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                 const fp8_delayed_recipe_t *recipe, const float *amax_history, const int32_t *step,
                                 const float *scale, const void *q, const void *qT, const fp8_stats_t *stats,
                                 const void *workspace, bool workspace_required)
{
    if (!recipe || !fmt_ok(recipe->fmt)) return FP8_ERR_INVALID_ARG;
    if (recipe->history_len < 1 || recipe->history_len > 1024) return FP8_ERR_INVALID_ARG;
    if (recipe->margin < -126 || recipe->margin > 126) return FP8_ERR_INVALID_ARG;
    if (recipe->algo != FP8_AMAX_MAX && recipe->algo != FP8_AMAX_MOST_RECENT) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % 128 != 0) return FP8_ERR_SHAPE;
    if (qT && rows % 128 != 0) return FP8_ERR_SHAPE;
    if (!amax_history || !step || !scale || (workspace_required && !workspace)) return FP8_ERR_INVALID_ARG;
    if (rows > 0 && cols > 0 && (!x || !q)) return FP8_ERR_INVALID_ARG;
    if (rows > 0 && cols > 0 && ldx < cols) return FP8_ERR_SHAPE;
    if ((x && !aligned16(x)) || (q && !aligned16(q)) || ldx % 8 != 0) return FP8_ERR_ALIGNMENT;
    if ((qT && !aligned16(qT)) || (workspace && !aligned16(workspace)) || (stats && !aligned16(stats)))
        return FP8_ERR_ALIGNMENT;
    return FP8_OK;
}

}  // namespace fp8fg

extern "C" {

FP8FG_API int fp8_abi_version(void) { return FP8FG_ABI_VERSION; }

FP8FG_API const char *fp8_status_string(int status)
{
    switch (status) {
    case FP8_OK: return "FP8_OK";
    case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
    case FP8_ERR_SHAPE: return "FP8_ERR_SHAPE";
    case FP8_ERR_ALIGNMENT: return "FP8_ERR_ALIGNMENT";
    case FP8_ERR_UNSUPPORTED: return "FP8_ERR_UNSUPPORTED";
    case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
    case FP8_ERR_NONFINITE: return "FP8_ERR_NONFINITE";
    case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT";
    case FP8_ERR_BOUNDS: return "FP8_ERR_BOUNDS";
    default: return "FP8_ERR_UNKNOWN";
    }
}

FP8FG_API int fp8_device_status(void *stream, int *out)
{
    if (!out) return FP8_ERR_INVALID_ARG;
    FP8FG_STATUS_OR_RETURN(st);
    if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return FP8_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, st, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return FP8_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(st, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return FP8_ERR_CUDA;
    *out = v;
    return FP8_OK;
}

FP8FG_API int fp8_selftest_wait_timeout(int timeout_ms, void *stream)
{
    if (timeout_ms < 1 || timeout_ms > 2000) return FP8_ERR_INVALID_ARG;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_selftest_wait(timeout_ms, st, S(stream));
}

FP8FG_API int fp8_debug_build(void)
{
#ifdef FP8FG_DEBUG
    return 1;
#else
    return 0;
#endif
}

FP8FG_API int fp8_selftest_bounds(float *buf, int64_t n_claimed, int64_t n_write, void *stream)
{
    if (n_claimed < 0 || n_write < n_claimed) return FP8_ERR_INVALID_ARG;
    if (n_write == 0) return FP8_OK;
    if (!buf) return FP8_ERR_INVALID_ARG;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_selftest_bounds(buf, n_claimed, n_write, st, S(stream));
}

FP8FG_API int fp8_quant_1x128(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, void *q, float *s,
                              void *qT, float *sT, void *stream)
{
    if (!fmt_ok(fmt)) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % 128 != 0) return FP8_ERR_SHAPE;
    if ((qT == nullptr) != (sT == nullptr)) return FP8_ERR_INVALID_ARG;
    if (qT && rows % 128 != 0) return FP8_ERR_SHAPE;
    if (rows * (cols / 128) >= (int64_t)1 << 31) return FP8_ERR_SHAPE;
    if (rows == 0 || cols == 0) return FP8_OK;
    if (!x || !q || !s) return FP8_ERR_INVALID_ARG;
    if (ldx < cols) return FP8_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s) || ldx % 8 != 0) return FP8_ERR_ALIGNMENT;
    if (qT && (!aligned16(qT) || !aligned16(sT))) return FP8_ERR_ALIGNMENT;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_quant_1x128(x, rows, cols, ldx, fmt, q, s, qT, sT, st, S(stream));
}

FP8FG_API int fp8_quant_128x128(const void *w, int64_t rows, int64_t cols, int64_t ldw, int fmt, void *q, float *s,
                                void *qT, float *sT, void *stream)
{
    if (!fmt_ok(fmt)) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0) return FP8_ERR_SHAPE;
    if ((qT == nullptr) != (sT == nullptr)) return FP8_ERR_INVALID_ARG;
    if (rows / 128 >= 65536 || cols / 128 >= ((int64_t)1 << 31)) return FP8_ERR_SHAPE;
    if (rows == 0 || cols == 0) return FP8_OK;
    if (!w || !q || !s) return FP8_ERR_INVALID_ARG;
    if (ldw < cols) return FP8_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(q) || ldw % 8 != 0) return FP8_ERR_ALIGNMENT;
    if (qT && !aligned16(qT)) return FP8_ERR_ALIGNMENT;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_quant_128x128(w, rows, cols, ldw, fmt, q, s, qT, sT, st, S(stream));
}

FP8FG_API int fp8_transpose_128x128(const void *q, const float *s, int64_t rows, int64_t cols, void *qT, float *sT,
                                    void *stream)
{
    if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0) return FP8_ERR_SHAPE;
    if (rows / 128 >= 65536) return FP8_ERR_SHAPE;
    if (rows == 0 || cols == 0) return FP8_OK;
    if (!q || !s || !qT || !sT) return FP8_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(qT)) return FP8_ERR_ALIGNMENT;
    return launch_transpose_128x128(q, s, rows, cols, qT, sT, S(stream));
}

FP8FG_API int fp8_transpose_128x128_batched(const void *q, const float *s, int batch, int64_t rows, int64_t cols,
                                            void *qT, float *sT, void *stream)
{
    if (batch < 0 || batch > 65535) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0) return FP8_ERR_SHAPE;
    if (rows / 128 >= 65536 || cols / 128 >= ((int64_t)1 << 31)) return FP8_ERR_SHAPE;
    if (batch == 0 || rows == 0 || cols == 0) return FP8_OK;
    if (!q || !s || !qT || !sT) return FP8_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(qT)) return FP8_ERR_ALIGNMENT;
    return launch_transpose_128x128(q, s, rows, cols, qT, sT, S(stream), batch);
}

FP8FG_API size_t fp8_pertensor_workspace_bytes(void) { return pertensor_workspace_bytes(); }

FP8FG_API int fp8_quant_pertensor_delayed(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                          const fp8_delayed_recipe_t *recipe, float *amax_history, int32_t *step,
                                          float *scale, void *q, void *qT, fp8_stats_t *stats, void *workspace,
                                          void *stream)
{
    const int rc = check_pertensor_delayed_args(x, rows, cols, ldx, recipe, amax_history, step, scale, q, qT, stats,
                                                workspace, true);
    if (rc != FP8_OK) return rc;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_pertensor_delayed(x, rows, cols, ldx, recipe->fmt, recipe->history_len, recipe->margin,
                                    recipe->algo, amax_history, step, scale, q, qT, stats, workspace, st, S(stream));
}

FP8FG_API int fp8_quant_pertensor_current(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                                          float *scale, void *q, void *workspace, void *stream)
{
    if (!fmt_ok(fmt)) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % 8 != 0 || ldx < cols) return FP8_ERR_SHAPE;
    if (!scale || !workspace) return FP8_ERR_INVALID_ARG;
    if (rows > 0 && cols > 0 && (!x || !q)) return FP8_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (q && (reinterpret_cast<uintptr_t>(q) & 7u)) || ldx % 8 != 0 || !aligned16(workspace))
        return FP8_ERR_ALIGNMENT;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_pertensor_current(x, rows, cols, ldx, fmt, scale, q, workspace, st, S(stream));
}

FP8FG_API int fp8_quant_mx(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, void *q, uint8_t *e8,
                           void *stream)
{
    if (!fmt_ok(fmt)) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % 32 != 0) return FP8_ERR_SHAPE;
    if (rows == 0 || cols == 0) return FP8_OK;
    if (!x || !q || !e8) return FP8_ERR_INVALID_ARG;
    if (ldx < cols) return FP8_ERR_SHAPE;
    if (!aligned16(x) || ldx % 8 != 0 || (reinterpret_cast<uintptr_t>(q) & 7u)) return FP8_ERR_ALIGNMENT;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_quant_mx(x, rows, cols, ldx, fmt, q, e8, false, st, S(stream));
}

FP8FG_API int fp8_quant_mx_tiled(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, void *q,
                                 uint8_t *e8_tiled, void *stream)
{
    if (!fmt_ok(fmt)) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0) return FP8_ERR_SHAPE;
    if (rows == 0 || cols == 0) return FP8_OK;
    if (!x || !q || !e8_tiled) return FP8_ERR_INVALID_ARG;
    if (ldx < cols) return FP8_ERR_SHAPE;
    if (!aligned16(x) || ldx % 8 != 0 || (reinterpret_cast<uintptr_t>(q) & 7u)) return FP8_ERR_ALIGNMENT;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_quant_mx(x, rows, cols, ldx, fmt, q, e8_tiled, true, st, S(stream));
}

FP8FG_API int fp8_quant_stats(const void *x, int64_t rows, int64_t cols, int64_t ldx, const void *q, const float *s,
                              int gran, int fmt, fp8_stats_t *stats, void *workspace, void *stream)
{
    if (!fmt_ok(fmt)) return FP8_ERR_INVALID_ARG;
    if (gran < FP8_GRAN_1x128 || gran > FP8_GRAN_128x1) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return FP8_ERR_SHAPE;
    if (gran == FP8_GRAN_1x128 && cols % 128 != 0) return FP8_ERR_SHAPE;
    if (gran != FP8_GRAN_1x128 && (rows % 128 != 0 || cols % 128 != 0)) return FP8_ERR_SHAPE;
    if (rows == 0 || cols == 0) return FP8_OK;
    if (!x || !q || !s || !stats) return FP8_ERR_INVALID_ARG;
    if (gran == FP8_GRAN_TENSOR && !workspace) return FP8_ERR_INVALID_ARG;
    if (ldx < cols) return FP8_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || ldx % 8 != 0 || !aligned16(stats)) return FP8_ERR_ALIGNMENT;
    if (workspace && !aligned16(workspace)) return FP8_ERR_ALIGNMENT;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_quant_stats(x, rows, cols, ldx, q, s, gran, fmt, stats, workspace, st, S(stream));
}

FP8FG_API int fp8_blockscaled_gemm(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const float *sA,
                                   int granA, const void *B, int fmtB, const float *sB, int granB, void *D,
                                   int out_dtype, int64_t ldD, void *stream)
{
    if (!fmt_ok(fmtA) || !fmt_ok(fmtB)) return FP8_ERR_INVALID_ARG;
    if (out_dtype != FP8_OUT_BF16 && out_dtype != FP8_OUT_F32) return FP8_ERR_INVALID_ARG;
    auto gran_ok = [](int g) { return g == FP8_GRAN_1x128 || g == FP8_GRAN_128x128 || g == FP8_GRAN_TENSOR; };
    if (!gran_ok(granA) || !gran_ok(granB)) return FP8_ERR_INVALID_ARG;
    if ((granA == FP8_GRAN_TENSOR) != (granB == FP8_GRAN_TENSOR)) return FP8_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0 || M % 128 != 0 || N % 128 != 0 || K % 128 != 0) return FP8_ERR_SHAPE;
    if (M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31)) return FP8_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8_OK;
    if (!D) return FP8_ERR_INVALID_ARG;
    if (ldD < N) return FP8_ERR_SHAPE;
    const int64_t esz = out_dtype == FP8_OUT_F32 ? 4 : 2;
    if (!aligned16(D) || (ldD * esz) % 16 != 0) return FP8_ERR_ALIGNMENT;
    if (K == 0) {
        FP8FG_STATUS_OR_RETURN(st0);
        return launch_gemm(M, N, K, A, fmtA, sA, granA, B, fmtB, sB, granB, D, out_dtype, ldD, st0, S(stream));
    }
    if (!A || !B || !sA || !sB) return FP8_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(sA) || !aligned16(sB)) return FP8_ERR_ALIGNMENT;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_gemm(M, N, K, A, fmtA, sA, granA, B, fmtB, sB, granB, D, out_dtype, ldD, st, S(stream));
}

static int mx_gemm_checked(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const uint8_t *eA,
                           const void *B, int fmtB, const uint8_t *eB, bool tiled, void *D, int out_dtype,
                           int64_t ldD, void *stream)
{
    if (!fmt_ok(fmtA) || !fmt_ok(fmtB)) return FP8_ERR_INVALID_ARG;
    if (out_dtype != FP8_OUT_BF16 && out_dtype != FP8_OUT_F32) return FP8_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || M % 128 != 0 || N % 128 != 0 || K % 128 != 0) return FP8_ERR_SHAPE;
    if (M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31)) return FP8_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8_OK;
    if (!D) return FP8_ERR_INVALID_ARG;
    if (ldD < N) return FP8_ERR_SHAPE;
    const int64_t esz = out_dtype == FP8_OUT_F32 ? 4 : 2;
    if (!aligned16(D) || (ldD * esz) % 16 != 0) return FP8_ERR_ALIGNMENT;
    if (K > 0) {
        if (!A || !B || !eA || !eB) return FP8_ERR_INVALID_ARG;
        const uintptr_t emask = tiled ? 15u : 3u;   // tiles are fetched by 16-byte bulk copies
        if (!aligned16(A) || !aligned16(B) || (reinterpret_cast<uintptr_t>(eA) & emask) ||
            (reinterpret_cast<uintptr_t>(eB) & emask))
            return FP8_ERR_ALIGNMENT;
    }
    FP8FG_STATUS_OR_RETURN(st);
    return launch_gemm_mx(M, N, K, A, fmtA, eA, B, fmtB, eB, tiled, D, out_dtype, ldD, st, S(stream));
}

FP8FG_API int fp8_mx_gemm(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const uint8_t *eA,
                          const void *B, int fmtB, const uint8_t *eB, void *D, int out_dtype, int64_t ldD,
                          void *stream)
{
    return mx_gemm_checked(M, N, K, A, fmtA, eA, B, fmtB, eB, false, D, out_dtype, ldD, stream);
}

FP8FG_API int fp8_mx_gemm_tiled(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const uint8_t *eA_tiled,
                                const void *B, int fmtB, const uint8_t *eB_tiled, void *D, int out_dtype,
                                int64_t ldD, void *stream)
{
    return mx_gemm_checked(M, N, K, A, fmtA, eA_tiled, B, fmtB, eB_tiled, true, D, out_dtype, ldD, stream);
}

FP8FG_API int fp8_grouped_gemm(int G, const int32_t *group_offsets, int64_t M_capacity, int64_t N, int64_t K,
                               const void *A, const float *sA, const void *B, const float *sB, void *D, int out_dtype,
                               int64_t ldD, void *stream)
{
    if (G < 1 || G > 1024) return FP8_ERR_INVALID_ARG;
    if (out_dtype != FP8_OUT_BF16 && out_dtype != FP8_OUT_F32) return FP8_ERR_INVALID_ARG;
    if (M_capacity < 0 || N < 0 || K < 0 || M_capacity % 128 != 0 || N % 128 != 0 || K % 128 != 0)
        return FP8_ERR_SHAPE;
    if (M_capacity >= ((int64_t)1 << 31) || (int64_t)G * N >= ((int64_t)1 << 31)) return FP8_ERR_SHAPE;
    if (M_capacity == 0 || N == 0 || K == 0) return FP8_OK;
    if (!group_offsets || !A || !sA || !B || !sB || !D) return FP8_ERR_INVALID_ARG;
    if (ldD < N) return FP8_ERR_SHAPE;
    const int64_t esz = out_dtype == FP8_OUT_F32 ? 4 : 2;
    if (!aligned16(A) || !aligned16(B) || !aligned16(sA) || !aligned16(sB) || !aligned16(D) ||
        (ldD * esz) % 16 != 0)
        return FP8_ERR_ALIGNMENT;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_grouped_gemm(G, group_offsets, M_capacity, N, K, A, sA, B, sB, D, out_dtype, ldD, st, S(stream));
}

FP8FG_API int fp8_grouped_gemm_wgrad(int G, const int32_t *group_offsets, int64_t M_capacity, int64_t N, int64_t K,
                                     const void *AT, int fmtA, const float *sAT, const void *BT, int fmtB,
                                     const float *sBT, void *D, int out_dtype, int64_t ldD, void *stream)
{
    if (G < 1 || G > 1024) return FP8_ERR_INVALID_ARG;
    if (!fmt_ok(fmtA) || !fmt_ok(fmtB)) return FP8_ERR_INVALID_ARG;
    if (out_dtype != FP8_OUT_BF16 && out_dtype != FP8_OUT_F32) return FP8_ERR_INVALID_ARG;
    if (M_capacity < 0 || N < 0 || K < 0 || M_capacity % 128 != 0 || N % 128 != 0 || K % 128 != 0)
        return FP8_ERR_SHAPE;
    if (M_capacity >= ((int64_t)1 << 31) || (int64_t)G * N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31))
        return FP8_ERR_SHAPE;
    if (N == 0 || K == 0) return FP8_OK;
    if (!D) return FP8_ERR_INVALID_ARG;
    if (ldD < K) return FP8_ERR_SHAPE;
    const int64_t esz = out_dtype == FP8_OUT_F32 ? 4 : 2;
    if (!aligned16(D) || (ldD * esz) % 16 != 0) return FP8_ERR_ALIGNMENT;
    if (M_capacity > 0) {
        if (!group_offsets || !AT || !sAT || !BT || !sBT) return FP8_ERR_INVALID_ARG;
        if (!aligned16(AT) || !aligned16(BT) || !aligned16(sAT) || !aligned16(sBT)) return FP8_ERR_ALIGNMENT;
    }
    FP8FG_STATUS_OR_RETURN(st);
    return launch_grouped_wgrad(G, group_offsets, M_capacity, N, K, AT, fmtA, sAT, BT, fmtB, sBT, D, out_dtype, ldD,
                                st, S(stream));
}

FP8FG_API int fp8_wgrad_recompute_error(int64_t M, int64_t N, int64_t K, const void *dY, const void *X, const float *D,
                                        int64_t ldD, float *ref_workspace, fp8_wgrad_err_t *err, void *stream)
{
    if (M < 0 || N < 0 || K < 0 || M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31))
        return FP8_ERR_SHAPE;
    if (N % 128 != 0 || K % 128 != 0) return FP8_ERR_SHAPE;
    if (!err) return FP8_ERR_INVALID_ARG;
    if (N > 0 && K > 0) {
        if (ldD < K) return FP8_ERR_SHAPE;
        if (!D || !ref_workspace || (M > 0 && (!dY || !X))) return FP8_ERR_INVALID_ARG;
        if ((M > 0 && (!aligned16(dY) || !aligned16(X))) || !aligned16(D) || ldD % 4 != 0 ||
            !aligned16(ref_workspace) || (reinterpret_cast<uintptr_t>(err) & 7u))
            return FP8_ERR_ALIGNMENT;
    }
    FP8FG_STATUS_OR_RETURN(st);
    return launch_wgrad_recompute_error(M, N, K, dY, X, D, ldD, ref_workspace, err, st, S(stream));
}

FP8FG_API int fp8_adamw_step_fp8_states(float *param, const void *grad, uint8_t *m, float *m_scales, uint8_t *v,
                                        float *v_scales, int64_t n, const fp8_adamw_hparams_t *hparams, void *stream)
{
    if (!hparams) return FP8_ERR_INVALID_ARG;
    if (n < 0 || n % 128 != 0) return FP8_ERR_SHAPE;
    if (n == 0) return FP8_OK;
    if (!param || !grad || !m || !m_scales || !v || !v_scales) return FP8_ERR_INVALID_ARG;
    if (!aligned16(param) || !aligned16(grad) || !aligned16(m) || !aligned16(v)) return FP8_ERR_ALIGNMENT;
    return launch_adamw_fp8(param, grad, m, m_scales, v, v_scales, n, *hparams, S(stream));
}

FP8FG_API int fp8_moe_route_pad(const float *logits, int64_t T, int E, int topk, int align, int64_t M_capacity,
                                int32_t *topk_idx, float *topk_prob, int32_t *counts, int32_t *group_offsets,
                                int32_t *row_token, float *row_prob, uint8_t *row_is_pad, void *stream)
{
    if (E < 1 || E > 256 || topk < 1 || topk > 8 || topk > E || align < 1 || align > 1024) return FP8_ERR_INVALID_ARG;
    if (T < 0 || M_capacity < 0 || T >= ((int64_t)1 << 31) || M_capacity >= ((int64_t)1 << 31)) return FP8_ERR_SHAPE;
    if (!counts || !group_offsets) return FP8_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_idx || !topk_prob)) return FP8_ERR_INVALID_ARG;
    if (M_capacity > 0 && (!row_token || !row_prob)) return FP8_ERR_INVALID_ARG;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_moe_route_pad(logits, T, E, topk, align, M_capacity, topk_idx, topk_prob, counts, group_offsets,
                                row_token, row_prob, row_is_pad, st, S(stream));
}

FP8FG_API int fp8_moe_gather(const void *q, const float *s, int64_t T, int64_t K, const int32_t *row_token,
                             const int32_t *group_offsets, int E, int64_t M_capacity, void *qg, float *sg,
                             void *stream)
{
    if (E < 1 || E > 256) return FP8_ERR_INVALID_ARG;
    if (T < 0 || K < 0 || K % 128 != 0 || M_capacity < 0) return FP8_ERR_SHAPE;
    if (T == 0 || K == 0 || M_capacity == 0) return FP8_OK;
    if (!q || !s || !row_token || !group_offsets || !qg || !sg) return FP8_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(qg)) return FP8_ERR_ALIGNMENT;
    return launch_moe_gather(q, s, T, K, row_token, group_offsets, E, M_capacity, qg, sg, S(stream));
}

FP8FG_API int fp8_swiglu_fwd(const void *gu, int64_t rows, int64_t F, void *h, void *stream)
{
    if (rows < 0 || F < 0 || F % 8 != 0) return FP8_ERR_SHAPE;
    if (rows == 0 || F == 0) return FP8_OK;
    if (!gu || !h) return FP8_ERR_INVALID_ARG;
    if (!aligned16(gu) || !aligned16(h)) return FP8_ERR_ALIGNMENT;
    return launch_swiglu_fwd(gu, rows, F, h, S(stream));
}

FP8FG_API int fp8_swiglu_bwd(const void *gu, const void *dh, int64_t rows, int64_t F, void *dgu, void *stream)
{
    if (rows < 0 || F < 0 || F % 8 != 0) return FP8_ERR_SHAPE;
    if (rows == 0 || F == 0) return FP8_OK;
    if (!gu || !dh || !dgu) return FP8_ERR_INVALID_ARG;
    if (!aligned16(gu) || !aligned16(dh) || !aligned16(dgu)) return FP8_ERR_ALIGNMENT;
    return launch_swiglu_bwd(gu, dh, rows, F, dgu, S(stream));
}

static int swiglu_quant_checks(const void *gu, const void *dh, bool bwd, int64_t rows, int64_t F, int fmt,
                               const void *q, const float *s, const void *qT, const float *sT)
{
    if (!fmt_ok(fmt)) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || F < 0 || rows % 128 != 0 || F % 128 != 0) return FP8_ERR_SHAPE;
    const int64_t cols = bwd ? 2 * F : F;
    if (rows * (cols / 128) >= (int64_t)1 << 31) return FP8_ERR_SHAPE;
    if (rows == 0 || F == 0) return FP8_OK;
    if (!gu || (bwd && !dh) || !q || !s || !qT || !sT) return FP8_ERR_INVALID_ARG;
    if (!aligned16(gu) || (bwd && !aligned16(dh)) || !aligned16(q) || !aligned16(s) || !aligned16(qT) ||
        !aligned16(sT))
        return FP8_ERR_ALIGNMENT;
    return FP8_OK;
}

FP8FG_API int fp8_swiglu_quant_fwd(const void *gu, int64_t rows, int64_t F, int fmt, void *q, float *s, void *qT,
                                   float *sT, void *stream)
{
    const int rc = swiglu_quant_checks(gu, nullptr, false, rows, F, fmt, q, s, qT, sT);
    if (rc != FP8_OK || rows == 0 || F == 0) return rc;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_swiglu_quant(gu, nullptr, rows, F, fmt, q, s, qT, sT, st, S(stream));
}

FP8FG_API int fp8_swiglu_bwd_quant(const void *gu, const void *dh, int64_t rows, int64_t F, int fmt, void *q,
                                   float *s, void *qT, float *sT, void *stream)
{
    const int rc = swiglu_quant_checks(gu, dh, true, rows, F, fmt, q, s, qT, sT);
    if (rc != FP8_OK || rows == 0 || F == 0) return rc;
    FP8FG_STATUS_OR_RETURN(st);
    return launch_swiglu_quant(gu, dh, rows, F, fmt, q, s, qT, sT, st, S(stream));
}

}  // extern "C"
