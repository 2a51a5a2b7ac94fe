// noalloc.cu -- a variant of the per-tensor delayed-scaling quantizer for
// callers that cannot allocate device memory.
//
// fp8_quant_pertensor_delayed needs a small scratch workspace (the cross-CTA
// amax, the presence bitmaps of the distortion monitor and the last-CTA
// ticket) that the caller normally allocates.  Some callers cannot call
// cudaMalloc at all: code running under another framework's fixed memory
// plan or arena, plugins and hooks that are handed buffers but no allocator,
// or real-time loops where an allocation could block or fail.  This entry
// point keeps that scratch in a file-scope device array instead, so the
// caller passes only its tensors and its delayed-scaling state.
//
// Trade-offs: the array is part of the library image (every GPU that loads
// the library holds it until the process exits), and all calls share it, so
// two calls that overlap on the GPU (different streams, no ordering between
// them) race on it.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

// Scratch for the no-allocation entry point: 16 KiB per GPU.  The delayed-
// scaling kernel needs pertensor_workspace_bytes() of it, whatever the size
// of the tensor.
constexpr size_t kNoAllocScratchBytes = 16384;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[64] = {};

// Device address of this device's scratch array.  In host code the array's
// name only stands for the symbol; the address a kernel may use must be
// looked up with the device current, once per device.
static int noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FP8_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FP8_OK;
}

}  // namespace fp8fg

using namespace fp8fg;

extern "C" FP8FG_API int fp8_quant_pertensor_delayed_noalloc(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                                             const fp8_delayed_recipe_t *recipe, float *amax_history,
                                                             int32_t *step, float *scale, void *q, void *qT,
                                                             fp8_stats_t *stats, void *stream)
{
    const size_t need = pertensor_workspace_bytes();
    if (need > kNoAllocScratchBytes) return FP8_ERR_UNSUPPORTED;   // scratch block too small for this kernel
    // the argument contract of fp8_quant_pertensor_delayed (the same check), minus the workspace
    const int arg_rc = check_pertensor_delayed_args(x, rows, cols, ldx, recipe, amax_history, step, scale, q, qT,
                                                    stats, nullptr, false);
    if (arg_rc != FP8_OK) return arg_rc;

    void *ws = nullptr;
    const int rc = noalloc_scratch(&ws);
    if (rc != FP8_OK) return rc;
    int *status_word = status_word_ptr();   // where kernels record device-side errors
    if (!status_word) return FP8_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the array keeps whatever the previous call left: start from zero
    if (cudaMemsetAsync(ws, 0, need, st) != cudaSuccess) return FP8_ERR_CUDA;
    return launch_pertensor_delayed(x, rows, cols, ldx, recipe->fmt, recipe->history_len, recipe->margin,
                                    recipe->algo, amax_history, step, scale, q, qT, stats, ws, status_word, st);
}
