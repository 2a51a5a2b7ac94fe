// monitor_dw.cu -- high-precision dw recompute monitor (sm_103a).
//
// Ling 2.0 FP8 pretraining blog, "Where does the error come from?": the
// tensors that the underflow / distortion monitors flag get their dw
// recomputed in high precision and compared with the FP8 one.  The reference
// wgrad R = dY^T . X of the BF16 operands is a plain BF16 GEMM with FP32
// accumulation, left to cuBLAS (loaded at run time, so the library itself
// does not depend on it); the comparison is this file's kernel, which
// reduces {sum (D - R)^2, sum R^2} in FP64 and {max |D - R|, max |R|}.
#include <dlfcn.h>

#include <mutex>

#include <cublas_v2.h>   // types and prototypes only; the symbols are looked up at run time

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

namespace {

// the exported C entry point (the C++ header also declares an overload)
typedef cublasStatus_t (*GemmExFn)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void *,
                                   const void *, cudaDataType, int, const void *, cudaDataType, int, const void *,
                                   void *, cudaDataType, int, cublasComputeType_t, cublasGemmAlgo_t);

struct CublasApi {
    decltype(&cublasCreate_v2) create = nullptr;
    decltype(&cublasSetStream_v2) set_stream = nullptr;
    GemmExFn gemm = nullptr;
    bool ok = false;
};

const CublasApi &cublas_api()
{
    static CublasApi api;
    static std::once_flag once;
    std::call_once(once, [] {
        void *h = dlopen("libcublas.so.13", RTLD_NOW | RTLD_GLOBAL);
        if (!h) h = dlopen("/usr/local/cuda/lib64/libcublas.so.13", RTLD_NOW | RTLD_GLOBAL);
        if (!h) return;
        api.create = reinterpret_cast<decltype(api.create)>(dlsym(h, "cublasCreate_v2"));
        api.set_stream = reinterpret_cast<decltype(api.set_stream)>(dlsym(h, "cublasSetStream_v2"));
        api.gemm = reinterpret_cast<decltype(api.gemm)>(dlsym(h, "cublasGemmEx"));
        api.ok = api.create && api.set_stream && api.gemm;
    });
    return api;
}

// One handle per device, created with that device current.
cublasHandle_t cublas_handle()
{
    static std::mutex mu;
    static cublasHandle_t handles[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!handles[dev] && cublas_api().create(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
    return handles[dev];
}

}  // namespace

// Row n of D against row n of R, threads across the columns.
__global__ void __launch_bounds__(256) k_wgrad_err(const float *__restrict__ D, int64_t ldD, const float *__restrict__ R,
                                                   int64_t N, int64_t K, fp8_wgrad_err_t *err)
{
    __shared__ double sd[8], sr[8];
    __shared__ float md[8], mr[8];
    double sdd = 0.0, srr = 0.0;
    float mdd = 0.0f, mrr = 0.0f;
    for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
        for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
            const double r = R[n * K + k];
            const double d = (double)D[n * ldD + k] - r;
            sdd += d * d;
            srr += r * r;
            mdd = fmaxf(mdd, (float)fabs(d));
            mrr = fmaxf(mrr, (float)fabs(r));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sdd += __shfl_xor_sync(0xffffffffu, sdd, o);
        srr += __shfl_xor_sync(0xffffffffu, srr, o);
        mdd = fmaxf(mdd, __shfl_xor_sync(0xffffffffu, mdd, o));
        mrr = fmaxf(mrr, __shfl_xor_sync(0xffffffffu, mrr, o));
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        sd[w] = sdd;
        sr[w] = srr;
        md[w] = mdd;
        mr[w] = mrr;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < (int)(blockDim.x >> 5); ++i) {
            sdd += sd[i];
            srr += sr[i];
            mdd = fmaxf(mdd, md[i]);
            mrr = fmaxf(mrr, mr[i]);
        }
        atomicAdd(&err->sum_sq_diff, sdd);
        atomicAdd(&err->sum_sq_ref, srr);
        // non-negative floats order like their bit patterns
        atomicMax(reinterpret_cast<unsigned int *>(&err->max_abs_diff), __float_as_uint(mdd));
        atomicMax(reinterpret_cast<unsigned int *>(&err->max_abs_ref), __float_as_uint(mrr));
    }
}

int launch_wgrad_recompute_error(int64_t M, int64_t N, int64_t K, const void *dY, const void *X, const float *D,
                                 int64_t ldD, float *R, fp8_wgrad_err_t *err, cudaStream_t st)
{
    if (cudaMemsetAsync(err, 0, sizeof(fp8_wgrad_err_t), st) != cudaSuccess) return FP8_ERR_CUDA;
    if (N == 0 || K == 0) return FP8_OK;
    if (M == 0) {
        if (cudaMemsetAsync(R, 0, (size_t)N * K * sizeof(float), st) != cudaSuccess) return FP8_ERR_CUDA;
    } else {
        if (!cublas_api().ok) return FP8_ERR_UNSUPPORTED;
        cublasHandle_t h = cublas_handle();
        if (!h || cublas_api().set_stream(h, st) != CUBLAS_STATUS_SUCCESS) return FP8_ERR_CUDA;
        // column-major view: R^T [K x N] = X^T [K x M] . dY [M x N]
        const float one = 1.0f, zero = 0.0f;
        if (cublas_api().gemm(h, CUBLAS_OP_N, CUBLAS_OP_T, (int)K, (int)N, (int)M, &one, X, CUDA_R_16BF, (int)K, dY,
                              CUDA_R_16BF, (int)N, &zero, R, CUDA_R_32F, (int)K, CUBLAS_COMPUTE_32F,
                              CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
            return FP8_ERR_CUDA;
    }
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)sm_count() * 8));
    k_wgrad_err<<<blocks, 256, 0, st>>>(D, ldD, R, N, K, err);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8fg
