// monitor_dw.cu -- high-precision dw recompute monitor (sm_103a).
//
// Ling 2.0 FP8 pretraining blog, "Where does the error come from?": the
// tensors that the underflow / distortion monitors flag get their dw
// recomputed in high precision and compared with the FP8 one.  The reference
// wgrad R = dY^T . X is a plain BF16 GEMM with FP32 accumulation over the
// tokens, run here on the tensor cores (tcgen05.mma kind::f16) straight from
// the token-major BF16 operands: dY [M][N] and X [M][K] are row-major with
// the contraction (token) index as the row, so both enter the MMA MN-major --
// TMA copies 64-token x 64-column boxes, whose 128-byte rows are 64
// consecutive output rows (dY) or columns (X).  The epilogue writes R and,
// from the same registers, reduces the comparison with the FP8 wgrad D:
// {sum (D - R)^2, sum R^2} (D - R in FP32, the squares and sums in FP64) and
// {max |D - R|, max |R|}; it overlaps the next tile's MMAs, so the slow FP64
// rate of this part stays hidden for token counts in the thousands.
//
// Structure (one persistent CTA per SM, 6 warps): warp 0 TMA producer
// (4 stages of 64 tokens), warp 1 owns the tensor memory (two accumulators of
// BN columns alternating per output tile) and issues 4 MMAs (K = 16) per
// stage from one thread, warps 2..5 drain the accumulator (one TMEM lane
// quarter each).  Every mbarrier wait is bounded as in the FP8 GEMM.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8fg {

constexpr int kDwThreads = 192;
constexpr int kDwBK = 64;             // tokens per stage
constexpr int kDwStages = 4;
constexpr int kDwEpiWarp0 = 2;

template <int BN>
struct DwSmem {
    static constexpr int kA = 128 * kDwBK * 2;   // two boxes of 64 rows of R x 64 tokens
    static constexpr int kB = BN * kDwBK * 2;    // BN / 64 boxes of 64 columns of R x 64 tokens
    static constexpr int kStage = kA + kB;
    static constexpr int kBars = 2 * kDwStages + 2 * 2 + 1;
    static constexpr int kBytes = 1024 + kDwStages * kStage + kBars * 8 + 16;
    static constexpr int kTmemCols = 2 * BN;
};

struct DwArgs {
    int N, K, M;            // R is [N][K]; M tokens are contracted
    float *R;
    const float *D;
    int64_t ldD;
    fp8_wgrad_err_t *err;
    int *status;
    int raster_gm;
};

template <int BN>
__global__ void __launch_bounds__(kDwThreads, 1)
    k_dw_reference(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, DwArgs a)
{
    using L = DwSmem<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kDwStages * L::kStage);
    uint64_t *empty = full + kDwStages;
    uint64_t *tfull = empty + kDwStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDwStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_mt = a.N / 128, num_nt = a.K / BN;
    const int ntiles = num_mt * num_nt;
    const int nkb = (a.M + kDwBK - 1) / kDwBK;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            int mt, nt;
            tile_coords_raster(tile, num_mt, num_nt, a.raster_gm, mt, nt);
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = it % kDwStages;
                if (!wait_or_abort(&empty[s], ((it / kDwStages) & 1) ^ 1, abort_flag, a.status)) { ok = false; break; }
                uint8_t *st = smem + s * L::kStage;
                // tokens past M read as zeros and still count their bytes
                mbar_arrive_expect_tx(&full[s], L::kStage);
#pragma unroll
                for (int j = 0; j < 2; ++j) tma_load_2d(st + j * 8192, &tmA, &full[s], mt * 128 + 64 * j, kb * kDwBK);
#pragma unroll
                for (int j = 0; j < BN / 64; ++j)
                    tma_load_2d(st + L::kA + j * 8192, &tmB, &full[s], nt * BN + 64 * j, kb * kDwBK);
                ++it;
            }
        }
        const uint32_t first = it > (uint32_t)kDwStages ? it - kDwStages : 0;
        for (uint32_t j = first; j < it; ++j) mbar_wait_bounded(&full[j % kDwStages], (j / kDwStages) & 1, nullptr);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16_mnmajor(128, BN);
        uint32_t it = 0, tc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++tc) {
            const uint32_t buf = tc & 1;
            if (!wait_or_abort(&tempty[buf], ((tc >> 1) & 1) ^ 1, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + buf * BN;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = it % kDwStages;
                if (!wait_or_abort(&full[s], (it / kDwStages) & 1, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * L::kStage), sb = sa + L::kA;
#pragma unroll
                for (int k = 0; k < kDwBK / 16; ++k) {
                    // 16 tokens = two 1024-byte swizzle atoms further along K
                    const uint64_t ad = sdesc_mnmajor_sw128(sa + k * 2048, 8192, 1024);
                    const uint64_t bd = sdesc_mnmajor_sw128(sb + k * 2048, 8192, 1024);
                    tc_mma_f16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                }
                tc_commit(&empty[s]);
                ++it;
            }
            if (!ok) break;
            tc_commit(&tfull[buf]);
        }
        tc_commit(mma_done);
        mbar_wait_bounded(mma_done, 0, nullptr);
    } else if (warp >= kDwEpiWarp0) {
        // ------------------------------------------------------ epilogue
        const int lq = warp & 3;                 // TMEM lane quarter of this warp
        const uint32_t tm_lane = tmem_base + ((uint32_t)(lq * 32) << 16);
        double sdd = 0.0, srr = 0.0;
        float mdd = 0.0f, mrr = 0.0f;
        uint32_t tc = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tc) {
            int mt, nt;
            tile_coords_raster(tile, num_mt, num_nt, a.raster_gm, mt, nt);
            const uint32_t buf = tc & 1;
            if (!warp_wait_or_abort(&tfull[buf], (tc >> 1) & 1, abort_flag, a.status)) break;
            tc_fence_after();
            const int64_t row = (int64_t)mt * 128 + lq * 32 + lane;
#pragma unroll 1
            for (int j = 0; j < BN / 32; ++j) {
                uint32_t r[32];
                tc_ld_32x32b_x32(tm_lane + buf * BN + j * 32, r);
                tc_wait_ld();
                const int64_t col = (int64_t)nt * BN + j * 32;
                float *Rp = a.R + row * a.K + col;
                const float *Dp = a.D + row * a.ldD + col;
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 rv = make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]),
                                                  __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
                    const float4 dv = *reinterpret_cast<const float4 *>(Dp + c);   // read before R is written
                    if (dbg_cell(row, col + c, 4, a.N, a.K, a.status)) *reinterpret_cast<float4 *>(Rp + c) = rv;
                    const float dd[4] = {dv.x - rv.x, dv.y - rv.y, dv.z - rv.z, dv.w - rv.w};
                    const float rr[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // squares of binary32 values are exact in FP64
                        sdd = fma((double)dd[e], (double)dd[e], sdd);
                        srr = fma((double)rr[e], (double)rr[e], srr);
                        mdd = fmaxf(mdd, fabsf(dd[e]));
                        mrr = fmaxf(mrr, fabsf(rr[e]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sdd += __shfl_xor_sync(0xffffffffu, sdd, o);
            srr += __shfl_xor_sync(0xffffffffu, srr, o);
            mdd = fmaxf(mdd, __shfl_xor_sync(0xffffffffu, mdd, o));
            mrr = fmaxf(mrr, __shfl_xor_sync(0xffffffffu, mrr, o));
        }
        if (lane == 0 && !*abort_flag) {
            atomicAdd(&a.err->sum_sq_diff, sdd);
            atomicAdd(&a.err->sum_sq_ref, srr);
            // non-negative floats order like their bit patterns
            atomicMax(reinterpret_cast<unsigned int *>(&a.err->max_abs_diff), __float_as_uint(mdd));
            atomicMax(reinterpret_cast<unsigned int *>(&a.err->max_abs_ref), __float_as_uint(mrr));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

// Row n of D against row n of R (R all zero when there are no tokens), threads
// across the columns.
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
        atomicMax(reinterpret_cast<unsigned int *>(&err->max_abs_diff), __float_as_uint(mdd));
        atomicMax(reinterpret_cast<unsigned int *>(&err->max_abs_ref), __float_as_uint(mrr));
    }
}

template <int BN>
static int run_dw(const CUtensorMap &mA, const CUtensorMap &mB, const DwArgs &args, int grid, cudaStream_t st)
{
    using L = DwSmem<BN>;
    static_assert(L::kBytes <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done[dev & 63]) {
        if (cudaFuncSetAttribute(k_dw_reference<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) !=
            cudaSuccess)
            return FP8_ERR_CUDA;
        attr_done[dev & 63] = true;
    }
    k_dw_reference<BN><<<grid, kDwThreads, L::kBytes, st>>>(mA, mB, args);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

int launch_wgrad_recompute_error(int64_t M, int64_t N, int64_t K, const void *dY, const void *X, const float *D,
                                 int64_t ldD, float *R, fp8_wgrad_err_t *err, int *status, cudaStream_t st)
{
    if (cudaMemsetAsync(err, 0, sizeof(fp8_wgrad_err_t), st) != cudaSuccess) return FP8_ERR_CUDA;
    if (N == 0 || K == 0) return FP8_OK;
    if (M == 0) {   // no tokens: R = 0
        if (cudaMemsetAsync(R, 0, (size_t)N * K * sizeof(float), st) != cudaSuccess) return FP8_ERR_CUDA;
        const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)sm_count() * 8));
        k_wgrad_err<<<blocks, 256, 0, st>>>(D, ldD, R, N, K, err);
        return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
    }
    const int BN = (K % 256 == 0) ? 256 : 128;
    CUtensorMap mA, mB;
    // dY [M][N] and X [M][K] row-major BF16: boxes of 64 columns (128 bytes) x 64 tokens
    if (!make_map_2d(&mA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2, 64, kDwBK,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
        !make_map_2d(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64, kDwBK,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
        return FP8_ERR_CUDA;
    DwArgs g{};
    g.N = (int)N;
    g.K = (int)K;
    g.M = (int)M;
    g.R = R;
    g.D = D;
    g.ldD = ldD;
    g.err = err;
    g.status = status;
    g.raster_gm = raster_band(N, N * M * 2, K * M * 2);
    const int64_t ntiles = (N / 128) * (K / BN);
    const int grid = (int)std::min<int64_t>(ntiles, sm_count());
    if (BN == 256) return run_dw<256>(mA, mB, g, grid, st);
    return run_dw<128>(mA, mB, g, grid, st);
}

}  // namespace fp8fg
