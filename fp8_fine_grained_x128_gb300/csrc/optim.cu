// optim.cu -- AdamW step with the moments kept in FP8 (sm_103a).
//
// Ling 2.0 FP8 pretraining blog, "FP8 Optimizer": Adam's first and second
// moments are stored in FP8 with fine-grained compression / decompression,
// which saves 75% of the optimizer-state memory; "FP8-LM" review, "Level 2:
// FP8 optimizer": momentum and variance in FP8.  Here m is E4M3 and v is E5M2
// (v holds squared gradients, the widest-ranged quantity), each with one
// binary32 scale per 128 consecutive parameters, s = amax / fmax.  The update
// is Adam (Kingma and Ba) with AdamW's decoupled weight decay (Loshchilov and
// Hutter), every operation a correctly rounded binary32 one in a fixed order:
//   m = dec(qm) * sm;  m = b1 * m + omb1 * g
//   v = dec(qv) * sv;  v = b2 * v + omb2 * (g * g)
//   u = (m / bc1) / (sqrt(v / bc2) + eps);  p = p - lr * (u + wd * p)
// then the new m and v are re-quantized with their blocks' new scales.  One
// pass over HBM: the parameters (read + write), the BF16 gradient and both
// code arrays.
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

// The 4 FP8 codes of w as binary32 (exact: FP8 values are binary16 values).
template <int FMT>
__device__ __forceinline__ void fp8x4_to_f32(uint32_t w, float (&f)[4])
{
    uint32_t h01, h23;
    const uint16_t lo = (uint16_t)(w & 0xFFFFu), hi = (uint16_t)(w >> 16);
    if (FMT == FP8_E4M3) {
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(lo));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(hi));
    } else {
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h01) : "h"(lo));
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h23) : "h"(hi));
    }
    f[0] = __half2float(__ushort_as_half((unsigned short)(h01 & 0xFFFFu)));
    f[1] = __half2float(__ushort_as_half((unsigned short)(h01 >> 16)));
    f[2] = __half2float(__ushort_as_half((unsigned short)(h23 & 0xFFFFu)));
    f[3] = __half2float(__ushort_as_half((unsigned short)(h23 >> 16)));
}

// Codes of 4 binary32 values with the block scale s (q = enc(x / s)).  The
// scale comes from the block's own amax, so no |x / s| exceeds fmax by more
// than a rounding and no quotient overflows; inside the fast range of s the
// packed Markstein quotients are the correctly rounded ones wherever they can
// decide a code, and they carry the sign of x even when zero.  A scale outside
// that range (an all-tiny block: one per warp, so the branch is uniform) takes
// the IEEE division.
template <int FMT>
__device__ __forceinline__ uint32_t f32x4_to_fp8(const float (&x)[4], const Divider2 &d)
{
    if (d.fast) {
        float q[4];
        d.fast_div_f32(x[0], x[1], q[0], q[1]);
        d.fast_div_f32(x[2], x[3], q[2], q[3]);
        return cvt2<FMT>(q[0], q[1]) | (cvt2<FMT>(q[2], q[3]) << 16);
    }
    return cvt2<FMT>(__fdiv_rn(x[0], d.s), __fdiv_rn(x[1], d.s)) |
           (cvt2<FMT>(__fdiv_rn(x[2], d.s), __fdiv_rn(x[3], d.s)) << 16);
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// What a lane reads of one 128-parameter block.
struct AdamBlockIn {
    float4 p4;
    uint2 g4;
    uint32_t cm, cv;
    float s_m, s_v;
};

__device__ __forceinline__ void load_block(AdamBlockIn &in, const float *p, const uint16_t *g, const uint8_t *qm,
                                           const float *sm, const uint8_t *qv, const float *sv, int64_t b, int lane)
{
    const int64_t k = b * 128 + lane * 4;
    in.p4 = __ldcs(reinterpret_cast<const float4 *>(p + k));
    in.g4 = __ldcs(reinterpret_cast<const uint2 *>(g + k));
    in.cm = *reinterpret_cast<const uint32_t *>(qm + k);
    in.cv = *reinterpret_cast<const uint32_t *>(qv + k);
    in.s_m = sm[b];
    in.s_v = sv[b];
}

// One warp per block of 128 parameters, 4 consecutive parameters per lane;
// the warp's next block is read while the current one is computed.
__global__ void __launch_bounds__(256) k_adamw_fp8(float *__restrict__ p, const uint16_t *__restrict__ g,
                                                   uint8_t *__restrict__ qm, float *__restrict__ sm,
                                                   uint8_t *__restrict__ qv, float *__restrict__ sv, int64_t nblk,
                                                   fp8_adamw_hparams_t h, int *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    AdamBlockIn cur;
    if (w0 < nblk) load_block(cur, p, g, qm, sm, qv, sv, w0, lane);
    for (int64_t b = w0; b < nblk; b += nw) {
        AdamBlockIn nxt;
        if (b + nw < nblk) load_block(nxt, p, g, qm, sm, qv, sv, b + nw, lane);
        const int64_t k = b * 128 + lane * 4;
        const float4 p4 = cur.p4;
        const uint2 g4 = cur.g4;
        const uint32_t cm = cur.cm, cv = cur.cv;
        const float s_m = cur.s_m, s_v = cur.s_v;
        float pp[4] = {p4.x, p4.y, p4.z, p4.w};
        const float gg[4] = {bf16_lo(g4.x), bf16_hi(g4.x), bf16_lo(g4.y), bf16_hi(g4.y)};
        float m[4], v[4];
        fp8x4_to_f32<FP8_E4M3>(cm, m);
        fp8x4_to_f32<FP8_E5M2>(cv, v);
        float am = 0.0f, av = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            m[e] = __fmul_rn(m[e], s_m);
            v[e] = __fmul_rn(v[e], s_v);
            m[e] = __fadd_rn(__fmul_rn(h.beta1, m[e]), __fmul_rn(h.one_minus_beta1, gg[e]));
            v[e] = __fadd_rn(__fmul_rn(h.beta2, v[e]), __fmul_rn(h.one_minus_beta2, __fmul_rn(gg[e], gg[e])));
            const float mh = __fdiv_rn(m[e], h.bias_correction1);
            const float vh = __fdiv_rn(v[e], h.bias_correction2);
            const float u = __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), h.eps));
            const float t = __fmul_rn(h.lr, __fadd_rn(u, __fmul_rn(h.weight_decay, pp[e])));
            pp[e] = __fsub_rn(pp[e], t);
            am = fmaxf(am, fabsf(m[e]));
            av = fmaxf(av, fabsf(v[e]));
        }
        am = warp_max(am);
        av = warp_max(av);
        const float nsm = am == 0.0f ? 1.0f : __fdiv_rn(am, 448.0f);
        const float nsv = av == 0.0f ? 1.0f : __fdiv_rn(av, 57344.0f);
        if (dbg_span(k, 4, nblk * 128, status)) {
            __stcs(reinterpret_cast<float4 *>(p + k), make_float4(pp[0], pp[1], pp[2], pp[3]));
            *reinterpret_cast<uint32_t *>(qm + k) = f32x4_to_fp8<FP8_E4M3>(m, Divider2(nsm));
            *reinterpret_cast<uint32_t *>(qv + k) = f32x4_to_fp8<FP8_E5M2>(v, Divider2(nsv));
        }
        if (lane == 0 && dbg_span(b, 1, nblk, status)) {
            sm[b] = nsm;
            sv[b] = nsv;
        }
        cur = nxt;
    }
}

int launch_adamw_fp8(float *p, const void *g, uint8_t *qm, float *sm, uint8_t *qv, float *sv, int64_t n,
                     const fp8_adamw_hparams_t &h, cudaStream_t st)
{
    const int64_t nblk = n / 128;
    if (nblk == 0) return FP8_OK;
    // one wave of resident blocks, each warp striding over the 128-blocks
    static int per_sm[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (per_sm[dev & 63] == 0 &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[dev & 63], k_adamw_fp8, 256, 0) != cudaSuccess)
        return FP8_ERR_CUDA;
    int64_t blocks = (nblk + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * std::max(1, per_sm[dev & 63]);
    if (blocks > cap) blocks = cap;
    k_adamw_fp8<<<(unsigned)blocks, 256, 0, st>>>(p, static_cast<const uint16_t *>(g), qm, sm, qv, sv, nblk, h,
                                              status_word_ptr());
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8fg
