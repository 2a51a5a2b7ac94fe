// mx.cu -- MXFP8 (micro-scaled FP8) quantizer: 1x32 blocks with power-of-two
// scales (sm_103a).
//
// "FP8 training infrastructure" guide: Blackwell adds MXFP8, micro-scaled FP8
// ("Hardware requirements for FP8 training"); every block inside a tensor gets
// its own scale factor ("Scaling strategies and stability"); block scaling in
// hardware replaces per-tensor scaling ("Blackwell MXFP8 and NVFP4: looking
// ahead").  The pages give neither the block size nor the scale encoding; this
// library reads them as: a block is 32 consecutive elements of a row, and its
// scale is a power of two X = 2^(e8 - 127), stored as an 8-bit exponent code,
// the smallest with amax / X <= fmax (the amax / fmax scale rounded up to a
// power of two, so no element saturates); an all-zero block gets X = 1.  The
// codes are RNE_satfinite(x / X), and x / X = x * 2^-e is an exact product.
//
// The scale codes go out either row-major [rows][cols/32] or in the layout the
// MXFP8 GEMM copies straight into tensor memory ("tiled"): for rows and cols
// multiples of 128, the codes of rows 128 rb .. 128 rb + 127 and 32-blocks
// 4 kc .. 4 kc + 3 form a 512-byte tile at (kc * rows/128 + rb) * 512, row r
// at byte 16 (r % 32) + 4 ((r % 128) / 32) + (block % 4) inside it.
//
// A streaming kernel (HBM-bound: 2 B read, 1 + 1/32 B written per element):
// every lane loads 16 bytes (8 BF16), four consecutive lanes hold one block
// and reduce its amax with two shuffles, and the exponent is read off the
// amax's BF16 bits -- no division, no transcendental.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

// Smallest e with fmax * 2^e >= a, for a = |amax| as BF16 bits (finite, > 0),
// clamped to the exponent code's range [-127, 127].  fmax = 1.75 * 2^kEmax, so
// with a = m * 2^p (m in [1, 2)): e = p - kEmax if m <= 1.75, else one more.
template <int FMT>
__device__ __forceinline__ int mx_exponent(uint32_t a)
{
    constexpr int kEmax = FMT == FP8_E4M3 ? 8 : 15;
    int p;
    uint32_t frac;   // the 7 fraction bits of m; 1.75 has 0x60
    const uint32_t ex = a >> 7, man = a & 0x7Fu;
    if (ex != 0) {
        p = (int)ex - 127;
        frac = man;
    } else {   // subnormal BF16: man * 2^-133, man in 1..127
        const int msb = 31 - __clz(man);
        p = msb - 133;
        frac = (man << (7 - msb)) & 0x7Fu;
    }
    const int e = p - kEmax + (frac > 0x60u ? 1 : 0);
    return max(-127, min(127, e));
}

// 8 BF16 values times 2^-e (exact) -> 8 FP8 codes.
template <int FMT>
__device__ __forceinline__ uint2 mx_codes8(uint4 v, float inv)
{
    uint2 o;
    o.x = cvt2<FMT>(bf16_lo(v.x) * inv, bf16_hi(v.x) * inv) | (cvt2<FMT>(bf16_lo(v.y) * inv, bf16_hi(v.y) * inv) << 16);
    o.y = cvt2<FMT>(bf16_lo(v.z) * inv, bf16_hi(v.z) * inv) | (cvt2<FMT>(bf16_lo(v.w) * inv, bf16_hi(v.w) * inv) << 16);
    return o;
}

// Each warp takes 128 consecutive 16-byte vectors per iteration (four per
// lane, loaded before any is used).  A row holds cols / 8 vectors, a multiple
// of 4, so the four lanes of a quad always share one block; all 32 lanes run
// every iteration (lanes past the end carry zeros) so the shuffles are full.
template <int FMT, bool TILED>
__global__ void __launch_bounds__(256) k_quant_mx(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                  int64_t ldx, uint8_t *__restrict__ q, uint8_t *__restrict__ e8,
                                                  int *status)
{
    constexpr int U = 4;
    const int lane = threadIdx.x & 31;
    const int64_t vpr = cols / 8, nvec = rows * vpr;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const bool flat = ldx == cols;
    for (int64_t base = w0 * (32 * U); base < nvec; base += nw * (32 * U)) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + u * 32 + lane;
            v[u] = make_uint4(0, 0, 0, 0);
            if (i < nvec) {
                const int64_t r = flat ? 0 : i / vpr;
                v[u] = ldg_stream(flat ? x + i * 8 : x + r * ldx + (i - r * vpr) * 8);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + u * 32 + lane;
            uint32_t a = absmax8(v[u]);
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
            if (i >= nvec) continue;
            if (a >= 0x7F80u && (lane & 3) == 0) set_status(status, FP8_ERR_NONFINITE);
            const int e = a == 0 ? 0 : mx_exponent<FMT>(min(a, 0x7F7Fu));
            const float inv = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e, e in [-127, 120]
            const uint2 codes = mx_codes8<FMT>(v[u], inv);
            if (dbg_span(i * 8, 8, rows * cols, status)) *reinterpret_cast<uint2 *>(q + i * 8) = codes;
            if ((lane & 3) == 0) {
                int64_t off = i >> 2;   // block index, row-major
                if (TILED) {
                    const int64_t kb = cols / 32, r = off / kb, k = off - r * kb;
                    off = ((k >> 2) * (rows >> 7) + (r >> 7)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (k & 3);
                }
                if (dbg_span(off, 1, rows * (cols / 32), status)) e8[off] = (uint8_t)(e + 127);
            }
        }
    }
}

int launch_quant_mx(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, void *q, uint8_t *e8,
                    bool tiled, int *status, cudaStream_t st)
{
    const int64_t nvec = rows * (cols / 8);
    if (nvec == 0) return FP8_OK;
    const int64_t per_block = 256 * 4;
    const unsigned grid =
        (unsigned)std::max<int64_t>(1, std::min<int64_t>((nvec + per_block - 1) / per_block, (int64_t)sm_count() * 4));
    auto X = static_cast<const uint16_t *>(x);
    auto Q = static_cast<uint8_t *>(q);
    if (fmt == FP8_E5M2) {
        if (tiled) k_quant_mx<FP8_E5M2, true><<<grid, 256, 0, st>>>(X, rows, cols, ldx, Q, e8, status);
        else k_quant_mx<FP8_E5M2, false><<<grid, 256, 0, st>>>(X, rows, cols, ldx, Q, e8, status);
    } else {
        if (tiled) k_quant_mx<FP8_E4M3, true><<<grid, 256, 0, st>>>(X, rows, cols, ldx, Q, e8, status);
        else k_quant_mx<FP8_E4M3, false><<<grid, 256, 0, st>>>(X, rows, cols, ldx, Q, e8, status);
    }
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8fg
