// common.cuh -- device helpers shared by the sm_103a kernels of the fine-grained
// FP8 Linear library: FP8 conversion, the per-element IEEE division x / s,
// BF16 unpacking, the device status word, and the inline-PTX wrappers for
// mbarriers, TMA and the tcgen05 tensor-core / tensor-memory instructions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8fg.h"

#ifndef __CUDA_ARCH__
#define FP8FG_HOST_ONLY 1
#endif

namespace fp8fg {

// Largest finite magnitude of the two formats ([FP8-LM] "FP8 data formats";
// E4M3 spans [-448, 448] per the FP8-RL article).
__host__ __device__ constexpr float fmax_of(int fmt) { return fmt == FP8_E5M2 ? 57344.0f : 448.0f; }

// Default bound for every spin-wait on the device (nanoseconds).
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;

// ------------------------------------------------------------------ status

// Records the first error seen by any thread in the device status word.
__device__ __forceinline__ void set_status(int *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------- debug build
// In the debug build (compiled with FP8FG_DEBUG) every global store of the
// kernels first checks its index against the extent of the buffer it writes,
// so a write outside an output -- what a memory checker would report -- is
// caught where it would happen: the check records FP8_ERR_BOUNDS in the
// status word and the store is skipped.  In the release build the checks are
// constant true and compile away.
#ifdef FP8FG_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// Elements [i, i + n) lie inside a buffer of `extent` elements.
__device__ __forceinline__ bool dbg_span(int64_t i, int64_t n, int64_t extent, int *status)
{
    if (!kDebugChecks) return true;
    const bool ok = i >= 0 && n >= 0 && i + n <= extent;
    if (!ok) set_status(status, FP8_ERR_BOUNDS);
    return ok;
}

// Row r and columns [c, c + n) lie inside a [rows][cols] matrix.
__device__ __forceinline__ bool dbg_cell(int64_t r, int64_t c, int64_t n, int64_t rows, int64_t cols, int *status)
{
    if (!kDebugChecks) return true;
    const bool ok = r >= 0 && r < rows && c >= 0 && n >= 0 && c + n <= cols;
    if (!ok) set_status(status, FP8_ERR_BOUNDS);
    return ok;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ numbers

// The two BF16 halves of a 32-bit word, widened exactly to FP32.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two FP32 values rounded to nearest-even BF16 and packed (lo in bits 0..15).
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// |x| of both BF16 halves, as bit patterns (unsigned order = magnitude order
// for everything but NaN, which sorts above +Inf and is caught separately).
__device__ __forceinline__ uint32_t bf16x2_abs(uint32_t w) { return w & 0x7FFF7FFFu; }
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) { return __vmaxu2(a, b); }
__device__ __forceinline__ uint32_t halfmax(uint32_t w) { return max(w & 0xFFFFu, w >> 16); }

// Scale of a group from its amax (as BF16 magnitude bits): s = fp32(amax / fmax),
// 1 for an all-zero group ([FP8-LM] "Tensor scaling"; s = amax / fmax).
__device__ __forceinline__ float scale_from_amax_bits(uint32_t amax_bf16_bits, int fmt)
{
    float amax = __uint_as_float(amax_bf16_bits << 16);
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, fmax_of(fmt));
}

// Scales for which the quotient x / s is taken from the reciprocal with
// Markstein's correction (below).  The correction needs the remainder
// e = x - q0*s exactly: e is a multiple of ulp(q0)*ulp(s) below ulp(q0)*s, so
// it fits binary32 while ulp(q0)*ulp(s) >= 2^-149, i.e. exponent(q) +
// exponent(s) >= -103.  Every quotient that can decide an FP8 code lies at or
// above 2^-18 (half of E5M2's smallest subnormal 2^-16 is 2^-17; E4M3's is
// 2^-10), so s >= 2^-84 keeps those remainders exact; below it, or for a
// smaller quotient, a misrounded q stays far from every code boundary.  With
// s just above the binary32 normal range instead (2^-125), BF16 subnormal x
// gave quotients one ulp off that changed 186 E4M3 / 92 E5M2 codes of the
// exhaustive (amax, x) check.  Above 2^125, 1/s would be subnormal.
constexpr float kFastDivMinScale = 0x1p-84f;
constexpr float kFastDivMaxScale = 0x1p125f;
__host__ __device__ __forceinline__ bool fast_div_scale(float s)
{
    return s >= kFastDivMinScale && s <= kFastDivMaxScale;
}

// Division x / s rounded to nearest binary32, computed from r = RN(1/s) with
// Markstein's correction (P. Markstein, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// r within half an ulp of 1/s and q0 within one ulp of x/s, the remainder
// e = x - q0*s is exact under FMA and RN(q0 + e*r) is the correctly rounded
// quotient.  Valid while s and 1/s are normal, e does not underflow and
// nothing overflows; callers use it only when fast_div_scale(s) and fall back
// to __fdiv_rn otherwise.  A quotient that overflows (or x = +-Inf) turns q0
// into +-Inf and q into NaN.
//
// Packed form for two dividends (the BF16 halves of a 32-bit word, or two
// binary32 values): q0 = x*r, e = x - q0*s (exact), q = q0 + e*r, two lanes
// per instruction (the f32x2 forms round each lane like the scalar
// instructions).  The remainder is taken rounding toward minus infinity: a
// nonzero e is exact, so its rounding mode changes nothing, and a zero x gives
// e = (+-0) * (-s) + x, a sum of opposite zeros, which rounds to -0 in that
// mode.  Then for x = -0, q = -0 * r + (-0) = -0, and for x = +0,
// q = -0 * r + (+0) = +0 (nearest): every zero quotient carries the sign of x,
// as in the IEEE division, and the FP8 conversion keeps it (-0 -> 0x80) with
// no sign fix-up on the codes.  Quantizers whose scale cannot make x / s
// overflow (scales from the group's own amax) need no NaN check; the others
// redo a group whose codes hold a NaN with __fdiv_rn (has_nan_code).
struct Divider2 {
    uint64_t r2, ns2;
    float s;
    bool fast;
    __device__ __forceinline__ explicit Divider2(float s_) : s(s_)
    {
        fast = fast_div_scale(s_);
        const float r = fast ? __frcp_rn(s_) : 0.0f;
        asm("mov.b64 %0, {%1, %1};" : "=l"(r2) : "f"(r));
        asm("mov.b64 %0, {%1, %1};" : "=l"(ns2) : "f"(-s_));
    }
    // from a scale and its reciprocal computed elsewhere (r = 0: not fast)
    __device__ __forceinline__ Divider2(float s_, float r) : s(s_)
    {
        fast = r != 0.0f;
        asm("mov.b64 %0, {%1, %1};" : "=l"(r2) : "f"(r));
        asm("mov.b64 %0, {%1, %1};" : "=l"(ns2) : "f"(-s_));
    }
    // the packed Markstein quotients alone (callers have checked `fast`)
    __device__ __forceinline__ void fast_div(uint32_t w, float &qlo, float &qhi) const
    {
        const float xlo = __uint_as_float(w << 16), xhi = __uint_as_float(w & 0xFFFF0000u);
        uint64_t x2, q0, e, q;
        asm("mov.b64 %0, {%1, %2};" : "=l"(x2) : "f"(xlo), "f"(xhi));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x2), "l"(r2));
        asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q0), "l"(ns2), "l"(x2));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(e), "l"(r2), "l"(q0));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(qlo), "=f"(qhi) : "l"(q));
    }
    // the same for two binary32 dividends
    __device__ __forceinline__ void fast_div_f32(float xlo, float xhi, float &qlo, float &qhi) const
    {
        uint64_t x2, q0, e, q;
        asm("mov.b64 %0, {%1, %2};" : "=l"(x2) : "f"(xlo), "f"(xhi));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x2), "l"(r2));
        asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q0), "l"(ns2), "l"(x2));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(e), "l"(r2), "l"(q0));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(qlo), "=f"(qhi) : "l"(q));
    }
    // quotients of (lo, hi) BF16 halves of w
    __device__ __forceinline__ void operator()(uint32_t w, float &qlo, float &qhi) const
    {
        const float xlo = __uint_as_float(w << 16), xhi = __uint_as_float(w & 0xFFFF0000u);
        if (fast) {
            uint64_t x2, q0, e, q;
            asm("mov.b64 %0, {%1, %2};" : "=l"(x2) : "f"(xlo), "f"(xhi));
            asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x2), "l"(r2));
            asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q0), "l"(ns2), "l"(x2));
            asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(e), "l"(r2), "l"(q0));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(qlo), "=f"(qhi) : "l"(q));
        } else {
            qlo = __fdiv_rn(xlo, s);
            qhi = __fdiv_rn(xhi, s);
        }
    }
};

// SwiGLU element math (SwiGLU(g, u) = g * sigmoid(g) * u and its gradients),
// shared by the standalone SwiGLU kernels and the quantizers that compute
// SwiGLU while loading, so both round identically.  The 8-wide forms below
// take 8 packed BF16 values per operand.
// sigmoid(g) = 1 / (1 + e^-g), with e^-g = 2^(-g log2 e) from the hardware
// base-2 exponential and the reciprocal from the hardware reciprocal (PTX
// ex2.approx.ftz.f32, rcp.approx.ftz.f32).  For g >= -64 the relative error is
// below 1e-5: rounding the argument -g log2 e (|arg| <= 128) to binary32 moves
// 2^arg by at most 128 * 7.3e-8 * ln 2 = 6.5e-6, and the two approximations
// add about 2^-22 and 2^-23.  That stays far inside half a BF16 ulp, so the
// BF16 results are within one ulp of the correctly rounded ones.  Neither
// flush to zero changes a result there: a 2^arg below the normal range leaves
// 1 + 2^arg == 1, and 1 + 2^arg < 2^93 keeps its reciprocal normal.
// Below g = -64, 1 + e^g rounds to 1, so sigmoid(g) = e^g, taken from the
// accurate exponential: e^-g itself would overflow FP32 below g = -88.7, while
// e^g keeps its value down into the subnormals, where g * sigmoid(g) * u can
// still be a nonzero BF16.  Groups of 8 with no gate below -64 (all but
// extreme inputs) run without a branch; the others go out of line.
__device__ __forceinline__ float ex2_approx_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx_ftz(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool LEFT>
__device__ __forceinline__ float swiglu_sigmoid(float g)
{
    constexpr float kLog2e = 1.44269504f;   // log2(e) rounded to binary32
    if (LEFT && g < -64.0f) return expf(g);
    return rcp_approx_ftz(1.0f + ex2_approx_ftz(g * -kLog2e));
}

template <bool LEFT>
__device__ __forceinline__ void swiglu_grad(float g, float u, float d, float &dg, float &du)
{
    const float sg = swiglu_sigmoid<LEFT>(g);
    dg = d * u * sg * (1.0f + g * (1.0f - sg));
    du = d * g * sg;
}

__device__ __forceinline__ float min_gate8(uint4 g4)
{
    const uint32_t w[4] = {g4.x, g4.y, g4.z, g4.w};
    float m = bf16_lo(w[0]);
#pragma unroll
    for (int k = 0; k < 4; ++k) m = fminf(m, fminf(bf16_lo(w[k]), bf16_hi(w[k])));
    return m;
}

// Packed FP32 pair helpers for the SwiGLU gradient (each lane rounds like the
// scalar instruction).  The gradient's eight multiplies and adds per value run
// as four packed ones (the fused backward quantizer: 298 -> 287 us on dGU
// 8192x28672); the forward's three are faster scalar (161 vs 170 us packed).
__device__ __forceinline__ uint64_t p2(float lo, float hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ uint64_t p2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t p2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint32_t p2_bf16(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return bf16x2_rn(lo, hi);
}
// the (lo, hi) BF16 halves of a word as a packed FP32 pair
__device__ __forceinline__ uint64_t p2_bf16x2(uint32_t w) { return p2(bf16_lo(w), bf16_hi(w)); }

template <bool LEFT>
__device__ __forceinline__ uint4 swiglu8_impl(uint4 g4, uint4 u4)
{
    const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, uw[4] = {u4.x, u4.y, u4.z, u4.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float g0 = bf16_lo(gw[k]), g1 = bf16_hi(gw[k]);
        o[k] = bf16x2_rn(g0 * swiglu_sigmoid<LEFT>(g0) * bf16_lo(uw[k]), g1 * swiglu_sigmoid<LEFT>(g1) * bf16_hi(uw[k]));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

static __device__ __noinline__ uint4 swiglu8_left(uint4 g4, uint4 u4) { return swiglu8_impl<true>(g4, u4); }

// H = SwiGLU(gate, up) for 8 values, BF16 round to nearest even.
__device__ __forceinline__ uint4 swiglu8(uint4 g4, uint4 u4)
{
    if (min_gate8(g4) < -64.0f) return swiglu8_left(g4, u4);
    return swiglu8_impl<false>(g4, u4);
}

struct Uint4x2 { uint4 a, b; };

template <bool LEFT>
__device__ __forceinline__ Uint4x2 swiglu_grad8_impl(uint4 g4, uint4 u4, uint4 d4)
{
    const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, uw[4] = {u4.x, u4.y, u4.z, u4.w},
                   dw[4] = {d4.x, d4.y, d4.z, d4.w};
    uint32_t og[4], ou[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (LEFT) {
            float dg0, du0, dg1, du1;
            swiglu_grad<true>(bf16_lo(gw[k]), bf16_lo(uw[k]), bf16_lo(dw[k]), dg0, du0);
            swiglu_grad<true>(bf16_hi(gw[k]), bf16_hi(uw[k]), bf16_hi(dw[k]), dg1, du1);
            og[k] = bf16x2_rn(dg0, dg1);
            ou[k] = bf16x2_rn(du0, du1);
        } else {
            // dg = d * u * sig * (1 + g * (1 - sig)), du = d * g * sig on packed pairs
            const float g0 = bf16_lo(gw[k]), g1 = bf16_hi(gw[k]);
            const uint64_t g = p2(g0, g1), u = p2_bf16x2(uw[k]), d = p2_bf16x2(dw[k]);
            const uint64_t sg = p2(swiglu_sigmoid<false>(g0), swiglu_sigmoid<false>(g1));
            const uint64_t one = p2(1.0f, 1.0f);
            const uint64_t oms = p2_fma(sg, p2(-1.0f, -1.0f), one);   // 1 - sig
            const uint64_t w = p2_fma(g, oms, one);                   // 1 + g (1 - sig)
            og[k] = p2_bf16(p2_mul(p2_mul(p2_mul(d, u), sg), w));
            ou[k] = p2_bf16(p2_mul(p2_mul(d, g), sg));
        }
    }
    return {make_uint4(og[0], og[1], og[2], og[3]), make_uint4(ou[0], ou[1], ou[2], ou[3])};
}

static __device__ __noinline__ Uint4x2 swiglu_grad8_left(uint4 g4, uint4 u4, uint4 d4)
{
    return swiglu_grad8_impl<true>(g4, u4, d4);
}

// dGate = dH * up * sig * (1 + gate * (1 - sig)) and dUp = dH * gate * sig
// for 8 values, BF16 round to nearest even.
__device__ __forceinline__ void swiglu_grad8(uint4 g4, uint4 u4, uint4 d4, uint4 &dg4, uint4 &du4)
{
    const Uint4x2 r = min_gate8(g4) < -64.0f ? swiglu_grad8_left(g4, u4, d4) : swiglu_grad8_impl<false>(g4, u4, d4);
    dg4 = r.a;
    du4 = r.b;
}

// Scales of 8 groups of 128 values spread over the 16 lanes of a half-warp
// (each lane holds 8 values of every group; m[u] = the lane's amax bits of
// group u).  The maxima are reduce-scattered (xor 8 and 4 split the groups,
// xor 2 and 1 finish them, two 16-bit maxima per word), so the quad of lanes
// 4p..4p+3 ends with groups 2p and 2p+1, and lane 4p+e (e = 0, 1) computes
// the scale s of group 2p+e and its reciprocal r (0 where the packed
// division must fall back to __fdiv_rn).  Group u's pair then lives in lane
// half_group_lane(u) of the half-warp.  Every lane of the warp must call it.
struct GroupScale {
    float s, r;
    uint32_t amax;   // BF16 magnitude bits of this lane's group
    int u;           // the group this lane computed
};

__device__ __forceinline__ int half_group_lane(int u) { return 4 * (u >> 1) + (u & 1); }

template <int FMT>
__device__ __forceinline__ GroupScale half_warp_scales8(const uint32_t (&m)[8], int l16)
{
    const bool b3 = (l16 & 8) != 0, b2 = (l16 & 4) != 0;
    const uint32_t M0 = m[0] | (m[1] << 16), M1 = m[2] | (m[3] << 16);
    const uint32_t M2 = m[4] | (m[5] << 16), M3 = m[6] | (m[7] << 16);
    uint32_t K0 = b3 ? M2 : M0, K1 = b3 ? M3 : M1;
    const uint32_t S0 = b3 ? M0 : M2, S1 = b3 ? M1 : M3;
    K0 = __vmaxu2(K0, __shfl_xor_sync(0xffffffffu, S0, 8));
    K1 = __vmaxu2(K1, __shfl_xor_sync(0xffffffffu, S1, 8));
    uint32_t K = b2 ? K1 : K0;
    const uint32_t S = b2 ? K0 : K1;
    K = __vmaxu2(K, __shfl_xor_sync(0xffffffffu, S, 4));
    K = __vmaxu2(K, __shfl_xor_sync(0xffffffffu, K, 2));
    K = __vmaxu2(K, __shfl_xor_sync(0xffffffffu, K, 1));
    GroupScale g;
    g.amax = (l16 & 1) ? (K >> 16) : (K & 0xFFFFu);
    g.u = 2 * (l16 >> 2) + (l16 & 1);
    g.s = scale_from_amax_bits(g.amax, FMT);
    g.r = fast_div_scale(g.s) ? __frcp_rn(g.s) : 0.0f;
    return g;
}

// Sign bits of the 4 BF16 values in (w0 = x0,x1 ; w1 = x2,x3) placed at bit 7
// of bytes 0..3: OR-ed into the 4 codes of the out-of-line IEEE paths, this
// sets the sign of every code from its value (the packed fast paths need no
// fix-up: their zero quotients already carry the sign).
__device__ __forceinline__ uint32_t sign_bits4(uint32_t w0, uint32_t w1)
{
    return __byte_perm(w0, w1, 0x7531) & 0x80808080u;
}

// True if one of the four codes in w is a NaN code (E4M3 S.1111.111, E5M2
// S.11111.xx with xx != 0; satfinite conversion produces no E5M2 infinity, so
// every code with an all-ones exponent is a NaN).
template <int FMT>
__device__ __forceinline__ bool has_nan_code(uint32_t w)
{
    constexpr uint32_t kMask = FMT == FP8_E4M3 ? 0x7F7F7F7Fu : 0x7C7C7C7Cu;
    constexpr uint32_t kAdd = FMT == FP8_E4M3 ? 0x01010101u : 0x04040404u;
    return (((w & kMask) + kAdd) & 0x80808080u) != 0;
}

// FP8 encode of two binary32 values (round to nearest even, saturating to
// +-fmax): the byte of `lo` lands in bits 0..7, `hi` in bits 8..15.
template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi)
{
    uint16_t r;
    if (FMT == FP8_E5M2)
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// Quantize BF16 values with the packed divider.  The fast path is inlined; a
// scale outside its range (rare: an all-tiny or non-finite group) takes one
// out-of-line call for the whole group, which keeps the unrolled loops small.
template <int FMT>
__device__ __forceinline__ uint32_t quant4p_fast(uint32_t w0, uint32_t w1, const Divider2 &d)
{
    float a, b, c, e;
    d.fast_div(w0, a, b);
    d.fast_div(w1, c, e);
    return cvt2<FMT>(a, b) | (cvt2<FMT>(c, e) << 16);
}

template <int FMT>
__device__ __noinline__ uint2 quant8p_slow(uint4 v, float s)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
    for (int j = 0; j < 4; ++j)
        c[j] = cvt2<FMT>(__fdiv_rn(__uint_as_float(w[j] << 16), s), __fdiv_rn(__uint_as_float(w[j] & 0xFFFF0000u), s));
    return make_uint2((c[0] | (c[1] << 16)) | sign_bits4(w[0], w[1]), (c[2] | (c[3] << 16)) | sign_bits4(w[2], w[3]));
}

template <int FMT>
__device__ __forceinline__ uint2 quant8p(uint4 v, const Divider2 &d)
{
    if (!d.fast) return quant8p_slow<FMT>(v, d.s);
    return make_uint2(quant4p_fast<FMT>(v.x, v.y, d), quant4p_fast<FMT>(v.z, v.w, d));
}

__device__ __forceinline__ uint32_t absmax8(uint4 v)
{
    uint32_t m = bf16x2_absmax(bf16x2_abs(v.x), bf16x2_abs(v.y));
    m = bf16x2_absmax(m, bf16x2_abs(v.z));
    m = bf16x2_absmax(m, bf16x2_abs(v.w));
    return halfmax(m);
}

__device__ __forceinline__ uint4 ldg_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// --------------------------------------------------------- shared / barriers

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global -> shared copy (L2 only) and the wait for all of
// the calling thread's copies; after the wait they are visible to that thread.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits until the phase with parity `parity` of `bar` has completed.  Gives
// up (returns false) after `timeout_ns`, or early when *abort becomes
// nonzero; it never spins without bound.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                  uint64_t timeout_ns = kWaitTimeoutNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u) {
            if (abort && *abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) return false;
        }
    }
}

// Bounded wait on an mbarrier phase shared by the roles of a warp-specialised
// kernel: on a timeout the first role to give up records FP8_ERR_TIMEOUT and
// raises the CTA's abort flag, which the other roles' waits poll.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int *status)
{
    if (mbar_wait_bounded(bar, parity, abort_flag)) return true;
    if (!*abort_flag) {
        *abort_flag = 1;
        set_status(status, FP8_ERR_TIMEOUT);
    }
    return false;
}

// Barrier operations on a shared-memory address computed once (the hot loops
// keep barrier and buffer addresses as 32-bit shared addresses).
__device__ __forceinline__ bool mbar_try_wait_a(uint32_t addr, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_arrive_a(uint32_t addr)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}

// The slow path of warp_wait_a: every lane polls with the bounded-wait rules
// of mbar_wait_bounded; out of line so the hot loop stays small.
static __device__ __noinline__ bool warp_wait_slow_a(uint32_t addr, uint32_t parity, volatile int *abort_flag,
                                                     int *status)
{
    const uint64_t t0 = globaltimer_ns();
    bool ok = false;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_a(addr, parity)) {
            ok = true;
            break;
        }
        if ((i & 63u) == 0u) {
            if (*abort_flag) break;
            if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                if (!*abort_flag) {
                    *abort_flag = 1;
                    set_status(status, FP8_ERR_TIMEOUT);
                }
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// A whole warp waits on the barrier at `addr` (see warp_wait_or_abort).
__device__ __forceinline__ bool warp_wait_a(uint32_t addr, uint32_t parity, volatile int *abort_flag, int *status)
{
    if (__all_sync(0xffffffffu, mbar_try_wait_a(addr, parity))) return true;
    return warp_wait_slow_a(addr, parity, abort_flag, status);
}

// Shared-memory loads at a 32-bit shared address plus a constant offset.
template <int OFF>
__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(addr), "n"(OFF) : "memory");
    return v;
}

template <int OFF>
__device__ __forceinline__ uint64_t lds_b64(uint32_t addr)
{
    uint64_t v;
    asm volatile("ld.shared.b64 %0, [%1+%2];" : "=l"(v) : "r"(addr), "n"(OFF) : "memory");
    return v;
}

// A whole warp waits: every lane polls the barrier, so the warp never splits
// into a single-lane spin loop, and a vote makes the outcome warp-uniform so
// the warp stays converged for the .sync.aligned tcgen05 instructions that
// follow.  (Polling through lane 0 and broadcasting the result was 7-12%
// slower on the GEMMs: the single-lane loop and its reconvergence took issue
// slots from the epilogue warps on the same sub-partition.)
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                   int *status)
{
    bool ok = mbar_try_wait(bar, parity);
    if (!__all_sync(0xffffffffu, ok)) {
        ok = wait_or_abort(bar, parity, abort_flag, status);
        ok = __all_sync(0xffffffffu, ok);
    }
    return ok;
}


// ---------------------------------------------------------------------- TMA

// 2-D tiled bulk tensor load global -> shared, completion counted in bytes
// on `bar`.  x is the innermost coordinate (elements of the map's type).
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// 2-D tiled bulk tensor store shared -> global (bulk-group completion).  The
// coordinates must be non-negative and x * element size a multiple of 16.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *smem_src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(smem_src)), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// The thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// The thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Barrier `id` (1..15) over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Untiled bulk copy global -> shared memory, completing `bytes` on the
// mbarrier.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(reinterpret_cast<uint64_t>(gmem_src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05

// Tiles are walked in bands of GM M-tiles, M fastest: a band's A rows stay in
// L2 while every B tile is streamed through it once per band.  GM = 0 walks N
// fastest instead (each M-tile's row of tiles in turn), which keeps all of B
// in L2 and streams A once.
__device__ __forceinline__ void tile_coords_raster(int tile, int num_mt, int num_nt, int GM, int &mt, int &nt)
{
    if (GM == 0) {
        mt = tile / num_nt;
        nt = tile - mt * num_nt;
        return;
    }
    const int group = tile / (GM * num_nt);
    const int first = group * GM;
    const int gm = min(GM, num_mt - first);
    const int local = tile - group * GM * num_nt;
    mt = first + local % gm;
    nt = local / gm;
}


__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem) (+)= A(smem desc) x B(smem desc)^T, FP8 operands, FP32 accumulator.
__device__ __forceinline__ void tc_mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(smem desc) x B(smem desc)^T with MXFP8 block scaling: FP8
// operands, one UE8M0 scale per 32-deep block of every row of A and of B read
// from tensor memory (sfa_tmem, sfb_tmem; which byte of the 32-bit word is in
// the instruction descriptor), FP32 accumulator.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Shared memory -> tensor memory: 32 rows of 16 bytes (row r at byte 16 r of
// the source) land in lane r of every one of the four lane quarters, columns
// [col, col + 4).  Ordered before the tcgen05.mma instructions this thread
// issues after it.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D(tmem) (+)= A(smem desc) x B(smem desc)^T, 16-bit operands (F16 or BF16 as
// the instruction descriptor says), FP32 accumulator.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 columns of 32-bit TMEM words: thread i of the warp receives
// lane (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 16 columns (16 registers per thread).
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// 16 lanes x 8 repetitions of 256 bits (8 columns of 32-bit words each, 64
// columns): thread i of the warp receives, for repetition j < 8, lane
// (base + i/4) columns col + 8j + 2(i%4) + {0, 1} in r[4j], r[4j+1] and lane
// (base + 8 + i/4), the same columns, in r[4j+2], r[4j+3].
__device__ __forceinline__ void tc_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Packed FP32 pair arithmetic (two IEEE binary32 lanes, each rounded to
// nearest like the scalar instruction).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// acc + (lo, hi) * s2, lane-wise
__device__ __forceinline__ uint64_t f2_fma_bits(uint32_t lo, uint32_t hi, uint64_t s2, uint64_t acc)
{
    uint64_t d;
    asm("{\n\t.reg .b64 p;\n\tmov.b64 p, {%1, %2};\n\tfma.rn.f32x2 %0, p, %3, %4;\n\t}"
        : "=l"(d)
        : "r"(lo), "r"(hi), "l"(s2), "l"(acc));
    return d;
}

// (lo, hi) * b2, lane-wise
__device__ __forceinline__ uint64_t f2_mul_bits(uint32_t lo, uint32_t hi, uint64_t b2)
{
    uint64_t d;
    asm("{\n\t.reg .b64 p;\n\tmov.b64 p, {%1, %2};\n\tmul.rn.f32x2 %0, p, %3;\n\t}"
        : "=l"(d)
        : "r"(lo), "r"(hi), "l"(b2));
    return d;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Per-warpgroup register budget changes (all threads of the warpgroup).
template <int N>
__device__ __forceinline__ void regs_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Shared-memory matrix descriptor for a K-major operand tile stored in the
// 128-byte swizzle layout that a TMA load with CU_TENSOR_MAP_SWIZZLE_128B
// writes: rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte
// offset), leading byte offset unused (1), descriptor version 1, swizzle mode
// 2 = 128B.  The tile base must be 1024-byte aligned; advancing along K
// inside the 128-byte row is done by adding the byte offset to the start.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Shared-memory descriptor of a plain (unswizzled) source for tcgen05.cp:
// rows of 16 bytes stored contiguously, 8-row core matrices 128 bytes apart
// (both byte offsets 128), version 1, no swizzle; 16-byte aligned start.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}

// Shared-memory matrix descriptor for an MN-major operand tile in the
// 128-byte swizzle layout a TMA load writes from a row-major matrix whose
// rows run along K: each K index is a 128-byte row of 64 consecutive M (or
// N) elements (16-bit types), 8 such rows form a 1024-byte swizzle atom.
// Stride byte offset = distance between atoms along K (1024 for consecutive
// rows), leading byte offset = distance between the 64-element slabs along
// M / N (one TMA box each).  Version 1, swizzle mode 2 = 128B; the base must
// be 1024-byte aligned and a K step advances the start by whole atoms.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma .kind::f16 with BF16 A and B (type
// code 1 at bits 7-9 and 10-12), an FP32 accumulator (bits 4-5 = 1), both
// operands MN-major (bits 15 and 16), N/8 at bits 17-22, M/16 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_mnmajor(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma .kind::f8f6f4 with an FP32
// accumulator, both operands K-major, dense: D format bits 4-5 (1 = F32),
// A type bits 7-9 and B type bits 10-12 (0 = E4M3, 1 = E5M2), N/8 at bits
// 17-22, M/16 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f8f6f4(int fmtA, int fmtB, int M, int N)
{
    return (1u << 4) | ((uint32_t)(fmtA == FP8_E5M2 ? 1 : 0) << 7) | ((uint32_t)(fmtB == FP8_E5M2 ? 1 : 0) << 10) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma .kind::mxf8f6f4.block_scale: A type
// bits 7-9 and B type bits 10-12 (0 = E4M3, 1 = E5M2), both operands K-major,
// dense, N/8 at bits 17-22, scale type UE8M0 (bit 23 = 1), M/16 at bits
// 24-28.  The byte of the 32-bit scale word each operand reads goes in bits
// 29-30 (A) and 4-5 (B): idesc_mx_block(d, j) for the j-th 32-deep block.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(int fmtA, int fmtB, int M, int N)
{
    return ((uint32_t)(fmtA == FP8_E5M2 ? 1 : 0) << 7) | ((uint32_t)(fmtB == FP8_E5M2 ? 1 : 0) << 10) |
           ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_mx_block(uint32_t idesc, uint32_t j)
{
    return idesc | (j << 4) | (j << 29);
}

}  // namespace fp8fg
