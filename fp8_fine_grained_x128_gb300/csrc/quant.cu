// quant.cu -- BF16 -> FP8 quantizers of the fine-grained FP8 Linear (sm_103a).
//
//   * 1x128 activation/gradient tiles (Ling 2.0 FP8 pretraining blog,
//     "Fine-grained quantization (per-tile/block wise scaling)"; activations
//     are quantized dynamically, FP8-RL article "dynamic weight sync").
//   * the same plus the transposed copy quantized along the token dimension
//     for the wgrad operand ("grad (transpose)" in the blog's monitor table),
//     from ONE read of the input -- also with SwiGLU computed while loading,
//     so that the MLP's H (forward) and dGU (backward) are quantized without
//     ever being written in BF16.
//   * 128x128 weight blocks (FP8-RL article, "dynamic weight sync"), with an
//     optional transposed copy written in the same pass.
//   * the on-demand FP8 weight transpose (blog, "FP8 on-demand transpose
//     weight").
// Quantization rule ("FP8-LM: Training FP8 Large Language Models", "Tensor
// scaling"): s = fp32(amax / fmax), q = RNE_satfinite(fp32(x) / s).
//
// All of these are streaming kernels (HBM-bound, or bound by instruction issue
// where SwiGLU and the transposed copy add work): 16-byte vector loads, amax
// by warp shuffles, coalesced FP8 stores, no tensor-core work.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

// ---------------------------------------------------------------------------
// 1x128 along rows only.  A half-warp owns a run of U consecutive 1x128 tiles
// of one row (16 lanes x 8 BF16 per tile), so every thread keeps U 16-byte
// loads in flight; the only division per run is the run -> (row, chunk) map.
// ---------------------------------------------------------------------------
template <int FMT, int U>
__global__ void __launch_bounds__(256, 4) k_quant_1x128_rows(const uint16_t *__restrict__ x, uint32_t rows,
                                                          uint32_t ncb, int64_t ldx, uint8_t *__restrict__ q,
                                                          float *__restrict__ s, int *status)
{
    const int l16 = threadIdx.x & 15;
    const uint32_t hw0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 4;
    const uint32_t nhw = (gridDim.x * blockDim.x) >> 4;
    const uint32_t ngrp = (ncb + U - 1) / U;        // runs per row
    const uint32_t nitems = rows * ngrp;
    const int64_t cols = (int64_t)ncb * 128;
    // both half-warps of a warp share the loop test (shuffles use the full mask)
    for (uint32_t it = hw0; (it & ~1u) < nitems; it += nhw) {
        const bool valid = it < nitems;
        const uint32_t r = valid ? it / ngrp : 0;
        const uint32_t c0 = valid ? (it - r * ngrp) * U : ncb;
        const uint16_t *xr = x + (int64_t)r * ldx + l16 * 8;
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = (c0 + u < ncb) ? ldg_stream(xr + (int64_t)(c0 + u) * 128) : make_uint4(0, 0, 0, 0);
        uint32_t m[U];
#pragma unroll
        for (int u = 0; u < U; ++u) m[u] = absmax8(v[u]);
        // each tile's scale is computed by one lane and shuffled to the others
        const GroupScale gs = half_warp_scales8<FMT>(m, l16);
        if (!(l16 & 2) && c0 + gs.u < ncb) {
            if (gs.amax >= 0x7F80u) set_status(status, FP8_ERR_NONFINITE);
            if (dbg_cell(c0 + gs.u, r, 1, ncb, rows, status)) s[(int64_t)(c0 + gs.u) * rows + r] = gs.s;
        }
        const int hbase = threadIdx.x & 16;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float su = __shfl_sync(0xffffffffu, gs.s, hbase + half_group_lane(u));
            const float ru = __shfl_sync(0xffffffffu, gs.r, hbase + half_group_lane(u));
            const uint32_t cb = c0 + u;
            if (cb < ncb) {
                const Divider2 d(su, ru);
                const uint2 c = quant8p<FMT>(v[u], d);
                if (dbg_cell(r, (int64_t)cb * 128 + l16 * 8, 8, rows, cols, status))
                    *reinterpret_cast<uint2 *>(q + (int64_t)r * cols + (int64_t)cb * 128 + l16 * 8) = c;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Fused 1x128 + transposed 128x1.  Persistent CTAs walk 128x128 tiles of x:
//  1. each thread holds 8 rows x 8 columns (16 B per row) of the tile in
//     registers -- the tile's only HBM read;
//  2. row scales by half-warp shuffles, row codes stored straight from
//     registers; the raw tile goes to shared memory (16-B chunks XOR-
//     swizzled by row so the row stores and the 4x4 column reads are both
//     bank-conflict free); per-column amax partials go to shared memory;
//  3. the 128 column scales and their reciprocals;
//  4. the loads of the NEXT tile are issued, then each thread quantizes 4x4
//     sub-blocks with the column scales and writes 4 words of the transposed
//     codes (full 32-byte segments per 8 lanes) while those loads fly.
// ---------------------------------------------------------------------------
struct ColDiv2 {
    uint64_t r2, ns2;    // (1/s_j, 1/s_j+1), (-s_j, -s_j+1)
    float s0, s1;
    int fast;
};

// Codes of the column pair (lo, hi) of w, each with its own column scale.
template <int FMT>
__device__ __forceinline__ uint32_t quant_pair_cols_fast(uint32_t w, const ColDiv2 &c)
{
    float qlo, qhi;
    const float xlo = __uint_as_float(w << 16), xhi = __uint_as_float(w & 0xFFFF0000u);
    uint64_t x2, q0, e, qq;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x2) : "f"(xlo), "f"(xhi));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x2), "l"(c.r2));
    asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q0), "l"(c.ns2), "l"(x2));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(qq) : "l"(e), "l"(c.r2), "l"(q0));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(qlo), "=f"(qhi) : "l"(qq));
    return cvt2<FMT>(qlo, qhi);
}

// The same for 4 rows x 4 columns when a column scale is outside the fast
// division's range (out of line: rare).
template <int FMT>
__device__ __noinline__ uint4 quant_cols4x4_slow(uint4 lo, uint4 hi, float s0, float s1, float s2, float s3)
{
    const uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w}, b[4] = {hi.x, hi.y, hi.z, hi.w};
    uint32_t rw[4];
    for (int i = 0; i < 4; ++i) {
        const uint32_t c01 = cvt2<FMT>(__fdiv_rn(__uint_as_float(a[i] << 16), s0),
                                       __fdiv_rn(__uint_as_float(a[i] & 0xFFFF0000u), s1));
        const uint32_t c23 = cvt2<FMT>(__fdiv_rn(__uint_as_float(b[i] << 16), s2),
                                       __fdiv_rn(__uint_as_float(b[i] & 0xFFFF0000u), s3));
        rw[i] = (c01 | (c23 << 16)) | sign_bits4(a[i], b[i]);
    }
    return make_uint4(rw[0], rw[1], rw[2], rw[3]);
}

constexpr int kFusedSmem = 32768 + 4096 + 64 * sizeof(ColDiv2);

// What the fused quantizer reads: x itself, or SwiGLU computed while loading
// from the gate/up projection GU [rows][2F] (forward: H [rows][F]) or from GU
// and dH [rows][F] (backward: dGU [rows][2F], gate-gradient half then up
// half), so the BF16 H / dGU never go to HBM.
enum { SRC_X = 0, SRC_SWIGLU_FWD = 1, SRC_SWIGLU_BWD = 2 };

// One thread's raw loads for one work unit: rows rr + 16i (i < 8), columns
// 8g .. 8g+7 of the unit's 128-column block.  A unit is one 128x128 tile of
// x or of H; for the backward it is a column block of the gate half together
// with the same block of the up half (both need gate, up and dH there).  The
// backward's dH goes to shared memory by asynchronous copies (32 more
// registers of prefetch would not fit next to the quantizer's).
template <int SRC> struct RawUnit;
template <> struct RawUnit<SRC_X> { uint4 x[8]; };
template <> struct RawUnit<SRC_SWIGLU_FWD> { uint4 g[8], u[8]; };
template <> struct RawUnit<SRC_SWIGLU_BWD> { uint4 g[8], u[8]; };

__device__ __forceinline__ void load_unit(RawUnit<SRC_X> &ru, const uint16_t *x, const uint16_t *, int64_t ldx,
                                          int64_t, int64_t r, int64_t c, uint4 *)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) ru.x[i] = ldg_stream(x + (r + 16 * i) * ldx + c);
}

__device__ __forceinline__ void load_unit(RawUnit<SRC_SWIGLU_FWD> &ru, const uint16_t *gu, const uint16_t *,
                                          int64_t, int64_t F, int64_t r, int64_t c, uint4 *)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ru.g[i] = ldg_stream(gu + (r + 16 * i) * 2 * F + c);
        ru.u[i] = ldg_stream(gu + (r + 16 * i) * 2 * F + F + c);
    }
}

// dstage: this thread's 8 staging slots (stride 256 slots: a warp's copies
// fill 512 contiguous bytes).
__device__ __forceinline__ void load_unit(RawUnit<SRC_SWIGLU_BWD> &ru, const uint16_t *gu, const uint16_t *dh,
                                          int64_t, int64_t F, int64_t r, int64_t c, uint4 *dstage)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ru.g[i] = ldg_stream(gu + (r + 16 * i) * 2 * F + c);
        ru.u[i] = ldg_stream(gu + (r + 16 * i) * 2 * F + F + c);
        cp_async16(dstage + 256 * i, dh + (r + 16 * i) * F + c);
    }
}

// The plain quantizer keeps 3 CTAs per SM; the SwiGLU sources hold 64
// registers of raw prefetch and run 2.
template <int SRC> constexpr int fused_ctas_per_sm() { return SRC == SRC_X ? 3 : 2; }
template <int SRC> constexpr int fused_smem() { return kFusedSmem + (SRC == SRC_SWIGLU_BWD ? 32768 : 0); }

template <int FMT, int SRC>
__global__ void __launch_bounds__(256, fused_ctas_per_sm<SRC>()) k_quant_1x128_fused_t(
    const uint16_t *__restrict__ x, const uint16_t *__restrict__ dh, int64_t F, int64_t rows, int64_t cols,
    int64_t ldx, uint8_t *__restrict__ q, float *__restrict__ s, uint8_t *__restrict__ qT, float *__restrict__ sT,
    int *status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *tile = smem;                                              // [128][256 B], swizzled 16-B chunks
    uint32_t *colpart = reinterpret_cast<uint32_t *>(smem + 32768);    // [8 warps][128]
    ColDiv2 *cdiv = reinterpret_cast<ColDiv2 *>(smem + 32768 + 4096);  // [64 column pairs]
    uint4 *dstage = reinterpret_cast<uint4 *>(smem + kFusedSmem) + threadIdx.x;   // backward: dH [8][256]

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int g = t & 15, rr = t >> 4;
    const int64_t nmb = rows / 128;
    const int64_t ncb = (SRC == SRC_X ? cols : F) / 128;   // column blocks of a unit
    const int64_t nunits = ncb * nmb;

    // Quantizes the 128x128 tile at (r0, c0) whose values this thread holds in
    // v (rows rr + 16i, columns c0 + 8g ..): codes and row scales, then the
    // transposed codes and column scales through shared memory.  prefetch()
    // runs once the tile is in shared memory.
    auto quant_tile = [&](const uint4(&v)[8], int64_t r0, int64_t c0, int64_t mb, auto &&prefetch) {
        const int64_t cb = c0 / 128;
        uint32_t cm0 = 0, cm1 = 0, cm2 = 0, cm3 = 0;
        GroupScale gs;
        {
            uint32_t m[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = absmax8(v[i]);
            gs = half_warp_scales8<FMT>(m, g);   // the half-warp's 8 rows rr + 16i
        }
        if (!(g & 2)) {
            if (gs.amax >= 0x7F80u) set_status(status, FP8_ERR_NONFINITE);
            if (dbg_cell(cb, r0 + rr + 16 * gs.u, 1, cols / 128, rows, status)) s[cb * rows + r0 + rr + 16 * gs.u] = gs.s;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = rr + 16 * i;
            const float si = __shfl_sync(0xffffffffu, gs.s, (lane & 16) + half_group_lane(i));
            const float ri = __shfl_sync(0xffffffffu, gs.r, (lane & 16) + half_group_lane(i));
            const Divider2 d(si, ri);
            const uint2 code = quant8p<FMT>(v[i], d);
            if (dbg_cell(r0 + row, c0 + g * 8, 8, rows, cols, status))
                *reinterpret_cast<uint2 *>(q + (r0 + row) * cols + c0 + g * 8) = code;
            *reinterpret_cast<uint4 *>(tile + row * 256 + ((g ^ ((row >> 2) & 7)) << 4)) = v[i];
            cm0 = bf16x2_absmax(cm0, bf16x2_abs(v[i].x));
            cm1 = bf16x2_absmax(cm1, bf16x2_abs(v[i].y));
            cm2 = bf16x2_absmax(cm2, bf16x2_abs(v[i].z));
            cm3 = bf16x2_absmax(cm3, bf16x2_abs(v[i].w));
        }
        // lanes l and l^16 hold rows rr and rr+1 of the same columns
        cm0 = bf16x2_absmax(cm0, __shfl_xor_sync(0xffffffffu, cm0, 16));
        cm1 = bf16x2_absmax(cm1, __shfl_xor_sync(0xffffffffu, cm1, 16));
        cm2 = bf16x2_absmax(cm2, __shfl_xor_sync(0xffffffffu, cm2, 16));
        cm3 = bf16x2_absmax(cm3, __shfl_xor_sync(0xffffffffu, cm3, 16));
        if (lane < 16) {
            uint32_t *p = colpart + warp * 128 + g * 8;
            p[0] = cm0 & 0xFFFFu; p[1] = cm0 >> 16;
            p[2] = cm1 & 0xFFFFu; p[3] = cm1 >> 16;
            p[4] = cm2 & 0xFFFFu; p[5] = cm2 >> 16;
            p[6] = cm3 & 0xFFFFu; p[7] = cm3 >> 16;
        }
        __syncthreads();
        if (t < 64) {
            float sc[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t m = 0;
#pragma unroll
                for (int w = 0; w < 8; ++w) m = max(m, colpart[w * 128 + 2 * t + h]);
                if (m >= 0x7F80u) set_status(status, FP8_ERR_NONFINITE);
                sc[h] = scale_from_amax_bits(m, FMT);
            }
            ColDiv2 c;
            c.s0 = sc[0];
            c.s1 = sc[1];
            c.fast = fast_div_scale(sc[0]) && fast_div_scale(sc[1]);
            const float ra = c.fast ? __frcp_rn(sc[0]) : 0.0f, rb = c.fast ? __frcp_rn(sc[1]) : 0.0f;
            c.r2 = f2_pack(ra, rb);
            c.ns2 = f2_pack(-sc[0], -sc[1]);
            cdiv[t] = c;
            if (dbg_cell(mb, c0 + 2 * t, 2, rows / 128, cols, status))
                *reinterpret_cast<float2 *>(sT + mb * cols + c0 + 2 * t) = make_float2(sc[0], sc[1]);
        }
        __syncthreads();
        // the next unit's loads fly during the transposed quantization
        prefetch();

        const int cw = (lane >> 3) + 4 * warp;   // columns 4cw .. 4cw+3
        const ColDiv2 d01 = cdiv[2 * cw], d23 = cdiv[2 * cw + 1];
        const bool cfast = d01.fast && d23.fast;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int mg = (lane & 7) + 8 * k;   // rows 4mg .. 4mg+3
            uint2 pr[4];                         // BF16 of row 4mg+i, columns 4cw..4cw+3
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = 4 * mg + i;
                pr[i] = *reinterpret_cast<const uint2 *>(
                    tile + row * 256 + (((cw >> 1) ^ ((row >> 2) & 7)) << 4) + ((cw & 1) << 3));
            }
            uint32_t rw[4];                      // codes of row 4mg+i, columns 4cw..4cw+3
            if (cfast) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    rw[i] = quant_pair_cols_fast<FMT>(pr[i].x, d01) | (quant_pair_cols_fast<FMT>(pr[i].y, d23) << 16);
            } else {
                const uint4 c = quant_cols4x4_slow<FMT>(make_uint4(pr[0].x, pr[1].x, pr[2].x, pr[3].x),
                                                        make_uint4(pr[0].y, pr[1].y, pr[2].y, pr[3].y), d01.s0,
                                                        d01.s1, d23.s0, d23.s1);
                rw[0] = c.x; rw[1] = c.y; rw[2] = c.z; rw[3] = c.w;
            }
            const uint32_t t0 = __byte_perm(rw[0], rw[1], 0x5140), t1 = __byte_perm(rw[2], rw[3], 0x5140);
            const uint32_t t2 = __byte_perm(rw[0], rw[1], 0x7362), t3 = __byte_perm(rw[2], rw[3], 0x7362);
            uint8_t *dst = qT + (c0 + 4 * cw) * rows + r0 + 4 * mg;
            if (dbg_cell(c0 + 4 * cw + 3, r0 + 4 * mg, 4, cols, rows, status)) {
                *reinterpret_cast<uint32_t *>(dst) = __byte_perm(t0, t1, 0x5410);
                *reinterpret_cast<uint32_t *>(dst + rows) = __byte_perm(t0, t1, 0x7632);
                *reinterpret_cast<uint32_t *>(dst + 2 * rows) = __byte_perm(t2, t3, 0x5410);
                *reinterpret_cast<uint32_t *>(dst + 3 * rows) = __byte_perm(t2, t3, 0x7632);
            }
        }
        __syncthreads();   // the tile buffer is rewritten by the next iteration
    };

    int64_t unit = blockIdx.x;
    RawUnit<SRC> ru;
    if (unit < nunits) load_unit(ru, x, dh, ldx, F, (unit / ncb) * 128 + rr, (unit % ncb) * 128 + g * 8, dstage);

    for (; unit < nunits; unit += gridDim.x) {
        const int64_t mb = unit / ncb, cb = unit - mb * ncb;
        const int64_t next = unit + gridDim.x;
        auto prefetch = [&] {
            if (next < nunits)
                load_unit(ru, x, dh, ldx, F, (next / ncb) * 128 + rr, (next % ncb) * 128 + g * 8, dstage);
        };
        if constexpr (SRC == SRC_X) {
            uint4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = ru.x[i];
            quant_tile(v, mb * 128, cb * 128, mb, prefetch);
        } else if constexpr (SRC == SRC_SWIGLU_FWD) {
            uint4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = swiglu8(ru.g[i], ru.u[i]);
            quant_tile(v, mb * 128, cb * 128, mb, prefetch);
        } else {
            // the up-half gradient waits in this thread's dH slots while the
            // gate half is quantized (its registers would not fit beside it)
            uint4 vg[8], vu[8];
            cp_async_wait_all();   // this thread's dH copies (it reads only its own slots)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint4 du;
                swiglu_grad8(ru.g[i], ru.u[i], dstage[256 * i], vg[i], du);
                dstage[256 * i] = du;
            }
            quant_tile(vg, mb * 128, cb * 128, mb, [] {});
#pragma unroll
            for (int i = 0; i < 8; ++i) vu[i] = dstage[256 * i];
            quant_tile(vu, mb * 128, F + cb * 128, mb, prefetch);
        }
    }
}

// ---------------------------------------------------------------------------
// Transposed write of a 128x128 tile of codes held in shared memory as
// [128 rows][33 words] (one pad word per row): each thread byte-transposes
// 4x4 sub-blocks and stores 4 words of the transposed tile.  Lane mapping
// (mg = lane & 7, cw = lane >> 3) keeps the shared reads conflict free and
// gives full 32-byte segments on the global stores.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_code_tile_transposed(const uint32_t *ct, uint8_t *qT, int64_t ldT,
                                                           int64_t c0, int64_t r0, int64_t qt_rows, int *status)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cw = (lane >> 3) + 4 * warp;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int mg = (lane & 7) + 8 * k;
        const uint32_t w0 = ct[(4 * mg + 0) * 33 + cw];
        const uint32_t w1 = ct[(4 * mg + 1) * 33 + cw];
        const uint32_t w2 = ct[(4 * mg + 2) * 33 + cw];
        const uint32_t w3 = ct[(4 * mg + 3) * 33 + cw];
        const uint32_t t0 = __byte_perm(w0, w1, 0x5140), t1 = __byte_perm(w2, w3, 0x5140);
        const uint32_t t2 = __byte_perm(w0, w1, 0x7362), t3 = __byte_perm(w2, w3, 0x7362);
        uint8_t *dst = qT + (c0 + 4 * cw) * ldT + r0 + 4 * mg;
        if (!dbg_cell(c0 + 4 * cw + 3, r0 + 4 * mg, 4, qt_rows, ldT, status)) continue;
        *reinterpret_cast<uint32_t *>(dst) = __byte_perm(t0, t1, 0x5410);
        *reinterpret_cast<uint32_t *>(dst + ldT) = __byte_perm(t0, t1, 0x7632);
        *reinterpret_cast<uint32_t *>(dst + 2 * ldT) = __byte_perm(t2, t3, 0x5410);
        *reinterpret_cast<uint32_t *>(dst + 3 * ldT) = __byte_perm(t2, t3, 0x7632);
    }
}

// ---------------------------------------------------------------------------
// 128x128 blocks: one CTA per block, 8 rows x 16 B per thread, block amax by
// shuffles + shared, codes stored from registers; optionally the codes are
// staged in shared memory and written transposed too.
// ---------------------------------------------------------------------------
template <int FMT, bool TRANS>
__global__ void __launch_bounds__(256) k_quant_128x128(const uint16_t *__restrict__ w, int64_t rows, int64_t cols,
                                                       int64_t ldw, uint8_t *__restrict__ q, float *__restrict__ s,
                                                       uint8_t *__restrict__ qT, float *__restrict__ sT, int *status)
{
    __shared__ uint32_t red[8];
    __shared__ uint32_t ct[TRANS ? 128 * 33 : 1];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int g = t & 15, rr = t >> 4;
    const int64_t cb = blockIdx.x, rb = blockIdx.y;
    const int64_t r0 = rb * 128, c0 = cb * 128;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ldg_stream(w + (r0 + rr + 16 * i) * ldw + c0 + g * 8);
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = max(m, absmax8(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = max(m, red[i]);
    if (m >= 0x7F80u && t == 0) set_status(status, FP8_ERR_NONFINITE);
    const float sc = scale_from_amax_bits(m, FMT);
    const Divider2 d(sc);
    const int64_t ncb = cols / 128, nrb = rows / 128;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = rr + 16 * i;
        const uint2 c = quant8p<FMT>(v[i], d);
        if (dbg_cell(r0 + row, c0 + g * 8, 8, rows, cols, status))
            *reinterpret_cast<uint2 *>(q + (r0 + row) * cols + c0 + g * 8) = c;
        if (TRANS) {
            ct[row * 33 + 2 * g] = c.x;
            ct[row * 33 + 2 * g + 1] = c.y;
        }
    }
    if (t == 0) {
        if (dbg_span(rb * ncb + cb, 1, nrb * ncb, status)) s[rb * ncb + cb] = sc;
        if (TRANS && dbg_span(cb * nrb + rb, 1, nrb * ncb, status)) sT[cb * nrb + rb] = sc;
    }
    if (TRANS) {
        __syncthreads();
        store_code_tile_transposed(ct, qT, rows, c0, r0, cols, status);
    }
}

// ---------------------------------------------------------------------------
// On-demand FP8 transpose of a 128x128-block-quantized weight.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_transpose_128x128(const uint8_t *__restrict__ q, const float *__restrict__ s,
                                                           int64_t rows, int64_t cols, uint8_t *__restrict__ qT,
                                                           float *__restrict__ sT, int *status)
{
    __shared__ uint32_t ct[128 * 33];
    const int t = threadIdx.x;
    const int64_t cb = blockIdx.x, rb = blockIdx.y;
    const int64_t r0 = rb * 128, c0 = cb * 128;
    // blockIdx.z: matrix of a batch of equally shaped ones, stored back to back
    q += (int64_t)blockIdx.z * rows * cols;
    qT += (int64_t)blockIdx.z * rows * cols;
    s += (int64_t)blockIdx.z * (rows / 128) * (cols / 128);
    sT += (int64_t)blockIdx.z * (rows / 128) * (cols / 128);
    // 128 rows x 8 chunks of 16 B: 4 chunks per thread
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int idx = t + 256 * k;
        const int row = idx >> 3, ch = idx & 7;
        const uint4 v = ldg_stream(q + (r0 + row) * cols + c0 + ch * 16);
        uint32_t *p = ct + row * 33 + ch * 4;
        p[0] = v.x; p[1] = v.y; p[2] = v.z; p[3] = v.w;
    }
    if (t == 0 && dbg_span(cb * (rows / 128) + rb, 1, (rows / 128) * (cols / 128), status))
        sT[cb * (rows / 128) + rb] = s[rb * (cols / 128) + cb];
    __syncthreads();
    store_code_tile_transposed(ct, qT, rows, c0, r0, cols, status);
}

// ------------------------------------------------------------------ launchers

static int check_launch()
{
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

template <int FMT, int SRC>
static int launch_fused_t(const void *x, const void *dh, int64_t F, int64_t rows, int64_t cols, int64_t ldx, void *q,
                          float *s, void *qT, float *sT, int *status, cudaStream_t st)
{
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done[dev & 63]) {
        if (cudaFuncSetAttribute(k_quant_1x128_fused_t<FMT, SRC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 fused_smem<SRC>()) != cudaSuccess)
            return FP8_ERR_CUDA;
        attr_done[dev & 63] = true;
    }
    const int64_t nunits = (rows / 128) * ((SRC == SRC_X ? cols : F) / 128);
    if (nunits == 0) return FP8_OK;
    const int64_t grid = std::min<int64_t>(nunits, (int64_t)sm_count() * fused_ctas_per_sm<SRC>());
    k_quant_1x128_fused_t<FMT, SRC><<<(unsigned)grid, 256, fused_smem<SRC>(), st>>>(
        static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(dh), F, rows, cols, ldx,
        static_cast<uint8_t *>(q), s, static_cast<uint8_t *>(qT), sT, status);
    return check_launch();
}

int launch_swiglu_quant(const void *gu, const void *dh, int64_t rows, int64_t F, int fmt, void *q, float *s, void *qT,
                        float *sT, int *status, cudaStream_t st)
{
    if (rows == 0 || F == 0) return FP8_OK;
    if (dh == nullptr)   // forward: H [rows][F]
        return fmt == FP8_E5M2 ? launch_fused_t<FP8_E5M2, SRC_SWIGLU_FWD>(gu, nullptr, F, rows, F, 2 * F, q, s, qT, sT, status, st)
                               : launch_fused_t<FP8_E4M3, SRC_SWIGLU_FWD>(gu, nullptr, F, rows, F, 2 * F, q, s, qT, sT, status, st);
    // backward: dGU [rows][2F]
    return fmt == FP8_E5M2 ? launch_fused_t<FP8_E5M2, SRC_SWIGLU_BWD>(gu, dh, F, rows, 2 * F, 2 * F, q, s, qT, sT, status, st)
                           : launch_fused_t<FP8_E4M3, SRC_SWIGLU_BWD>(gu, dh, F, rows, 2 * F, 2 * F, q, s, qT, sT, status, st);
}

template <int FMT>
static int quant_1x128_fmt(const void *x, int64_t rows, int64_t cols, int64_t ldx, void *q, float *s, void *qT,
                           float *sT, int *status, cudaStream_t st)
{
    if (qT) return launch_fused_t<FMT, SRC_X>(x, nullptr, 0, rows, cols, ldx, q, s, qT, sT, status, st);
    constexpr int U = 8;
    const int64_t items = rows * ((cols / 128 + U - 1) / U);
    // one run per half-warp: the block scheduler balances the load (a
    // persistent grid leaves whole runs of imbalance at this size)
    int64_t blocks = (items + 15) / 16;
    const int64_t cap = (int64_t)1 << 20;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_quant_1x128_rows<FMT, U><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const uint16_t *>(x), (uint32_t)rows, (uint32_t)(cols / 128), ldx, static_cast<uint8_t *>(q), s,
        status);
    return check_launch();
}

int launch_quant_1x128(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, void *q, float *s,
                       void *qT, float *sT, int *status, cudaStream_t st)
{
    if (rows == 0 || cols == 0) return FP8_OK;
    return fmt == FP8_E5M2 ? quant_1x128_fmt<FP8_E5M2>(x, rows, cols, ldx, q, s, qT, sT, status, st)
                           : quant_1x128_fmt<FP8_E4M3>(x, rows, cols, ldx, q, s, qT, sT, status, st);
}

int launch_quant_128x128(const void *w, int64_t rows, int64_t cols, int64_t ldw, int fmt, void *q, float *s,
                         void *qT, float *sT, int *status, cudaStream_t st)
{
    if (rows == 0 || cols == 0) return FP8_OK;
    dim3 grid((unsigned)(cols / 128), (unsigned)(rows / 128));
    auto W = static_cast<const uint16_t *>(w);
    auto Q = static_cast<uint8_t *>(q);
    auto QT = static_cast<uint8_t *>(qT);
    if (fmt == FP8_E5M2) {
        if (qT) k_quant_128x128<FP8_E5M2, true><<<grid, 256, 0, st>>>(W, rows, cols, ldw, Q, s, QT, sT, status);
        else k_quant_128x128<FP8_E5M2, false><<<grid, 256, 0, st>>>(W, rows, cols, ldw, Q, s, QT, sT, status);
    } else {
        if (qT) k_quant_128x128<FP8_E4M3, true><<<grid, 256, 0, st>>>(W, rows, cols, ldw, Q, s, QT, sT, status);
        else k_quant_128x128<FP8_E4M3, false><<<grid, 256, 0, st>>>(W, rows, cols, ldw, Q, s, QT, sT, status);
    }
    return check_launch();
}

int launch_transpose_128x128(const void *q, const float *s, int64_t rows, int64_t cols, void *qT, float *sT,
                             cudaStream_t st, int batch)
{
    if (rows == 0 || cols == 0 || batch == 0) return FP8_OK;
    dim3 grid((unsigned)(cols / 128), (unsigned)(rows / 128), (unsigned)batch);
    k_transpose_128x128<<<grid, 256, 0, st>>>(static_cast<const uint8_t *>(q), s, rows, cols,
                                              static_cast<uint8_t *>(qT), sT, status_word_ptr());
    return check_launch();
}

}  // namespace fp8fg
