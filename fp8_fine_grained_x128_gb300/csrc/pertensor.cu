// pertensor.cu -- per-tensor delayed scaling with fused monitors, and the
// standalone monitor kernels (sm_103a).
//
// Delayed scaling ("FP8 training infrastructure" guide, "Transformer Engine"
// DelayedScaling and "Scaling strategies: delayed scaling"): the scale of
// step t comes from the amax history of earlier steps, so quantization needs
// no grid-wide reduction before it starts.  One persistent pass quantizes
// with s_t, reduces this step's amax and the monitors, and the last CTA to
// finish (atomic ticket, no spinning) writes the history slot, the next scale
// and the step counter, and re-zeroes the workspace.
//
// Monitors (Ling 2.0 FP8 pretraining blog, "Where does the error come
// from?" and the underflow / distortion monitor table): nonzero, underflow
// (nonzero -> +-0), saturated (|x/s| > fmax), distinct values in and out per
// scaling group (+-0 counted once).
//
// Per-tensor current scaling (FP8-RL article, "KV cache compression": one
// scale per cache tensor from its own amax): an amax pass whose last CTA
// writes s = amax / fmax to device memory, then a quantize pass that reads it
// -- two launches, no host round trip.
#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

// Caller-owned workspace for tensor-wide reductions.  Zeroed by the caller
// once; every call that completes leaves it zeroed again.
struct PtWorkspace {
    unsigned int ticket;
    unsigned int amax_bits;
    unsigned int pad[2];
    unsigned int bmx[2048];   // presence of the 65536 BF16 keys
    unsigned int bmq[8];      // presence of the 256 FP8 keys
};

size_t pertensor_workspace_bytes() { return sizeof(PtWorkspace); }

__device__ __forceinline__ uint32_t key_bf16(uint32_t b) { return (b & 0x7FFFu) == 0 ? 0u : b; }
__device__ __forceinline__ uint32_t key_fp8(uint32_t c) { return (c & 0x7Fu) == 0 ? 0u : c; }

__device__ __forceinline__ void bitmap_set(uint32_t *bm, uint32_t key)
{
    const uint32_t bit = 1u << (key & 31);
    uint32_t *w = bm + (key >> 5);
    if (!(*reinterpret_cast<volatile uint32_t *>(w) & bit)) atomicOr(w, bit);
}

struct Counts {
    uint32_t nz = 0, uf = 0, sat = 0;
};

// Quantize 8 BF16 values with one scale and (optionally) account the monitors.
// The distinct-code count of a quantization done here needs no per-element
// code bitmap: q = enc(x / s) is a function of x, so the distinct codes are the
// image of the distinct inputs, which the last CTA derives once from the merged
// presence bitmap.
struct Quot8 {
    float q[8];
};

// IEEE quotients of 8 BF16 values (out of line: the rare path).
__device__ __noinline__ Quot8 quot8_ieee(uint4 v, float s)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    Quot8 r;
    for (int j = 0; j < 4; ++j) {
        r.q[2 * j] = __fdiv_rn(__uint_as_float(w[j] << 16), s);
        r.q[2 * j + 1] = __fdiv_rn(__uint_as_float(w[j] & 0xFFFF0000u), s);
    }
    return r;
}

// NaN codes carry no sign: every byte that encodes a NaN (E4M3 S.1111.111,
// E5M2 S.11111.xx with xx != 0) becomes 0x7F, whatever the sign of x.
template <int FMT>
__device__ __forceinline__ uint32_t canon_nan4(uint32_t w)
{
    constexpr uint32_t kAdd = FMT == FP8_E4M3 ? 0x01010101u : 0x03030303u;   // bit 7 set <=> low 7 bits are a NaN
    const uint32_t nan7 = ((w & 0x7F7F7F7Fu) + kAdd) & 0x80808080u;
    const uint32_t m = (nan7 >> 7) * 0xFFu;                                    // 0xFF in every NaN byte
    return (w & ~m) | (m & 0x7F7F7F7Fu);
}

template <int FMT, bool STATS>
__device__ __forceinline__ uint2 quant8_mon(uint4 v, const Divider2 &d, Counts &c, uint8_t *seen)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float qv[8];
    if (d.fast) {
#pragma unroll
        for (int j = 0; j < 4; ++j) d.fast_div(w[j], qv[2 * j], qv[2 * j + 1]);
    } else {
        const Quot8 r = quot8_ieee(v, d.s);
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] = r.q[e];
    }
    uint2 out;
    out.x = cvt2<FMT>(qv[0], qv[1]) | (cvt2<FMT>(qv[2], qv[3]) << 16);
    out.y = cvt2<FMT>(qv[4], qv[5]) | (cvt2<FMT>(qv[6], qv[7]) << 16);
    if (has_nan_code<FMT>(out.x) || has_nan_code<FMT>(out.y)) {
        // x NaN, x = +-Inf, or x / s overflowed in the fast division (the
        // scale comes from earlier steps): the IEEE quotients decide
        const Quot8 r = quot8_ieee(v, d.s);
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] = r.q[e];
        out.x = canon_nan4<FMT>((cvt2<FMT>(qv[0], qv[1]) | (cvt2<FMT>(qv[2], qv[3]) << 16)) | sign_bits4(v.x, v.y));
        out.y = canon_nan4<FMT>((cvt2<FMT>(qv[4], qv[5]) | (cvt2<FMT>(qv[6], qv[7]) << 16)) | sign_bits4(v.z, v.w));
    }
    if (STATS) {
        // four elements at a time: bit 7 of byte i flags element i
        constexpr uint32_t kMaxMag = (FMT == FP8_E4M3 ? 0x7Eu : 0x7Bu) * 0x01010101u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t w0 = w[2 * h], w1 = w[2 * h + 1], cw = h ? out.y : out.x;
            const uint32_t nzb = __byte_perm((w0 & 0x7FFF7FFFu) + 0x7FFF7FFFu, (w1 & 0x7FFF7FFFu) + 0x7FFF7FFFu,
                                             0x7531) & 0x80808080u;                       // x != +-0
            const uint32_t zc = ~((cw & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) & 0x80808080u;       // code +-0
            c.nz += __popc(nzb);
            c.uf += __popc(nzb & zc);
            // |x/s| > fmax only where the code saturated to the largest magnitude
            const uint32_t y = (cw & 0x7F7F7F7Fu) ^ kMaxMag;
            if ((y - 0x01010101u) & ~y & 0x80808080u) {
                const float fm = fmax_of(FMT);
#pragma unroll
                for (int e = 0; e < 4; ++e) c.sat += fabsf(qv[4 * h + e]) > fm;
            }
        }
        // presence of the raw BF16 patterns, one byte each (a plain store, no
        // read or branch); +0 and -0 are merged in the count
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            seen[w[j] & 0xFFFFu] = 1;
            seen[w[j] >> 16] = 1;
        }
    }
    return out;
}

// Block-wide sum / max of per-thread values (256 threads), result in thread 0.
__device__ __forceinline__ uint32_t block_reduce_sum(uint32_t v, uint32_t *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = 0;
    if (threadIdx.x == 0)
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r += red[i];
    return r;
}

__device__ __forceinline__ uint32_t block_reduce_max(uint32_t v, uint32_t *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = 0;
    if (threadIdx.x == 0)
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = max(r, red[i]);
    return r;
}

// Merges this CTA's counts and presence bitmaps into the stats / workspace,
// takes a ticket, and returns true in every thread of the last CTA.
template <bool STATS>
__device__ bool merge_and_ticket(const Counts &c, uint32_t amax, const uint32_t *bmx, const uint32_t *bmq,
                                 fp8_stats_t *stats, PtWorkspace *ws, uint32_t *red, int *is_last)
{
    const uint32_t a = block_reduce_max(amax, red);
    if (threadIdx.x == 0) atomicMax(&ws->amax_bits, a);
    if (STATS) {
        const uint32_t nz = block_reduce_sum(c.nz, red);
        const uint32_t uf = block_reduce_sum(c.uf, red);
        const uint32_t sat = block_reduce_sum(c.sat, red);
        if (threadIdx.x == 0) {
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->nonzero), (unsigned long long)nz);
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->underflow), (unsigned long long)uf);
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->saturated), (unsigned long long)sat);
        }
        for (int i = threadIdx.x; i < 2048; i += blockDim.x)
            if (bmx[i]) atomicOr(&ws->bmx[i], bmx[i]);
        if (threadIdx.x < 8 && bmq[threadIdx.x]) atomicOr(&ws->bmq[threadIdx.x], bmq[threadIdx.x]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *is_last = (atomicAdd(&ws->ticket, 1u) == gridDim.x - 1);
    __syncthreads();
    return *is_last != 0;
}

// In the last CTA of a delayed-scaling step: the codes of the distinct inputs
// are marked in the workspace's code bitmap before the counts are taken, one
// key at a time (the path for scales outside (0, Inf)).
template <int FMT>
__device__ void mark_codes_per_key(PtWorkspace *ws, const Divider2 &d)
{
    uint32_t m[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // this thread's 256-bit code set
    for (int i = threadIdx.x; i < 2048; i += blockDim.x) {
        uint32_t w = __ldcg(&ws->bmx[i]);
        while (w) {
            const int bit = __ffs(w) - 1;
            w &= w - 1;
            const uint32_t key = (uint32_t)i * 32 + bit;      // BF16 bits (+-0 folded to +0)
            float lo, hi;
            d(key, lo, hi);                                   // the key is the low half of the word
            if (lo != lo) lo = __fdiv_rn(__uint_as_float(key << 16), d.s);   // overflow, Inf or NaN
            const uint32_t code = key_fp8(canon_nan4<FMT>(cvt2<FMT>(lo, lo) & 0xFFu) & 0xFFu);
#pragma unroll
            for (int j = 0; j < 8; ++j) m[j] |= ((code >> 5) == (uint32_t)j) ? (1u << (code & 31)) : 0u;
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m[j] |= __shfl_xor_sync(0xffffffffu, m[j], o);
        if ((threadIdx.x & 31) == 0 && m[j]) atomicOr(&ws->bmq[j], m[j]);
    }
    __syncthreads();
}

// The distinct counts of a delayed-scaling step in its last CTA, for a scale s
// in (0, Inf), with the code set found by intervals instead of key by key.
// The code of |x| is a non-decreasing function of |x| over the finite and
// infinite magnitudes 0 .. 0x7F80 (an IEEE quotient by s, then a rounding,
// saturating conversion), so the magnitudes of code c form an interval
// [L_c, L_c+1) and c occurs with sign b exactly when the merged presence
// bitmap holds a key of sign b in it.  128 threads find the interval starts by
// bisection (15 IEEE quotients each) while the bitmap loads are in flight;
// prefix popcounts give each interval's key count in O(1).  NaN keys, whose
// code is the conversion's NaN code, are checked per sign apart.  The
// bitmap is read once: counted, copied to shared memory and zeroed for the
// next call.  Shared scratch: words[2048], pre[2049], L[129], cq[8].
template <int FMT>
__device__ void delayed_distinct_by_intervals(PtWorkspace *ws, float s, fp8_stats_t *stats, uint32_t *words,
                                              uint32_t *pre, uint32_t *L, uint32_t *cq, uint32_t *red)
{
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;   // 256 threads
    uint32_t wv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) wv[j] = __ldcg(&ws->bmx[8 * t + j]);
    if (t < 8) cq[t] = 0;
    if (t < 128) {
        uint32_t lo = 0, hi = 0x7F81u;   // L_t: the smallest magnitude whose code is >= t
        while (lo < hi) {
            const uint32_t mid = (lo + hi) >> 1;
            const uint32_t c = cvt2<FMT>(__fdiv_rn(__uint_as_float(mid << 16), s), 0.0f) & 0xFFu;
            if (c >= (uint32_t)t) hi = mid;
            else lo = mid + 1;
        }
        L[t] = lo;
    }
    if (t == 0) L[128] = 0x7F81u;
    uint32_t loc[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        words[8 * t + j] = wv[j];
        ws->bmx[8 * t + j] = 0;
        loc[j] = sum;
        sum += __popc(wv[j]);
    }
    uint32_t incl = sum;   // inclusive scan of the per-thread sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    uint32_t base = incl - sum, total = 0;
    for (int w = 0; w < 8; ++w) {
        if (w < warp) base += red[w];
        total += red[w];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) pre[8 * t + j] = base + loc[j];
    if (t == 255) pre[2048] = base + sum;
    __syncthreads();
    auto below = [&](uint32_t k) -> uint32_t {   // present keys < k, 0 <= k <= 65536
        const uint32_t w = k >> 5, b = k & 31;
        return b ? pre[w] + __popc(words[w] & ((1u << b) - 1u)) : pre[w];
    };
    const uint32_t sg = (uint32_t)t >> 7, c = (uint32_t)t & 127;   // sign, magnitude code
    if (L[c] < L[c + 1] && below((sg << 15) | L[c + 1]) > below((sg << 15) | L[c])) {
        const uint32_t code = key_fp8((sg << 7) | c);
        atomicOr(&cq[code >> 5], 1u << (code & 31));
    }
    if (t < 2 && below(((uint32_t)t << 15) + 0x8000u) > below(((uint32_t)t << 15) | 0x7F81u)) {
        // a NaN key of either sign: its quotient is NaN, whose code is 0x7F
        const float nan = __uint_as_float(((uint32_t)t << 31) | 0x7FC00000u);
        const uint32_t code = key_fp8(canon_nan4<FMT>(cvt2<FMT>(__fdiv_rn(nan, s), 0.0f) & 0xFFu) & 0xFFu);
        atomicOr(&cq[code >> 5], 1u << (code & 31));
    }
    __syncthreads();
    if (t == 0) {
        // +0 and -0 are one value: bit 0 of words 0 and 1024 (keys 0x0000, 0x8000)
        const uint32_t din = total - (words[0] & words[1024] & 1u);
        uint32_t dout = 0;
        for (int j = 0; j < 8; ++j) dout += __popc(cq[j]);
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats->distinct_in), (unsigned long long)din);
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats->distinct_out), (unsigned long long)dout);
        ws->ticket = 0;
    }
}

// In the last CTA: distinct counts from the merged bitmaps, workspace reset.
template <bool STATS>
__device__ void finalize_distinct_and_reset(fp8_stats_t *stats, PtWorkspace *ws, uint32_t *red)
{
    __threadfence();
    if (STATS) {
        uint32_t din = 0, dout = 0;
        // +0 and -0 are one value: bit 0 of words 0 and 1024 (keys 0x0000, 0x8000)
        if (threadIdx.x == 0 && (__ldcg(&ws->bmx[0]) & __ldcg(&ws->bmx[1024]) & 1u)) din = (uint32_t)-1;
        __syncthreads();
        for (int i = threadIdx.x; i < 2048; i += blockDim.x) {
            din += __popc(__ldcg(&ws->bmx[i]));
            ws->bmx[i] = 0;
        }
        if (threadIdx.x < 8) {
            dout = __popc(__ldcg(&ws->bmq[threadIdx.x]));
            ws->bmq[threadIdx.x] = 0;
        }
        din = block_reduce_sum(din, red);
        dout = block_reduce_sum(dout, red);
        if (threadIdx.x == 0) {
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->distinct_in), (unsigned long long)din);
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->distinct_out), (unsigned long long)dout);
        }
    }
    if (threadIdx.x == 0) ws->ticket = 0;
}

// ---------------------------------------------------------------------------
// Delayed-scaling quantization of one tensor, one step.
// ---------------------------------------------------------------------------
template <int FMT, bool TRANS, bool STATS>
__global__ void __launch_bounds__(256, STATS ? 2 : 4) k_pertensor_delayed(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                           int64_t ldx, int hist_len, int margin, int algo,
                                                           float *hist, int32_t *step, float *scale,
                                                           uint8_t *__restrict__ q, uint8_t *__restrict__ qT,
                                                           fp8_stats_t *stats, PtWorkspace *ws, int *status)
{
    __shared__ uint32_t ct[TRANS ? 128 * 33 : 1];
    __shared__ uint32_t bmx[STATS ? 2048 : 1];
    __shared__ uint32_t bmq[8];
    __shared__ uint32_t red[32];
    __shared__ int is_last;
    extern __shared__ __align__(16) uint8_t seen[];   // STATS: one byte per BF16 pattern (64 KB)

    const int t = threadIdx.x;
    const int g = t & 15, rr = t >> 4;
    if (STATS) {
        for (int i = t; i < 65536 / 16; i += 256) reinterpret_cast<uint4 *>(seen)[i] = make_uint4(0, 0, 0, 0);
        if (t < 8) bmq[t] = 0;
    }
    const float s_t = *scale;   // chosen from the amax of earlier steps
    const Divider2 d(s_t);
    __syncthreads();

    Counts c;
    uint32_t amax = 0;
    const int64_t ncb = cols / 128, nrb = (rows + 127) / 128;
    const int64_t ntiles = nrb * ncb;
    // With monitors (two CTAs per SM, held back by the 64 KB presence table)
    // the next tile is loaded into registers while this one is processed.
    uint4 vn[8];
    if (STATS && blockIdx.x < ntiles) {
        const int64_t rbn = blockIdx.x / ncb, cbn = blockIdx.x - rbn * ncb;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t r = rbn * 128 + rr + 16 * i;
            vn[i] = r < rows ? ldg_stream(x + r * ldx + cbn * 128 + g * 8) : make_uint4(0, 0, 0, 0);
        }
    }
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t rb = tile / ncb, cb = tile - rb * ncb;
        const int64_t r0 = rb * 128, c0 = cb * 128;
        uint4 v[8];
        if (STATS) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = vn[i];
            if (tile + gridDim.x < ntiles) {
                const int64_t tn = tile + gridDim.x, rbn = tn / ncb, cbn = tn - rbn * ncb;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int64_t r = rbn * 128 + rr + 16 * i;
                    vn[i] = r < rows ? ldg_stream(x + r * ldx + cbn * 128 + g * 8) : make_uint4(0, 0, 0, 0);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t r = r0 + rr + 16 * i;
                v[i] = r < rows ? ldg_stream(x + r * ldx + c0 + g * 8) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = rr + 16 * i;
            if (r0 + row < rows) {
                amax = max(amax, absmax8(v[i]));
                const uint2 code = quant8_mon<FMT, STATS>(v[i], d, c, seen);
                if (dbg_cell(r0 + row, c0 + g * 8, 8, rows, cols, status))
                    *reinterpret_cast<uint2 *>(q + (r0 + row) * cols + c0 + g * 8) = code;
                if (TRANS) {
                    ct[row * 33 + 2 * g] = code.x;
                    ct[row * 33 + 2 * g + 1] = code.y;
                }
            }
        }
        if (TRANS) {
            __syncthreads();
            // transposed copy: same scale, so exactly q^T
            const int lane = t & 31, warp = t >> 5;
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
                uint8_t *dst = qT + (c0 + 4 * cw) * rows + r0 + 4 * mg;
                if (!dbg_cell(c0 + 4 * cw + 3, r0 + 4 * mg, 4, cols, rows, status)) continue;
                *reinterpret_cast<uint32_t *>(dst) = __byte_perm(t0, t1, 0x5410);
                *reinterpret_cast<uint32_t *>(dst + rows) = __byte_perm(t0, t1, 0x7632);
                *reinterpret_cast<uint32_t *>(dst + 2 * rows) = __byte_perm(t2, t3, 0x5410);
                *reinterpret_cast<uint32_t *>(dst + 3 * rows) = __byte_perm(t2, t3, 0x7632);
            }
            __syncthreads();
        }
    }

    if (STATS) {
        // presence bytes -> presence bits (bytes are 0 or 1)
        __syncthreads();
        for (int i = t; i < 2048; i += 256) {
            const uint4 a = reinterpret_cast<const uint4 *>(seen)[2 * i], b = reinterpret_cast<const uint4 *>(seen)[2 * i + 1];
            const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t bits = 0;
            // bytes b0..b3 of 0 / 1: the product's top byte is b0 + 2 b1 + 4 b2 + 8 b3 (b_i lands
            // on bit 24 + i; every other partial product is below bit 24 and on a bit of its own,
            // or above bit 31)
#pragma unroll
            for (int j = 0; j < 8; ++j) bits |= ((wv[j] * 0x01020408u) >> 24) << (4 * j);
            bmx[i] = bits;
        }
    }
    if (!merge_and_ticket<STATS>(c, amax, bmx, bmq, stats, ws, red, &is_last)) return;

    // ---- last CTA: state update (history slot, next scale, step) ----
    if (STATS && s_t > 0.0f && s_t < __uint_as_float(0x7F800000u)) {
        __threadfence();
        uint32_t *scratch = reinterpret_cast<uint32_t *>(seen);
        delayed_distinct_by_intervals<FMT>(ws, s_t, stats, bmx, scratch, scratch + 2049, scratch + 2049 + 129, red);
    } else {
        if (STATS) {
            __threadfence();
            mark_codes_per_key<FMT>(ws, d);
        }
        finalize_distinct_and_reset<STATS>(stats, ws, red);
    }
    if (t == 0) {
        const uint32_t a = atomicExch(&ws->amax_bits, 0u);
        if (a >= 0x7F80u) {
            // Inf/NaN in this step: report it and leave the state untouched
            set_status(status, FP8_ERR_NONFINITE);
        } else {
            const float amax_t = __uint_as_float(a << 16);
            const int32_t st = *step;
            hist[st % hist_len] = amax_t;
            float m = amax_t;
            if (algo == FP8_AMAX_MAX) {
                m = 0.0f;
                for (int i = 0; i < hist_len; ++i) m = fmaxf(m, hist[i]);
            }
            if (m > 0.0f) {
                const float p2 = __uint_as_float((uint32_t)(127 + margin) << 23);   // 2^margin, exact
                *scale = __fdiv_rn(__fmul_rn(m, p2), fmax_of(FMT));
            }
            *step = st + 1;
        }
    }
}

// ---------------------------------------------------------------------------
// Monitors of an existing quantization.
// ---------------------------------------------------------------------------

// Saturation of a scaling group without a division.  |x / s| rounded to
// binary32 exceeds fmax exactly when the real quotient exceeds
// fmax + ulp(fmax) / 2 (a tie rounds to fmax, whose last significand bit is
// 0), i.e. when |x| > |s| (fmax + ulp(fmax) / 2).  That product has at most
// 24 + 25 significant bits, so it is exact in binary64; the largest BF16 at or
// below it is its toward-zero binary32 rounding with the low 16 bits cut off,
// and |x| exceeds the product exactly when its BF16 magnitude bits exceed
// those.  Returned as the per-half addend of sat_bits, (0x8000 - T) in both
// halves with T = those bits + 1.  Scales of 0 (every nonzero x saturates),
// Inf (only a quotient Inf / Inf = NaN could reach it: none does) and NaN
// (T = 0x8000: none) follow from the same rule.
template <int FMT>
__device__ __forceinline__ uint32_t sat_addend(float s)
{
    const double b = FMT == FP8_E4M3 ? 448.0 + 0x1p-16 : 57344.0 + 0x1p-9;
    const uint32_t hi = __float_as_uint(__double2float_rz(fabs((double)s) * b)) >> 16;
    const uint32_t t = min(hi + 1u, 0x8000u);
    return (0x8000u - t) * 0x00010001u;
}

// Bits 15 and 31: the BF16 halves of w that saturate, T <= |x| <= Inf (a NaN
// x gives a NaN quotient, which never exceeds fmax).  Neither sum carries
// across the halves: each half of the magnitude is at most 0x7FFF.
__device__ __forceinline__ uint32_t sat_bits(uint32_t w, uint32_t addend)
{
    const uint32_t t = w & 0x7FFF7FFFu;
    return (t + addend) & ~(t + 0x007F007Fu) & 0x80008000u;
}

// Bit 7 of byte e: element e of the 4 BF16 values (w0 = x0, x1; w1 = x2, x3)
// from the per-half flags at bits 15 and 31 of f0 / f1.
__device__ __forceinline__ uint32_t halves_to_bytes(uint32_t f0, uint32_t f1)
{
    return __byte_perm(f0, f1, 0x7531) & 0x80808080u;
}

// Per-warp scratch of the 128-element group monitors: a presence bitmap of the
// 65536 BF16 keys and one flag byte per FP8 key.  Both are all zero between
// groups: every group clears exactly what it set.
struct GroupScratch {
    uint32_t bx[2048];
    uint32_t fq[64];
};

// Monitors of one group of 128 elements, 4 per lane: x as BF16 bits
// (elements 0, 1 in xv.x and 2, 3 in xv.y, low half first) and q as FP8 codes
// (byte e = element e); the order of the elements within the group does not
// matter.  Nonzero, underflow and saturation are counted four elements at a
// time on packed flags.  A BF16 key counts as distinct for the lane whose
// atomic OR set its bit first (bitmap word from the key's low 11 bits, bit
// from its top 5: a group's values share a few binades, and this spreads them
// over words and banks); the distinct FP8 keys are the flag bytes set, at the
// code rotated left by one so that +-c share a word (a store of both signs of
// one magnitude is then no bank conflict).
__device__ __forceinline__ void mon_group(uint2 xv, uint32_t qv, uint32_t sat_add, GroupScratch &g, int lane,
                                          uint32_t &nz, uint32_t &uf, uint32_t &sat, uint32_t &din, uint32_t &dout)
{
    const uint32_t n0 = (xv.x & 0x7FFF7FFFu) + 0x7FFF7FFFu;   // bit 15 of a half: that x is nonzero
    const uint32_t n1 = (xv.y & 0x7FFF7FFFu) + 0x7FFF7FFFu;
    const uint32_t nzb = halves_to_bytes(n0, n1);
    const uint32_t qn = (qv & 0x7F7F7F7Fu) + 0x7F7F7F7Fu;      // bit 7 of a byte: that code is nonzero
    nz += __popc(nzb);
    uf += __popc(nzb & ~qn);
    sat += __popc(halves_to_bytes(sat_bits(xv.x, sat_add), sat_bits(xv.y, sat_add)));
    // keys: -0 -> +0 on both sides
    const uint32_t k0 = xv.x & (n0 | 0x7FFF7FFFu), k1 = xv.y & (n1 | 0x7FFF7FFFu);
    const uint32_t kq = qv & (qn | 0x7F7F7F7Fu);
    const uint32_t key[4] = {k0, k0 >> 16, k1, k1 >> 16};     // bits above 15 of the low keys are masked below
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t bit = __funnelshift_l(1u, 1u, key[e] >> 11);   // 1 << bits 11..15 of the key
        din += (atomicOr(&g.bx[key[e] & 2047u], bit) & bit) == 0;
    }
    const uint32_t rq = ((kq << 1) & 0xFEFEFEFEu) | ((kq >> 7) & 0x01010101u);
    uint8_t *fqb = reinterpret_cast<uint8_t *>(g.fq);
    fqb[rq & 0xFFu] = 1;
    fqb[(rq >> 8) & 0xFFu] = 1;
    fqb[(rq >> 16) & 0xFFu] = 1;
    fqb[rq >> 24] = 1;
    __syncwarp();
    uint2 *fq2 = reinterpret_cast<uint2 *>(g.fq);
    const uint2 f = fq2[lane];
    dout += __popc(f.x) + __popc(f.y);                         // flag bytes are 0 or 1
    fq2[lane] = make_uint2(0u, 0u);
#pragma unroll
    for (int e = 0; e < 4; ++e) g.bx[key[e] & 2047u] = 0;
    __syncwarp();
}

__device__ __forceinline__ void warp_stats_flush(fp8_stats_t *stats, int lane, uint32_t nz, uint32_t uf, uint32_t sat,
                                                 uint32_t din, uint32_t dout)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        nz += __shfl_xor_sync(0xffffffffu, nz, o);
        uf += __shfl_xor_sync(0xffffffffu, uf, o);
        sat += __shfl_xor_sync(0xffffffffu, sat, o);
        din += __shfl_xor_sync(0xffffffffu, din, o);
        dout += __shfl_xor_sync(0xffffffffu, dout, o);
    }
    if (lane == 0 && nz + sat + din + dout > 0) {
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats->nonzero), (unsigned long long)nz);
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats->underflow), (unsigned long long)uf);
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats->saturated), (unsigned long long)sat);
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats->distinct_in), (unsigned long long)din);
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats->distinct_out), (unsigned long long)dout);
    }
}

constexpr int kG128Warps = 4;   // 128 threads, 33 KB of group scratch per CTA

__device__ __forceinline__ void clear_group_scratch(GroupScratch &g, int lane)
{
    for (int i = lane; i < 2048; i += 32) g.bx[i] = 0;
    for (int i = lane; i < 64; i += 32) g.fq[i] = 0;
    __syncwarp();
}

// 1x128 groups (one row, 128 consecutive columns): one warp per group.  Each
// warp takes a contiguous range of groups in the order of the scales
// S[C/128][R] (group i = row i % R of column block i / R) and walks it in
// batches of 32: lane j computes the saturation threshold of the batch's
// group j from one coalesced load of scales, and four groups are loaded
// ahead of their processing.
template <int FMT>
__global__ void __launch_bounds__(kG128Warps * 32) k_stats_1x128(const uint16_t *__restrict__ x, int64_t rows,
                                                                 int64_t cols, int64_t ldx,
                                                                 const uint8_t *__restrict__ q,
                                                                 const float *__restrict__ s, fp8_stats_t *stats)
{
    __shared__ GroupScratch scr[kG128Warps];
    const int lane = threadIdx.x & 31;
    GroupScratch &g = scr[threadIdx.x >> 5];
    clear_group_scratch(g, lane);
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t ngroups = rows * (cols / 128);
    const int64_t gbeg = ngroups * warp0 / nwarps, gend = ngroups * (warp0 + 1) / nwarps;
    constexpr int U = 4;
    uint32_t nz = 0, uf = 0, sat = 0, din = 0, dout = 0;
    int64_t cb = gbeg / rows, r = gbeg - cb * rows;
    for (int64_t b0 = gbeg; b0 < gend; b0 += 32) {
        const int n = gend - b0 < 32 ? (int)(gend - b0) : 32;
        const uint32_t add_l = lane < n ? sat_addend<FMT>(s[b0 + lane]) : 0u;
        for (int j = 0; j < n; j += U) {
            uint2 xv[U];
            uint32_t qv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (j + u < n) {
                    xv[u] = __ldcs(reinterpret_cast<const uint2 *>(x + r * ldx + cb * 128) + lane);
                    qv[u] = __ldcs(reinterpret_cast<const uint32_t *>(q + r * cols + cb * 128) + lane);
                }
                if (++r == rows) {
                    r = 0;
                    ++cb;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j + u < n)
                    mon_group(xv[u], qv[u], __shfl_sync(0xffffffffu, add_l, j + u), g, lane, nz, uf, sat, din, dout);
        }
    }
    warp_stats_flush(stats, lane, nz, uf, sat, din, dout);
}

// 128x1 groups (128 rows of one column; q is the transposed copy qT[C][R] and
// s is S[R/128][C]).  A CTA stages 128 rows x 32 columns of x in shared
// memory, transposed, so that every warp reads its columns contiguously; lane
// j computes the saturation threshold of the tile's column j.
template <int FMT>
__global__ void __launch_bounds__(kG128Warps * 32) k_stats_128x1(const uint16_t *__restrict__ x, int64_t rows,
                                                                 int64_t cols, int64_t ldx,
                                                                 const uint8_t *__restrict__ q,
                                                                 const float *__restrict__ s, fp8_stats_t *stats)
{
    constexpr int kPitch = 65;                  // words per staged column: conflict-free transposing stores
    __shared__ GroupScratch scr[kG128Warps];
    __shared__ uint32_t xs[32 * kPitch];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    GroupScratch &g = scr[warp];
    clear_group_scratch(g, lane);
    uint16_t *xs16 = reinterpret_cast<uint16_t *>(xs);
    const int64_t ncs = cols / 32, ntiles = (rows / 128) * ncs;
    uint32_t nz = 0, uf = 0, sat = 0, din = 0, dout = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t mb = tile / ncs, c0 = (tile - mb * ncs) * 32;
        uint4 v[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)                // row p*32 + t/4, columns (t%4)*8 .. +7
            v[p] = ldg_stream(x + (mb * 128 + p * 32 + (t >> 2)) * ldx + c0 + (t & 3) * 8);
        const uint32_t add_l = sat_addend<FMT>(s[mb * cols + c0 + lane]);
        __syncthreads();                           // the previous tile's columns are consumed
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int r = p * 32 + (t >> 2), cc = (t & 3) * 8;
            const uint32_t w[4] = {v[p].x, v[p].y, v[p].z, v[p].w};
#pragma unroll
            for (int k = 0; k < 8; ++k)
                xs16[(cc + k) * (2 * kPitch) + r] = (uint16_t)((k & 1) ? (w[k >> 1] >> 16) : (w[k >> 1] & 0xFFFFu));
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 32 / kG128Warps; ++j) {
            const int c = warp * (32 / kG128Warps) + j;
            const uint2 xv = make_uint2(xs[c * kPitch + 2 * lane], xs[c * kPitch + 2 * lane + 1]);
            const uint32_t qv = __ldcs(reinterpret_cast<const uint32_t *>(q + (c0 + c) * rows + mb * 128) + lane);
            mon_group(xv, qv, __shfl_sync(0xffffffffu, add_l, c), g, lane, nz, uf, sat, din, dout);
        }
    }
    warp_stats_flush(stats, lane, nz, uf, sat, din, dout);
}

// 128x128 blocks (one CTA per block, shared presence bitmaps) and the whole
// tensor as one group (persistent grid, bitmaps merged in the workspace).
template <int FMT, bool TENSOR>
__global__ void __launch_bounds__(256) k_stats_blocks(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                      int64_t ldx, const uint8_t *__restrict__ q,
                                                      const float *__restrict__ s, fp8_stats_t *stats,
                                                      PtWorkspace *ws)
{
    __shared__ uint32_t bmx[2048];
    __shared__ uint32_t bmq[8];
    __shared__ uint32_t red[32];
    __shared__ int is_last;
    const int t = threadIdx.x, g = t & 15, rr = t >> 4;
    const int64_t ncb = cols / 128, nrb = rows / 128, ntiles = ncb * nrb;
    Counts c;
    uint32_t din = 0, dout = 0;
    if (TENSOR) {
        for (int i = t; i < 2048; i += 256) bmx[i] = 0;
        if (t < 8) bmq[t] = 0;
        __syncthreads();
    }
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t rb = tile / ncb, cb = tile - rb * ncb;
        if (!TENSOR) {
            __syncthreads();
            for (int i = t; i < 2048; i += 256) bmx[i] = 0;
            if (t < 8) bmq[t] = 0;
            __syncthreads();
        }
        const uint32_t sat_add = sat_addend<FMT>(TENSOR ? s[0] : s[rb * ncb + cb]);
#pragma unroll 2
        for (int i = 0; i < 8; ++i) {
            const int64_t r = rb * 128 + rr + 16 * i;
            const uint4 v = ldg_stream(x + r * ldx + cb * 128 + g * 8);
            const uint2 qq = *reinterpret_cast<const uint2 *>(q + r * cols + cb * 128 + g * 8);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // four elements at a time, as in mon_group
                const uint32_t w0 = w[2 * h], w1 = w[2 * h + 1], cw = h ? qq.y : qq.x;
                const uint32_t n0 = (w0 & 0x7FFF7FFFu) + 0x7FFF7FFFu, n1 = (w1 & 0x7FFF7FFFu) + 0x7FFF7FFFu;
                const uint32_t nzb = halves_to_bytes(n0, n1);
                const uint32_t qn = (cw & 0x7F7F7F7Fu) + 0x7F7F7F7Fu;
                c.nz += __popc(nzb);
                c.uf += __popc(nzb & ~qn);
                c.sat += __popc(halves_to_bytes(sat_bits(w0, sat_add), sat_bits(w1, sat_add)));
                const uint32_t k0 = w0 & (n0 | 0x7FFF7FFFu), k1 = w1 & (n1 | 0x7FFF7FFFu);
                const uint32_t kq = cw & (qn | 0x7F7F7F7Fu);
                bitmap_set(bmx, k0 & 0xFFFFu);
                bitmap_set(bmx, k0 >> 16);
                bitmap_set(bmx, k1 & 0xFFFFu);
                bitmap_set(bmx, k1 >> 16);
#pragma unroll
                for (int e = 0; e < 4; ++e) bitmap_set(bmq, (kq >> (8 * e)) & 0xFFu);
            }
        }
        if (!TENSOR) {
            __syncthreads();
            for (int i = t; i < 2048; i += 256) din += __popc(bmx[i]);
            if (t < 8) dout += __popc(bmq[t]);
        }
    }
    if (!TENSOR) {
        const uint32_t nz = block_reduce_sum(c.nz, red);
        const uint32_t uf = block_reduce_sum(c.uf, red);
        const uint32_t sat = block_reduce_sum(c.sat, red);
        din = block_reduce_sum(din, red);
        dout = block_reduce_sum(dout, red);
        if (t == 0) {
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->nonzero), (unsigned long long)nz);
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->underflow), (unsigned long long)uf);
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->saturated), (unsigned long long)sat);
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->distinct_in), (unsigned long long)din);
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats->distinct_out), (unsigned long long)dout);
        }
        return;
    }
    if (!merge_and_ticket<true>(c, 0u, bmx, bmq, stats, ws, red, &is_last)) return;
    finalize_distinct_and_reset<true>(stats, ws, red);
    if (t == 0) ws->amax_bits = 0;
}

// ---------------------------------------------------------------------------
// Per-tensor current scaling (FP8-RL article, "KV cache compression": the
// scaling factor of the FP8 KV cache is recomputed from the current tensor
// after every model update).  Pass 1 reduces the tensor's amax and its last
// CTA writes s = amax / fmax to the device (no host round trip); pass 2
// quantizes with that s.  Pass 2 is a programmatic dependent launch: pass 1
// lets it be scheduled as soon as every pass-1 CTA is running, and each pass-2
// thread waits (griddepcontrol.wait: pass 1 complete, its writes visible)
// before it reads s or x or writes q, so only the launch latency overlaps.
//
// Pass 2 re-reads x, which pass 1 has just brought through L2 (129 MB).  With
// plain streaming loads much of a 64 MB tensor is evicted before pass 2 gets
// to it; pass 1 therefore loads with an L2 evict_last policy, and pass 2, as it
// consumes each 128-byte line, puts the line back to normal priority
// (applypriority), so nothing stays pinned for the kernels that follow.  This
// is done only when x is contiguous and 128-byte aligned: then every line
// pass 1 marks starts at one of pass 2's vectors and is reset.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool keep_in_l2(const uint16_t *x, int64_t cols, int64_t ldx)
{
    return ldx == cols && (reinterpret_cast<uintptr_t>(x) & 127u) == 0;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ldg_stream_policy(const void *ptr, uint64_t policy)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr), "l"(policy));
    return v;
}

// Back to normal eviction priority for the line that starts at p (no-op for a
// p inside a line).
__device__ __forceinline__ void l2_priority_normal(const void *p)
{
    if ((reinterpret_cast<uintptr_t>(p) & 127u) == 0)
        asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(p) : "memory");
}

// Contiguous x: every CTA takes kCurVecs consecutive 16-byte vectors, all of
// a thread's loads in flight at once (no serial remainder), and the grid
// covers the tensor in as many waves as it needs.
constexpr int kCurU = 8;
constexpr int64_t kCurVecs = 256 * kCurU;

template <bool KEEP>
__device__ __forceinline__ uint32_t amax_cta(const uint16_t *__restrict__ x, int64_t nvec)
{
    const uint64_t pol = KEEP ? l2_policy_evict_last() : 0;
    const int64_t base = (int64_t)blockIdx.x * kCurVecs + threadIdx.x;
    uint4 v[kCurU];
#pragma unroll
    for (int u = 0; u < kCurU; ++u) {
        const int64_t i = base + u * 256;
        v[u] = make_uint4(0, 0, 0, 0);
        if (i < nvec) v[u] = KEEP ? ldg_stream_policy(x + i * 8, pol) : ldg_stream(x + i * 8);
    }
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < kCurU; ++u) m = max(m, absmax8(v[u]));
    return m;
}

template <int FMT>
__global__ void __launch_bounds__(256) k_amax_scale(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                    int64_t ldx, float *scale, PtWorkspace *ws, int *status)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ uint32_t red[32];
    __shared__ int is_last;
    const int64_t vpr = cols / 8, nvec = rows * vpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t m = 0;
    if (keep_in_l2(x, cols, ldx)) {
        m = amax_cta<true>(x, nvec);
    } else if (ldx == cols) {
        m = amax_cta<false>(x, nvec);
    } else {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
            const int64_t r = i / vpr, c = (i - r * vpr) * 8;
            m = max(m, absmax8(ldg_stream(x + r * ldx + c)));
        }
    }
    const uint32_t a = block_reduce_max(m, red);
    if (threadIdx.x == 0) atomicMax(&ws->amax_bits, a);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(&ws->ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (is_last && threadIdx.x == 0) {
        __threadfence();
        const uint32_t am = __ldcg(&ws->amax_bits);
        if (am >= 0x7F80u) set_status(status, FP8_ERR_NONFINITE);
        *scale = scale_from_amax_bits(am, FMT);
        ws->amax_bits = 0;
        ws->ticket = 0;
    }
}

template <int FMT>
__global__ void __launch_bounds__(256) k_quant_scale(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                     int64_t ldx, const float *scale, uint8_t *__restrict__ q,
                                                     int *status)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const Divider2 d(*scale);
    const int64_t vpr = cols / 8, nvec = rows * vpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (ldx == cols) {   // contiguous: kCurVecs vectors per CTA, as in pass 1
        const bool keep = keep_in_l2(x, cols, ldx);
        const int64_t base = (int64_t)blockIdx.x * kCurVecs + threadIdx.x;
        uint4 v[kCurU];
#pragma unroll
        for (int u = 0; u < kCurU; ++u) {
            const int64_t i = base + u * 256;
            v[u] = make_uint4(0, 0, 0, 0);
            if (i < nvec) v[u] = ldg_stream(x + i * 8);
        }
        if (keep) {
#pragma unroll
            for (int u = 0; u < kCurU; ++u)
                if (base + u * 256 < nvec) l2_priority_normal(x + (base + u * 256) * 8);
        }
#pragma unroll
        for (int u = 0; u < kCurU; ++u) {
            const int64_t i = base + u * 256;
            if (i >= nvec) break;
            const uint2 c = quant8p<FMT>(v[u], d);
            if (dbg_span(i * 8, 8, nvec * 8, status)) *reinterpret_cast<uint2 *>(q + i * 8) = c;
        }
    } else {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
            const int64_t r = i / vpr, c = (i - r * vpr) * 8;
            const uint2 code = quant8p<FMT>(ldg_stream(x + r * ldx + c), d);
            if (dbg_cell(r, c, 8, rows, cols, status)) *reinterpret_cast<uint2 *>(q + r * cols + c) = code;
        }
    }
}

// ---------------------------------------------------------------------------
// Bounded-wait self-test: one thread waits on a barrier nothing arrives at.
// ---------------------------------------------------------------------------
__global__ void k_selftest_wait(uint64_t timeout_ns, int *status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait_bounded(&bar, 0, nullptr, timeout_ns)) set_status(status, FP8_ERR_TIMEOUT);
        // complete the phase so the barrier is left in a clean state
        mbar_arrive(&bar);
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// Index-check self-test: writes 1.0f to buf[0, n_write) through the checked
// store, against a claimed extent of n_claimed elements.  The caller owns all
// n_write elements, so every store lands inside real memory in either build;
// the debug build skips those at and past n_claimed and records the error.
// ---------------------------------------------------------------------------
__global__ void k_selftest_bounds(float *buf, int64_t n_claimed, int64_t n_write, int *status)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_write; i += (int64_t)gridDim.x * blockDim.x)
        if (dbg_span(i, 1, n_claimed, status)) buf[i] = 1.0f;
}

// ------------------------------------------------------------------ launchers

static int check_launch() { return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

template <int FMT, bool TRANS, bool STATS>
static void delayed_launch(int blocks, cudaStream_t st, const void *x, int64_t rows, int64_t cols, int64_t ldx,
                           int hist_len, int margin, int algo, float *hist, int32_t *step, float *scale, void *q,
                           void *qT, void *stats, void *ws, int *status)
{
    constexpr int kSeen = STATS ? 65536 : 0;
    if (STATS) {
        static bool attr_done[64] = {};
        int dev = 0;
        cudaGetDevice(&dev);
        if (!attr_done[dev & 63]) {
            cudaFuncSetAttribute(k_pertensor_delayed<FMT, TRANS, STATS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSeen);
            attr_done[dev & 63] = true;
        }
    }
    k_pertensor_delayed<FMT, TRANS, STATS><<<blocks, 256, kSeen, st>>>(
        static_cast<const uint16_t *>(x), rows, cols, ldx, hist_len, margin, algo, hist, step, scale,
        static_cast<uint8_t *>(q), static_cast<uint8_t *>(qT), static_cast<fp8_stats_t *>(stats),
        static_cast<PtWorkspace *>(ws), status);
}

int launch_pertensor_delayed(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, int hist_len,
                             int margin, int algo, float *hist, int32_t *step, float *scale, void *q, void *qT,
                             void *stats, void *ws, int *status, cudaStream_t st)
{
    const int64_t ntiles = ((rows + 127) / 128) * (cols / 128);
    // with monitors a CTA holds 64 KB of presence bytes: two per SM
    int64_t blocks = (int64_t)sm_count() * (stats ? 2 : 4);
    if (blocks > ntiles) blocks = ntiles;
    if (blocks < 1) blocks = 1;   // an empty tensor still runs the state update
    const int b = (int)blocks;
    const bool tr = qT != nullptr, stt = stats != nullptr;
#define FP8FG_DL(F, T, S) delayed_launch<F, T, S>(b, st, x, rows, cols, ldx, hist_len, margin, algo, hist, step, scale, q, qT, stats, ws, status)
    if (fmt == FP8_E5M2) {
        if (tr) { if (stt) FP8FG_DL(FP8_E5M2, true, true); else FP8FG_DL(FP8_E5M2, true, false); }
        else { if (stt) FP8FG_DL(FP8_E5M2, false, true); else FP8FG_DL(FP8_E5M2, false, false); }
    } else {
        if (tr) { if (stt) FP8FG_DL(FP8_E4M3, true, true); else FP8FG_DL(FP8_E4M3, true, false); }
        else { if (stt) FP8FG_DL(FP8_E4M3, false, true); else FP8FG_DL(FP8_E4M3, false, false); }
    }
#undef FP8FG_DL
    return check_launch();
}

int launch_quant_stats(const void *x, int64_t rows, int64_t cols, int64_t ldx, const void *q, const float *s,
                       int gran, int fmt, void *stats, void *ws, int *status, cudaStream_t st)
{
    (void)status;
    if (rows == 0 || cols == 0) return FP8_OK;
    auto X = static_cast<const uint16_t *>(x);
    auto Q = static_cast<const uint8_t *>(q);
    auto S = static_cast<fp8_stats_t *>(stats);
    auto W = static_cast<PtWorkspace *>(ws);
    if (gran == FP8_GRAN_1x128 || gran == FP8_GRAN_128x1) {
        const bool cols_mode = gran == FP8_GRAN_128x1;
        const int64_t units = cols_mode ? (rows / 128) * (cols / 32) : (rows * (cols / 128) + kG128Warps * 4 - 1) /
                                                                         (kG128Warps * 4);
        const int64_t cap = (int64_t)sm_count() * (cols_mode ? 5 : 6);   // CTAs that fit an SM's shared memory
        const unsigned b = (unsigned)std::max<int64_t>(1, std::min<int64_t>(units, cap));
        if (fmt == FP8_E5M2) {
            if (cols_mode) k_stats_128x1<FP8_E5M2><<<b, kG128Warps * 32, 0, st>>>(X, rows, cols, ldx, Q, s, S);
            else k_stats_1x128<FP8_E5M2><<<b, kG128Warps * 32, 0, st>>>(X, rows, cols, ldx, Q, s, S);
        } else {
            if (cols_mode) k_stats_128x1<FP8_E4M3><<<b, kG128Warps * 32, 0, st>>>(X, rows, cols, ldx, Q, s, S);
            else k_stats_1x128<FP8_E4M3><<<b, kG128Warps * 32, 0, st>>>(X, rows, cols, ldx, Q, s, S);
        }
        return check_launch();
    }
    const int64_t ntiles = (rows / 128) * (cols / 128);
    int64_t blocks = gran == FP8_GRAN_TENSOR ? std::min<int64_t>(ntiles, (int64_t)sm_count() * 4) : ntiles;
    const unsigned b = (unsigned)blocks;
    if (fmt == FP8_E5M2) {
        if (gran == FP8_GRAN_TENSOR) k_stats_blocks<FP8_E5M2, true><<<b, 256, 0, st>>>(X, rows, cols, ldx, Q, s, S, W);
        else k_stats_blocks<FP8_E5M2, false><<<b, 256, 0, st>>>(X, rows, cols, ldx, Q, s, S, W);
    } else {
        if (gran == FP8_GRAN_TENSOR) k_stats_blocks<FP8_E4M3, true><<<b, 256, 0, st>>>(X, rows, cols, ldx, Q, s, S, W);
        else k_stats_blocks<FP8_E4M3, false><<<b, 256, 0, st>>>(X, rows, cols, ldx, Q, s, S, W);
    }
    return check_launch();
}

int launch_pertensor_current(const void *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, float *scale, void *q,
                             void *ws, int *status, cudaStream_t st)
{
    const int64_t nvec = rows * (cols / 8);
    // contiguous x: one CTA per kCurVecs vectors; strided x: a grid-strided loop
    const bool flat = ldx == cols;
    const int64_t flat_grid = std::max<int64_t>(1, (nvec + kCurVecs - 1) / kCurVecs);
    const unsigned ba = (unsigned)(flat ? flat_grid
                                        : std::max<int64_t>(1, std::min<int64_t>((nvec + 255) / 256,
                                                                                 (int64_t)sm_count() * 4)));
    const unsigned bq = (unsigned)(flat ? flat_grid
                                        : std::max<int64_t>(1, std::min<int64_t>((nvec + 255) / 256,
                                                                                 (int64_t)sm_count() * 8)));
    auto X = static_cast<const uint16_t *>(x);
    auto W = static_cast<PtWorkspace *>(ws);
    auto Q = static_cast<uint8_t *>(q);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(bq);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    const float *S = scale;
    cudaError_t e = cudaSuccess;
    if (fmt == FP8_E5M2) {
        k_amax_scale<FP8_E5M2><<<ba, 256, 0, st>>>(X, rows, cols, ldx, scale, W, status);
        if (nvec > 0) e = cudaLaunchKernelEx(&cfg, k_quant_scale<FP8_E5M2>, X, rows, cols, ldx, S, Q, status);
    } else {
        k_amax_scale<FP8_E4M3><<<ba, 256, 0, st>>>(X, rows, cols, ldx, scale, W, status);
        if (nvec > 0) e = cudaLaunchKernelEx(&cfg, k_quant_scale<FP8_E4M3>, X, rows, cols, ldx, S, Q, status);
    }
    if (e != cudaSuccess) return FP8_ERR_CUDA;
    return check_launch();
}

int launch_selftest_wait(int timeout_ms, int *status, cudaStream_t st)
{
    k_selftest_wait<<<1, 32, 0, st>>>((uint64_t)timeout_ms * 1000000ull, status);
    return check_launch();
}

int launch_selftest_bounds(float *buf, int64_t n_claimed, int64_t n_write, int *status, cudaStream_t st)
{
    const int64_t blocks = std::min<int64_t>((n_write + 255) / 256, 1024);
    k_selftest_bounds<<<(unsigned)blocks, 256, 0, st>>>(buf, n_claimed, n_write, status);
    return check_launch();
}

}  // namespace fp8fg
