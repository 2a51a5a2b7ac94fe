// moe.cu -- MoE routing with the padded routing map, FP8 dispatch gather, and
// the SwiGLU glue between the up and down projections (sm_103a).
//
// Ling 2.0 FP8 pretraining blog, "FP8 padding routing map": instead of
// padding/unpadding layers around the FP8 GEMM, the routing map itself is
// edited before dispatch so every expert's token count meets the GEMM's
// multiple; the added entries carry router probability 0, so the result is
// mathematically unchanged.  Here the multiple is 128 (the GEMM's M tile and
// the 1x128 scale group), the added entries are the lowest-index tokens not
// already routed to that expert, and the rows of an expert are its tokens in
// ascending order -- all decided on the device, no host round trip.  The
// SwiGLU element math lives in common.cuh, shared with the quantizer that
// computes SwiGLU while loading, so both give the same BF16 values.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

// ---------------------------------------------------------------- top-k

// Unsigned key with the order of the logits (-0 and +0 share one key so they
// tie; NaN gets the lowest key and is chosen last).
__device__ __forceinline__ uint32_t logit_key(float z)
{
    if (z != z) return 0u;
    const uint32_t u = z == 0.0f ? 0u : __float_as_uint(z);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int EPL>
__global__ void __launch_bounds__(256) k_moe_topk(const float *__restrict__ logits, int64_t T, int E, int topk,
                                                  int32_t *__restrict__ topk_idx, float *__restrict__ topk_prob,
                                                  int32_t *__restrict__ counts)
{
    // per-expert counts of this block's choices (E <= 256), merged into
    // counts[] (zeroed by the launcher) at the end
    __shared__ int hist[256];
    for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = w0; t < T; t += nw) {
        float z[EPL];
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = j * 32 + lane;
            z[j] = e < E ? logits[t * E + e] : -INFINITY;
            m = fmaxf(m, z[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (j * 32 + lane < E) sum += expf(z[j] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        // each round: the largest remaining logit, ties to the lower expert
        // index, by two warp reductions on an order-preserving key
        uint32_t taken = 0, my_key = 0, my_idx = 0;   // lane k keeps round k's choice
        for (int k = 0; k < topk; ++k) {
            uint32_t bk = 0, be = 0xffffffffu;
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const int e = j * 32 + lane;
                const uint32_t key = logit_key(z[j]);
                if (e < E && !((taken >> j) & 1u) && key > bk) {
                    bk = key;
                    be = (uint32_t)e;
                }
            }
            const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t bi = __reduce_min_sync(0xffffffffu, bk == mk ? be : 0xffffffffu);
            if (bi < (uint32_t)E && (int)(bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == k) {
                my_key = mk;
                my_idx = bi;
            }
        }
        if (lane < topk) {
            topk_idx[t * topk + lane] = (int32_t)my_idx;
            topk_prob[t * topk + lane] = expf(key_logit(my_key) - m) / sum;
            if (my_idx < (uint32_t)E) atomicAdd(&hist[my_idx], 1);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x)
        if (hist[i]) atomicAdd(&counts[i], hist[i]);
}

// Block-wide exclusive prefix sum of per-thread counts and the total.
__device__ __forceinline__ int block_excl_scan_count(int v, int *warp_tot, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
    total = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        if (w < warp) before += warp_tot[w];
        total += warp_tot[w];
    }
    return before + incl - v;
}

__device__ __forceinline__ int64_t padded_count(int c, int align) { return ((int64_t)c + align - 1) / align * align; }

// One CTA per expert: offset from the padded counts of earlier experts, the
// routing-map edit (first `need` free tokens), and the dispatch rows.  The
// tokens are walked in ascending order, kFillTokens consecutive ones per
// thread and round.
constexpr int kFillThreads = 1024;
constexpr int kFillTokens = 2;

__global__ void __launch_bounds__(kFillThreads) k_moe_fill(const int32_t *__restrict__ topk_idx,
                                                  const float *__restrict__ topk_prob, const int32_t *__restrict__ counts,
                                                  int64_t T, int E, int topk, int align, int64_t Mcap,
                                                  int32_t *__restrict__ offsets, int32_t *__restrict__ row_token,
                                                  float *__restrict__ row_prob, uint8_t *__restrict__ row_is_pad,
                                                  int *status)
{
    __shared__ int warp_tot[kFillThreads / 32];
    __shared__ int64_t red[kFillThreads / 32];
    const int e = blockIdx.x;
    // offset of this expert and the total, from the counts of all experts
    int64_t before = 0, all = 0;
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        const int64_t p = padded_count(counts[i], align);
        if (i < e) before += p;
        all += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = before;
    __syncthreads();
    int64_t off = 0;
    for (int w = 0; w < kFillThreads / 32; ++w) off += red[w];
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = all;
    __syncthreads();
    int64_t total = 0;
    for (int w = 0; w < kFillThreads / 32; ++w) total += red[w];

    const int c = counts[e];
    const int64_t need = padded_count(c, align) - c;
    if (threadIdx.x == 0) {
        offsets[e] = (int32_t)off;
        if (e == E - 1) {
            offsets[E] = (int32_t)total;
            if (total > Mcap) set_status(status, FP8_ERR_INVALID_ARG);
        }
    }
    // The padding entries are the first `need` tokens not routed to e, and the
    // rows are the members in token order, so with r_t = tokens before t
    // routed to e (and t - r_t free ones): a routed token's row is
    // off + r_t + min(need, t - r_t), a free token is padding iff
    // t - r_t < need, and then its row is off + t.  One block-wide scan of
    // the routed counts per round of kFillThreads x kFillTokens tokens.
    if (threadIdx.x == 0 && need > T - c) set_status(status, FP8_ERR_INVALID_ARG);   // too few free tokens
    // which of token t's choices is e (-1: none); top-8 rows are read as two
    // coalesced 16-byte loads when aligned
    const bool vec8 = topk == 8 && (reinterpret_cast<uintptr_t>(topk_idx) & 15u) == 0;
    auto choices = [&](int64_t t, int4 &a, int4 &b) {
        if (t < T && vec8) {
            a = __ldg(reinterpret_cast<const int4 *>(topk_idx + t * 8));
            b = __ldg(reinterpret_cast<const int4 *>(topk_idx + t * 8) + 1);
        } else if (t < T) {
            int v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = k < topk ? __ldg(topk_idx + t * topk + k) : -1;
            a = make_int4(v[0], v[1], v[2], v[3]);
            b = make_int4(v[4], v[5], v[6], v[7]);
        } else {
            a = b = make_int4(-1, -1, -1, -1);
        }
    };
    int64_t r_prev = 0;
    int4 cv[kFillTokens][2];
#pragma unroll
    for (int i = 0; i < kFillTokens; ++i) choices((int64_t)threadIdx.x * kFillTokens + i, cv[i][0], cv[i][1]);
    for (int64_t t0 = 0; t0 < T; t0 += (int64_t)kFillThreads * kFillTokens) {
        const int64_t tb = t0 + (int64_t)threadIdx.x * kFillTokens;
        int k_hit[kFillTokens];
#pragma unroll
        for (int i = 0; i < kFillTokens; ++i) {
            const int v[8] = {cv[i][0].x, cv[i][0].y, cv[i][0].z, cv[i][0].w,
                              cv[i][1].x, cv[i][1].y, cv[i][1].z, cv[i][1].w};
            k_hit[i] = -1;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (v[k] == e) k_hit[i] = k;
        }
        // the next iteration's loads fly during the scan
#pragma unroll
        for (int i = 0; i < kFillTokens; ++i)
            choices(tb + (int64_t)kFillThreads * kFillTokens + i, cv[i][0], cv[i][1]);
        int nr = 0;
#pragma unroll
        for (int i = 0; i < kFillTokens; ++i) nr += k_hit[i] >= 0;
        int nround = 0;
        int64_t rt = r_prev + block_excl_scan_count(nr, warp_tot, nround);
#pragma unroll
        for (int i = 0; i < kFillTokens; ++i) {
            const int64_t t = tb + i;
            const bool routed = k_hit[i] >= 0;
            const int64_t ft = t - rt;
            if (t < T && (routed || ft < need)) {
                const int64_t r = off + (routed ? rt + (ft < need ? ft : need) : t);
                if (r < Mcap) {
                    row_token[r] = (int32_t)t;
                    row_prob[r] = routed ? topk_prob[t * topk + k_hit[i]] : 0.0f;
                    if (row_is_pad) row_is_pad[r] = routed ? 0 : 1;
                }
            }
            rt += routed;
        }
        r_prev += nround;
    }
    // rows past the last expert
    for (int64_t r = total + (int64_t)e * blockDim.x + threadIdx.x; r < Mcap; r += (int64_t)E * blockDim.x) {
        row_token[r] = -1;
        row_prob[r] = 0.0f;
        if (row_is_pad) row_is_pad[r] = 0;
    }
}

// ---------------------------------------------------------------- gather

// One warp per dispatched row: K FP8 bytes and K/128 scales of its token.
// Each lane has its 16-byte vectors of a row (four per 2048 bytes) and its
// scale in flight at once before any is stored (35.6 against 36.9 us for
// one load and store at a time on 73728 rows x 2048; the bulk-copy engine
// through per-lane shared buffers measured 37.0 us, and loads without L1
// allocation with streaming stores 42.8 us).
__global__ void __launch_bounds__(256) k_moe_gather(const uint8_t *__restrict__ q, const float *__restrict__ s,
                                                    int64_t T, int64_t K, const int32_t *__restrict__ row_token,
                                                    const int32_t *__restrict__ offsets, int E, int64_t Mcap,
                                                    uint8_t *__restrict__ qg, float *__restrict__ sg, int *status)
{
    constexpr int U = 4;
    const int lane = threadIdx.x & 31;
    const int64_t total = min((int64_t)offsets[E], Mcap);
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t nv = K / 16, nkb = K / 128;
    for (int64_t r = w0; r < total; r += nw) {
        const int64_t t = row_token[r];
        if (t < 0 || t >= T) continue;
        const uint4 *src = reinterpret_cast<const uint4 *>(q + t * K);
        uint4 *dst = reinterpret_cast<uint4 *>(qg + r * K);
        for (int64_t i0 = 0; i0 < nv; i0 += 32 * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + 32 * u + lane;
                if (i < nv) v[u] = src[i];
            }
            float sc = 0.0f;
            const int64_t kb = i0 / 8 + lane;   // this round's scales: 32 U vectors = 4 U chunks of 128
            const bool has_sc = lane < 4 * U && kb < nkb;
            if (has_sc) sc = s[kb * T + t];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + 32 * u + lane;
                if (i < nv && dbg_cell(r, i * 16, 16, Mcap, K, status)) dst[i] = v[u];
            }
            if (has_sc && dbg_cell(kb, r, 1, nkb, Mcap, status)) sg[kb * Mcap + r] = sc;
        }
    }
}

// ---------------------------------------------------------------- SwiGLU

__global__ void __launch_bounds__(256) k_swiglu_fwd(const uint16_t *__restrict__ gu, int64_t rows, int64_t F,
                                                    uint16_t *__restrict__ h, int *status)
{
    const int64_t nvec = rows * (F / 8);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / (F / 8), j = (i - r * (F / 8)) * 8;
        const uint4 g4 = *reinterpret_cast<const uint4 *>(gu + r * 2 * F + j);
        const uint4 u4 = *reinterpret_cast<const uint4 *>(gu + r * 2 * F + F + j);
        const uint4 hv = swiglu8(g4, u4);
        if (dbg_cell(r, j, 8, rows, F, status)) *reinterpret_cast<uint4 *>(h + r * F + j) = hv;
    }
}

__global__ void __launch_bounds__(256) k_swiglu_bwd(const uint16_t *__restrict__ gu, const uint16_t *__restrict__ dh,
                                                    int64_t rows, int64_t F, uint16_t *__restrict__ dgu, int *status)
{
    const int64_t nvec = rows * (F / 8);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / (F / 8), j = (i - r * (F / 8)) * 8;
        const uint4 g4 = *reinterpret_cast<const uint4 *>(gu + r * 2 * F + j);
        const uint4 u4 = *reinterpret_cast<const uint4 *>(gu + r * 2 * F + F + j);
        const uint4 d4 = *reinterpret_cast<const uint4 *>(dh + r * F + j);
        uint4 dg4, du4;
        swiglu_grad8(g4, u4, d4, dg4, du4);
        if (dbg_cell(r, j, 8, rows, 2 * F, status) && dbg_cell(r, F + j, 8, rows, 2 * F, status)) {
            *reinterpret_cast<uint4 *>(dgu + r * 2 * F + j) = dg4;
            *reinterpret_cast<uint4 *>(dgu + r * 2 * F + F + j) = du4;
        }
    }
}

// ------------------------------------------------------------------ launchers

static int check_launch() { return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

int launch_moe_route_pad(const float *logits, int64_t T, int E, int topk, int align, int64_t Mcap, int32_t *topk_idx,
                         float *topk_prob, int32_t *counts, int32_t *offsets, int32_t *row_token, float *row_prob,
                         uint8_t *row_is_pad, int *status, cudaStream_t st)
{
    int64_t blocks = (T + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const unsigned b = (unsigned)blocks;
    const int epl = (E + 31) / 32;
    // the top-k kernel also counts each expert's tokens
    if (cudaMemsetAsync(counts, 0, (size_t)E * sizeof(int32_t), st) != cudaSuccess) return FP8_ERR_CUDA;
    if (epl <= 1) k_moe_topk<1><<<b, 256, 0, st>>>(logits, T, E, topk, topk_idx, topk_prob, counts);
    else if (epl <= 2) k_moe_topk<2><<<b, 256, 0, st>>>(logits, T, E, topk, topk_idx, topk_prob, counts);
    else if (epl <= 4) k_moe_topk<4><<<b, 256, 0, st>>>(logits, T, E, topk, topk_idx, topk_prob, counts);
    else k_moe_topk<8><<<b, 256, 0, st>>>(logits, T, E, topk, topk_idx, topk_prob, counts);
    k_moe_fill<<<E, kFillThreads, 0, st>>>(topk_idx, topk_prob, counts, T, E, topk, align, Mcap, offsets, row_token, row_prob,
                                  row_is_pad, status);
    return check_launch();
}

int launch_moe_gather(const void *q, const float *s, int64_t T, int64_t K, const int32_t *row_token,
                      const int32_t *offsets, int E, int64_t Mcap, void *qg, float *sg, cudaStream_t st)
{
    int64_t blocks = (Mcap + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_moe_gather<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint8_t *>(q), s, T, K, row_token, offsets, E,
                                                   Mcap, static_cast<uint8_t *>(qg), sg, status_word_ptr());
    return check_launch();
}

int launch_swiglu_fwd(const void *gu, int64_t rows, int64_t F, void *h, cudaStream_t st)
{
    const int64_t nvec = rows * (F / 8);
    if (nvec == 0) return FP8_OK;
    int64_t blocks = (nvec + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    k_swiglu_fwd<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t *>(gu), rows, F,
                                                   static_cast<uint16_t *>(h), status_word_ptr());
    return check_launch();
}

int launch_swiglu_bwd(const void *gu, const void *dh, int64_t rows, int64_t F, void *dgu, cudaStream_t st)
{
    const int64_t nvec = rows * (F / 8);
    if (nvec == 0) return FP8_OK;
    int64_t blocks = (nvec + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    k_swiglu_bwd<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t *>(gu),
                                                   static_cast<const uint16_t *>(dh), rows, F,
                                                   static_cast<uint16_t *>(dgu), status_word_ptr());
    return check_launch();
}

}  // namespace fp8fg
