// gemm.cu -- block-scaled / per-tensor / grouped FP8 GEMM on the sm_103a
// tensor cores (tcgen05), D = A . B^T with A [M][K] and B [N][K] K-major.
//
// Method (Ling 2.0 FP8 pretraining blog, "Where does the error come from?":
// an FP8 GEMM whose accumulator is kept in FP32 adds negligible error;
// "Fine-grained quantization": one scale per 1x128 activation tile / 128x128
// weight block): every 128-deep K chunk is multiplied on the tensor cores into
// its own FP32 accumulator in tensor memory, then promoted into an FP32
// running sum in registers with the chunk's two scales:
//     acc[m][n] += sA(m, kb) * sB(n, kb) * P_kb[m][n].
// For per-tensor scales (the coarse delayed-scaling recipe) the whole K is
// accumulated in tensor memory and sA*sB applied once.  MXFP8 (power-of-two
// scales per 32-deep block of every row) needs no promotion in registers:
// the tensor cores apply the scales themselves (kind::mxf8f6f4.block_scale)
// and the whole K accumulates in one tensor-memory accumulator.
//
// Structure (one persistent CTA per SM, 384 threads = 3 warpgroups):
//   warp 0      TMA producer: A tile 128x128 B and B tile BNx128 B per stage,
//               128-byte swizzle, STAGES-deep ring of shared-memory stages.
//   warp 1      owns the tensor memory (2 accumulators of BN columns) and
//               issues tcgen05.mma kind::f8f6f4 (M=128, N=BN, K=32, 4 per
//               chunk) from one thread; tcgen05.commit frees the stage and
//               publishes the accumulator.
//   warp 2      scale producer: runs up to 4 chunks ahead and copies each
//               chunk's scales into a shared-memory ring -- the tile's row
//               scales sA(m,kb), and either the two column-half scalars
//               sB(n-block,kb) (128x128 B) or the per-column sB(n,kb) (1x128
//               B) -- so the epilogue never waits on a global load.  (Warp 3
//               idles.)  This warpgroup gives registers away (setmaxnreg.dec).
//   warps 4..11 epilogue, two warpgroups raised to 176 registers (216 for the
//               per-column mode): the tile's FP32 running sum lives in their
//               registers.  With 128x128 B scales each thread owns one row and
//               half of the columns and drains 16 columns per tcgen05.ld /
//               wait (32x32b.x16), promoting them with packed fma.rn.f32x2;
//               with per-column scales each thread owns 4 rows x 32 columns of
//               16x256b fragments and drains 32 columns of one 16-lane half per
//               wait (the small rounds keep the staging registers beside the
//               accumulators).  At the end of a tile BF16 output leaves through
//               swizzled shared memory and TMA stores (K <= 8192), otherwise
//               straight from registers.  The two accumulators alternate per
//               chunk, so the tensor cores fill one while the epilogue drains
//               the other.
// MXFP8 mode: warp 1 first copies each stage's scale words from shared into
// tensor memory (tcgen05.cp) and issues kind::mxf8f6f4.block_scale MMAs;
// the scale words reach shared memory by two bulk copies per stage from the
// producer (tiled codes) or from warp 2, which reorders row-major codes; one
// accumulator per tile, which the epilogue drains at once and hands back
// before it stores the tile.
// Every mbarrier wait is bounded (about 1 s): on a timeout the CTA records
// FP8_ERR_TIMEOUT, tells the other roles through a shared flag, waits for
// its own copies and MMAs in flight (bounded again), frees the tensor memory
// and returns.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8fg {

constexpr int kGemmThreads = 384;
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 4;          // first epilogue warp (warpgroups 1 and 2)
// setmaxnreg of the control warpgroup and of the two epilogue warpgroups,
// per scale mode (the 1x128 x 1x128 epilogue holds per-row and per-column
// scales beside its accumulators)
template <int SBG> struct RegSplit { static constexpr int kCtrl = 144, kEpi = 176; };
template <> struct RegSplit<1> { static constexpr int kCtrl = 64, kEpi = 216; };
template <> struct RegSplit<2> { static constexpr int kCtrl = 128, kEpi = 184; };  // MXFP8: the scale warp prefetches
// the split must fit the registers the CTA is launched with
template <int SBG>
constexpr int regs_needed_at_launch()
{
    return (128 * RegSplit<SBG>::kCtrl + 256 * RegSplit<SBG>::kEpi + kGemmThreads - 1) / kGemmThreads;
}
constexpr int kMaxGroups = 1024;
// Up to this K a BF16 tile is short enough (<= 64 chunks) that storing it
// through shared memory with TMA, at the price of one operand stage, pays:
// measured +5..+41% at K = 768..4096, -3..-5% at K = 14336..28672.
constexpr int64_t kTmaStoreMaxK = 8192;

struct GemmArgs {
    int M, N, K;          // M = rows of A (the capacity for the grouped GEMM)
    const float *sA;      // scale arrays, layouts per granularity
    int64_t ldsA;
    int granA;
    const float *sB;
    int64_t ldsB;
    int64_t sB_group_stride;
    void *D;
    int64_t ldD;
    int out_f32;
    const int32_t *offsets;
    int G;
    int *status;
    int raster_gm;        // M-tiles per raster band (0: N fastest)
    const uint8_t *eA;    // MXFP8: scale exponents [M][K/32] and [N][K/32] (X = 2^(e - 127))
    const uint8_t *eB;
    int64_t ldE;          // K / 32
    int mx_vec;           // MXFP8: rows of exponents 16-byte aligned (16-byte loads of four chunks)
    int mx_tiled;         // MXFP8: exponents in 512-byte tiles, fetched by the TMA producer
};

// Scale modes: the 1x128 recipe with 128x128 B (one scalar per column half)
// and with 1x128 B (one value per column), both promoted in registers; and
// MXFP8 (one power-of-two scale per 32-block of each row of A and of B),
// applied by the tensor cores from scale words staged in tensor memory.
enum { SB_BLOCK = 0, SB_ROW = 1, SB_MX = 2 };
// Grouping of the tiles: none; by rows of A (MoE forward/dgrad: each M tile
// belongs to one expert, whose B it uses); by K (MoE wgrad: each expert's
// output is a full M x N matrix contracted over that expert's K chunks only).
enum { G_NONE = 0, G_ROWS = 1, G_K = 2 };

constexpr int kScaleDepth = 4;     // chunks of scales staged ahead of the epilogue

template <int BN, int STAGES, bool TSTORE, bool MX = false>
struct GemmSmem {
    static constexpr int kA = 128 * 128;
    static constexpr int kB = BN * 128;
    static constexpr int kStage = kA + kB;
    // BF16 output tile staged for the TMA store (4 boxes of 64 columns x 128 rows)
    static constexpr int kStg = TSTORE ? 128 * BN * 2 : 0;
    // per scale slot: row values for the two column halves + BN column values
    static constexpr int kScaleSlotFloats = 2 * 128 + BN;
    // MXFP8: per operand stage, one 32-bit word of four block exponents for
    // each of the 128 rows of A and BN rows of B, in blocks of 128 rows laid
    // out for tcgen05.cp 32x128b.warpx4 (row i at byte 512 (i / 128) +
    // 16 (i % 32) + 4 ((i / 32) % 4))
    static constexpr int kSfStage = (128 + BN) * 4;
    static constexpr int kScaleBytes = MX ? STAGES * kSfStage : kScaleDepth * kScaleSlotFloats * 4;
    // TMEM accumulators of BN columns: for the promotion modes two or four
    // alternating per chunk over all 512 columns; for MXFP8 one (BN = 256) or
    // two (BN = 128) per tile, followed by a ring of scale words, one set per
    // operand stage: A in 4 columns (row m at lane m, column m / 32), B in
    // BN / 32 columns (row n at lane n % 32 of every lane quarter, column n / 32)
    static constexpr int kNbuf = MX ? (BN == 256 ? 1 : 2) : 512 / BN;
    static constexpr int kSfCol0 = kNbuf * BN;
    static constexpr int kSfCols = 4 + BN / 32;
    static_assert(!MX || kSfCol0 + STAGES * kSfCols <= 512, "MXFP8 scale ring beyond the tensor memory");
    static constexpr int kBars = 2 * STAGES + 2 * kNbuf + 1 + 2 * kScaleDepth;
    static constexpr int kCtrl = kBars * 8 + 16;
    static constexpr int kBytes = 1024 + STAGES * kStage + kStg + kScaleBytes + kCtrl + 4 * (kMaxGroups + 1);
    static constexpr int kTmemCols = 512;
};

// Largest g with off[g] <= row (skips empty groups).
__device__ __forceinline__ int group_of_row(const int32_t *off, int G, int row)
{
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= row) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// What one output tile reads and writes; every role decodes tiles with it.
struct TileInfo {
    int a_row;        // first row of the A tile
    int b_row;        // first row of the B tile (in the stacked B for G_ROWS)
    int n0;           // first output column
    int kg0;          // first K chunk (global index into K and the scale arrays)
    int nk;           // K chunks of this tile (0 for an empty group in G_K)
    int grp;          // group
    int64_t out_row;  // first output row
};

template <int BN, int GMODE>
__device__ __forceinline__ TileInfo tile_info(int tile, int num_mt, int num_nt, const GemmArgs &a,
                                              const int32_t *off)
{
    TileInfo t;
    int mt, nt;
    if (GMODE == G_K) {
        const int per = num_mt * num_nt;
        t.grp = tile / per;
        const int rem = tile - t.grp * per;
        mt = rem / num_nt;
        nt = rem - mt * num_nt;
        t.kg0 = off[t.grp] >> 7;
        t.nk = (off[t.grp + 1] - off[t.grp]) >> 7;
        t.out_row = (int64_t)t.grp * a.M + mt * 128;
        t.b_row = nt * BN;
    } else if (GMODE == G_ROWS) {
        mt = tile / num_nt;
        nt = tile - mt * num_nt;
        t.grp = group_of_row(off, a.G, mt * 128);
        t.kg0 = 0;
        t.nk = a.K / 128;
        t.out_row = mt * 128;
        t.b_row = t.grp * a.N + nt * BN;
    } else {
        tile_coords_raster(tile, num_mt, num_nt, a.raster_gm, mt, nt);
        t.grp = 0;
        t.kg0 = 0;
        t.nk = a.K / 128;
        t.out_row = mt * 128;
        t.b_row = nt * BN;
    }
    t.a_row = mt * 128;
    t.n0 = nt * BN;
    return t;
}

template <int NCOL>
__device__ __forceinline__ void store_row(void *D, int64_t ldD, int out_f32, int64_t row, int64_t col0,
                                          const float (&v)[NCOL])
{
    if (out_f32) {
        float *p = static_cast<float *>(D) + row * ldD + col0;
#pragma unroll
        for (int c = 0; c < NCOL; c += 4)
            *reinterpret_cast<float4 *>(p + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
    } else {
        uint16_t *p = static_cast<uint16_t *>(D) + row * ldD + col0;
#pragma unroll
        for (int c = 0; c < NCOL; c += 8) {
            uint4 w;
            w.x = bf16x2_rn(v[c], v[c + 1]);
            w.y = bf16x2_rn(v[c + 2], v[c + 3]);
            w.z = bf16x2_rn(v[c + 4], v[c + 5]);
            w.w = bf16x2_rn(v[c + 6], v[c + 7]);
            *reinterpret_cast<uint4 *>(p + c) = w;
        }
    }
}

// Two adjacent output columns (row, col), (row, col + 1) from a packed pair.
__device__ __forceinline__ void store_pair(void *D, int64_t ldD, int out_f32, int64_t row, int64_t col, uint64_t v)
{
    float lo, hi;
    f2_unpack(v, lo, hi);
    if (out_f32) *reinterpret_cast<float2 *>(static_cast<float *>(D) + row * ldD + col) = make_float2(lo, hi);
    else *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(D) + row * ldD + col) = bf16x2_rn(lo, hi);
}

// MXFP8 scale words of one group of up to four consecutive 128-deep chunks
// [c0, c0 + size) of a tile: w[i] holds, for this lane's row of slot i (rows
// lane + 32 i of A for i < 4, rows lane + 32 (i - 4) of B after), the words of
// the group's chunks in .x .. .w -- one 16-byte load per row when the rows are
// 16-byte aligned and the group is whole, else one 4-byte load per chunk.
template <int BN>
__device__ __forceinline__ void mx_load_group(uint4 (&w)[4 + BN / 32], const GemmArgs &a, const TileInfo &ti, int c0,
                                              int size, int lane)
{
    const bool vec = a.mx_vec && size == 4;
#pragma unroll
    for (int i = 0; i < 4 + BN / 32; ++i) {
        const int64_t r = i < 4 ? ti.a_row + lane + 32 * i : ti.b_row + lane + 32 * (i - 4);
        const uint8_t *p = (i < 4 ? a.eA : a.eB) + r * a.ldE + 4 * c0;
        if (vec) {
            w[i] = __ldg(reinterpret_cast<const uint4 *>(p));
        } else {
            const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
            w[i].x = __ldg(q);
            w[i].y = size > 1 ? __ldg(q + 1) : 0u;
            w[i].z = size > 2 ? __ldg(q + 2) : 0u;
            w[i].w = size > 3 ? __ldg(q + 3) : 0u;
        }
    }
}

// Writes the group's stages [it0, it0 + size) into their shared-memory slots
// in the tcgen05.cp layout, each once its stage is free, and arrives on the
// stage's full barrier.  False on an abort.
template <int BN, int STAGES>
__device__ __forceinline__ bool mx_write_group(const uint4 (&w)[4 + BN / 32], uint32_t it0, int size, uint8_t *sfw,
                                               int sf_stage_bytes, uint64_t *full, uint64_t *empty,
                                               volatile int *abort_flag, int *status, int lane)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j >= size) break;
        const uint32_t it = it0 + j;
        const int s = it % STAGES;
        if (!warp_wait_or_abort(&empty[s], ((it / STAGES) & 1) ^ 1, abort_flag, status)) return false;
        uint4 *dst = reinterpret_cast<uint4 *>(sfw + s * sf_stage_bytes);
#pragma unroll
        for (int b = 0; b < 1 + BN / 128; ++b) {
            const uint32_t *c0 = &w[4 * b].x, *c1 = &w[4 * b + 1].x, *c2 = &w[4 * b + 2].x, *c3 = &w[4 * b + 3].x;
            dst[32 * b + lane] = make_uint4(c0[j], c1[j], c2[j], c3[j]);
        }
        fence_proxy_async_smem();   // visible to the tensor memory copy
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
    }
    return true;
}

template <int BN, int STAGES, bool PROMOTE, int SBG, int GMODE, bool TSTORE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmD, uint32_t idesc, GemmArgs a)
{
    using L = GemmSmem<BN, STAGES, TSTORE, SBG == SB_MX>;
    constexpr int HALF = BN / 2;        // columns per epilogue thread
    constexpr int NP = HALF / 2;        // packed FP32 pairs per epilogue thread
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stg = smem + STAGES * L::kStage;                                  // TMA-store staging
    float *scl = reinterpret_cast<float *>(stg + L::kStg);                    // [kScaleDepth][slot floats]
    uint8_t *sfw = stg + L::kStg;                                             // MXFP8: [STAGES][kSfStage]
    uint64_t *full = reinterpret_cast<uint64_t *>(stg + L::kStg + L::kScaleBytes);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + L::kNbuf;
    uint64_t *mma_done = tempty + L::kNbuf;
    uint64_t *sc_full = mma_done + 1;
    uint64_t *sc_empty = sc_full + kScaleDepth;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sc_empty + kScaleDepth);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *bad_offsets = reinterpret_cast<int *>(tmem_slot + 2);
    volatile int *tile_go = reinterpret_cast<volatile int *>(tmem_slot + 3);
    int32_t *sh_off = reinterpret_cast<int32_t *>(stg + L::kStg + L::kScaleBytes + L::kCtrl);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // MXFP8 with row-major exponents: the stage's scale words arrive
            // from warp 2 beside the TMA bytes
            mbar_init(&full[s], SBG == SB_MX && !a.mx_tiled ? 2 : 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < L::kNbuf; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
        }
        mbar_init(mma_done, 1);
        for (int i = 0; i < kScaleDepth; ++i) {
            mbar_init(&sc_full[i], 1);
            mbar_init(&sc_empty[i], kEpiWarps);
        }
        *abort_flag = 0;
        *bad_offsets = 0;
        fence_barrier_init();
    }
    if (GMODE != G_NONE) {
        for (int i = threadIdx.x; i <= a.G; i += blockDim.x) sh_off[i] = a.offsets[i];
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (TSTORE) prefetch_tensormap(&tmD);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (GMODE != G_NONE && threadIdx.x == 0) {
        bool ok = sh_off[0] == 0;
        for (int i = 0; i < a.G; ++i) ok = ok && (sh_off[i] <= sh_off[i + 1]) && ((sh_off[i + 1] & 127) == 0);
        ok = ok && sh_off[a.G] <= (GMODE == G_K ? a.K : a.M);   // the grouped extent's capacity
        if (!ok) {
            *bad_offsets = 1;
            set_status(a.status, FP8_ERR_INVALID_ARG);
        }
    }
    if (GMODE != G_NONE) __syncthreads();

    const int num_nt = a.N / BN;
    const int num_mt = GMODE == G_ROWS ? sh_off[a.G] / 128 : a.M / 128;
    int ntiles = GMODE == G_K ? a.G * num_mt * num_nt : num_mt * num_nt;
    const int64_t out_rows = GMODE == G_K ? (int64_t)a.G * a.M : (int64_t)a.M;   // rows of D
    if (GMODE != G_NONE && *bad_offsets) ntiles = 0;

    if (warp < kEpiWarp0) {
        regs_dec<RegSplit<SBG>::kCtrl>();
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------- TMA producer
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const TileInfo ti = tile_info<BN, GMODE>(tile, num_mt, num_nt, a, sh_off);
                for (int kb = 0; kb < ti.nk; ++kb) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!wait_or_abort(&empty[s], ph ^ 1, abort_flag, a.status)) { ok = false; break; }
                    uint8_t *st = smem + s * L::kStage;
                    const bool sf_bulk = SBG == SB_MX && a.mx_tiled;
                    mbar_arrive_expect_tx(&full[s], L::kStage + (sf_bulk ? L::kSfStage : 0));
                    tma_load_2d(st, &tmA, &full[s], (ti.kg0 + kb) * 128, ti.a_row);
                    tma_load_2d(st + L::kA, &tmB, &full[s], (ti.kg0 + kb) * 128, ti.b_row);
                    if (sf_bulk) {
                        // MXFP8, tiled exponents: the chunk's 512-byte tile of A's 128 rows
                        // and the BN / 128 consecutive tiles of B's rows, already in the
                        // tcgen05.cp layout
                        const int64_t kc = ti.kg0 + kb;
                        bulk_load(sfw + s * L::kSfStage, a.eA + (kc * (a.M / 128) + ti.a_row / 128) * 512, 512,
                                  &full[s]);
                        bulk_load(sfw + s * L::kSfStage + 512, a.eB + (kc * (a.N / 128) + ti.b_row / 128) * 512,
                                  BN * 4, &full[s]);
                    }
                    ++it;
                }
            }
            // copies still in flight land before the CTA may exit
            const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0;
            for (uint32_t j = first; j < it; ++j) mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1, nullptr);
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------- MMA issuer
            uint32_t it = 0, cc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const int nk = tile_info<BN, GMODE>(tile, num_mt, num_nt, a, sh_off).nk;
                uint32_t buf = cc % L::kNbuf;
                if (!PROMOTE) {
                    if (!wait_or_abort(&tempty[buf], ((cc / L::kNbuf) & 1) ^ 1, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                }
                for (int kb = 0; kb < nk; ++kb) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (PROMOTE) {
                        buf = cc % L::kNbuf;
                        if (!wait_or_abort(&tempty[buf], ((cc / L::kNbuf) & 1) ^ 1, abort_flag, a.status)) { ok = false; break; }
                    }
                    if (!wait_or_abort(&full[s], ph, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(smem + s * L::kStage));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smem + s * L::kStage + L::kA));
                    if (SBG == SB_MX) {
                        // the stage's scale words into its tensor-memory slot (ordered
                        // before the MMAs below), then one block-scaled MMA per
                        // 32-deep block reading byte k of every row's word
                        const uint32_t sf_a = tmem_base + L::kSfCol0 + s * L::kSfCols, sf_b = sf_a + 4;
                        const uint64_t sd = sdesc_rows16(smem_u32(sfw + s * L::kSfStage));
                        tc_cp_32x128b_warpx4(sf_a, sd);
#pragma unroll
                        for (int b = 0; b < BN / 128; ++b) tc_cp_32x128b_warpx4(sf_b + 4 * b, sd + 32 * (1 + b));
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma_mx(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mx_block(idesc, k), sf_a, sf_b,
                                      (k > 0 || kb > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            // advance 32 bytes (K = 32 FP8) inside the 128-byte swizzled row
                            tc_mma_f8f6f4(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc,
                                          (k > 0 || (!PROMOTE && kb > 0)) ? 1u : 0u);
                        }
                    }
                    // the stage goes back to the producer as soon as these MMAs
                    // have read it, whatever the epilogue is doing
                    tc_commit(&empty[s]);
                    if (PROMOTE) {
                        tc_commit(&tfull[buf]);   // one accumulator per chunk
                        ++cc;
                    }
                    ++it;
                }
                if (!ok) break;
                if (!PROMOTE) {
                    tc_commit(&tfull[buf]);
                    ++cc;
                }
            }
            // every MMA issued by this thread completes before the CTA frees TMEM
            tc_commit(mma_done);
            mbar_wait_bounded(mma_done, 0, nullptr);
        } else if (SBG == SB_MX && warp == 2 && !a.mx_tiled) {
            // -------------------------------------------------- MX scale producer
            // The whole warp, in step with the operand stages: per 128-deep stage
            // it writes the 32-bit word of four block exponents of each of the
            // tile's 128 rows of A and BN rows of B ([rows][K/32] bytes) in the
            // tcgen05.cp layout -- lane j stores the words of rows j, j + 32,
            // j + 64, j + 96 of each block of 128 rows as one 16-byte row -- once
            // the stage is free, then arrives on the stage's full barrier (the
            // second of its two arrivals).  The words are loaded a group of four
            // stages at a time (one 16-byte load per row: each row's word sits
            // in a line of its own, so per-stage 4-byte loads cost four times
            // the requests), double-buffered in registers: the next group's
            // loads are in flight while this group is written.
            constexpr int kW = 4 + BN / 32;
            const int nk = a.K / 128, ng = (nk + 3) / 4;   // chunks and groups per tile
            const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
            const int ngroups = my_tiles * ng;
            uint4 w0[kW], w1[kW];
            // group g: tile g / ng of this CTA, chunks [4 (g % ng), +4) of it
#define FP8FG_MX_GROUP(g, tl, q, ti) \
    const int tl = (g) / ng, q = (g) - tl * ng; \
    const TileInfo ti = tile_info<BN, GMODE>(blockIdx.x + tl * gridDim.x, num_mt, num_nt, a, sh_off)
            if (ngroups > 0) {
                FP8FG_MX_GROUP(0, tl, q, ti);
                mx_load_group<BN>(w0, a, ti, 4 * q, min(4, nk - 4 * q), lane);
            }
            for (int g = 0; g < ngroups; g += 2) {
                if (g + 1 < ngroups) {
                    FP8FG_MX_GROUP(g + 1, tl, q, ti);
                    mx_load_group<BN>(w1, a, ti, 4 * q, min(4, nk - 4 * q), lane);
                }
                {
                    FP8FG_MX_GROUP(g, tl, q, ti);
                    if (!mx_write_group<BN, STAGES>(w0, (uint32_t)(tl * nk + 4 * q), min(4, nk - 4 * q), sfw,
                                                    L::kSfStage, full, empty, abort_flag, a.status, lane))
                        break;
                }
                if (g + 1 >= ngroups) break;
                if (g + 2 < ngroups) {
                    FP8FG_MX_GROUP(g + 2, tl, q, ti);
                    mx_load_group<BN>(w0, a, ti, 4 * q, min(4, nk - 4 * q), lane);
                }
                {
                    FP8FG_MX_GROUP(g + 1, tl, q, ti);
                    if (!mx_write_group<BN, STAGES>(w1, (uint32_t)(tl * nk + 4 * q), min(4, nk - 4 * q), sfw,
                                                    L::kSfStage, full, empty, abort_flag, a.status, lane))
                        break;
                }
            }
#undef FP8FG_MX_GROUP
        } else if (PROMOTE && warp == 2 && lane == 0) {
            // -------------------------------------------------- scale producer
            // Slot layout: [0, 128) sA of the tile's rows (1x128 A) or [128]
            // the tile's sA (128x128 A); [256, 256 + BN) sB of the tile's
            // columns (1x128 B) or [256], [257] the sB of the two column halves
            // (128x128 B).  Vectors arrive by bulk copy, scalars are loaded
            // before the slot is free and stored after.
            const bool a_rows = a.granA == FP8_GRAN_1x128;
            uint32_t cs = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const TileInfo ti = tile_info<BN, GMODE>(tile, num_mt, num_nt, a, sh_off);
                const int m0 = ti.a_row, n0 = ti.n0;
                const float *sB = a.sB;
                if (GMODE == G_ROWS) sB += (int64_t)ti.grp * a.sB_group_stride;
                for (int kb = ti.kg0; kb < ti.kg0 + ti.nk; ++kb, ++cs) {
                    const int slot = cs % kScaleDepth;
                    float b0 = 0.0f, b1 = 0.0f, av = 0.0f;
                    if (SBG == SB_BLOCK) {
                        b0 = sB[(int64_t)(n0 >> 7) * a.ldsB + kb];
                        b1 = sB[(int64_t)((n0 + HALF) >> 7) * a.ldsB + kb];
                    }
                    if (!a_rows) av = a.sA[(int64_t)(m0 >> 7) * a.ldsA + kb];
                    if (!wait_or_abort(&sc_empty[slot], ((cs / kScaleDepth) & 1) ^ 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    float *sv = scl + slot * L::kScaleSlotFloats;
                    if (SBG == SB_BLOCK) {
                        sv[256] = b0;
                        sv[257] = b1;
                    }
                    if (!a_rows) sv[128] = av;
                    // the arrive releases the stores above; the copies complete the phase
                    mbar_arrive_expect_tx(&sc_full[slot], (a_rows ? 512u : 0u) + (SBG == SB_ROW ? BN * 4u : 0u));
                    if (a_rows) bulk_load(sv, a.sA + (int64_t)kb * a.ldsA + m0, 512, &sc_full[slot]);
                    if (SBG == SB_ROW) bulk_load(sv + 256, sB + (int64_t)kb * a.ldsB + n0, BN * 4, &sc_full[slot]);
                }
            }
            // copies still in flight land before the CTA may exit
            const uint32_t first = cs > (uint32_t)kScaleDepth ? cs - kScaleDepth : 0;
            for (uint32_t j = first; j < cs; ++j)
                mbar_wait_bounded(&sc_full[j % kScaleDepth], (j / kScaleDepth) & 1, nullptr);
        }
    } else {
        regs_inc<RegSplit<SBG>::kEpi>();
        // ------------------------------------------------------ epilogue
        const int ew = warp - kEpiWarp0;
        const int lg = warp & 3;             // TMEM lane quarter this warp may access
        const int colbase = (ew >> 2) * HALF;
        const int row = lg * 32 + lane;
        const uint32_t tm_lane = tmem_base + ((uint32_t)(lg * 32) << 16);
        // Addresses the chunk loop uses, computed once: barriers and the scale
        // ring as 32-bit shared addresses, this thread's byte offsets inside a
        // scale slot (row scale, column-half scale, the 4 row scales and the
        // column-scale pairs of the 16x256b fragments), and its TMEM columns.
        const uint32_t tfull_a = smem_u32(tfull), tempty_a = smem_u32(tempty);
        const uint32_t scf_a = smem_u32(sc_full), sce_a = smem_u32(sc_empty);
        const uint32_t scl_a = smem_u32(scl);
        const uint32_t off_ra = 4u * (a.granA == FP8_GRAN_1x128 ? row : 128);
        const uint32_t off_rb = 4u * (256 + (colbase >> 7));
        const uint32_t off_rq = 4u * (a.granA == FP8_GRAN_1x128 ? (lg * 32 + (lane >> 2)) : 128);
        const uint32_t rq_step = a.granA == FP8_GRAN_1x128 ? 32u : 0u;
        const uint32_t off_col = 4u * (256 + colbase + 2 * (lane & 3));
        const uint32_t tm_row = tm_lane + colbase;                          // 32x32b: this warp's lanes
        const uint32_t tm_q0 = tm_lane + colbase, tm_q1 = tm_q0 + (16u << 16);   // 16x256b: lanes 0-15, 16-31
        uint32_t cc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const TileInfo ti = tile_info<BN, GMODE>(tile, num_mt, num_nt, a, sh_off);
            const int64_t m0 = ti.out_row;   // output row of the tile
            const int n0 = ti.n0;
            if (PROMOTE) {
                uint64_t acc[NP];
#pragma unroll
                for (int i = 0; i < NP; ++i) acc[i] = 0ull;
                const int nchunks = ti.nk;
                for (int kb = 0; kb < nchunks; ++kb) {
                    const uint32_t buf = cc & (L::kNbuf - 1);
                    const uint32_t slot = cc & (kScaleDepth - 1);
                    const uint32_t bpar = (cc / L::kNbuf) & 1, spar = (cc / kScaleDepth) & 1;
                    if (!warp_wait_a(scf_a + 8 * slot, spar, abort_flag, a.status)) { ok = false; break; }
                    const uint32_t sva = scl_a + slot * (L::kScaleSlotFloats * 4);
                    if (SBG == SB_BLOCK) {
                        // sA * sB of this thread's row and column half
                        const float sr = lds_f32<0>(sva + off_ra) * lds_f32<0>(sva + off_rb);
                        if (!warp_wait_a(tfull_a + 8 * buf, bpar, abort_flag, a.status)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t s2 = f2_pack(sr, sr);
                        const uint32_t tb = tm_row + buf * BN;
                        // 16 columns per wait: the 128 accumulator registers and the
                        // staging registers fit the epilogue's budget with room to spare
                        // (two x32 loads per wait measured 8% slower, x8 loads 13%, and
                        // loading the next 16 columns before the current group's FMAs 12%)
#pragma unroll
                        for (int j = 0; j < HALF / 16; ++j) {
                            uint32_t r0[16];
                            tc_ld_32x32b_x16(tb + j * 16, r0);
                            tc_wait_ld();
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                acc[j * 8 + i] = f2_fma_bits(r0[2 * i], r0[2 * i + 1], s2, acc[j * 8 + i]);
                        }
                    } else {
                        // per-column scales sB(n, kb).  16x256b fragments: each
                        // thread holds rows {16h + q, 16h + q + 8} (q = lane / 4,
                        // h = 0, 1) of its lane quarter and columns 8i + 2(lane % 4)
                        // + {0, 1}, so it reads 1/4 of the column scales.  64
                        // columns of one 16-lane half per wait (x8); 32 per wait
                        // (x4) measured 4% slower on the dense wgrad.
                        uint64_t sa2[4];
#pragma unroll
                        for (int rr = 0; rr < 4; ++rr) {
                            const float v = lds_f32<0>(sva + off_rq + rr * rq_step);
                            sa2[rr] = f2_pack(v, v);
                        }
                        if (!warp_wait_a(tfull_a + 8 * buf, bpar, abort_flag, a.status)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t scol = sva + off_col;
                        static_assert(HALF % 64 == 0, "the per-column drain reads 64 columns per load");
#pragma unroll
                        for (int c4 = 0; c4 < HALF / 64; ++c4) {
                            uint64_t sbv[8];   // column-scale pairs of this thread's 8 eight-column groups
#pragma unroll
                            for (int i = 0; i < 8; ++i) sbv[i] = lds_b64<0>(scol + 256 * c4 + 32 * i);
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                uint32_t p0[32];
                                tc_ld_16x256b_x8((hh ? tm_q1 : tm_q0) + buf * BN + 64 * c4, p0);
                                tc_wait_ld();
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    uint64_t *ac = acc + 8 * c4 + i;
                                    ac[(2 * hh) * (HALF / 8)] = f2_fma(f2_mul_bits(p0[4 * i], p0[4 * i + 1], sbv[i]),
                                                                       sa2[2 * hh], ac[(2 * hh) * (HALF / 8)]);
                                    ac[(2 * hh + 1) * (HALF / 8)] =
                                        f2_fma(f2_mul_bits(p0[4 * i + 2], p0[4 * i + 3], sbv[i]), sa2[2 * hh + 1],
                                               ac[(2 * hh + 1) * (HALF / 8)]);
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive_a(tempty_a + 8 * buf);
                        mbar_arrive_a(sce_a + 8 * slot);
                    }
                    ++cc;
                }
                if (TSTORE) {
                    // The BF16 tile goes to shared memory in the 128-byte-swizzled
                    // layout of the output map (boxes of 64 columns x 128 rows) and
                    // one thread stores it with TMA, so the next tile's drain starts
                    // at once.  Every epilogue warp passes the same three barriers
                    // per tile, aborted or not, and leaves on a shared decision.
                    const bool elected = threadIdx.x == kEpiWarp0 * 32;
                    if (elected) bulk_wait_read_all();   // the previous tile's store has read the buffer
                    named_bar_sync(1, kEpiWarps * 32);
                    if (ok) {
#pragma unroll
                        for (int k = 0; k < HALF / 8; ++k) {
                            const int col = colbase + 8 * k;
                            float f[8];
#pragma unroll
                            for (int e = 0; e < 4; ++e) f2_unpack(acc[4 * k + e], f[2 * e], f[2 * e + 1]);
                            const uint4 w = make_uint4(bf16x2_rn(f[0], f[1]), bf16x2_rn(f[2], f[3]),
                                                       bf16x2_rn(f[4], f[5]), bf16x2_rn(f[6], f[7]));
                            *reinterpret_cast<uint4 *>(stg + (col >> 6) * 16384 + row * 128 +
                                                       ((((col >> 3) & 7) ^ (row & 7)) << 4)) = w;
                        }
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1, kEpiWarps * 32);
                    if (elected) {
                        const int go = *abort_flag == 0;
                        *tile_go = go;
                        if (go) {
#pragma unroll
                            for (int b = 0; b < BN / 64; ++b) tma_store_2d(&tmD, stg + b * 16384, n0 + 64 * b, (int)m0);
                            bulk_commit_group();
                        }
                    }
                    named_bar_sync(1, kEpiWarps * 32);
                    if (!*tile_go) {
                        ok = false;
                        break;
                    }
                    continue;
                }
                if (!ok) break;
                if (SBG == SB_BLOCK) {
                    float v[HALF];
#pragma unroll
                    for (int i = 0; i < NP; ++i) f2_unpack(acc[i], v[2 * i], v[2 * i + 1]);
                    if (dbg_cell((int64_t)m0 + row, (int64_t)n0 + colbase, HALF, out_rows, a.N, a.status))
                        store_row<HALF>(a.D, a.ldD, a.out_f32, (int64_t)m0 + row, (int64_t)n0 + colbase, v);
                } else {
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) {
                        const int64_t orow = (int64_t)m0 + lg * 32 + rr * 8 + (lane >> 2);
#pragma unroll
                        for (int i = 0; i < HALF / 8; ++i) {
                            const int64_t ocol = (int64_t)n0 + colbase + 8 * i + 2 * (lane & 3);
                            if (dbg_cell(orow, ocol, 2, out_rows, a.N, a.status))
                                store_pair(a.D, a.ldD, a.out_f32, orow, ocol, acc[rr * (HALF / 8) + i]);
                        }
                    }
                }
            } else if (SBG == SB_MX) {
                // The tile's accumulator is read into registers at once and handed
                // back, so the next tile's MMAs run while this one is converted
                // and stored.
                const uint32_t buf = cc % L::kNbuf;
                uint32_t r[HALF / 32][32];
                if (warp_wait_or_abort(&tfull[buf], (cc / L::kNbuf) & 1, abort_flag, a.status)) {
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < HALF / 32; ++j) tc_ld_32x32b_x32(tm_row + buf * BN + 32 * j, r[j]);
                    tc_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[buf]);
                    ++cc;
                } else {
                    ok = false;
                }
                if (TSTORE) {
                    // same protocol as the promotion modes' staged store
                    const bool elected = threadIdx.x == kEpiWarp0 * 32;
                    if (elected) bulk_wait_read_all();
                    named_bar_sync(1, kEpiWarps * 32);
                    if (ok) {
#pragma unroll
                        for (int k = 0; k < HALF / 8; ++k) {
                            const int col = colbase + 8 * k;
                            const uint32_t *v = &r[k / 4][8 * (k % 4)];
                            const uint4 w = make_uint4(
                                bf16x2_rn(__uint_as_float(v[0]), __uint_as_float(v[1])),
                                bf16x2_rn(__uint_as_float(v[2]), __uint_as_float(v[3])),
                                bf16x2_rn(__uint_as_float(v[4]), __uint_as_float(v[5])),
                                bf16x2_rn(__uint_as_float(v[6]), __uint_as_float(v[7])));
                            *reinterpret_cast<uint4 *>(stg + (col >> 6) * 16384 + row * 128 +
                                                       ((((col >> 3) & 7) ^ (row & 7)) << 4)) = w;
                        }
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1, kEpiWarps * 32);
                    if (elected) {
                        const int go = *abort_flag == 0;
                        *tile_go = go;
                        if (go) {
#pragma unroll
                            for (int b = 0; b < BN / 64; ++b) tma_store_2d(&tmD, stg + b * 16384, n0 + 64 * b, (int)m0);
                            bulk_commit_group();
                        }
                    }
                    named_bar_sync(1, kEpiWarps * 32);
                    if (!*tile_go) {
                        ok = false;
                        break;
                    }
                    continue;
                }
                if (!ok) break;
#pragma unroll
                for (int j = 0; j < HALF / 32; ++j) {
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[j][i]);
                    if (dbg_cell((int64_t)m0 + row, (int64_t)n0 + colbase + j * 32, 32, out_rows, a.N, a.status))
                        store_row<32>(a.D, a.ldD, a.out_f32, (int64_t)m0 + row, (int64_t)n0 + colbase + j * 32, v);
                }
            } else {
                const uint32_t buf = cc % L::kNbuf;
                const float sab = a.sA[0] * a.sB[0];
                if (!warp_wait_or_abort(&tfull[buf], (cc / L::kNbuf) & 1, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < HALF / 32; ++j) {
                    uint32_t r[32];
                    tc_ld_32x32b_x32(tm_lane + buf * BN + colbase + j * 32, r);
                    tc_wait_ld();
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * sab;
                    if (dbg_cell((int64_t)m0 + row, (int64_t)n0 + colbase + j * 32, 32, out_rows, a.N, a.status))
                        store_row<32>(a.D, a.ldD, a.out_f32, (int64_t)m0 + row, (int64_t)n0 + colbase + j * 32, v);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
                ++cc;
            }
        }
    }

    // the output tiles' TMA stores complete before the CTA exits
    if (TSTORE && threadIdx.x == kEpiWarp0 * 32) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool make_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *ptr, uint64_t inner, uint64_t rows,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapL2promotion l2)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over an FP8 (byte) matrix [rows][inner], box 128 (K) x box_rows,
// 128-byte swizzle (the layout the MMA descriptors expect).
static bool make_map(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t rows, uint32_t box_rows)
{
    return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, inner, rows, inner, 128, box_rows,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// 2-D map over a BF16 output matrix [rows][cols] with row stride ld
// elements: boxes of 64 columns x 128 rows, 128-byte swizzle (the staging
// layout of the epilogue).
static bool make_out_map(CUtensorMap *map, void *ptr, uint64_t cols, uint64_t rows, uint64_t ld)
{
    return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, cols, rows, ld * 2, 64, 128,
                       CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

template <int BN, int STAGES, bool PROMOTE, int SBG, int GMODE, bool TSTORE = false>
static int run_gemm(const CUtensorMap &mA, const CUtensorMap &mB, const CUtensorMap &mD, uint32_t idesc,
                    const GemmArgs &args, int grid, cudaStream_t st)
{
    using L = GemmSmem<BN, STAGES, TSTORE, SBG == SB_MX>;
    static_assert(L::kBytes <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
    auto kern = k_gemm<BN, STAGES, PROMOTE, SBG, GMODE, TSTORE>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done[dev & 63]) {
        // The warpgroups re-split their registers with setmaxnreg; the split
        // only completes if the CTA was launched with at least that many.
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return FP8_ERR_CUDA;
        if (fa.numRegs < regs_needed_at_launch<SBG>()) return FP8_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) != cudaSuccess)
            return FP8_ERR_CUDA;
        attr_done[dev & 63] = true;
    }
    kern<<<grid, kGemmThreads, L::kBytes, st>>>(mA, mB, mD, idesc, args);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

int launch_gemm(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const float *sA, int granA, const void *B,
                int fmtB, const float *sB, int granB, void *D, int out_dtype, int64_t ldD, int *status,
                cudaStream_t st)
{
    if (M == 0 || N == 0) return FP8_OK;
    if (K == 0) {
        const size_t esz = out_dtype == FP8_OUT_F32 ? 4 : 2;
        return cudaMemset2DAsync(D, (size_t)ldD * esz, 0, (size_t)N * esz, (size_t)M, st) == cudaSuccess
                   ? FP8_OK
                   : FP8_ERR_CUDA;
    }
    const int BN = (N % 256 == 0) ? 256 : 128;
    CUtensorMap mA, mB;
    if (!make_map(&mA, A, (uint64_t)K, (uint64_t)M, 128) || !make_map(&mB, B, (uint64_t)K, (uint64_t)N, BN))
        return FP8_ERR_CUDA;
    GemmArgs g{};
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    g.sA = sA;
    g.granA = granA;
    g.ldsA = granA == FP8_GRAN_1x128 ? M : K / 128;
    g.sB = sB;
    g.ldsB = granB == FP8_GRAN_1x128 ? N : K / 128;
    g.D = D;
    g.ldD = ldD;
    g.out_f32 = out_dtype == FP8_OUT_F32;
    g.status = status;
    g.raster_gm = raster_band(M, M * K, N * K);
    const int64_t ntiles = (M / 128) * (N / BN);
    const int grid = (int)std::min<int64_t>(ntiles, sm_count());
    const bool tensor = granA == FP8_GRAN_TENSOR;
    if (BN == 256) {
        const uint32_t idesc = idesc_f8f6f4(fmtA, fmtB, 128, 256);
        if (tensor) return run_gemm<256, 4, false, SB_BLOCK, G_NONE>(mA, mB, mA, idesc, g, grid, st);
        if (granB == FP8_GRAN_1x128) return run_gemm<256, 4, true, SB_ROW, G_NONE>(mA, mB, mA, idesc, g, grid, st);
        if (!g.out_f32 && K <= kTmaStoreMaxK) {
            // BF16 output leaves through shared memory and TMA stores (one
            // operand stage fewer makes room for the staged tile)
            CUtensorMap mD;
            if (!make_out_map(&mD, D, (uint64_t)N, (uint64_t)M, (uint64_t)ldD)) return FP8_ERR_CUDA;
            return run_gemm<256, 3, true, SB_BLOCK, G_NONE, true>(mA, mB, mD, idesc, g, grid, st);
        }
        return run_gemm<256, 4, true, SB_BLOCK, G_NONE>(mA, mB, mA, idesc, g, grid, st);
    } else {
        const uint32_t idesc = idesc_f8f6f4(fmtA, fmtB, 128, 128);
        if (tensor) return run_gemm<128, 6, false, SB_BLOCK, G_NONE>(mA, mB, mA, idesc, g, grid, st);
        if (granB == FP8_GRAN_1x128) return run_gemm<128, 6, true, SB_ROW, G_NONE>(mA, mB, mA, idesc, g, grid, st);
        return run_gemm<128, 6, true, SB_BLOCK, G_NONE>(mA, mB, mA, idesc, g, grid, st);
    }
}

// MXFP8: the tensor cores apply X_A(m, b) * X_B(n, b) = 2^(eA + eB - 254) to
// every 32-deep block (kind::mxf8f6f4.block_scale) and the whole K accumulates
// in tensor memory.
int launch_gemm_mx(int64_t M, int64_t N, int64_t K, const void *A, int fmtA, const uint8_t *eA, const void *B,
                   int fmtB, const uint8_t *eB, bool tiled, void *D, int out_dtype, int64_t ldD, int *status,
                   cudaStream_t st)
{
    if (M == 0 || N == 0) return FP8_OK;
    if (K == 0) {
        const size_t esz = out_dtype == FP8_OUT_F32 ? 4 : 2;
        return cudaMemset2DAsync(D, (size_t)ldD * esz, 0, (size_t)N * esz, (size_t)M, st) == cudaSuccess
                   ? FP8_OK
                   : FP8_ERR_CUDA;
    }
    const int BN = (N % 256 == 0) ? 256 : 128;
    CUtensorMap mA, mB;
    if (!make_map(&mA, A, (uint64_t)K, (uint64_t)M, 128) || !make_map(&mB, B, (uint64_t)K, (uint64_t)N, BN))
        return FP8_ERR_CUDA;
    GemmArgs g{};
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    g.granA = FP8_GRAN_1x128;
    g.D = D;
    g.ldD = ldD;
    g.out_f32 = out_dtype == FP8_OUT_F32;
    g.status = status;
    g.eA = eA;
    g.eB = eB;
    g.ldE = K / 32;
    g.mx_vec = (K % 512 == 0) && (reinterpret_cast<uintptr_t>(eA) % 16 == 0) && (reinterpret_cast<uintptr_t>(eB) % 16 == 0);
    g.mx_tiled = tiled;
    g.raster_gm = raster_band(M, M * K, N * K);
    const int64_t ntiles = (M / 128) * (N / BN);
    const int grid = (int)std::min<int64_t>(ntiles, sm_count());
    const uint32_t idesc = idesc_mxf8f6f4(fmtA, fmtB, 128, BN);
    if (BN == 256) {
        // Tiled codes: four operand stages and stores straight from registers
        // (the epilogue hands the accumulator back before it stores, so the
        // stores overlap the next tile's MMAs): 674 against 686 us with three
        // stages and the TMA-store epilogue on 8192x28672x4096.  Row-major
        // codes: the scale warp's loads share the load/store path with
        // register stores, so the BF16 tile leaves through TMA stores instead
        // (730 against 790 us).
        if (!tiled && !g.out_f32 && K <= kTmaStoreMaxK) {
            CUtensorMap mD;
            if (!make_out_map(&mD, D, (uint64_t)N, (uint64_t)M, (uint64_t)ldD)) return FP8_ERR_CUDA;
            return run_gemm<256, 3, false, SB_MX, G_NONE, true>(mA, mB, mD, idesc, g, grid, st);
        }
        return run_gemm<256, 4, false, SB_MX, G_NONE>(mA, mB, mA, idesc, g, grid, st);
    }
    return run_gemm<128, 6, false, SB_MX, G_NONE>(mA, mB, mA, idesc, g, grid, st);
}

int launch_grouped_gemm(int G, const int32_t *offsets, int64_t Mcap, int64_t N, int64_t K, const void *A,
                        const float *sA, const void *B, const float *sB, void *D, int out_dtype, int64_t ldD,
                        int *status, cudaStream_t st)
{
    if (Mcap == 0 || N == 0 || K == 0) return FP8_OK;
    const int BN = (N % 256 == 0) ? 256 : 128;
    CUtensorMap mA, mB;
    if (!make_map(&mA, A, (uint64_t)K, (uint64_t)Mcap, 128) ||
        !make_map(&mB, B, (uint64_t)K, (uint64_t)G * (uint64_t)N, BN))
        return FP8_ERR_CUDA;
    GemmArgs g{};
    g.M = (int)Mcap;
    g.N = (int)N;
    g.K = (int)K;
    g.sA = sA;
    g.granA = FP8_GRAN_1x128;
    g.ldsA = Mcap;
    g.sB = sB;
    g.ldsB = K / 128;
    g.sB_group_stride = (N / 128) * (K / 128);
    g.D = D;
    g.ldD = ldD;
    g.out_f32 = out_dtype == FP8_OUT_F32;
    g.offsets = offsets;
    g.G = G;
    g.status = status;
    g.raster_gm = 1;
    const int64_t ntiles_max = (Mcap / 128) * (N / BN);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ntiles_max, sm_count()));
    if (BN == 256) {
        const uint32_t idesc = idesc_f8f6f4(FP8_E4M3, FP8_E4M3, 128, 256);
        if (!g.out_f32 && K <= kTmaStoreMaxK) {
            CUtensorMap mD;
            if (!make_out_map(&mD, D, (uint64_t)N, (uint64_t)Mcap, (uint64_t)ldD)) return FP8_ERR_CUDA;
            return run_gemm<256, 3, true, SB_BLOCK, G_ROWS, true>(mA, mB, mD, idesc, g, grid, st);
        }
        return run_gemm<256, 4, true, SB_BLOCK, G_ROWS>(mA, mB, mA, idesc, g, grid, st);
    }
    return run_gemm<128, 6, true, SB_BLOCK, G_ROWS>(mA, mB, mA, idesc_f8f6f4(FP8_E4M3, FP8_E4M3, 128, 128), g, grid,
                                                  st);
}

// MoE wgrad: expert g's D[g] [N][K] contracts the transposed copies AT [N][Mcap]
// and BT [K][Mcap] over the dispatch rows [off[g], off[g+1]) only.
int launch_grouped_wgrad(int G, const int32_t *offsets, int64_t Mcap, int64_t N, int64_t K, const void *AT, int fmtA,
                         const float *sAT, const void *BT, int fmtB, const float *sBT, void *D, int out_dtype,
                         int64_t ldD, int *status, cudaStream_t st)
{
    if (N == 0 || K == 0) return FP8_OK;
    if (Mcap == 0) {   // every expert is empty: D = 0
        const size_t esz = out_dtype == FP8_OUT_F32 ? 4 : 2;
        return cudaMemset2DAsync(D, (size_t)ldD * esz, 0, (size_t)K * esz, (size_t)G * N, st) == cudaSuccess
                   ? FP8_OK
                   : FP8_ERR_CUDA;
    }
    const int BN = (K % 256 == 0) ? 256 : 128;
    CUtensorMap mA, mB;
    if (!make_map(&mA, AT, (uint64_t)Mcap, (uint64_t)N, 128) || !make_map(&mB, BT, (uint64_t)Mcap, (uint64_t)K, BN))
        return FP8_ERR_CUDA;
    GemmArgs g{};
    g.M = (int)N;        // rows of each expert's output
    g.N = (int)K;        // columns of each expert's output
    g.K = (int)Mcap;     // contraction capacity; expert g uses [off[g], off[g+1])
    g.sA = sAT;
    g.granA = FP8_GRAN_1x128;
    g.ldsA = N;
    g.sB = sBT;
    g.ldsB = K;
    g.D = D;
    g.ldD = ldD;
    g.out_f32 = out_dtype == FP8_OUT_F32;
    g.offsets = offsets;
    g.G = G;
    g.status = status;
    g.raster_gm = 1;
    const int64_t ntiles = (int64_t)G * (N / 128) * (K / BN);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ntiles, sm_count()));
    const uint32_t idesc = idesc_f8f6f4(fmtA, fmtB, 128, BN);
    if (BN == 256) return run_gemm<256, 4, true, SB_ROW, G_K>(mA, mB, mA, idesc, g, grid, st);
    return run_gemm<128, 6, true, SB_ROW, G_K>(mA, mB, mA, idesc, g, grid, st);
}

}  // namespace fp8fg
