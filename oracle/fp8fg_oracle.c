/*
 * fp8fg_oracle.c -- plain, slow CPU oracle for the fine-grained FP8 Linear.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * bench's CPU-baseline leg may load this file's library.  It shares no code,
 * header, table or constant generator with the CUDA library, and includes no
 * CUDA header.  Every quantity is computed the obvious way, in FP64 where the
 * definition is a real-valued formula, and in IEEE binary32 exactly where the
 * method fixes binary32 (the scale s = amax / fmax and the quotient x / s).
 *
 * Sources (web pages on FP8 training), cited by title and section:
 *  [FP8-LM]  "FP8-LM: Training FP8 Large Language Models" (paper review),
 *            section "Core formulas": the two FP8 formats (E4M3 forward,
 *            E5M2 gradients) and tensor scaling x_fp8 = Cast_fp8(x / s).
 *  [Ling]    "Ling 2.0 FP8 pretraining" blog: "Where does the error come
 *            from?" (underflow: nonzero -> 0; distortion: nearby values made
 *            equal; FP32-accumulated GEMM), "Fine-grained quantization
 *            (per-tile/block wise scaling)", the underflow/distortion monitor
 *            table ("smaller is better" / "larger is better"), "FP8 on-demand
 *            transpose weight" and "FP8 padding routing map".
 *  [FP8-RL]  FP8-RL article, "Core breakthrough: dynamic weight sync":
 *            128x128 weight blocks with one scale each, E4M3 range [-448,448],
 *            activations quantized dynamically.
 *  [Infra]   "FP8 training infrastructure" guide, "Transformer Engine" and
 *            "Scaling strategies": delayed scaling from an amax history
 *            (margin 0, history 16, max algorithm, HYBRID = E4M3 forward /
 *            E5M2 backward), E4M3 max +-448, E5M2 for gradients.
 *
 * Readings where the pages are silent:
 *  R1  FP8 encode: round to nearest, ties to even mantissa; |v| >= fmax
 *      saturates to +-fmax (never inf/NaN for a finite input); sign kept, so
 *      -0 -> 0x80; NaN -> 0x7F.
 *  R2  s = fp32(amax / fmax); a group whose amax is 0 gets s = 1.
 *  R3  q = enc(fp32(x) / s) with an IEEE binary32 division (divide, not a
 *      multiply by a reciprocal); denormals are kept.
 *  R4  E5M2 max = 57344; E4M3 max = 448.
 *  R5  Delayed scaling: s_0 = 1; at step t quantize with s_t, write amax_t
 *      into history slot t mod L, s_{t+1} = max(history) * 2^margin / fmax
 *      (or the most recent amax for the "most recent" algorithm); if that
 *      amax is 0, s_{t+1} = s_t.  A step whose tensor holds Inf/NaN is
 *      reported and leaves history, scale and step unchanged.
 *  R6  Monitors: underflow = #(x != 0 and q is +-0) ; distortion is reported
 *      as a retention ratio distinct(q) / distinct(x) summed over scaling
 *      groups, +-0 counted as one value on both sides; saturated =
 *      #(|fp32(x)/s| > fmax).
 *  R7  GEMM: D = sum_kb sA*sB * (sum over the 128-chunk of qA*qB), all in
 *      FP64 (exact per chunk for E4M3 x E4M3), rounded once at the end.
 *  R8  Routing: top-k by logit (softmax is monotone), ties to the lower
 *      expert index; pad every expert to a multiple of `align` with the
 *      lowest-index tokens not already routed to it, router prob 0; the rows
 *      of an expert are its tokens in ascending order.
 *  R12 FP8 optimizer states: Adam's m in E4M3 and v in E5M2 (v holds squared
 *      gradients, the widest-ranged quantity), one R2 scale per 128
 *      consecutive parameters; the AdamW update in binary32 in a fixed order
 *      (see orc_adam_fp8_step).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_E4M3 0
#define ORC_E5M2 1

#define ORC_GRAN_1x128 0   /* scales S[cols/128][rows]                       */
#define ORC_GRAN_128x128 1 /* scales S[rows/128][cols/128]                   */
#define ORC_GRAN_TENSOR 2  /* one scale                                      */
#define ORC_GRAN_128x1 3   /* groups of 128 rows in one column; q is [cols][rows],
                              scales S[rows/128][cols]                        */

#define ORC_OK 0
#define ORC_NONFINITE 1
#define ORC_BADARG 2

int orc_version(void) { return 1; }

/* ---------------------------------------------------------------------------
 * Number formats
 * ------------------------------------------------------------------------- */

/* BF16 is the upper half of an IEEE binary32: exact widening. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

typedef struct {
    int mbits;      /* mantissa bits                        */
    int ebits;      /* exponent bits                        */
    int bias;       /* exponent bias                        */
    int emin;       /* exponent of the smallest normal      */
    double fmax;    /* largest finite magnitude             */
    uint8_t maxcode;
} fmt_t;

/* [FP8-LM] "FP8 data formats": E4M3 = 4 exponent + 3 mantissa bits, E5M2 =
 * 5 + 2.  [FP8-RL]/[Infra]: E4M3 max 448 (R4). */
static fmt_t fmt_of(int fmt)
{
    fmt_t f;
    if (fmt == ORC_E5M2) {
        f.mbits = 2; f.ebits = 5; f.bias = 15; f.emin = -14;
        f.fmax = 57344.0; f.maxcode = 0x7B;
    } else {
        f.mbits = 3; f.ebits = 4; f.bias = 7; f.emin = -6;
        f.fmax = 448.0; f.maxcode = 0x7E;
    }
    return f;
}

float orc_fmax(int fmt) { return (float)fmt_of(fmt).fmax; }

/* Decode one FP8 code to its real value. */
double orc_fp8_decode(uint8_t c, int fmt)
{
    fmt_t f = fmt_of(fmt);
    int sign = c >> 7;
    int e = (c >> f.mbits) & ((1 << f.ebits) - 1);
    int m = c & ((1 << f.mbits) - 1);
    double v;
    if (fmt == ORC_E4M3 && e == 15 && m == 7) return NAN;
    if (fmt == ORC_E5M2 && e == 31) {
        if (m != 0) return NAN;
        return sign ? -INFINITY : INFINITY;
    }
    if (e == 0)
        v = ldexp((double)m, f.emin - f.mbits);
    else
        v = ldexp(1.0 + (double)m / (double)(1 << f.mbits), e - f.bias);
    return sign ? -v : v;
}

/* Encode a binary32 value to FP8 (R1): nearest representable value, ties to
 * the even mantissa, saturating at +-fmax. */
uint8_t orc_fp8_encode(float v, int fmt)
{
    fmt_t f = fmt_of(fmt);
    uint8_t sign;
    double a, quantum, r, fl, n, val;
    int e, E;

    if (isnan(v)) return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs((double)v);
    if (a >= f.fmax) return sign | f.maxcode;
    if (a == 0.0) return sign;

    /* a = frac * 2^e with frac in [0.5, 1): floor(log2 a) = e - 1. */
    frexp(a, &e);
    E = e - 1;
    if (E < f.emin) E = f.emin;              /* subnormal binade */
    quantum = ldexp(1.0, E - f.mbits);       /* spacing of codes near a */
    r = a / quantum;                         /* exact: power-of-two scaling */
    fl = floor(r);
    if (r - fl > 0.5)
        n = fl + 1.0;
    else if (r - fl < 0.5)
        n = fl;
    else
        n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;   /* tie: even */
    val = n * quantum;                       /* the chosen value, <= fmax */
    if (val == 0.0) return sign;

    frexp(val, &e);
    E = e - 1;
    if (E < f.emin) {
        /* subnormal: exponent field 0, mantissa counts 2^(emin - mbits) */
        int mant = (int)(val / ldexp(1.0, f.emin - f.mbits));
        return sign | (uint8_t)mant;
    } else {
        int expf = E + f.bias;
        int mant = (int)((val / ldexp(1.0, E) - 1.0) * (double)(1 << f.mbits));
        return sign | (uint8_t)((expf << f.mbits) | mant);
    }
}

void orc_fp8_encode_array(const float *v, int64_t n, int fmt, uint8_t *out)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) out[i] = orc_fp8_encode(v[i], fmt);
}

void orc_fp8_encode_bits_range(uint32_t first, int64_t count, int fmt, uint8_t *out)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < count; ++i) {
        uint32_t u = first + (uint32_t)i;
        float f;
        memcpy(&f, &u, sizeof f);
        out[i] = orc_fp8_encode(f, fmt);
    }
}

/* Round a real value to BF16 (nearest, ties to even), returned as bits. */
uint16_t orc_f64_to_bf16(double v)
{
    double a, quantum, r, fl, n, val;
    int e, E;
    float f;
    uint32_t u;
    uint16_t sign;
    if (isnan(v)) return 0x7FC0;
    sign = signbit(v) ? 0x8000 : 0;
    a = fabs(v);
    if (a == 0.0) return sign;
    frexp(a, &e);
    E = e - 1;
    if (E < -126) E = -126;
    quantum = ldexp(1.0, E - 7);
    r = a / quantum;
    fl = floor(r);
    if (r - fl > 0.5) n = fl + 1.0;
    else if (r - fl < 0.5) n = fl;
    else n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    val = n * quantum;
    if (val >= ldexp(1.0, 128)) return sign | 0x7F80;   /* overflow -> inf */
    f = (float)val;                                      /* exact */
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ---------------------------------------------------------------------------
 * Scaling and quantization
 * ------------------------------------------------------------------------- */

/* R2: s = fp32(amax / fmax), 1 for an all-zero group. */
static float scale_of(float amax, int fmt)
{
    float fm = (float)fmt_of(fmt).fmax;
    if (amax == 0.0f) return 1.0f;
    return amax / fm;
}

/* R3 / [FP8-LM] "Tensor scaling": q = Cast_fp8(x / s). */
static uint8_t quant_one(float x, float s, int fmt)
{
    float quotient = x / s;
    return orc_fp8_encode(quotient, fmt);
}

/* [Ling] "Fine-grained quantization": one scale per 1x128 tile of a row
 * (activations / gradients).  Scales S[cols/128][rows]. */
int orc_quant_1x128(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                    uint8_t *q, float *s)
{
    int64_t r;
    int bad = 0;
    if (cols % 128 != 0 || rows < 0) return ORC_BADARG;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (r = 0; r < rows; ++r) {
        int64_t cb, k;
        for (cb = 0; cb < cols / 128; ++cb) {
            float amax = 0.0f, sc;
            for (k = 0; k < 128; ++k) {
                float v = orc_bf16_to_f32(x[r * ldx + cb * 128 + k]);
                if (!isfinite(v)) bad = 1;
                else if (fabsf(v) > amax) amax = fabsf(v);
            }
            sc = scale_of(amax, fmt);
            s[cb * rows + r] = sc;
            for (k = 0; k < 128; ++k)
                q[r * cols + cb * 128 + k] =
                    quant_one(orc_bf16_to_f32(x[r * ldx + cb * 128 + k]), sc, fmt);
        }
    }
    return bad ? ORC_NONFINITE : ORC_OK;
}

/* The wgrad operand ("grad (transpose)" in [Ling]'s monitor table): the same
 * per-128 quantization, but along the token (row) dimension of x[rows][cols]:
 * qT[c][m] = enc(x[m][c] / sT[m/128][c]), sT[mb][c] = amax of x[mb*128 ..
 * mb*128+127][c] / fmax. */
int orc_quant_128x1_transposed(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx,
                               int fmt, uint8_t *qT, float *sT)
{
    int64_t c;
    int bad = 0;
    if (rows % 128 != 0 || cols < 0) return ORC_BADARG;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (c = 0; c < cols; ++c) {
        int64_t mb, i;
        for (mb = 0; mb < rows / 128; ++mb) {
            float amax = 0.0f, sc;
            for (i = 0; i < 128; ++i) {
                float v = orc_bf16_to_f32(x[(mb * 128 + i) * ldx + c]);
                if (!isfinite(v)) bad = 1;
                else if (fabsf(v) > amax) amax = fabsf(v);
            }
            sc = scale_of(amax, fmt);
            sT[mb * cols + c] = sc;
            for (i = 0; i < 128; ++i)
                qT[c * rows + mb * 128 + i] =
                    quant_one(orc_bf16_to_f32(x[(mb * 128 + i) * ldx + c]), sc, fmt);
        }
    }
    return bad ? ORC_NONFINITE : ORC_OK;
}

/* [FP8-RL] "dynamic weight sync": each 128x128 weight block gets its own
 * scale.  Scales S[rows/128][cols/128]. */
int orc_quant_128x128(const uint16_t *w, int64_t rows, int64_t cols, int64_t ldw, int fmt,
                      uint8_t *q, float *s)
{
    int64_t blk;
    int64_t nrb = rows / 128, ncb = cols / 128;
    int bad = 0;
    if (rows % 128 != 0 || cols % 128 != 0) return ORC_BADARG;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (blk = 0; blk < nrb * ncb; ++blk) {
        int64_t rb = blk / ncb, cb = blk % ncb, i, j;
        float amax = 0.0f, sc;
        for (i = 0; i < 128; ++i)
            for (j = 0; j < 128; ++j) {
                float v = orc_bf16_to_f32(w[(rb * 128 + i) * ldw + cb * 128 + j]);
                if (!isfinite(v)) bad = 1;
                else if (fabsf(v) > amax) amax = fabsf(v);
            }
        sc = scale_of(amax, fmt);
        s[rb * ncb + cb] = sc;
        for (i = 0; i < 128; ++i)
            for (j = 0; j < 128; ++j)
                q[(rb * 128 + i) * cols + cb * 128 + j] =
                    quant_one(orc_bf16_to_f32(w[(rb * 128 + i) * ldw + cb * 128 + j]), sc, fmt);
    }
    return bad ? ORC_NONFINITE : ORC_OK;
}

/* [Ling] "FP8 on-demand transpose weight": the FP8 W^T for dgrad.  A
 * 128x128-block quantization is symmetric under transposition, so W^T's
 * bytes are W's bytes transposed and its scale grid is the transposed grid. */
void orc_fp8_transpose(const uint8_t *q, int64_t rows, int64_t cols, uint8_t *qT)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t c;
        for (c = 0; c < cols; ++c) qT[c * rows + r] = q[r * cols + c];
    }
}

void orc_f32_transpose(const float *s, int64_t rows, int64_t cols, float *sT)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c) sT[c * rows + r] = s[r * cols + c];
}

/* ---------------------------------------------------------------------------
 * Monitors ([Ling] "Where does the error come from?" and the monitor table)
 * ------------------------------------------------------------------------- */

/* Distinct values in a group, counted with a per-thread stamp table:
 * value v is new in the current group iff stamp[v] != group id. */
typedef struct {
    uint32_t *stamp;   /* 65536 entries */
    uint32_t gen;
} distinct_t;

static void distinct_init(distinct_t *d)
{
    d->stamp = (uint32_t *)calloc(65536, sizeof(uint32_t));
    d->gen = 0;
}

static void distinct_free(distinct_t *d) { free(d->stamp); }

static void distinct_new_group(distinct_t *d)
{
    d->gen++;
    if (d->gen == 0) {   /* wrapped: clear and restart */
        memset(d->stamp, 0, 65536 * sizeof(uint32_t));
        d->gen = 1;
    }
}

/* returns 1 if `key` had not been seen in this group */
static int distinct_add(distinct_t *d, uint32_t key)
{
    if (d->stamp[key] == d->gen) return 0;
    d->stamp[key] = d->gen;
    return 1;
}

/* +-0 are one value on both sides (R6). */
static uint32_t key_bf16(uint16_t b) { return (b & 0x7FFF) == 0 ? 0u : (uint32_t)b; }
static uint32_t key_fp8(uint8_t c) { return (c & 0x7F) == 0 ? 0u : (uint32_t)c; }

/* stats[0..4] += {nonzero, underflow, saturated, distinct_in, distinct_out}.
 * x: [rows][cols] BF16 with leading dimension ldx.  q and s follow `gran`:
 *   1x128, 128x128, TENSOR: q is [rows][cols];
 *   128x1:  q is the transposed copy [cols][rows], s is S[rows/128][cols]. */
int orc_quant_stats(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx,
                    const uint8_t *q, const float *s, int gran, int fmt, uint64_t *stats)
{
    fmt_t f = fmt_of(fmt);
    float fm = (float)f.fmax;
    int64_t ngroups, g;
    uint64_t nz = 0, uf = 0, sat = 0, din = 0, dout = 0;
    int64_t gr, gc; /* group extent in rows / cols of x */

    switch (gran) {
    case ORC_GRAN_1x128: gr = 1; gc = 128; break;
    case ORC_GRAN_128x128: gr = 128; gc = 128; break;
    case ORC_GRAN_128x1: gr = 128; gc = 1; break;
    case ORC_GRAN_TENSOR: gr = rows; gc = cols; break;
    default: return ORC_BADARG;
    }
    if (rows == 0 || cols == 0) return ORC_OK;
    if (rows % gr != 0 || cols % gc != 0) return ORC_BADARG;
    ngroups = (rows / gr) * (cols / gc);

    if (gran == ORC_GRAN_TENSOR) {
        /* One group: count in parallel, then merge per-thread presence sets. */
        uint8_t seen_x[65536], seen_q[256];
        float sc = s[0];
        int64_t r;
        memset(seen_x, 0, sizeof seen_x);
        memset(seen_q, 0, sizeof seen_q);
#pragma omp parallel reduction(+ : nz, uf, sat)
        {
            uint8_t *px = (uint8_t *)calloc(65536, 1), *pq = (uint8_t *)calloc(256, 1);
            int v;
#pragma omp for schedule(static)
            for (r = 0; r < rows; ++r) {
                int64_t c;
                for (c = 0; c < cols; ++c) {
                    uint16_t xb = x[r * ldx + c];
                    uint8_t qc = q[r * cols + c];
                    float xv = orc_bf16_to_f32(xb);
                    float quotient = xv / sc;
                    if (xv != 0.0f) {
                        nz++;
                        if ((qc & 0x7F) == 0) uf++;
                    }
                    if (fabsf(quotient) > fm) sat++;
                    px[key_bf16(xb)] = 1;
                    pq[key_fp8(qc)] = 1;
                }
            }
#pragma omp critical
            {
                for (v = 0; v < 65536; ++v) seen_x[v] |= px[v];
                for (v = 0; v < 256; ++v) seen_q[v] |= pq[v];
            }
            free(px);
            free(pq);
        }
        for (g = 0; g < 65536; ++g) din += seen_x[g];
        for (g = 0; g < 256; ++g) dout += seen_q[g];
        stats[0] += nz;
        stats[1] += uf;
        stats[2] += sat;
        stats[3] += din;
        stats[4] += dout;
        return ORC_OK;
    }

#pragma omp parallel reduction(+ : nz, uf, sat, din, dout)
    {
        distinct_t dx, dq;
        distinct_init(&dx);
        distinct_init(&dq);
#pragma omp for schedule(dynamic, 64)
        for (g = 0; g < ngroups; ++g) {
            int64_t grow = g / (cols / gc), gcol = g % (cols / gc);
            int64_t i, j;
            float sc;
            switch (gran) {
            case ORC_GRAN_1x128: sc = s[gcol * rows + grow]; break;
            case ORC_GRAN_128x128: sc = s[grow * (cols / 128) + gcol]; break;
            case ORC_GRAN_128x1: sc = s[grow * cols + gcol]; break;
            default: sc = s[0]; break;
            }
            distinct_new_group(&dx);
            distinct_new_group(&dq);
            for (i = 0; i < gr; ++i)
                for (j = 0; j < gc; ++j) {
                    int64_t r = grow * gr + i, c = gcol * gc + j;
                    uint16_t xb = x[r * ldx + c];
                    uint8_t qc = (gran == ORC_GRAN_128x1) ? q[c * rows + r] : q[r * cols + c];
                    float xv = orc_bf16_to_f32(xb);
                    float quotient = xv / sc;
                    if (xv != 0.0f) {
                        nz++;
                        if ((qc & 0x7F) == 0) uf++;
                    }
                    if (fabsf(quotient) > fm) sat++;
                    din += (uint64_t)distinct_add(&dx, key_bf16(xb));
                    dout += (uint64_t)distinct_add(&dq, key_fp8(qc));
                }
        }
        distinct_free(&dx);
        distinct_free(&dq);
    }
    stats[0] += nz;
    stats[1] += uf;
    stats[2] += sat;
    stats[3] += din;
    stats[4] += dout;
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Per-tensor current scaling ([FP8-RL] "KV cache compression": the scaling
 * factor of the FP8 KV cache is recomputed from the current tensor after every
 * model update, "inference-side calibration").  One group, the whole tensor:
 * s = fp32(amax / fmax) (1 if amax = 0), q = enc(fp32(x) / s).  A tensor that
 * holds Inf/NaN is reported (its outputs unspecified).
 * ------------------------------------------------------------------------- */
int orc_quant_pertensor_current(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                                float *scale, uint8_t *q)
{
    float amax = 0.0f, sc;
    int64_t r;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(max : amax) reduction(| : bad)
    for (r = 0; r < rows; ++r) {
        int64_t c;
        for (c = 0; c < cols; ++c) {
            const float v = orc_bf16_to_f32(x[r * ldx + c]);
            if (!isfinite(v)) bad = 1;
            else if (fabsf(v) > amax) amax = fabsf(v);
        }
    }
    sc = scale_of(amax, fmt);
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t c;
        for (c = 0; c < cols; ++c) q[r * cols + c] = quant_one(orc_bf16_to_f32(x[r * ldx + c]), sc, fmt);
    }
    *scale = sc;
    return bad ? ORC_NONFINITE : ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Per-tensor delayed scaling ([Infra] "Transformer Engine", "Scaling
 * strategies: delayed scaling") -- one step of the state machine (R5).
 * ------------------------------------------------------------------------- */

#define ORC_ALGO_MAX 0
#define ORC_ALGO_MOST_RECENT 1

int orc_delayed_step(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                     int hist_len, int margin, int algo, float *hist, int32_t *step,
                     float *scale, uint8_t *q, uint64_t *stats)
{
    float s_t = *scale;
    float amax = 0.0f, m;
    int64_t r;
    int bad = 0, i;
    if (hist_len <= 0) return ORC_BADARG;

    /* 1. quantize with the scale chosen from earlier steps */
#pragma omp parallel for schedule(static) reduction(max : amax) reduction(| : bad)
    for (r = 0; r < rows; ++r) {
        int64_t c;
        for (c = 0; c < cols; ++c) {
            float v = orc_bf16_to_f32(x[r * ldx + c]);
            if (!isfinite(v)) bad = 1;
            else if (fabsf(v) > amax) amax = fabsf(v);
            q[r * cols + c] = quant_one(v, s_t, fmt);
        }
    }
    /* monitors of this step, one group = the whole tensor */
    if (stats) {
        float one_scale = s_t;
        orc_quant_stats(x, rows, cols, ldx, q, &one_scale, ORC_GRAN_TENSOR, fmt, stats);
    }
    /* A step whose tensor holds Inf/NaN reports it and leaves the state as it
     * was (reading R5: a non-finite amax must not enter the history). */
    if (bad) return ORC_NONFINITE;
    /* 2. record this step's amax; 3. next scale from the history */
    hist[*step % hist_len] = amax;
    if (algo == ORC_ALGO_MOST_RECENT) {
        m = amax;
    } else {
        m = 0.0f;
        for (i = 0; i < hist_len; ++i)
            if (hist[i] > m) m = hist[i];
    }
    if (m > 0.0f) *scale = ldexpf(m, margin) / (float)fmt_of(fmt).fmax;
    *step += 1;
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * GEMM ([Ling] "FP8 gemm ... FP32 accumulate"; fine-grained scales applied per
 * 128-deep chunk of K).  D = A . B^T, A [M][K], B [N][K], K contiguous.
 * Returns unrounded FP64 values at the listed (m, n) points (R7).
 * ------------------------------------------------------------------------- */

static float scale_at(const float *sv, int gran, int64_t ld, int64_t row, int64_t kb)
{
    switch (gran) {
    case ORC_GRAN_1x128: return sv[kb * ld + row];          /* S[K/128][ld]     */
    case ORC_GRAN_128x128: return sv[(row / 128) * ld + kb]; /* S[rows/128][ld]  */
    default: return sv[0];
    }
}

static double gemm_point(int64_t K, const uint8_t *arow, int fmtA, const float *sA, int granA,
                         int64_t ldsA, int64_t m, const uint8_t *brow, int fmtB, const float *sB,
                         int granB, int64_t ldsB, int64_t n, const double *decA,
                         const double *decB)
{
    int64_t kb, k;
    double d = 0.0;
    (void)fmtA; (void)fmtB;
    if (granA == ORC_GRAN_TENSOR && granB == ORC_GRAN_TENSOR) {
        double p = 0.0;
        for (k = 0; k < K; ++k) p += decA[arow[k]] * decB[brow[k]];
        return (double)sA[0] * (double)sB[0] * p;
    }
    for (kb = 0; kb < K / 128; ++kb) {
        double p = 0.0;
        for (k = kb * 128; k < kb * 128 + 128; ++k) p += decA[arow[k]] * decB[brow[k]];
        d += (double)scale_at(sA, granA, ldsA, m, kb) * (double)scale_at(sB, granB, ldsB, n, kb) * p;
    }
    return d;
}

int orc_gemm_points(int64_t M, int64_t N, int64_t K,
                    const uint8_t *A, int64_t lda, int fmtA, const float *sA, int granA, int64_t ldsA,
                    const uint8_t *B, int64_t ldb, int fmtB, const float *sB, int granB, int64_t ldsB,
                    int64_t npts, const int64_t *pm, const int64_t *pn, double *out)
{
    double decA[256], decB[256];
    int64_t i;
    int c;
    if (K % 128 != 0) return ORC_BADARG;
    for (c = 0; c < 256; ++c) {
        decA[c] = orc_fp8_decode((uint8_t)c, fmtA);
        decB[c] = orc_fp8_decode((uint8_t)c, fmtB);
    }
#pragma omp parallel for schedule(dynamic, 256)
    for (i = 0; i < npts; ++i) {
        int64_t m = pm[i], n = pn[i];
        if (m < 0 || m >= M || n < 0 || n >= N) { out[i] = NAN; continue; }
        out[i] = gemm_point(K, A + m * lda, fmtA, sA, granA, ldsA, m, B + n * ldb, fmtB, sB, granB,
                            ldsB, n, decA, decB);
    }
    return ORC_OK;
}

/* Grouped (MoE expert) GEMM: rows [off[g], off[g+1]) of A use expert g's
 * weights B[g] ([N][K]) with 128x128 scales sB[g][N/128][K/128]; A's 1x128
 * scales are S[K/128][ldsA].  Points at rows >= off[G] give NaN. */
int orc_grouped_gemm_points(int G, const int32_t *off, int64_t N, int64_t K,
                            const uint8_t *A, const float *sA, int64_t ldsA,
                            const uint8_t *B, const float *sB,
                            int64_t npts, const int64_t *pm, const int64_t *pn, double *out)
{
    double dec[256];
    int64_t i;
    int c;
    if (K % 128 != 0 || N % 128 != 0) return ORC_BADARG;
    for (c = 0; c < 256; ++c) dec[c] = orc_fp8_decode((uint8_t)c, ORC_E4M3);
#pragma omp parallel for schedule(dynamic, 256)
    for (i = 0; i < npts; ++i) {
        int64_t m = pm[i], n = pn[i];
        int g = -1, e;
        for (e = 0; e < G; ++e)
            if (m >= off[e] && m < off[e + 1]) { g = e; break; }
        if (g < 0 || n < 0 || n >= N) { out[i] = NAN; continue; }
        out[i] = gemm_point(K, A + m * K, ORC_E4M3, sA, ORC_GRAN_1x128, ldsA, m,
                            B + ((int64_t)g * N + n) * K, ORC_E4M3, sB + (int64_t)g * (N / 128) * (K / 128),
                            ORC_GRAN_128x128, K / 128, n, dec, dec);
    }
    return ORC_OK;
}

/* Grouped wgrad of the MoE expert layers ([FP8-RL] MoE expert layers in FP8;
 * [Ling] "grad (transpose)": the wgrad operands are the transposed copies
 * quantized along the token dimension).  The dispatch rows of expert g are
 * [off[g], off[g+1]); the operands are the transposed copies AT [N][ldt] and
 * BT [K][ldt] of two dispatch-ordered tensors, with 1x128 scales along the
 * rows, S[ldt/128][N] and S[ldt/128][K].  Expert g's output is
 *   D_g[n][k] = sum over its 128-row chunks c of sA[c][n] * sB[c][k] *
 *               (sum over the chunk's rows r of AT[n][r] * BT[k][r]),
 * zero for an expert without rows.  Points (g, n, k); unrounded FP64. */
int orc_grouped_wgrad_points(int G, const int32_t *off, int64_t N, int64_t K, int64_t ldt,
                             const uint8_t *AT, int fmtA, const float *sA,
                             const uint8_t *BT, int fmtB, const float *sB,
                             int64_t npts, const int64_t *pg, const int64_t *pn, const int64_t *pk,
                             double *out)
{
    double decA[256], decB[256];
    int64_t i;
    int c;
    if (ldt % 128 != 0) return ORC_BADARG;
    for (c = 0; c < 256; ++c) {
        decA[c] = orc_fp8_decode((uint8_t)c, fmtA);
        decB[c] = orc_fp8_decode((uint8_t)c, fmtB);
    }
#pragma omp parallel for schedule(dynamic, 256)
    for (i = 0; i < npts; ++i) {
        int64_t g = pg[i], n = pn[i], k = pk[i], r0, rows;
        if (g < 0 || g >= G || n < 0 || n >= N || k < 0 || k >= K) { out[i] = NAN; continue; }
        r0 = off[g];
        rows = off[g + 1] - off[g];
        if (rows < 0 || r0 % 128 != 0 || rows % 128 != 0 || r0 + rows > ldt) { out[i] = NAN; continue; }
        /* the group's slice: its chunks start at chunk r0/128 of the scale arrays */
        out[i] = gemm_point(rows, AT + n * ldt + r0, fmtA, sA + (r0 / 128) * N, ORC_GRAN_1x128, N, n,
                            BT + k * ldt + r0, fmtB, sB + (r0 / 128) * K, ORC_GRAN_1x128, K, k, decA, decB);
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * High-precision dw recompute monitor ([Ling] "Where does the error come
 * from?": tensors flagged by the underflow / distortion monitors get their dw
 * recomputed in high precision and compared).  The reference is
 *   R[n][k] = sum_m dY[m][n] * X[m][k]
 * over the BF16 operands (token-major dY [M][N], X [M][K]), exact products
 * summed in FP64; against the FP8 wgrad D [N][ldD] the monitor reports
 *   out = { sum (D - R)^2, sum R^2, max |D - R|, max |R| }  (FP64).
 * ------------------------------------------------------------------------- */
int orc_wgrad_recompute_error(int64_t M, int64_t N, int64_t K, const uint16_t *dY, const uint16_t *X,
                              const float *D, int64_t ldD, double *out)
{
    double sdd = 0.0, srr = 0.0, mdd = 0.0, mrr = 0.0;
    int64_t n;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : sdd, srr) reduction(max : mdd, mrr)
    for (n = 0; n < N; ++n) {
        int64_t k, m;
        for (k = 0; k < K; ++k) {
            double r = 0.0, d;
            for (m = 0; m < M; ++m)
                r += (double)orc_bf16_to_f32(dY[m * N + n]) * (double)orc_bf16_to_f32(X[m * K + k]);
            d = (double)D[n * ldD + k] - r;
            sdd += d * d;
            srr += r * r;
            if (fabs(d) > mdd) mdd = fabs(d);
            if (fabs(r) > mrr) mrr = fabs(r);
        }
    }
    out[0] = sdd;
    out[1] = srr;
    out[2] = mdd;
    out[3] = mrr;
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * AdamW step with the moments kept in FP8 ([Ling] "FP8 Optimizer": both Adam
 * moments in FP8 with fine-grained compression / decompression; [FP8-LM]
 * "Level 2: FP8 optimizer": momentum and variance in FP8) -- R12.
 * m is E4M3 and v is E5M2, each with one binary32 scale per 128 consecutive
 * parameters (R2's rule).  Every step below is one IEEE binary32 operation,
 * in this order (Adam as published by Kingma and Ba, with the decoupled
 * weight decay of Loshchilov and Hutter's AdamW):
 *   m  = dec(qm) * sm                 v  = dec(qv) * sv
 *   m  = b1 * m + omb1 * g            v  = b2 * v + omb2 * (g * g)
 *   mh = m / bc1                      vh = v / bc2
 *   u  = mh / (sqrt(vh) + eps)
 *   p  = p - lr * (u + wd * p)
 * then per 128-block s = amax / fmax (1 if amax = 0) and q = enc(x / s) for
 * the new m and v.  omb1 = 1 - b1, omb2 = 1 - b2, bc1 = 1 - b1^t and
 * bc2 = 1 - b2^t are given as binary32 numbers.
 * ------------------------------------------------------------------------- */
int orc_adam_fp8_step(int64_t n, float *p, const uint16_t *g, uint8_t *qm, float *sm, uint8_t *qv, float *sv,
                      float lr, float b1, float b2, float omb1, float omb2, float eps, float wd, float bc1,
                      float bc2)
{
    int64_t blk;
    if (n % 128 != 0) return ORC_BADARG;
#pragma omp parallel for schedule(static)
    for (blk = 0; blk < n / 128; ++blk) {
        float mn[128], vn[128], am = 0.0f, av = 0.0f, s_m, s_v;
        int i;
        for (i = 0; i < 128; ++i) {
            const int64_t k = blk * 128 + i;
            const float gi = orc_bf16_to_f32(g[k]);
            float m = (float)orc_fp8_decode(qm[k], ORC_E4M3) * sm[blk];
            float v = (float)orc_fp8_decode(qv[k], ORC_E5M2) * sv[blk];
            float gg, mh, vh, den, u, t;
            m = b1 * m + omb1 * gi;
            gg = gi * gi;
            v = b2 * v + omb2 * gg;
            mh = m / bc1;
            vh = v / bc2;
            den = sqrtf(vh) + eps;
            u = mh / den;
            t = wd * p[k];
            t = u + t;
            t = lr * t;
            p[k] = p[k] - t;
            mn[i] = m;
            vn[i] = v;
            if (fabsf(m) > am) am = fabsf(m);
            if (fabsf(v) > av) av = fabsf(v);
        }
        s_m = am == 0.0f ? 1.0f : am / 448.0f;
        s_v = av == 0.0f ? 1.0f : av / 57344.0f;
        for (i = 0; i < 128; ++i) {
            qm[blk * 128 + i] = orc_fp8_encode(mn[i] / s_m, ORC_E4M3);
            qv[blk * 128 + i] = orc_fp8_encode(vn[i] / s_v, ORC_E5M2);
        }
        sm[blk] = s_m;
        sv[blk] = s_v;
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * MoE routing with the padded routing map ([Ling] "FP8 padding routing map";
 * [FP8-RL] MoE expert layers in FP8) -- R8.
 * ------------------------------------------------------------------------- */
int orc_moe_route(int64_t T, int E, int topk, int align, const float *logits,
                  int32_t *topk_idx, double *topk_prob, int32_t *counts, int32_t *padded,
                  int32_t *offsets, int64_t cap, int32_t *row_token, double *row_prob,
                  uint8_t *row_is_pad, int64_t *total)
{
    uint8_t *routed, *pad;
    double *prob;
    int64_t t;
    int e, k;
    if (topk <= 0 || topk > E || align <= 0) return ORC_BADARG;
    routed = (uint8_t *)calloc((size_t)(T * E), 1);
    pad = (uint8_t *)calloc((size_t)(T * E), 1);
    prob = (double *)calloc((size_t)(T * E), sizeof(double));

    /* softmax in FP64; top-k by logit, ties to the lower index */
    for (t = 0; t < T; ++t) {
        const float *z = logits + t * E;
        double mx = -INFINITY, sum = 0.0;
        for (e = 0; e < E; ++e) if ((double)z[e] > mx) mx = (double)z[e];
        for (e = 0; e < E; ++e) { prob[t * E + e] = exp((double)z[e] - mx); sum += prob[t * E + e]; }
        for (e = 0; e < E; ++e) prob[t * E + e] /= sum;
        for (k = 0; k < topk; ++k) {
            int best = -1;
            for (e = 0; e < E; ++e) {
                if (routed[t * E + e]) continue;
                if (best < 0 || z[e] > z[best]) best = e;   /* strict: keeps the lower index on ties */
            }
            routed[t * E + best] = 1;
            topk_idx[t * topk + k] = best;
            topk_prob[t * topk + k] = prob[t * E + best];
        }
    }
    /* per-expert counts, padded counts, and the routing-map edit */
    offsets[0] = 0;
    for (e = 0; e < E; ++e) {
        int64_t c = 0, need;
        for (t = 0; t < T; ++t) c += routed[t * E + e];
        counts[e] = (int32_t)c;
        padded[e] = (int32_t)(((c + align - 1) / align) * align);
        need = padded[e] - c;
        for (t = 0; t < T && need > 0; ++t)
            if (!routed[t * E + e]) { pad[t * E + e] = 1; need--; }
        if (need > 0) { free(routed); free(pad); free(prob); return ORC_BADARG; }
        offsets[e + 1] = offsets[e] + padded[e];
    }
    *total = offsets[E];
    if (*total > cap) { free(routed); free(pad); free(prob); return ORC_BADARG; }
    /* dispatch: rows of expert e = its tokens (routed or padding) in ascending order */
    for (e = 0; e < E; ++e) {
        int64_t r = offsets[e];
        for (t = 0; t < T; ++t) {
            if (routed[t * E + e] || pad[t * E + e]) {
                row_token[r] = (int32_t)t;
                row_prob[r] = routed[t * E + e] ? prob[t * E + e] : 0.0;
                row_is_pad[r] = pad[t * E + e];
                r++;
            }
        }
    }
    free(routed); free(pad); free(prob);
    return ORC_OK;
}

/* Gather FP8 rows and their 1x128 scales for the dispatched rows:
 * qg[r] = q[row_token[r]], sg[kb][r] = s[kb][row_token[r]] (s ld = T,
 * sg ld = cap). */
void orc_moe_gather(const uint8_t *q, const float *s, int64_t T, int64_t K,
                    const int32_t *row_token, int64_t total, int64_t cap, uint8_t *qg, float *sg)
{
    int64_t r, kb;
    for (r = 0; r < total; ++r) {
        memcpy(qg + r * K, q + (int64_t)row_token[r] * K, (size_t)K);
        for (kb = 0; kb < K / 128; ++kb) sg[kb * cap + r] = s[kb * T + row_token[r]];
    }
}

/* ---------------------------------------------------------------------------
 * SwiGLU glue between the two expert / MLP GEMMs (not an FP8 step).  The
 * fused [gate; up] GEMM output has gate in columns [0, F) and up in [F, 2F).
 * ------------------------------------------------------------------------- */
void orc_swiglu_fwd(const uint16_t *gu, int64_t rows, int64_t F, uint16_t *h)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t j;
        for (j = 0; j < F; ++j) {
            double g = orc_bf16_to_f32(gu[r * 2 * F + j]);
            double u = orc_bf16_to_f32(gu[r * 2 * F + F + j]);
            double sig = 1.0 / (1.0 + exp(-g));
            h[r * F + j] = orc_f64_to_bf16(g * sig * u);
        }
    }
}

/* d/dg [g*sig(g)*u] = u*sig*(1 + g*(1 - sig));  d/du = g*sig. */
void orc_swiglu_bwd(const uint16_t *gu, const uint16_t *dh, int64_t rows, int64_t F, uint16_t *dgu)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t j;
        for (j = 0; j < F; ++j) {
            double g = orc_bf16_to_f32(gu[r * 2 * F + j]);
            double u = orc_bf16_to_f32(gu[r * 2 * F + F + j]);
            double d = orc_bf16_to_f32(dh[r * F + j]);
            double sig = 1.0 / (1.0 + exp(-g));
            dgu[r * 2 * F + j] = orc_f64_to_bf16(d * u * sig * (1.0 + g * (1.0 - sig)));
            dgu[r * 2 * F + F + j] = orc_f64_to_bf16(d * g * sig);
        }
    }
}
