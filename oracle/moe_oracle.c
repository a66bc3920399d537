/*
 * moe_oracle.c -- CPU oracle for the routed MoE expert-FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * reference that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never links, calls or falls back to it.  It shares no code,
 * header, table or constant with the CUDA sources.
 *
 * Arithmetic is IEEE binary64 throughout.  Every routine is written as the
 * plain definition it implements (loops in the order of the definition, no
 * blocking, no fusion), with the passage it follows named in its comment.
 * Pages cited:
 *   [RB]  "Route-Block Membership Selects Packed-AWQ Arithmetic" (arXiv
 *         2607.26316): route flattening, alignment, block membership, the
 *         AWQ-g128 fixture, the split-K schedule derivation, stable
 *         construction.
 *   [SQ]  "Hardware-Native Joint Sparse-Quantization for Trillion-Scale
 *         Mixture-of-Experts" (arXiv 2610.02241): grouped expert products
 *         Y_e = X_e W_e^T (Sec. 3.4), 32-element activation scale blocks
 *         (Sec. 3.4, App. D.1), fused SwiGLU with requantization (App. D.1),
 *         the OCP microscaling formats it cites.
 *   [WD]  "Warp decode" (cursor.com blog, Spanish edition): the two-kernel
 *         output-centric decode, SiLU(gate) x up, routing weight folded into
 *         the down accumulation, MXFP8 weights converted to FP32 on the fly,
 *         BF16 activations kept un-quantized ("Mayor precision").
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - MXFP8 = OCP MX: E4M3 elements, one E8M0 power-of-two scale per 32
 *     consecutive elements along K.  Quantizer: X = floor(log2 amax) - 8,
 *     clamped to [-127,127]; amax = 0 gives X = -127; element = RNE(v/2^X)
 *     onto the E4M3 grid with saturation at +-448; the sign of v is kept
 *     (so a negative value that rounds to zero is -0, code 0x80).
 *   - AWQ-4bit: w = (q - z) * s, q and z unsigned nibbles, s fp16, one
 *     (s, z) per group of 128 along K; plain nibble order.
 *   - Paired 4:8 sparse NVFP4 ([SQ] App. A): per group of 8 weights along
 *     K, two kept adjacent pairs named by a nibble p0 | p1 << 2 (p0 < p1),
 *     four kept E2M1 codes, one UE4M3 scale per 32 weights, one binary32
 *     constant per matrix; quantizer by Eq. 5 with the pattern chosen by
 *     pair energy (the page chooses by learned logits).
 *   - Alignment: valid route = expert id in [0,E); order (expert, route id);
 *     pad each active expert to a multiple of b with sentinel M*k; experts
 *     with no route get no block; unused tails: sentinel rows, -1 blocks.
 *   - Top-k routing: select by logit (exact FP32 compare, ties to the lower
 *     expert id, slots in descending order), softmax over all E in binary64,
 *     renormalise the k selected probabilities to sum 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_MXFP8 0
#define ORC_AWQ4 1
#define ORC_NVFP4S 2

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3 (cited by [SQ] Sec. 2 for the MX formats; [WD] "Como
 * funcionan los dos kernels" for MXFP8 weights): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 is subnormal
 * (2^-6 * m/8); no infinities; S.1111.111 is NaN. */
double orc_e4m3_value(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* OCP E8M0 shared scale: 2^(c-127); 0xFF is NaN. */
double orc_e8m0_value(uint8_t c)
{
    if (c == 0xFF)
        return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* IEEE binary16 (fp16): 1-5-10, bias 15. */
double orc_fp16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double mag;
    if (e == 0x1F)
        return m ? NAN : (sign ? -INFINITY : INFINITY);
    if (e == 0)
        mag = ldexp((double)m / 1024.0, -14);
    else
        mag = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -mag : mag;
}

/* bfloat16: 1-8-7, bias 127 (the upper half of a binary32). */
double orc_bf16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int m = h & 0x7F;
    double mag;
    if (e == 0xFF)
        return m ? NAN : (sign ? -INFINITY : INFINITY);
    if (e == 0)
        mag = ldexp((double)m / 128.0, -126);
    else
        mag = ldexp(1.0 + (double)m / 128.0, e - 127);
    return sign ? -mag : mag;
}

/* FP4 E2M1, the value grid of [SQ] App. A, Figure 3 caption
 * ({0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}): 1 sign bit, 2 exponent bits
 * with bias 1, 1 mantissa bit; exponent field 0 is subnormal (m/2); every
 * code is finite. */
double orc_e2m1_value(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 0x3;
    int m = c & 0x1;
    double mag = e == 0 ? (double)m / 2.0 : ldexp(1.0 + (double)m / 2.0, e - 1);
    return sign ? -mag : mag;
}

/* UE4M3, the unsigned FP8 block scale of [SQ] App. A ("G_s contains UE4M3
 * scales"; Figure 3 caption "UE4M3 (unsigned FP8)"): the E4M3 codes with the
 * sign bit clear, 0x00..0x7E; 0x7F and codes with bit 7 set are not scales
 * (NaN). */
double orc_ue4m3_value(uint8_t c)
{
    if (c & 0x80)
        return NAN;
    return orc_e4m3_value(c);
}

/* Paired 4:8 sparsity metadata ([SQ] App. A: a group of m = 8 weights keeps
 * two of its four adjacent pairs, six patterns; 4 bits of metadata per
 * group, Eq. 7).  Encoding (a reading; the page fixes the count of bits, not
 * their meaning): nibble = p0 | p1 << 2 with p0 < p1 the indices of the kept
 * pairs (pair j = positions 2j, 2j+1 of the group).  Returns 1 and the two
 * indices for one of the six patterns, 0 for any other nibble. */
int orc_pair_pattern(uint8_t nib, int *p0, int *p1)
{
    int a = nib & 0x3, b = (nib >> 2) & 0x3;
    if ((nib & 0xF0) || a >= b)
        return 0;
    *p0 = a;
    *p1 = b;
    return 1;
}

/* The 127 non-negative finite E4M3 values, codes 0x00..0x7E, which are in
 * increasing order of value; filled once from orc_e4m3_value. */
static double e4m3_grid[127];

__attribute__((constructor)) static void e4m3_grid_init(void)
{
    int c;
    for (c = 0; c <= 0x7E; ++c)
        e4m3_grid[c] = orc_e4m3_value((uint8_t)c);
}

/* Round-to-nearest-even of a non-negative finite value onto the E4M3 grid,
 * saturating at 448.  A binary search finds the grid interval
 * [grid[lo], grid[lo+1]) holding the value; the nearer end wins, and on an
 * exact tie the code whose mantissa LSB is 0 (the even code) wins. */
static uint8_t e4m3_rne_magnitude(double a)
{
    int lo = 0, hi = 0x7E;
    double dlo, dhi;
    if (a >= 448.0)
        return 0x7E;
    while (hi - lo > 1) {           /* invariant: grid[lo] <= a < grid[hi] */
        int mid = (lo + hi) / 2;
        if (e4m3_grid[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    dlo = a - e4m3_grid[lo];
    dhi = e4m3_grid[hi] - a;
    if (dlo < dhi)
        return (uint8_t)lo;
    if (dhi < dlo)
        return (uint8_t)hi;
    return (uint8_t)((lo & 1) == 0 ? lo : hi);
}

/* MXFP8 quantizer over rows of K values (K a multiple of 32), per 32-element
 * block along K ([SQ] Sec. 3.4 and App. D.1: 32-element scale blocks; OCP MX
 * rule for the shared exponent, emax(E4M3) = 8).  q: [rows][K] E4M3 codes,
 * s: [rows][K/32] E8M0 bytes. */
void orc_mxfp8_quantize(const double *v, int64_t rows, int64_t K, uint8_t *q, uint8_t *s)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t blk, i;
        for (blk = 0; blk < K / 32; ++blk) {
            const double *vb = v + r * K + blk * 32;
            double amax = 0.0;
            int X;
            for (i = 0; i < 32; ++i)
                if (fabs(vb[i]) > amax)
                    amax = fabs(vb[i]);
            if (amax == 0.0) {
                X = -127;
            } else {
                int e2;
                frexp(amax, &e2);       /* amax = f * 2^e2, f in [0.5,1) */
                X = (e2 - 1) - 8;       /* floor(log2 amax) - emax(E4M3) */
                if (X < -127) X = -127;
                if (X > 127) X = 127;
            }
            s[r * (K / 32) + blk] = (uint8_t)(X + 127);
            for (i = 0; i < 32; ++i) {
                double u = ldexp(vb[i], -X);
                uint8_t code = e4m3_rne_magnitude(fabs(u));
                if (signbit(u))
                    code |= 0x80;
                q[r * K + blk * 32 + i] = code;
            }
        }
    }
}

/* Round-to-nearest-even of a non-negative finite value onto the E2M1
 * magnitudes (codes 0..7 in increasing order of value), saturating at 6; on
 * an exact tie the code whose mantissa bit is 0 wins. */
static uint8_t e2m1_rne_magnitude(double a)
{
    int c;
    if (a >= 6.0)
        return 7;
    for (c = 0; c < 7; ++c) {
        double lo = orc_e2m1_value((uint8_t)c), hi = orc_e2m1_value((uint8_t)(c + 1));
        if (a < hi) {
            if (a - lo < hi - a)
                return (uint8_t)c;
            if (hi - a < a - lo)
                return (uint8_t)(c + 1);
            return (uint8_t)((c & 1) == 0 ? c : c + 1);
        }
    }
    return 7;
}

/* Paired 4:8 sparse NVFP4 quantizer of one matrix W [N][K], K a multiple of
 * 32 ([SQ] App. A feasible set, Eq. 6; block scales by Eq. 5, Sec. 3.4):
 *  1. pattern: in every group of 8 consecutive weights along K, keep the two
 *     adjacent pairs of largest energy (sum of squares; ties to the lower
 *     pair index).  The page keeps the highest-logit pattern of a trained
 *     model; without training, magnitude is the plain reading.
 *  2. Y = W with the other pairs zeroed; amax_b = max |Y| over each block of
 *     32 weights; gamma = 448 / (max_b amax_b / 6) (Eq. 5); an all-zero Y
 *     takes gamma = 1.
 *  3. alpha = 1/gamma rounded to binary32: the per-matrix constant ("UE4M3
 *     scales up to a per-matrix constant", App. A), stored in FP32.
 *  4. block scale code = RNE_E4M3(gamma * amax_b / 6) (at most 448 by the
 *     choice of gamma).
 *  5. each kept weight: E2M1 code = RNE(|y| / (alpha * UE4M3(code))),
 *     saturating at 6, sign kept (a negative weight that rounds to zero is
 *     code 0x8); a zero scale gives code 0.
 * Layout: vals [N][K/4] (group g's four kept codes in bytes 2g, 2g+1, low
 * nibble first, pair p0's two values then pair p1's), meta [N][K/16]
 * (group g's pattern nibble in byte g/2, low nibble for even g), sc
 * [N][K/32] UE4M3 codes, *alpha. */
void orc_nvfp4s_quantize(const double *W, int64_t N, int64_t K, uint8_t *vals, uint8_t *meta,
                         uint8_t *sc, float *alpha)
{
    int64_t n, g, b;
    int *keep = (int *)malloc(sizeof(int) * (size_t)(N * (K / 8) * 2));
    double ymax = 0.0, gamma, a;
    /* 1. patterns */
    for (n = 0; n < N; ++n)
        for (g = 0; g < K / 8; ++g) {
            const double *w = W + n * K + 8 * g;
            double en[4];
            int j, p0 = 0, p1 = 1, t;
            for (j = 0; j < 4; ++j)
                en[j] = w[2 * j] * w[2 * j] + w[2 * j + 1] * w[2 * j + 1];
            /* the largest, then the largest of the rest (lower index on ties) */
            for (j = 1; j < 4; ++j)
                if (en[j] > en[p0])
                    p0 = j;
            p1 = p0 == 0 ? 1 : 0;
            for (j = 0; j < 4; ++j)
                if (j != p0 && en[j] > en[p1])
                    p1 = j;
            if (p1 < p0) {
                t = p0;
                p0 = p1;
                p1 = t;
            }
            keep[(n * (K / 8) + g) * 2] = p0;
            keep[(n * (K / 8) + g) * 2 + 1] = p1;
        }
    /* 2. block maxima of the pruned matrix, gamma */
    for (n = 0; n < N; ++n)
        for (g = 0; g < K / 8; ++g) {
            int i;
            for (i = 0; i < 4; ++i) {
                int pj = keep[(n * (K / 8) + g) * 2 + i / 2];
                double v = fabs(W[n * K + 8 * g + 2 * pj + i % 2]);
                if (v > ymax)
                    ymax = v;
            }
        }
    gamma = ymax > 0.0 ? 448.0 / (ymax / 6.0) : 1.0;
    /* 3. the per-matrix constant */
    *alpha = (float)(1.0 / gamma);
    a = (double)*alpha;
    for (n = 0; n < N; ++n) {
        for (b = 0; b < K / 32; ++b) {
            double amax = 0.0, s;
            uint8_t code;
            int64_t gg;
            for (gg = 4 * b; gg < 4 * b + 4; ++gg) {
                int i;
                for (i = 0; i < 4; ++i) {
                    int pj = keep[(n * (K / 8) + gg) * 2 + i / 2];
                    double v = fabs(W[n * K + 8 * gg + 2 * pj + i % 2]);
                    if (v > amax)
                        amax = v;
                }
            }
            /* 4. the block's scale code */
            code = e4m3_rne_magnitude(gamma * amax / 6.0);
            sc[n * (K / 32) + b] = code;
            s = a * orc_ue4m3_value(code);
            /* 5. the kept values */
            for (gg = 4 * b; gg < 4 * b + 4; ++gg) {
                int p0 = keep[(n * (K / 8) + gg) * 2], p1 = keep[(n * (K / 8) + gg) * 2 + 1], i;
                uint8_t *vb = vals + n * (K / 4) + 2 * gg;
                uint8_t *mb = meta + n * (K / 16) + gg / 2;
                uint8_t nib = (uint8_t)(p0 | (p1 << 2));
                if (gg % 2 == 0)
                    *mb = nib;
                else
                    *mb = (uint8_t)(*mb | (nib << 4));
                vb[0] = vb[1] = 0;
                for (i = 0; i < 4; ++i) {
                    int pj = i < 2 ? p0 : p1;
                    double y = W[n * K + 8 * gg + 2 * pj + i % 2];
                    uint8_t c = s > 0.0 ? e2m1_rne_magnitude(fabs(y) / s) : 0;
                    if (y < 0.0 || (y == 0.0 && signbit(y)))
                        c = (uint8_t)(c | 0x8);
                    vb[i / 2] = (uint8_t)(vb[i / 2] | (c << (4 * (i % 2))));
                }
            }
        }
    }
    free(keep);
}

/* Run-time activation quantizer Q_a onto NVFP4 with 32-element scale blocks
 * ([SQ] Sec. 3.4 and App. D.1: expert activations are quantized at run time
 * into 32-element blocks, each with one UE4M3 scale, before the first GEMM
 * and again after SwiGLU; the block scale follows Eq. 5).  Reading: Eq. 5's
 * tensor-wide factor gamma is 1 / alpha with alpha the activation's
 * tensor-wide scale, a constant of the layer (App. D.1 folds the tensor-wide
 * scales of both operands into one factor alpha_e per expert, so alpha does
 * not change from batch to batch).  The page does not fix the precision of
 * the rounding decisions; they are taken in binary32, in this order:
 *   r6   = binary32(1 / (6 alpha))              the quotient in binary64, rounded once
 *   t    = binary32(amax * r6)                  amax = max |v| over the block
 *   s    = t rounded to nearest (ties to even) onto UE4M3, saturating at 448
 *   S    = UE4M3(s); when S = 0 every magnitude code is 0
 *   q    = binary32(1 / binary32(alpha * S))
 *   code = sign bit of v | |binary32(v * q)| rounded to nearest (ties to
 *          even) onto the E2M1 magnitudes, saturating at 6
 * The activation it stands for is alpha * S * E2M1(code).
 * v: [rows][K] binary32 (K a multiple of 32); codes: [rows][K] one E2M1 code
 * per byte; scales: [rows][K/32] UE4M3 codes. */
void orc_nvfp4_act_quantize(const float *v, int64_t rows, int64_t K, float alpha, uint8_t *codes,
                            uint8_t *scales)
{
    const float r6 = (float)(1.0 / (6.0 * (double)alpha));
    int64_t r;
    for (r = 0; r < rows; ++r) {
        int64_t blk, i;
        for (blk = 0; blk < K / 32; ++blk) {
            const float *vb = v + r * K + blk * 32;
            float amax = 0.0f, t, S, q = 0.0f;
            uint8_t s;
            for (i = 0; i < 32; ++i)
                if (fabsf(vb[i]) > amax)
                    amax = fabsf(vb[i]);
            t = amax * r6;
            s = e4m3_rne_magnitude((double)t);
            scales[r * (K / 32) + blk] = s;
            S = (float)orc_ue4m3_value(s);
            if (S > 0.0f) {
                const float p = alpha * S;
                q = 1.0f / p;
            }
            for (i = 0; i < 32; ++i) {
                uint8_t c = 0;
                if (S > 0.0f) {
                    const float u = vb[i] * q;
                    c = e2m1_rne_magnitude((double)fabsf(u));
                }
                if (signbit(vb[i]))
                    c = (uint8_t)(c | 0x8);
                codes[r * K + blk * 32 + i] = c;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Expert weights                                                            */
/* ------------------------------------------------------------------------ */

/* One projection of every expert, [E][N][K].  `slot` maps an expert id to
 * the index of its slab in the arrays (NULL = identity), which lets a caller
 * hand over only the experts a routing touches; -1 = not supplied. */
typedef struct {
    int32_t fmt;             /* ORC_MXFP8, ORC_AWQ4 or ORC_NVFP4S */
    int32_t E;
    int64_t N, K;
    const uint8_t *q8;       /* MXFP8 codes   [slots][N][K]          */
    const uint8_t *s8;       /* MXFP8 scales  [slots][N][K/32]       */
    const int32_t *q4;       /* AWQ nibbles   [slots][N][K/8]        */
    const uint16_t *s16;     /* AWQ fp16 scale[slots][N][K/128]      */
    const int32_t *z4;       /* AWQ zeros     [slots][N/8][K/128]    */
    const int32_t *slot;     /* [E] or NULL                          */
    const uint8_t *v4;       /* NVFP4S kept E2M1 codes [slots][N][K/4]  */
    const uint8_t *m4;       /* NVFP4S pattern nibbles [slots][N][K/16] */
    const uint8_t *sc8;      /* NVFP4S UE4M3 scales    [slots][N][K/32] */
    const float *alpha;      /* NVFP4S per-matrix constant [slots]      */
} orc_weights;

static int64_t weight_slot(const orc_weights *w, int32_t e)
{
    return w->slot ? (int64_t)w->slot[e] : (int64_t)e;
}

/* Dequantize row n of expert e exactly.
 * MXFP8: w = E4M3(q) * 2^(s-127) ([WD] "Como funcionan los dos kernels").
 * AWQ:   w = (q - z) * s with group 128 along K ([RB] fixture paragraph:
 *        4-bit AWQ, group size 128).  Element 8c+i of a row sits in bits
 *        4i..4i+3 of word c; the zero of row 8a+i sits in nibble i of word a. */
int orc_dequant_row(const orc_weights *w, int32_t e, int64_t n, double *out)
{
    int64_t sl = weight_slot(w, e);
    int64_t kk;
    if (sl < 0)
        return -1;
    if (w->fmt == ORC_MXFP8) {
        const uint8_t *qr = w->q8 + (sl * w->N + n) * w->K;
        const uint8_t *sr = w->s8 + (sl * w->N + n) * (w->K / 32);
        for (kk = 0; kk < w->K; ++kk)
            out[kk] = orc_e4m3_value(qr[kk]) * orc_e8m0_value(sr[kk / 32]);
    } else if (w->fmt == ORC_NVFP4S) {
        /* w = alpha * UE4M3(scale of the 32-block) * E2M1(code) at the kept
         * positions of each group of 8, 0 elsewhere ([SQ] App. A, Eq. 6 and
         * Eq. 7 storage; layout as orc_nvfp4s_quantize writes it).  A pattern
         * nibble that is not one of the six returns -2. */
        const uint8_t *vr = w->v4 + (sl * w->N + n) * (w->K / 4);
        const uint8_t *mr = w->m4 + (sl * w->N + n) * (w->K / 16);
        const uint8_t *sr = w->sc8 + (sl * w->N + n) * (w->K / 32);
        const double a = (double)w->alpha[sl];
        int64_t g;
        for (kk = 0; kk < w->K; ++kk)
            out[kk] = 0.0;
        for (g = 0; g < w->K / 8; ++g) {
            int p0, p1, i;
            const double s = a * orc_ue4m3_value(sr[(8 * g) / 32]);
            if (!orc_pair_pattern((uint8_t)((mr[g / 2] >> (4 * (g % 2))) & 0xF), &p0, &p1))
                return -2;
            for (i = 0; i < 4; ++i) {
                int pj = i < 2 ? p0 : p1;
                uint8_t c = (uint8_t)((vr[2 * g + i / 2] >> (4 * (i % 2))) & 0xF);
                out[8 * g + 2 * pj + i % 2] = orc_e2m1_value(c) * s;
            }
        }
    } else {
        const int32_t *qr = w->q4 + (sl * w->N + n) * (w->K / 8);
        const uint16_t *sr = w->s16 + (sl * w->N + n) * (w->K / 128);
        const int32_t *zr = w->z4 + (sl * (w->N / 8) + n / 8) * (w->K / 128);
        for (kk = 0; kk < w->K; ++kk) {
            uint32_t word = (uint32_t)qr[kk / 8];
            int qv = (int)((word >> (4 * (kk % 8))) & 0xF);
            uint32_t zword = (uint32_t)zr[kk / 128];
            int zv = (int)((zword >> (4 * (n % 8))) & 0xF);
            out[kk] = (double)(qv - zv) * orc_fp16_value(sr[kk / 128]);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Routing                                                                   */
/* ------------------------------------------------------------------------ */

/* Top-k routing ([WD] "La ruta convencional de MoE": each token selects 8 of
 * 128 experts; [RB] opening paragraph: the router yields an M x k id array).
 * Selection compares the FP32 logits exactly (softmax is monotone, so this is
 * the top-k of the probabilities); ties go to the lower expert id; slots are
 * in descending order.  Weights: softmax over all E in binary64, then the k
 * selected probabilities renormalised to sum 1. */
void orc_topk_softmax(const float *logits, int64_t M, int32_t E, int32_t k,
                      int32_t *ids, double *wts)
{
    int64_t t;
    for (t = 0; t < M; ++t) {
        const float *l = logits + t * E;
        double mx = -INFINITY, z = 0.0, zsel = 0.0;
        int32_t j, e;
        for (j = 0; j < k; ++j) {
            int32_t best = -1;
            for (e = 0; e < E; ++e) {
                int taken = 0, jj;
                for (jj = 0; jj < j; ++jj)
                    if (ids[t * k + jj] == e)
                        taken = 1;
                if (taken)
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e;
            }
            ids[t * k + j] = best;
        }
        for (e = 0; e < E; ++e)
            if ((double)l[e] > mx)
                mx = (double)l[e];
        for (e = 0; e < E; ++e)
            z += exp((double)l[e] - mx);
        for (j = 0; j < k; ++j)
            zsel += exp((double)l[ids[t * k + j]] - mx) / z;
        for (j = 0; j < k; ++j)
            wts[t * k + j] = (exp((double)l[ids[t * k + j]] - mx) / z) / zsel;
    }
}

/* ------------------------------------------------------------------------ */
/* Alignment                                                                 */
/* ------------------------------------------------------------------------ */

/* Route alignment by stable construction ([RB] opening paragraph: group the
 * valid routes by expert, pad each expert's count to a multiple of b, emit a
 * parallel expert-block vector; [RB] stable-construction paragraph: order by
 * (expert id, flattened route id)).  Route id r = t*k + j (row-major flatten).
 * Returns 0, or -1 when the capacities are too small.  *n_invalid counts
 * routes whose id lies outside [0,E). */
int orc_align(const int32_t *ids, int64_t M, int32_t k, int32_t E, int32_t b,
              int32_t *sorted_route_ids, int32_t *expert_ids, int32_t *num_rows_post_pad,
              int64_t cap_rows, int64_t cap_blocks, int32_t *n_invalid)
{
    int64_t MK = M * k, r, row = 0, blk = 0;
    int32_t e;
    int32_t invalid = 0;
    for (r = 0; r < MK; ++r)
        if (ids[r] < 0 || ids[r] >= E)
            ++invalid;
    for (e = 0; e < E; ++e) {
        int64_t count = 0, padded, i;
        for (r = 0; r < MK; ++r) {
            if (ids[r] == e) {
                if (row >= cap_rows)
                    return -1;
                sorted_route_ids[row++] = (int32_t)r;
                ++count;
            }
        }
        if (count == 0)
            continue;
        padded = ((count + b - 1) / b) * b;
        for (i = count; i < padded; ++i) {
            if (row >= cap_rows)
                return -1;
            sorted_route_ids[row++] = (int32_t)MK;
        }
        for (i = 0; i < padded / b; ++i) {
            if (blk >= cap_blocks)
                return -1;
            expert_ids[blk++] = e;
        }
    }
    *num_rows_post_pad = (int32_t)row;
    for (; row < cap_rows; ++row)
        sorted_route_ids[row] = (int32_t)MK;
    for (; blk < cap_blocks; ++blk)
        expert_ids[blk] = -1;
    if (n_invalid)
        *n_invalid = invalid;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The layer                                                                 */
/* ------------------------------------------------------------------------ */

static double silu(double g)
{
    return g / (1.0 + exp(-g));
}

/* MXFP8 quantize-dequantize of one vector of n values (n a multiple of 32),
 * the activation quantizer of the block-scaled path ([SQ] Sec. 3.4, App. D.1:
 * run-time quantization into 32-element scale blocks, before the first GEMM
 * and again after SwiGLU).  Optional code/scale outputs. */
static void mx_roundtrip(const double *v, int64_t n, double *out, uint8_t *q, uint8_t *s)
{
    uint8_t *qq = q ? q : (uint8_t *)malloc((size_t)n);
    uint8_t *ss = s ? s : (uint8_t *)malloc((size_t)(n / 32));
    int64_t i;
    orc_mxfp8_quantize(v, 1, n, qq, ss);
    for (i = 0; i < n; ++i)
        out[i] = orc_e4m3_value(qq[i]) * orc_e8m0_value(ss[i / 32]);
    if (!q) free(qq);
    if (!s) free(ss);
}

/* Round a binary64 value to the nearest fp16 (ties to even), by search over
 * the binade: used for the fp16 intermediate of the AWQ grouped mode. */
static double round_to_fp16(double v)
{
    double a = fabs(v), q, lo, hi, ulp;
    int e2;
    if (a == 0.0)
        return v;
    if (a >= 65520.0)
        return v > 0 ? INFINITY : -INFINITY;
    frexp(a, &e2);                        /* a in [2^(e2-1), 2^e2) */
    if (e2 - 1 < -14)
        ulp = ldexp(1.0, -24);           /* subnormal spacing */
    else
        ulp = ldexp(1.0, (e2 - 1) - 10);
    lo = floor(a / ulp) * ulp;
    hi = lo + ulp;
    if (a - lo < hi - a)
        q = lo;
    else if (a - lo > hi - a)
        q = hi;
    else
        q = (fmod(lo / ulp, 2.0) == 0.0) ? lo : hi;
    return v < 0 ? -q : q;
}

/* Per-route modes of the intermediate activation. */
#define ORC_MODE_EXACT 0   /* x and h exact (output-centric decode, [WD]) */
#define ORC_MODE_MX 1      /* x and h MXFP8-quantized ([SQ] block-scaled path) */
#define ORC_MODE_H16 2     /* h rounded to fp16 (fp16 tensor-core AWQ path) */

/* The routed expert-FFN layer, for tokens t in [0, M).
 *   x      : [M][d] exact activation values
 *   ids, w : [M][k] routing
 *   w13    : N = 2I rows (gate rows 0..I-1, up rows I..2I-1), K = d
 *   w2     : N = d rows, K = I
 *   y      : [M][d] output
 *   h_out  : optional [M*k][I] intermediate SiLU(g)*u (before any
 *            quantization of h); rows of invalid routes are 0
 *   hq_in  : optional [M*k][I] codes + [M*k][I/32] scales: when given (MX
 *            mode), these replace the oracle's own quantized h (stage-wise
 *            check of the second projection)
 *   hq_out, hs_out: optional codes/scales of the oracle's own quantized h
 *
 * y[t] = sum_j w[t][j] * W2_{e_j} . h_{t,j},  h_{t,j} = SiLU(g) * u,
 * [g; u] = W13_{e_j} . x[t]   ([WD] "Como funcionan los dos kernels": SiLU
 * of gate times up; the routing weight folded into the down accumulation;
 * [SQ] Sec. 3.3: a gate-up-down expert block).  Routes whose expert id is
 * outside [0,E) contribute nothing.  Returns 0, or -1 if a routed expert's
 * weights were not supplied. */
int orc_moe_layer(const double *x, int64_t M, int64_t d, int64_t I,
                  const int32_t *ids, const double *w, int32_t k, int32_t E,
                  const orc_weights *w13, const orc_weights *w2, int32_t mode,
                  double *y, double *h_out,
                  const uint8_t *hq_in, const uint8_t *hs_in,
                  uint8_t *hq_out, uint8_t *hs_out)
{
    int64_t t;
    int err = 0;
    for (t = 0; t < M * d; ++t)
        y[t] = 0.0;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < M; ++t) {
        double *xt = (double *)malloc(sizeof(double) * (size_t)d);
        double *row = (double *)malloc(sizeof(double) * (size_t)(d > I ? d : I));
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *hx = (double *)malloc(sizeof(double) * (size_t)I);
        int32_t j;
        int64_t n, o, kk;
        if (mode == ORC_MODE_MX)
            mx_roundtrip(x + t * d, d, xt, NULL, NULL);
        else
            memcpy(xt, x + t * d, sizeof(double) * (size_t)d);
        for (j = 0; j < k; ++j) {
            int64_t r = t * k + j;
            int32_t e = ids[r];
            if (e < 0 || e >= E) {
                if (h_out)
                    for (n = 0; n < I; ++n) h_out[r * I + n] = 0.0;
                continue;
            }
            for (n = 0; n < I; ++n) {
                double g = 0.0, u = 0.0;
                if (orc_dequant_row(w13, e, n, row)) { err = -1; break; }
                for (kk = 0; kk < d; ++kk) g += row[kk] * xt[kk];
                if (orc_dequant_row(w13, e, I + n, row)) { err = -1; break; }
                for (kk = 0; kk < d; ++kk) u += row[kk] * xt[kk];
                h[n] = silu(g) * u;
            }
            if (h_out)
                memcpy(h_out + r * I, h, sizeof(double) * (size_t)I);
            if (mode == ORC_MODE_MX) {
                if (hq_in) {
                    for (n = 0; n < I; ++n)
                        hx[n] = orc_e4m3_value(hq_in[r * I + n]) *
                                orc_e8m0_value(hs_in[r * (I / 32) + n / 32]);
                } else {
                    mx_roundtrip(h, I, hx, hq_out ? hq_out + r * I : NULL,
                                 hs_out ? hs_out + r * (I / 32) : NULL);
                }
            } else if (mode == ORC_MODE_H16) {
                for (n = 0; n < I; ++n) hx[n] = round_to_fp16(h[n]);
            } else {
                memcpy(hx, h, sizeof(double) * (size_t)I);
            }
            for (o = 0; o < d; ++o) {
                double acc = 0.0;
                if (orc_dequant_row(w2, e, o, row)) { err = -1; break; }
                for (n = 0; n < I; ++n) acc += row[n] * hx[n];
                y[t * d + o] += w[r] * acc;
            }
        }
        free(xt); free(row); free(h); free(hx);
    }
    return err;
}

/* The routed expert-FFN layer with NVFP4-quantized activations, the W4A4
 * grouped path of [SQ] (Sec. 3.4, App. D.1): x is quantized by Q_a with the
 * constant alpha_x before the first projection, h = SiLU(g) * u by Q_a with
 * alpha_h before the second; the weights (any format; paired 4:8 sparse
 * NVFP4 on that path) are dequantized exactly, per-expert constant included.
 *   x      : [M][d] activation values, taken as binary32
 *   xv_out : optional [M][d], S * E2M1(code) of Q_a(x) (without alpha_x)
 *   h_out  : optional [M*k][I], h before quantization (binary64)
 *   hv_in  : optional [M*k][I], S * E2M1(code) values that replace the
 *            oracle's own Q_a(h) (stage-wise check of the second projection)
 *   hv_out : optional [M*k][I], S * E2M1(code) of the oracle's own Q_a(h),
 *            h rounded to binary32 first (the decisions are binary32)
 * Otherwise as orc_moe_layer: y[t] = sum_j w[t][j] * W2_{e_j} . (alpha_h hv),
 * binary64 sums; routes outside [0,E) contribute nothing; rows of invalid
 * routes in h_out / hv_out are 0.  Returns 0, or -1 if a routed expert's
 * weights were not supplied. */
int orc_moe_layer_a4(const double *x, int64_t M, int64_t d, int64_t I,
                     const int32_t *ids, const double *w, int32_t k, int32_t E,
                     const orc_weights *w13, const orc_weights *w2, float alpha_x, float alpha_h,
                     double *y, double *xv_out, double *h_out, const double *hv_in, double *hv_out)
{
    int64_t t;
    int err = 0;
    for (t = 0; t < M * d; ++t)
        y[t] = 0.0;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < M; ++t) {
        float *xf = (float *)malloc(sizeof(float) * (size_t)d);
        float *hf = (float *)malloc(sizeof(float) * (size_t)I);
        uint8_t *cd = (uint8_t *)malloc((size_t)(d > I ? d : I));
        uint8_t *sc = (uint8_t *)malloc((size_t)((d > I ? d : I) / 32));
        double *xt = (double *)malloc(sizeof(double) * (size_t)d);
        double *row = (double *)malloc(sizeof(double) * (size_t)(d > I ? d : I));
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *hx = (double *)malloc(sizeof(double) * (size_t)I);
        int32_t j;
        int64_t n, o, kk;
        for (kk = 0; kk < d; ++kk)
            xf[kk] = (float)x[t * d + kk];
        orc_nvfp4_act_quantize(xf, 1, d, alpha_x, cd, sc);
        for (kk = 0; kk < d; ++kk) {
            const double v = orc_e2m1_value(cd[kk]) * orc_ue4m3_value(sc[kk / 32]);
            if (xv_out)
                xv_out[t * d + kk] = v;
            xt[kk] = (double)alpha_x * v;
        }
        for (j = 0; j < k; ++j) {
            int64_t r = t * k + j;
            int32_t e = ids[r];
            if (e < 0 || e >= E) {
                for (n = 0; n < I; ++n) {
                    if (h_out) h_out[r * I + n] = 0.0;
                    if (hv_out) hv_out[r * I + n] = 0.0;
                }
                continue;
            }
            for (n = 0; n < I; ++n) {
                double g = 0.0, u = 0.0;
                if (orc_dequant_row(w13, e, n, row)) { err = -1; break; }
                for (kk = 0; kk < d; ++kk) g += row[kk] * xt[kk];
                if (orc_dequant_row(w13, e, I + n, row)) { err = -1; break; }
                for (kk = 0; kk < d; ++kk) u += row[kk] * xt[kk];
                h[n] = silu(g) * u;
            }
            if (h_out)
                memcpy(h_out + r * I, h, sizeof(double) * (size_t)I);
            if (hv_in) {
                for (n = 0; n < I; ++n) hx[n] = hv_in[r * I + n];
            } else {
                for (n = 0; n < I; ++n) hf[n] = (float)h[n];
                orc_nvfp4_act_quantize(hf, 1, I, alpha_h, cd, sc);
                for (n = 0; n < I; ++n) hx[n] = orc_e2m1_value(cd[n]) * orc_ue4m3_value(sc[n / 32]);
            }
            if (hv_out)
                memcpy(hv_out + r * I, hx, sizeof(double) * (size_t)I);
            for (o = 0; o < d; ++o) {
                double acc = 0.0;
                if (orc_dequant_row(w2, e, o, row)) { err = -1; break; }
                for (n = 0; n < I; ++n) acc += row[n] * ((double)alpha_h * hx[n]);
                y[t * d + o] += w[r] * acc;
            }
        }
        free(xf); free(hf); free(cd); free(sc); free(xt); free(row); free(h); free(hx);
    }
    return err;
}

/* Number of OpenMP threads the layer uses (1 when built without OpenMP). */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n);
#else
    (void)n;
#endif
}
