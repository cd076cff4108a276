/*
 * nvq_oracle.c -- the CPU oracle for block-scaled 4-bit quantisation.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is loaded by the test-suite, by the
 * smoke check and by the benchmark's CPU-baseline leg, and by nothing else.
 * The CUDA library never links, includes or calls it; the two share no code,
 * no header, no table and no constant generator.
 *
 * Every function is a plain, slow, single-threaded restatement of what the
 * path computes, in the order the sources describe it:
 *
 *   [P1] "Getting GLM-5.2 NVFP4 Post-Training off the ground" (Patronus AI),
 *        Part I, "Why can't we just transpose the one copy?" and
 *        "The bottom line" (NVFP4 format, rowwise/columnwise blocking,
 *        dequantised bf16 backward).
 *   [P4] "The 4-bitter Lesson: Balancing Stability and Performance in NVFP4 RL"
 *        (humans&), "Key claims" and "Method" (round-to-nearest, Four-Over-Six,
 *        per-token FP32 activation scales, FP32 error accumulation).
 *   [P5] "nf4moe -- QLoRA for a 743B Fused-MoE", "The fix: dequant-on-forward
 *        for routed experts" (NF4, blocksize 64, routed dequantisation, the
 *        "nested code" of the NF4 state).
 *
 * Where the sources leave a step open, the reading taken is stated at the
 * step.  Build: gcc -O2 -ffp-contract=off -fno-fast-math.  With contraction
 * off every float expression below is a sequence of IEEE-754 binary32
 * operations, each rounded to nearest-even; fmaf() is the correctly rounded
 * fused multiply-add and is used only where it is written.
 *
 * Parity pins: every function here is pinned by the host tests against
 * something other than itself (library conversions, hand-computed blocks, the
 * worked example of [P1], closed forms, invariants, brute force, and the NF4
 * values printed in the QLoRA paper's appendix).  The nested NF4 absmax
 * follows the published double quantisation with the readings stated at
 * it; its equality with a third-party nested code is not claimed.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* Flag and status bits of the boundary, restated (not shared) here. */
#define O_FLAG_4OVER6    1u
#define O_FLAG_AMAX_GIVEN 2u
#define O_STATUS_NONFINITE 1
#define O_STATUS_BAD_INDEX 2

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                           */
/* ------------------------------------------------------------------------ */

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the upper half of a binary32 word: widening is exact. */
ORACLE_API float oracle_bf16_to_f32(uint16_t h) { return from_bits((uint32_t)h << 16); }

/*
 * Round a binary32 value to the nearest bf16, ties to the even bf16 pattern.
 * Written as the definition: take the two bf16 neighbours that bracket x
 * (truncation towards zero and the next pattern away from zero), compare x
 * with their exact midpoint in double precision (exact: every operand has at
 * most 24 significant bits), and break a tie towards the even pattern.
 */
ORACLE_API uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u = to_bits(x);
    if (isnan(x)) return (uint16_t)((u >> 16) | 0x0040u);   /* quiet NaN */
    uint16_t lo = (uint16_t)(u >> 16);                        /* toward zero */
    if ((u & 0xffffu) == 0) return lo;                        /* exact */
    uint16_t hi = (uint16_t)(lo + 1u);                        /* away from zero */
    double ax = fabs((double)x);
    double vlo = fabs((double)oracle_bf16_to_f32(lo));
    double vhi;
    if (((hi >> 7) & 0xffu) == 0xffu)     /* stepping past the largest finite */
        vhi = vlo + ldexp(1.0, ilogb(vlo) - 7);              /* one bf16 ulp */
    else
        vhi = fabs((double)oracle_bf16_to_f32(hi));
    double mid = 0.5 * (vlo + vhi);
    if (ax < mid) return lo;
    if (ax > mid) return hi;
    return (lo & 1u) ? hi : lo;
}

/*
 * FP8 E4M3 (OCP): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities; pattern 0x7F is NaN, so the largest finite value is
 * 0x7E = 448.  Exponent field 0 holds subnormals m * 2^-9.
 */
ORACLE_API float oracle_e4m3_value(uint8_t c)
{
    int e = (c >> 3) & 0xF, m = c & 7;
    float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
    return (c & 0x80) ? -v : v;
}

/*
 * Round a non-negative binary32 value to E4M3, nearest with ties to the even
 * mantissa, saturating at 448 (the "satfinite" rule: no value maps to NaN).
 * Definition: scan the 127 non-negative finite values in increasing order,
 * find the pair that brackets x, and compare x with their midpoint (exact in
 * binary32: the midpoint has at most five significant bits).
 */
ORACLE_API uint8_t oracle_e4m3_encode(float x)
{
    if (!(x > 0.0f)) return 0;                 /* +0, -0 (and NaN: out of contract) */
    if (x >= 448.0f) return 0x7E;
    uint8_t k = 0;
    while (k < 0x7E && oracle_e4m3_value((uint8_t)(k + 1)) <= x) k++;
    float lo = oracle_e4m3_value(k), hi = oracle_e4m3_value((uint8_t)(k + 1));
    if (x == lo) return k;
    float mid = 0.5f * (lo + hi);
    if (x < mid) return k;
    if (x > mid) return (uint8_t)(k + 1);
    return (k & 1) ? (uint8_t)(k + 1) : k;
}

/*
 * FP4 E2M1: 1 sign bit (bit 3), 2 exponent bits with bias 1, 1 mantissa bit.
 * The eight magnitudes are {0, 0.5, 1, 1.5, 2, 3, 4, 6}; the 3-bit magnitude
 * code is the bit pattern itself.
 */
ORACLE_API float oracle_e2m1_value(uint8_t c)
{
    int e = (c >> 1) & 3, m = c & 1;
    float v = (e == 0) ? 0.5f * (float)m : ldexpf((float)(2 + m), e - 2);
    return (c & 8) ? -v : v;
}

/*
 * Round a binary32 value to E2M1: nearest magnitude with ties to the even
 * mantissa, saturating at 6; the sign bit is the sign of the input (so -0 and
 * negative values that round to zero give 0x8).  Same bracket-and-midpoint
 * definition as E4M3 over the eight magnitudes.
 */
ORACLE_API uint8_t oracle_e2m1_encode(float x)
{
    uint8_t sign = signbit(x) ? 8 : 0;
    float a = fabsf(x);
    if (a >= 6.0f) return sign | 7;
    uint8_t k = 0;
    while (k < 7 && oracle_e2m1_value((uint8_t)(k + 1)) <= a) k++;
    float lo = oracle_e2m1_value(k), hi = oracle_e2m1_value((uint8_t)(k + 1));
    if (a == lo) return sign | k;
    float mid = 0.5f * (lo + hi);
    if (a < mid) return sign | k;
    if (a > mid) return sign | (uint8_t)(k + 1);
    return sign | ((k & 1) ? (uint8_t)(k + 1) : k);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 with optional Four-Over-Six                                        */
/* ------------------------------------------------------------------------ */

/*
 * Largest E4M3 block scale the global scale aims at.  Without Four-Over-Six
 * it is the format maximum, 448, so the tensor scale is amax/(6*448) ([P1]
 * "Why can't we just transpose the one copy?": one FP32 global scale).  With
 * Four-Over-Six [P4] "Key claims" names a smaller E4M3 maximum
 * ("E4M3_4OVER6_MAX") without printing it; the reading taken is 256, the
 * largest power of two M with 1.5*M <= 448, so that the amax/4 candidate of
 * the block holding the tensor amax (1.5 times the amax/6 candidate) never
 * saturates.
 */
static float block_scale_max(int four_over_six) { return four_over_six ? 256.0f : 448.0f; }

/*
 * Global scales of one slice with absolute maximum amax.
 *   G = amax / (6 * M)          the stored FP32 tensor (or token) scale
 *   E = 1 / G, at most FLT_MAX  the encode factor applied once to the target
 * [P4] "Key claims": the target is scaled down once by the inverse of
 * amax/(E2M1_MAX * E4M3_4OVER6_MAX).  amax = 0 gives G = 0 and E = FLT_MAX
 * (1/0 = +inf, clamped), which maps every zero input to a zero target.
 */
ORACLE_API void oracle_tensor_scales(float amax, int four_over_six, float* G, float* E)
{
    float g = amax / (6.0f * block_scale_max(four_over_six));
    float e = 1.0f / g;
    if (e > FLT_MAX) e = FLT_MAX;
    *G = g;
    *E = e;
}

/* Codes of one candidate: c_i = E2M1(t_i * (1/S)); S = 0 keeps only signs. */
static void candidate_codes(const float t[16], float S, uint8_t c[16])
{
    if (S == 0.0f) {
        for (int i = 0; i < 16; i++) c[i] = signbit(t[i]) ? 8 : 0;
        return;
    }
    float r = 1.0f / S;
    for (int i = 0; i < 16; i++) c[i] = oracle_e2m1_encode(t[i] * r);
}

/*
 * Block squared error of one candidate, in FP32 ([P4] "Method": blockwise
 * error kept in FP32 against the original values, in the scaled domain).
 * d_i = t_i - c_i * S, where c_i * S is exact (at most six significant bits);
 * the squares are accumulated with fused multiply-adds in two interleaved
 * chains, even and odd element positions, which are added at the end.
 */
static float candidate_sse(const float t[16], float S, const uint8_t c[16])
{
    float acc_even = 0.0f, acc_odd = 0.0f;
    for (int k = 0; k < 8; k++) {
        float d0 = t[2 * k] - oracle_e2m1_value(c[2 * k]) * S;
        float d1 = t[2 * k + 1] - oracle_e2m1_value(c[2 * k + 1]) * S;
        acc_even = fmaf(d0, d0, acc_even);
        acc_odd = fmaf(d1, d1, acc_odd);
    }
    return acc_even + acc_odd;
}

/*
 * One 16-element NVFP4 block.  x holds the 16 bf16 inputs at the given
 * element stride (1 along a row; the row length down a column); E is the
 * slice's encode factor.
 *   t_i = x_i * E,  a = max |t_i|
 *   S6  = E4M3(a / 6)      (map the block amax to 6)
 *   S4  = E4M3(a / 4)      (Four-Over-Six: map it to 4)     [P4] "Method"
 * Without Four-Over-Six the block keeps S6.  With it, the candidate with the
 * strictly lower squared error wins and a tie keeps S6.  Outputs the chosen
 * E4M3 scale byte and the 16 codes; sse6/sse4 (if non-null) receive the two
 * errors (sse4 is NaN without Four-Over-Six).
 */
ORACLE_API void oracle_nvfp4_block(const uint16_t* x, int64_t stride, float E,
                                   int four_over_six, uint8_t* scale_byte,
                                   uint8_t codes[16], float* sse6, float* sse4)
{
    float t[16], a = 0.0f;
    for (int i = 0; i < 16; i++) {
        t[i] = oracle_bf16_to_f32(x[(int64_t)i * stride]) * E;
        if (fabsf(t[i]) > a) a = fabsf(t[i]);
    }
    uint8_t s6 = oracle_e4m3_encode(a / 6.0f);
    float S6 = oracle_e4m3_value(s6);
    uint8_t c6[16];
    candidate_codes(t, S6, c6);
    float e6 = candidate_sse(t, S6, c6);
    if (sse6) *sse6 = e6;
    if (!four_over_six) {
        if (sse4) *sse4 = NAN;
        *scale_byte = s6;
        memcpy(codes, c6, 16);
        return;
    }
    uint8_t s4 = oracle_e4m3_encode(a / 4.0f);
    float S4 = oracle_e4m3_value(s4);
    uint8_t c4[16];
    candidate_codes(t, S4, c4);
    float e4 = candidate_sse(t, S4, c4);
    if (sse4) *sse4 = e4;
    if (e4 < e6) {
        *scale_byte = s4;
        memcpy(codes, c4, 16);
    } else {
        *scale_byte = s6;
        memcpy(codes, c6, 16);
    }
}

/* max |x| over n bf16 values, as binary32 (exact). */
ORACLE_API float oracle_amax_bf16(const uint16_t* x, int64_t n)
{
    float a = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float v = fabsf(oracle_bf16_to_f32(x[i]));
        if (v > a || isnan(v)) a = v;
        if (isnan(a)) break;
    }
    return a;
}

/* Packs 16 codes, element 2j in the low nibble of byte j. */
static void pack_codes(const uint8_t c[16], uint8_t* dst)
{
    for (int j = 0; j < 8; j++) dst[j] = (uint8_t)((c[2 * j] & 0xF) | ((c[2 * j + 1] & 0xF) << 4));
}

/* Per-slice amax and scales; honours the amax-given flag; sets status bit 0. */
static void slice_scales(const uint16_t* w, int64_t n, uint32_t flags, float* amax_e,
                         float* G_e, float* E_out, int* status)
{
    float amax = (flags & O_FLAG_AMAX_GIVEN) ? *amax_e : oracle_amax_bf16(w, n);
    if (!(flags & O_FLAG_AMAX_GIVEN)) *amax_e = amax;
    if (!isfinite(amax) && status) *status |= O_STATUS_NONFINITE;
    oracle_tensor_scales(amax, (flags & O_FLAG_4OVER6) != 0, G_e, E_out);
}

/*
 * Rowwise NVFP4 quantisation of an expert stack w [nexp, rows, cols] (bf16,
 * row-major, cols contiguous): one FP32 tensor scale per expert slice, blocks
 * of 16 consecutive elements along cols ([P1]: rowwise blocks 1x16 along
 * "in").  codes [nexp, rows, cols/2], scales [nexp, rows, cols/16],
 * amax [nexp] (input with the amax-given flag, else output), G [nexp].
 */
ORACLE_API void oracle_nvfp4_quantize(const uint16_t* w, int64_t nexp, int64_t rows,
                                      int64_t cols, uint32_t flags, uint8_t* codes,
                                      uint8_t* scales, float* amax, float* G, int* status)
{
    int f46 = (flags & O_FLAG_4OVER6) != 0;
    for (int64_t e = 0; e < nexp; e++) {
        const uint16_t* we = w + e * rows * cols;
        float E;
        slice_scales(we, rows * cols, flags, &amax[e], &G[e], &E, status);
        for (int64_t r = 0; r < rows; r++)
            for (int64_t b = 0; b < cols / 16; b++) {
                uint8_t c[16];
                int64_t blk = (e * rows + r) * (cols / 16) + b;
                oracle_nvfp4_block(we + r * cols + b * 16, 1, E, f46, &scales[blk], c, 0, 0);
                pack_codes(c, codes + blk * 8);
            }
    }
}

/*
 * Columnwise NVFP4 quantisation: an independent quantisation of the same
 * slice with blocks of 16 consecutive rows at a fixed column ([P1]: 16x1
 * along "out"), using the same per-expert tensor scale, stored K-major for the
 * dgrad contraction, i.e. as the transpose: codes [nexp, cols, rows/2],
 * scales [nexp, cols, rows/16].
 */
ORACLE_API void oracle_nvfp4_quantize_colwise(const uint16_t* w, int64_t nexp, int64_t rows,
                                              int64_t cols, uint32_t flags, uint8_t* codes,
                                              uint8_t* scales, float* amax, float* G,
                                              int* status)
{
    int f46 = (flags & O_FLAG_4OVER6) != 0;
    for (int64_t e = 0; e < nexp; e++) {
        const uint16_t* we = w + e * rows * cols;
        float E;
        slice_scales(we, rows * cols, flags, &amax[e], &G[e], &E, status);
        for (int64_t col = 0; col < cols; col++)
            for (int64_t b = 0; b < rows / 16; b++) {
                uint8_t c[16];
                int64_t blk = (e * cols + col) * (rows / 16) + b;
                oracle_nvfp4_block(we + b * 16 * cols + col, cols, E, f46, &scales[blk], c, 0, 0);
                pack_codes(c, codes + blk * 8);
            }
    }
}

/*
 * Dequantised value of one code: bf16( (|c| * S) * G ) with the code's sign.
 * |c| * S is exact; the product with G is one binary32 rounding; the result is
 * rounded once more to bf16.  This is DQ(Q(w)), the tensor the dequantised
 * backward multiplies by ([P1] "The bottom line", [P4] "Method").
 */
static uint16_t dq_one(uint8_t c, uint8_t s, float G)
{
    float v = oracle_e2m1_value(c & 7) * oracle_e4m3_value(s);
    float y = v * G;
    if (c & 8) y = -y;
    return oracle_f32_to_bf16(y);
}

/* Rowwise dequantisation to bf16 [nexp, rows, cols]. */
ORACLE_API void oracle_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales,
                                     const float* G, int64_t nexp, int64_t rows, int64_t cols,
                                     uint16_t* dst)
{
    for (int64_t e = 0; e < nexp; e++)
        for (int64_t r = 0; r < rows; r++)
            for (int64_t c = 0; c < cols; c++) {
                int64_t i = (e * rows + r) * cols + c;
                uint8_t byte = codes[i / 2];
                uint8_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);
                dst[i] = dq_one(code, scales[i / 16], G[e]);
            }
}

/*
 * DQ(Q(w)) of the rowwise copy, written transposed as bf16 [nexp, cols, rows]
 * for the dgrad product dX = dY * W ([P1] "The bottom line": dequantise the
 * rowwise copy and run dgrad in bf16; the transpose is free in bf16).
 */
ORACLE_API void oracle_nvfp4_dequant_t(const uint8_t* codes, const uint8_t* scales,
                                       const float* G, int64_t nexp, int64_t rows,
                                       int64_t cols, uint16_t* dst)
{
    for (int64_t e = 0; e < nexp; e++)
        for (int64_t r = 0; r < rows; r++)
            for (int64_t c = 0; c < cols; c++) {
                int64_t i = (e * rows + r) * cols + c;
                uint8_t byte = codes[i / 2];
                uint8_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);
                dst[(e * cols + c) * rows + r] = dq_one(code, scales[i / 16], G[e]);
            }
}

/*
 * Per-token activation quantisation ([P4] "Method"): every token row of
 * x [T, H] gets its own FP32 scale computed over the hidden dimension, so no
 * state is shared across the batch; blocks of 16 along H as in the rowwise
 * weight path.  codes [T, H/2], scales [T, H/16], token_scale [T] = G_row.
 */
ORACLE_API void oracle_act_quantize_per_token(const uint16_t* x, int64_t T, int64_t H,
                                              uint32_t flags, uint8_t* codes, uint8_t* scales,
                                              float* token_scale, int* status)
{
    int f46 = (flags & O_FLAG_4OVER6) != 0;
    for (int64_t r = 0; r < T; r++) {
        const uint16_t* xr = x + r * H;
        float amax = oracle_amax_bf16(xr, H), G, E;
        if (!isfinite(amax) && status) *status |= O_STATUS_NONFINITE;
        oracle_tensor_scales(amax, f46, &G, &E);
        token_scale[r] = G;
        for (int64_t b = 0; b < H / 16; b++) {
            uint8_t c[16];
            int64_t blk = r * (H / 16) + b;
            oracle_nvfp4_block(xr + b * 16, 1, E, f46, &scales[blk], c, 0, 0);
            pack_codes(c, codes + blk * 8);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* NF4                                                                      */
/* ------------------------------------------------------------------------ */

/* Standard normal CDF and its inverse by bisection (double precision). */
static double std_normal_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

static double std_normal_quantile(double p)
{
    double lo = -40.0, hi = 40.0;
    for (int it = 0; it < 2000; it++) {
        double mid = 0.5 * (lo + hi);
        if (mid == lo || mid == hi) break;
        if (std_normal_cdf(mid) < p) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

/*
 * The 16 NF4 levels, ascending.  The pages name NF4 (bitsandbytes'
 * quant_type "nf4", [P5] "The fix") but print no values; NF4 is the 4-bit
 * NormalFloat data type of QLoRA (Dettmers et al. 2023, "4-bit NormalFloat
 * Quantization" and the NF4 value list in its appendix).  Construction, in
 * that paper's order:
 *   1. quantiles of N(0,1) at probabilities spaced evenly between the outer
 *      probability delta and 1/2: eight on the positive side (9 points,
 *      1/2 dropped) and seven on the negative side (8 points, 1/2 dropped),
 *      so that zero is an exact level and the type is asymmetric;
 *   2. the two sets joined with one zero and normalised by the largest
 *      level into [-1, 1].
 * delta is the published offset 0.9677083 (1 - (1/32 + 1/30)/2 to seven
 * digits).  Precision, the reading that reproduces the published binary32
 * values bit for bit: delta and the probabilities are binary32, stepped from
 * both ends (p_i = delta + i*s for the first half, 1/2 - (n-1-i)*s for the
 * rest, s = (1/2 - delta)/(n-1)); each quantile is computed in double and
 * rounded once to binary32; the normalisation is one binary32 division.
 */
static void nf4_probabilities(int n, float p[9])
{
    const float d = 0.9677083f, h = 0.5f;
    const float s = (h - d) / (float)(n - 1);
    for (int i = 0; i < n; i++) {
        if (i < n / 2) p[i] = d + s * (float)i;
        else p[i] = h - s * (float)(n - 1 - i);
    }
}

ORACLE_API void oracle_nf4_codebook(float cb[16])
{
    float pp[9], pn[9], q[16];
    nf4_probabilities(9, pp);   /* pp[0] = delta ... pp[8] = 1/2 */
    nf4_probabilities(8, pn);   /* pn[0] = delta ... pn[7] = 1/2 */
    /* ascending: -Phi^-1(pn[0]) ... -Phi^-1(pn[6]), 0, Phi^-1(pp[7]) ... Phi^-1(pp[0]) */
    for (int i = 0; i < 7; i++) q[i] = (float)(-std_normal_quantile((double)pn[i]));
    q[7] = 0.0f;
    for (int i = 0; i < 8; i++) q[8 + i] = (float)std_normal_quantile((double)pp[7 - i]);
    const float top = q[15];
    for (int i = 0; i < 16; i++) cb[i] = q[i] / top;
}

/*
 * NF4 blockwise quantisation with blocksize 64 ([P5] "The fix":
 * quantize_4bit, blocksize 64, one absmax per block).  Per block of 64
 * consecutive elements along cols:
 *   absmax = max |x_i|                  (binary32, exact)
 *   r      = absmax == 0 ? 0 : 1/absmax
 *   v_i    = x_i * r
 *   c_i    = number of midpoints m_j, j = 0..14, with v_i > m_j, where
 *            m_j = (cb[j] + cb[j+1]) * 0.5 in binary32
 * i.e. the nearest level, a value exactly on a midpoint going to the lower
 * index.  codes [nexp, rows, cols/2] (element 2j in the low nibble),
 * absmax [nexp, rows, cols/64] (binary32, no second-level quantisation).
 */
ORACLE_API void oracle_nf4_quantize(const uint16_t* w, int64_t nexp, int64_t rows, int64_t cols,
                                    uint8_t* codes, float* absmax, int* status)
{
    float cb[16], m[15];
    oracle_nf4_codebook(cb);
    for (int j = 0; j < 15; j++) m[j] = (cb[j] + cb[j + 1]) * 0.5f;
    int64_t nblk = nexp * rows * (cols / 64);
    for (int64_t b = 0; b < nblk; b++) {
        const uint16_t* xb = w + b * 64;
        float am = oracle_amax_bf16(xb, 64);
        if (!isfinite(am) && status) *status |= O_STATUS_NONFINITE;
        absmax[b] = am;
        float r = (am == 0.0f) ? 0.0f : 1.0f / am;
        for (int i = 0; i < 64; i += 2) {
            uint8_t c[2];
            for (int h = 0; h < 2; h++) {
                float v = oracle_bf16_to_f32(xb[i + h]) * r;
                uint8_t k = 0;
                for (int j = 0; j < 15; j++) if (v > m[j]) k++;
                c[h] = k;
            }
            codes[b * 32 + i / 2] = (uint8_t)(c[0] | (c[1] << 4));
        }
    }
}

/* NF4 dequantisation of one slice run: y = bf16(cb[c] * absmax). */
static void nf4_dequant_range(const uint8_t* codes, const float* absmax, int64_t n, uint16_t* dst)
{
    float cb[16];
    oracle_nf4_codebook(cb);
    for (int64_t i = 0; i < n; i++) {
        uint8_t byte = codes[i / 2];
        uint8_t c = (i & 1) ? (byte >> 4) : (byte & 0xF);
        dst[i] = oracle_f32_to_bf16(cb[c] * absmax[i / 64]);
    }
}

ORACLE_API void oracle_nf4_dequant(const uint8_t* codes, const float* absmax, int64_t nexp,
                                   int64_t rows, int64_t cols, uint16_t* dst)
{
    nf4_dequant_range(codes, absmax, nexp * rows * cols, dst);
}

/*
 * Union of the experts the router hit ([P5] "The fix": one-hot mask of
 * top_k_index, summed, the non-zero experts gathered in one host read).
 * hit_list receives the hit experts in ascending order, then -1 up to nexp
 * entries; *n_hit their number.  Indices outside [0, nexp) are ignored and
 * set status bit 1.
 */
ORACLE_API void oracle_routed_union(const int32_t* topk, int64_t T, int64_t k, int64_t nexp,
                                    int32_t* hit_list, int32_t* n_hit, int* status)
{
    unsigned char* hit = (unsigned char*)calloc((size_t)nexp, 1);
    for (int64_t i = 0; i < T * k; i++) {
        int32_t e = topk[i];
        if (e < 0 || e >= nexp) {
            if (status) *status |= O_STATUS_BAD_INDEX;
            continue;
        }
        hit[e] = 1;
    }
    int32_t n = 0;
    for (int64_t e = 0; e < nexp; e++)
        if (hit[e]) hit_list[n++] = (int32_t)e;
    for (int64_t e = n; e < nexp; e++) hit_list[e] = -1;
    *n_hit = n;
    free(hit);
}

/*
 * Routed dequant-on-forward ([P5] "The fix"): only the experts in the union
 * are dequantised, each into its own slice of dst [nexp, rows, cols]; the
 * slices of experts nobody routed to are left untouched.
 */
ORACLE_API void oracle_nf4_dequant_routed(const uint8_t* codes, const float* absmax, int64_t nexp,
                                          int64_t rows, int64_t cols, const int32_t* topk,
                                          int64_t T, int64_t k, uint16_t* dst,
                                          int32_t* hit_list, int32_t* n_hit, int* status)
{
    oracle_routed_union(topk, T, k, nexp, hit_list, n_hit, status);
    int64_t slice = rows * cols;
    for (int32_t h = 0; h < *n_hit; h++) {
        int64_t e = hit_list[h];
        nf4_dequant_range(codes + e * slice / 2, absmax + e * slice / 64, slice, dst + e * slice);
    }
}

/* ------------------------------------------------------------------------ */
/* Array forms of the scalar conversions (loops over the definitions above,  */
/* for conversion sweeps).                                                   */
/* ------------------------------------------------------------------------ */

ORACLE_API void oracle_e4m3_encode_n(const float* x, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode(x[i]);
}

ORACLE_API void oracle_e2m1_encode_n(const float* x, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e2m1_encode(x[i]);
}

ORACLE_API void oracle_f32_to_bf16_n(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* MXFP8: the format "The 4-bitter Lesson" ("Key claims") used to            */
/* validate the dequantised backward before NVFP4.  The pages name it only;  */
/* its definition is the OCP Microscaling (MX) one: blocks of 32 consecutive */
/* elements share one E8M0 scale X = 2^s, and each element is stored as the  */
/* E4M3 value of v / X.                                                     */
/*   s = floor(log2(amax)) - 8, 8 being the exponent of the largest power of */
/*       two in E4M3 (256); clamped to [-127, 127]; amax = 0 gives -127;     */
/*   scale byte = s + 127 (E8M0: the value 2^(byte - 127));                  */
/*   element = E4M3(v * 2^-s), nearest with ties to even, saturating at 448  */
/*       (values in (448, 512) clamp), carrying the sign of v (so -0 and     */
/*       negative values that round to zero give 0x80).                      */
/* v * 2^-s is exact in binary32 whenever its E4M3 value is not zero.        */
/* ------------------------------------------------------------------------ */

static int mx_shared_exp(float amax)
{
    if (!(amax > 0.0f)) return -127;
    int e;
    frexpf(amax, &e);            /* amax = m * 2^e, m in [0.5, 1): floor(log2 amax) = e - 1 */
    int s = (e - 1) - 8;
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

static uint8_t e4m3_signed(float x)
{
    uint8_t m = oracle_e4m3_encode(fabsf(x));
    return signbit(x) ? (uint8_t)(m | 0x80u) : m;
}

/* One block of 32 bf16 values x[0], x[stride], ...: the 32 codes and the
 * returned scale byte. */
ORACLE_API uint8_t oracle_mxfp8_block(const uint16_t* x, int64_t stride, uint8_t codes[32])
{
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(oracle_bf16_to_f32(x[i * stride]));
        if (a > amax) amax = a;
    }
    int s = mx_shared_exp(amax);
    float inv = ldexpf(1.0f, -s);
    for (int i = 0; i < 32; i++) codes[i] = e4m3_signed(oracle_bf16_to_f32(x[i * stride]) * inv);
    return (uint8_t)(s + 127);
}

/* Rowwise: blocks of 1x32 along cols.  codes [nexp, rows, cols], scales
 * [nexp, rows, cols/32]; cols % 32 == 0. */
ORACLE_API void oracle_mxfp8_quantize(const uint16_t* w, int64_t nexp, int64_t rows, int64_t cols,
                                      uint8_t* codes, uint8_t* scales)
{
    for (int64_t e = 0; e < nexp; e++)
        for (int64_t r = 0; r < rows; r++)
            for (int64_t b = 0; b < cols / 32; b++) {
                int64_t i = (e * rows + r) * cols + 32 * b;
                scales[(e * rows + r) * (cols / 32) + b] = oracle_mxfp8_block(w + i, 1, codes + i);
            }
}

/* Columnwise: blocks of 32x1 along rows, stored transposed (K-major for the
 * transposed product): codes [nexp, cols, rows], scales [nexp, cols, rows/32];
 * rows % 32 == 0. */
ORACLE_API void oracle_mxfp8_quantize_colwise(const uint16_t* w, int64_t nexp, int64_t rows,
                                              int64_t cols, uint8_t* codes, uint8_t* scales)
{
    for (int64_t e = 0; e < nexp; e++)
        for (int64_t c = 0; c < cols; c++)
            for (int64_t b = 0; b < rows / 32; b++) {
                const uint16_t* x = w + (e * rows + 32 * b) * cols + c;
                scales[(e * cols + c) * (rows / 32) + b] =
                    oracle_mxfp8_block(x, cols, codes + (e * cols + c) * rows + 32 * b);
            }
}

/* y = bf16(E4M3 value * 2^(byte - 127)) (the product is exact in binary32),
 * for n elements in the layout of the codes (one scale per 32). */
ORACLE_API void oracle_mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int64_t n,
                                     uint16_t* dst)
{
    for (int64_t i = 0; i < n; i++)
        dst[i] = oracle_f32_to_bf16(ldexpf(oracle_e4m3_value(codes[i]), (int)scales[i / 32] - 127));
}

/* ------------------------------------------------------------------------ */
/* NF4 double-quantised ("nested") absmax                                   */
/* ------------------------------------------------------------------------ */
/*
 * [P5] "The fix" names the NF4 quantisation state as holding the absmax and
 * a "nested code", and says no more.  The reading taken is the published
 * double quantisation of QLoRA (Dettmers et al., 2023, "Double
 * Quantization"): the first-level FP32 absmax values of one expert slice are
 * centred on their mean and quantised again to 8-bit floats in blocks of
 * 256.  Where that description is silent:
 *   - the mean is the FP32 sum of the slice's n absmax values taken as a
 *     pairwise tree (values padded with zeros to the next power of two,
 *     adjacent pairs added level by level), divided by n in binary64 and
 *     rounded to binary32;
 *   - the 8-bit float is OCP E4M3, and each block's largest centred
 *     magnitude c1 is mapped to 448 with the factor k = min(fl(448 / c1),
 *     FLT_MAX) (the same encode-by-multiplication as the NVFP4 global scale);
 *     codes are nearest-even, saturating, sign kept;
 *   - decoding is one fused multiply-add: value(code) * fl(c1 / 448) + mean.
 */

/* Pairwise tree sum of a[0..n-1] in binary32, zero padded to a power of two. */
ORACLE_API float oracle_tree_sum(const float* a, int64_t n)
{
    if (n <= 0) return 0.0f;
    int64_t P = 1;
    while (P < n) P *= 2;
    float* s = (float*)calloc((size_t)P, sizeof(float));
    if (!s) abort();
    memcpy(s, a, (size_t)n * sizeof(float));
    for (int64_t len = P; len > 1; len /= 2)
        for (int64_t i = 0; i < len / 2; i++) s[i] = s[2 * i] + s[2 * i + 1];
    float r = s[0];
    free(s);
    return r;
}

ORACLE_API float oracle_absmax_mean(const float* a, int64_t n)
{
    if (n <= 0) return 0.0f;
    return (float)((double)oracle_tree_sum(a, n) / (double)n);
}

/* absmax [nexp, n] -> codes [nexp, n], c1 [nexp, ceil(n/256)], mean [nexp]. */
ORACLE_API void oracle_nf4_absmax_nest(const float* absmax, int64_t nexp, int64_t n,
                                       uint8_t* codes, float* c1, float* mean)
{
    const int64_t nb = (n + 255) / 256;
    for (int64_t e = 0; e < nexp; e++) {
        const float* a = absmax + e * n;
        const float mu = oracle_absmax_mean(a, n);
        mean[e] = mu;
        for (int64_t b = 0; b < nb; b++) {
            const int64_t i0 = 256 * b, i1 = (i0 + 256 < n) ? i0 + 256 : n;
            float m = 0.0f;
            for (int64_t i = i0; i < i1; i++) {
                float v = fabsf(a[i] - mu);
                if (v > m) m = v;
            }
            c1[e * nb + b] = m;
            float k = 448.0f / m;
            if (k > FLT_MAX) k = FLT_MAX;
            for (int64_t i = i0; i < i1; i++) codes[e * n + i] = e4m3_signed((a[i] - mu) * k);
        }
    }
}

ORACLE_API void oracle_nf4_absmax_unnest(const uint8_t* codes, const float* c1, const float* mean,
                                         int64_t nexp, int64_t n, float* absmax)
{
    const int64_t nb = (n + 255) / 256;
    for (int64_t e = 0; e < nexp; e++)
        for (int64_t i = 0; i < n; i++) {
            const float r = c1[e * nb + i / 256] / 448.0f;
            absmax[e * n + i] = fmaf(oracle_e4m3_value(codes[e * n + i]), r, mean[e]);
        }
}
