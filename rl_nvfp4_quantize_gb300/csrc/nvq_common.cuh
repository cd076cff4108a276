// nvq_common.cuh -- device primitives shared by the libnvq kernels (sm_103a).
//
// The arithmetic restates the block-scaled 4-bit formats described in
// "Getting GLM-5.2 NVFP4 Post-Training off the ground", Part I ("Why can't we
// just transpose the one copy?": E2M1 values, one E4M3 scale per 16-element
// block, one FP32 global scale) and "The 4-bitter Lesson" ("Key claims",
// "Method": round to nearest even, Four-Over-Six with an FP32 block squared
// error, target scaled down once by the inverse global scale, E2M1 x E4M3
// products formed exactly in FP16).
//
// Every FP32 operation is an explicit round-to-nearest intrinsic (or a
// packed f32x2 / mixed f16-f32 PTX instruction with .rn), so the compiler
// cannot contract or reorder it.
#pragma once

#include <cfloat>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nvq {

constexpr int kStatusNonFinite = 1;
constexpr int kStatusBadIndex = 2;
constexpr int kStatusTimeout = 4;

// ---------------------------------------------------------------- bf16 words
// A 32-bit word holds two bf16 values; element 2k sits in the low half.
__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Per half: max(|a|, |b|) (sign bits of the result are meaningless).  A
// selection, hence exact; NaN halves are ignored.
__device__ __forceinline__ uint32_t maxabs2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per half: max(|a|, |b|), a NaN in either operand giving NaN (sign bits of
// the result are meaningless).
__device__ __forceinline__ uint32_t maxabs2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The larger of the two magnitudes of a max-abs word, as FP32.
__device__ __forceinline__ float amax_of(uint32_t m) {
  m &= 0x7fff7fffu;
  return fmaxf(lo_f(m), hi_f(m));
}

// ----------------------------------------------------------------- E4M3 table
// One 8-byte entry per E4M3 byte: the correctly rounded reciprocal 1/S (0 for
// S = 0, so a zero scale yields sign-only codes) and -S as an f16 pair for
// the residual FMA.  Bytes >= 0x80 never occur (scales are non-negative);
// 0x7F (NaN) only for a non-finite amax, whose outputs are unspecified.
struct __align__(8) ScaleEnt {
  float rcp;
  uint32_t negS2;
};
constexpr int kScaleTableBytes = 128 * 8;

// E4M3 (OCP): bias 7, 3 mantissa bits, subnormals m * 2^-9.
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  if (e == 0) return __fmul_rn((float)m, 0x1p-9f);
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

__device__ __forceinline__ void build_scale_table(ScaleEnt* tbl) {
  for (int b = threadIdx.x; b < 128; b += blockDim.x) {
    float S = e4m3_decode((uint32_t)b);
    ScaleEnt e;
    e.rcp = (b == 0) ? 0.0f : __frcp_rn(S);
    uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn(S)) ^ 0x8000u;
    e.negS2 = h | (h << 16);
    tbl[b] = e;
  }
}

// f16 pair (S, S) of an entry.
__device__ __forceinline__ uint32_t pos_s2(const ScaleEnt& e) { return e.negS2 ^ 0x80008000u; }

// ------------------------------------------------------------- block scales
// fl(a / 6): q0 = a * fl(1/6) followed by one FMA residual correction
// (Markstein's correction step for division by a constant known in advance;
// Brisebarre, Muller and Raina, "Accelerating correctly rounded
// floating-point division when the divisor is known in advance", 2004).
// Checked exhaustively on the host against IEEE division for every binary32
// a >= 2^-124; below that the E4M3 encoding of the quotient is 0 either way.
__device__ __forceinline__ float div6(float a) {
  const float y = 0x1.555556p-3f;  // fl(1/6)
  float q0 = __fmul_rn(a, y);
  float r = __fmaf_rn(-q0, 6.0f, a);
  return __fmaf_rn(r, y, q0);
}

// Two FP32 values -> two E4M3 bytes (RNE, saturating at 448).  Byte 0 of the
// result encodes `lo`, byte 1 encodes `hi`.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t s;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(s) : "f"(hi), "f"(lo));
  return (uint32_t)s;
}

// Scale bytes of one block with scaled amax a: byte 0 = E4M3(a/6) (amax
// mapped to 6), byte 1 = E4M3(a/4) (Four-Over-Six: amax mapped to 4).
__device__ __forceinline__ uint32_t block_scale_bytes(float a) {
  return e4m3x2(div6(a), __fmul_rn(a, 0.25f));
}

// ------------------------------------------------------------------- E2M1
// Two FP32 values -> one byte of two E2M1 codes (RNE, saturating at 6, sign
// kept), element `lo` in the low nibble; also returns the exact f16 pair of
// the two code values (low half = low nibble).
__device__ __forceinline__ uint32_t e2m1x2_enc_dec(float lo, float hi, uint32_t& h2) {
  uint32_t byte;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %2, %3;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, t;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(byte), "=r"(h2)
      : "f"(hi), "f"(lo));
  return byte;
}

// Eight FP32 values q[0..7] -> one word of eight E2M1 codes (q[j] in nibble
// j).  The conversions write their bytes straight into the word.
__device__ __forceinline__ uint32_t e2m1x8_enc(float q0, float q1, float q2, float q3, float q4,
                                               float q5, float q6, float q7) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(q0), "f"(q1), "f"(q2), "f"(q3), "f"(q4), "f"(q5), "f"(q6), "f"(q7));
  return w;
}

// Word of eight E2M1 codes -> the four exact f16 pairs (h[k] = codes 2k, 2k+1).
__device__ __forceinline__ void e2m1x8_dec(uint32_t w, uint32_t h[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t e2m1x8_enc_dec(float q0, float q1, float q2, float q3,
                                                   float q4, float q5, float q6, float q7,
                                                   uint32_t h[4]) {
  const uint32_t w = e2m1x8_enc(q0, q1, q2, q3, q4, q5, q6, q7);
  e2m1x8_dec(w, h);
  return w;
}

// Byte of two E2M1 codes -> exact f16 pair (low half = low nibble).
__device__ __forceinline__ uint32_t e2m1x2_dec(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.u8.u32 t, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(byte));
  return h2;
}

// Residuals t - c*S for the two halves of h2 (codes c as f16), with S given
// as -S in both halves of negS2: one fused multiply-add each, the product
// c*S being exact, so the result is the correctly rounded t - c*S.
__device__ __forceinline__ float2 resid2(uint32_t h2, uint32_t negS2, float tlo, float thi) {
  float dlo, dhi;
  asm("{\n\t.reg .b16 cl, ch, sl, sh;\n\t"
      "mov.b32 {cl, ch}, %2;\n\t"
      "mov.b32 {sl, sh}, %3;\n\t"
      "fma.rn.f32.f16 %0, cl, sl, %4;\n\t"
      "fma.rn.f32.f16 %1, ch, sh, %5;\n\t}"
      : "=f"(dlo), "=f"(dhi)
      : "r"(h2), "r"(negS2), "f"(tlo), "f"(thi));
  return make_float2(dlo, dhi);
}

// Exact f16 pair of the two codes in byte K of w (low half = low nibble).
template <int K>
__device__ __forceinline__ uint32_t e2m1x2_dec_byte(uint32_t w) {
  uint32_t h;
  if constexpr (K == 0)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}" : "=r"(h) : "r"(w));
  else if constexpr (K == 1)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b1;\n\t}" : "=r"(h) : "r"(w));
  else if constexpr (K == 2)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b2;\n\t}" : "=r"(h) : "r"(w));
  else
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b3;\n\t}" : "=r"(h) : "r"(w));
  return h;
}

// Exact products c*S of an f16 code pair and an f16 scale pair, as FP32
// (mixed-precision FMA c*S + (-0): the product has at most six significant
// bits, so nothing is rounded and the sign of zero is kept).
__device__ __forceinline__ float2 cs_exact(uint32_t h2, uint32_t S2) {
  float lo, hi;
  asm("{\n\t.reg .b16 cl, ch, sl, sh;\n\t"
      "mov.b32 {cl, ch}, %2;\n\t"
      "mov.b32 {sl, sh}, %3;\n\t"
      "fma.rn.f32.f16 %0, cl, sl, 0f80000000;\n\t"
      "fma.rn.f32.f16 %1, ch, sl, 0f80000000;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2), "r"(S2));
  return make_float2(lo, hi);
}

// E4M3 byte b -> the exact f16 pair (S, S) of its value (every E4M3 value,
// subnormals included, is an f16).
__device__ __forceinline__ uint32_t e4m3_to_f16x2(uint32_t b) {
  uint32_t h;
  const uint16_t two = (uint16_t)(b | (b << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  return h;
}

// Two FP32 -> bf16 pair (RNE); `lo` in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// bf16 pair -> FP32 pair, exactly: a mixed-precision FMA x*1 + (-0) per half
// runs on the FMA pipe and leaves the (half-rate) ALU pipe to the
// conversions; NVQ_WIDEN_LOGIC selects the two logic operations instead.
__device__ __forceinline__ float2 widen2(uint32_t w) {
#ifndef NVQ_WIDEN_LOGIC
  float lo, hi;
  asm("{\n\t.reg .b16 l, h, one;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "mov.b16 one, 0x3F80;\n\t"
      "fma.rn.f32.bf16 %0, l, one, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %1, h, one, 0f80000000;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w));
  return make_float2(lo, hi);
#else
  return make_float2(lo_f(w), hi_f(w));
#endif
}

// ------------------------------------------------------------ global scales
// G = amax / (6 M) and E = min(1/G, FLT_MAX), with 6M = 2688 (M = 448) or
// 1536 (M = 256 under Four-Over-Six).
__device__ __forceinline__ void global_scales(float amax, float six_m, float& G, float& E) {
  G = __fdiv_rn(amax, six_m);
  E = fminf(__frcp_rn(G), FLT_MAX);
}

// Larger magnitude of the two halves of a max-abs word, as FP32 (both halves
// of the swapped max hold it; the high half is already an FP32 pattern).
__device__ __forceinline__ float amax_fold(uint32_t m) {
  const uint32_t both = maxabs2(m, __byte_perm(m, 0, 0x1032));
  return __uint_as_float(both & 0x7fff0000u);
}

// ---------------------------------------------------------- one NVFP4 block
// Candidate of one rowwise block: t2[k] = (t_2k, t_2k+1).  Writes the 8 code
// bytes into two words and returns the FP32 squared error, accumulated as
// two fused multiply-add chains (even and odd positions) added at the end.
__device__ __forceinline__ float row_candidate(const float2 t2[8], const ScaleEnt se,
                                               uint32_t& c0, uint32_t& c1) {
  const float2 r2 = make_float2(se.rcp, se.rcp);
  float2 q[8];
#pragma unroll
  for (int k = 0; k < 8; k++) q[k] = __fmul2_rn(t2[k], r2);
  uint32_t h[8];
  c0 = e2m1x8_enc_dec(q[0].x, q[0].y, q[1].x, q[1].y, q[2].x, q[2].y, q[3].x, q[3].y, h);
  c1 = e2m1x8_enc_dec(q[4].x, q[4].y, q[5].x, q[5].y, q[6].x, q[6].y, q[7].x, q[7].y, h + 4);
  float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const float2 d = resid2(h[k], se.negS2, t2[k].x, t2[k].y);
    acc = __ffma2_rn(d, d, acc);
  }
  return __fadd_rn(acc.x, acc.y);
}

// Quantises one block given its scaled values t2[k] = (t_2k, t_2k+1) (t = x E)
// and its scaled amax a = fl(bamax E).  Outputs the two code words and the
// scale byte.
template <bool F46>
__device__ __forceinline__ void quant_block_t2(const float2 t2[8], float a, const ScaleEnt* tbl,
                                               uint32_t& c0, uint32_t& c1, uint32_t& sb) {
  const uint32_t sbytes = block_scale_bytes(a);
  const uint32_t s6 = sbytes & 0x7fu;
  const float e6 = row_candidate(t2, tbl[s6], c0, c1);
  sb = s6;
  if (F46) {
    const uint32_t s4 = (sbytes >> 8) & 0x7fu;
    uint32_t d0, d1;
    const float e4 = row_candidate(t2, tbl[s4], d0, d1);
    if (e4 < e6) {
      c0 = d0;
      c1 = d1;
      sb = s4;
    }
  }
}

// Quantises one rowwise block given its 8 bf16x2 words, the block amax (FP32)
// and the slice's encode factor E.  Outputs the two code words and the scale
// byte.
template <bool F46>
__device__ __forceinline__ void quant_row_block_amax(const uint32_t w[8], float bamax, float E,
                                                     const ScaleEnt* tbl, uint32_t& c0,
                                                     uint32_t& c1, uint32_t& sb) {
  float2 t2[8];
  const float2 E2 = make_float2(E, E);
#pragma unroll
  for (int k = 0; k < 8; k++) t2[k] = __fmul2_rn(widen2(w[k]), E2);
  quant_block_t2<F46>(t2, __fmul_rn(bamax, E), tbl, c0, c1, sb);
}

template <bool F46>
__device__ __forceinline__ void quant_row_block(const uint32_t w[8], float E, const ScaleEnt* tbl,
                                                uint32_t& c0, uint32_t& c1, uint32_t& sb) {
  const uint32_t m = maxabs2(maxabs2(maxabs2(w[0], w[1]), maxabs2(w[2], w[3])),
                             maxabs2(maxabs2(w[4], w[5]), maxabs2(w[6], w[7])));
  quant_row_block_amax<F46>(w, amax_fold(m), E, tbl, c0, c1, sb);
}

// ------------------------------------------------------- tiled scale layout
// Byte offset of block scale (r, c) -- row r of the quantised matrix, block
// column c -- in the tensor-core layout of block scales: tiles of 128 rows x
// 4 block columns (512 bytes), row-major over tiles with `ctiles` tiles per
// tile row; inside a tile, row r sits at (r % 32) * 16 + ((r / 32) % 4) * 4
// and column c at c % 4.
__device__ __forceinline__ int64_t scale_off_tiled(int64_t r, int c, int ctiles) {
  return ((r >> 7) * ctiles + (c >> 2)) * 512 + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (c & 3);
}

// ------------------------------------------------------------ small helpers
// Unsigned division by a divisor fixed at launch, for dividends below 2^31:
// n / d = (umulhi(n, m) + n) >> s with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1 (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994).  Built on the host by
// make_fastdiv(); the sum cannot overflow because umulhi(n, m) <= n < 2^31.
struct FastDiv {
  uint32_t d, m, s;
  __device__ __forceinline__ uint32_t div(uint32_t n) const { return (__umulhi(n, m) + n) >> s; }
};

// ---------------------------------------------------- TMA and mbarriers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Plain arrival (release at CTA scope): one of the barrier's expected arrivals.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// No legitimate wait of these kernels lasts more than milliseconds; a wait
// still open after this long is a stall, reported instead of waited out.
constexpr uint64_t kMaxWaitNs = 500000000ull;

// Waits for the phase of `bar` with the given parity to complete, giving up
// after `max_tries` polls or kMaxWaitNs of wall-clock time, whichever comes
// first (a poll may itself block for a short, hardware-defined time, so the
// count alone does not bound the time).  Returns false on giving up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_tries) {
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < max_tries; i++) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    const uint64_t now = globaltimer_ns();
    if (i == 0) t0 = now;
    else if (now - t0 > kMaxWaitNs) return false;
  }
  return false;
}

// Non-blocking: whether the phase of `bar` with the given parity has completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Barrier `id` (1 .. 15) over the first `n` threads that reach it: a group
// of warps synchronising without the rest of the CTA.
__device__ __forceinline__ void named_barrier(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// named_barrier that also returns whether `pred` held for any of the n threads.
__device__ __forceinline__ bool named_barrier_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// 1-D bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`, with an L2
// eviction policy.
__device__ __forceinline__ void bulk_load_hint(void* smem_dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 2-D tiled TMA load of one box at element coordinates (x, y) into shared
// memory, completing on `bar` (x * element size must be a multiple of 16).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// L2 eviction policies for the cache-hinted loads below: evict-first for
// data read for the last time, evict-last for data that is read again soon.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_2d with an L2 eviction policy.
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map, int x,
                                                 int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------ grid-wide arrival counts
// Words shared by the CTAs of one co-resident grid.
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Returns the old value; the release orders the thread's earlier memory
// operations (and those ordered before them in its CTA) before the add.
__device__ __forceinline__ uint32_t atom_add_release(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ float ld_relaxed_f32(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// A per-slice word holding a finished result has its sign bit set.
constexpr uint32_t kSliceDone = 0x80000000u;

// Polls *p until its kSliceDone bit is set (the word is returned in `w`),
// giving up after `max_polls` polls or kMaxWaitNs of wall-clock time,
// whichever comes first.  Returns false on giving up.
__device__ __forceinline__ bool wait_done(const uint32_t* p, uint32_t& w,
                                          uint32_t max_polls = 1u << 24) {
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < max_polls; i++) {
    w = ld_relaxed_u32(p);
    if (w & kSliceDone) return true;
    const uint64_t now = globaltimer_ns();
    if (i == 0) t0 = now;
    else if (now - t0 > kMaxWaitNs) return false;
    __nanosleep(32);
  }
  return false;
}

// Orders generic-proxy shared-memory writes before later TMA reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32-byte vector load (read-only path, no L1 allocation).
__device__ __forceinline__ void ldg32(const void* p, uint32_t v[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "l"(p));
}

// 32-byte store (one whole L2 sector per lane; 32-byte aligned address).
__device__ __forceinline__ void stg256(void* p, const uint32_t v[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// The same with the streaming (evict-first) hint.
__device__ __forceinline__ void stg256_stream(void* p, const uint32_t v[8]) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Streaming 16-byte store (evict-first: the output is not read back soon).
__device__ __forceinline__ void stg_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Streaming (evict-first) 8-, 4- and 1-byte stores.
__device__ __forceinline__ void stg_stream_v2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void stg_stream_u32(void* p, uint32_t a) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}
__device__ __forceinline__ void stg_stream_u8(void* p, uint32_t a) {
  asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace nvq
