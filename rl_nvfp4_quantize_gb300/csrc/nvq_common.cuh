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
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nvq {

constexpr int kStatusNonFinite = 1;
constexpr int kStatusBadIndex = 2;

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

// Per half: unsigned 16-bit max of the magnitude bits.  NaN patterns compare
// above infinity, so a NaN anywhere propagates to the result.
__device__ __forceinline__ uint32_t umaxmag2(uint32_t m, uint32_t w) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(m), "r"(w & 0x7fff7fffu));
  return d;
}

// The larger of the two magnitudes of a max-abs word, as FP32.
__device__ __forceinline__ float amax_of(uint32_t m) {
  m &= 0x7fff7fffu;
  return fmaxf(lo_f(m), hi_f(m));
}

// ----------------------------------------------------------------- E4M3 table
// One entry per non-negative E4M3 byte: its value S, the correctly rounded
// reciprocal 1/S (0 for S = 0, so a zero scale yields sign-only codes), and
// -S as an f16 pair for the residual FMA.
struct __align__(16) ScaleEnt {
  float S;
  float rcp;
  uint32_t negS2;
  uint32_t pad;
};

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
    e.S = S;
    e.rcp = (b == 0) ? 0.0f : __frcp_rn(S);
    uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn(S)) ^ 0x8000u;
    e.negS2 = h | (h << 16);
    e.pad = 0;
    tbl[b] = e;
  }
}

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

__device__ __forceinline__ float2 div6x2(float2 a) {
  const float2 y = make_float2(0x1.555556p-3f, 0x1.555556p-3f);
  const float2 m6 = make_float2(-6.0f, -6.0f);
  float2 q0 = __fmul2_rn(a, y);
  float2 r = __ffma2_rn(q0, m6, a);
  return __ffma2_rn(r, y, q0);
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

// Two FP32 -> bf16 pair (RNE); `lo` in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// ------------------------------------------------------------ global scales
// G = amax / (6 M) and E = min(1/G, FLT_MAX), with 6M = 2688 (M = 448) or
// 1536 (M = 256 under Four-Over-Six).
__device__ __forceinline__ void global_scales(float amax, float six_m, float& G, float& E) {
  G = __fdiv_rn(amax, six_m);
  E = fminf(__frcp_rn(G), FLT_MAX);
}

// ---------------------------------------------------------- one NVFP4 block
// Candidate of one rowwise block: t2[k] = (t_2k, t_2k+1).  Writes the 8 code
// bytes into two words and returns the FP32 squared error, accumulated as
// two fused multiply-add chains (even and odd positions) added at the end.
__device__ __forceinline__ float row_candidate(const float2 t2[8], const ScaleEnt& se,
                                               uint32_t& c0, uint32_t& c1) {
  const float2 r2 = make_float2(se.rcp, se.rcp);
  float2 acc = make_float2(0.0f, 0.0f);
  c0 = 0;
  c1 = 0;
#pragma unroll
  for (int k = 0; k < 8; k++) {
    float2 q = __fmul2_rn(t2[k], r2);
    uint32_t h2;
    uint32_t b = e2m1x2_enc_dec(q.x, q.y, h2);
    float2 d = resid2(h2, se.negS2, t2[k].x, t2[k].y);
    acc = __ffma2_rn(d, d, acc);
    if (k < 4) c0 |= b << (8 * k); else c1 |= b << (8 * (k - 4));
  }
  return __fadd_rn(acc.x, acc.y);
}

// Quantises one rowwise block given its 8 bf16x2 words and the slice's
// encode factor E.  Outputs the two code words and the scale byte.
template <bool F46>
__device__ __forceinline__ void quant_row_block(const uint32_t w[8], float E, const ScaleEnt* tbl,
                                                uint32_t& c0, uint32_t& c1, uint32_t& sb) {
  uint32_t m = maxabs2(maxabs2(maxabs2(w[0], w[1]), maxabs2(w[2], w[3])),
                       maxabs2(maxabs2(w[4], w[5]), maxabs2(w[6], w[7])));
  float a = __fmul_rn(amax_of(m), E);
  uint32_t sbytes = block_scale_bytes(a);
  float2 t2[8];
  const float2 E2 = make_float2(E, E);
#pragma unroll
  for (int k = 0; k < 8; k++) t2[k] = __fmul2_rn(make_float2(lo_f(w[k]), hi_f(w[k])), E2);
  const uint32_t s6 = sbytes & 0x7fu;
  float e6 = row_candidate(t2, tbl[s6], c0, c1);
  sb = s6;
  if (F46) {
    const uint32_t s4 = (sbytes >> 8) & 0x7fu;
    uint32_t d0, d1;
    float e4 = row_candidate(t2, tbl[s4], d0, d1);
    if (e4 < e6) {
      c0 = d0;
      c1 = d1;
      sb = s4;
    }
  }
}

// Same as quant_row_block but with the block amax already known (as FP32).
template <bool F46>
__device__ __forceinline__ void quant_row_block_amax(const uint32_t w[8], float bamax, float E,
                                                     const ScaleEnt* tbl, uint32_t& c0,
                                                     uint32_t& c1, uint32_t& sb) {
  float a = __fmul_rn(bamax, E);
  uint32_t sbytes = block_scale_bytes(a);
  float2 t2[8];
  const float2 E2 = make_float2(E, E);
#pragma unroll
  for (int k = 0; k < 8; k++) t2[k] = __fmul2_rn(make_float2(lo_f(w[k]), hi_f(w[k])), E2);
  const uint32_t s6 = sbytes & 0x7fu;
  float e6 = row_candidate(t2, tbl[s6], c0, c1);
  sb = s6;
  if (F46) {
    const uint32_t s4 = (sbytes >> 8) & 0x7fu;
    uint32_t d0, d1;
    float e4 = row_candidate(t2, tbl[s4], d0, d1);
    if (e4 < e6) {
      c0 = d0;
      c1 = d1;
      sb = s4;
    }
  }
}

// Candidate of two columnwise blocks side by side (columns j and j+1):
// u[i] = (t_ij, t_i,j+1) for the 16 rows i of the block.  Codes of column j
// go to cj0/cj1 and of column j+1 to ck0/ck1, each packed along the block
// (element 2k in the low nibble of byte k).  Returns both errors.
__device__ __forceinline__ float2 col_candidate(const float2 u[16], const ScaleEnt& sj,
                                                const ScaleEnt& sk, uint32_t& cj0, uint32_t& cj1,
                                                uint32_t& ck0, uint32_t& ck1) {
  const float2 r2 = make_float2(sj.rcp, sk.rcp);
  float2 accE = make_float2(0.0f, 0.0f), accO = make_float2(0.0f, 0.0f);
  cj0 = cj1 = ck0 = ck1 = 0;
#pragma unroll
  for (int k = 0; k < 8; k++) {
    float2 q0 = __fmul2_rn(u[2 * k], r2);
    float2 q1 = __fmul2_rn(u[2 * k + 1], r2);
    uint32_t hj, hk;
    uint32_t bj = e2m1x2_enc_dec(q0.x, q1.x, hj);
    uint32_t bk = e2m1x2_enc_dec(q0.y, q1.y, hk);
    float2 dj = resid2(hj, sj.negS2, u[2 * k].x, u[2 * k + 1].x);
    float2 dk = resid2(hk, sk.negS2, u[2 * k].y, u[2 * k + 1].y);
    float2 de = make_float2(dj.x, dk.x), dod = make_float2(dj.y, dk.y);
    accE = __ffma2_rn(de, de, accE);
    accO = __ffma2_rn(dod, dod, accO);
    if (k < 4) {
      cj0 |= bj << (8 * k);
      ck0 |= bk << (8 * k);
    } else {
      cj1 |= bj << (8 * (k - 4));
      ck1 |= bk << (8 * (k - 4));
    }
  }
  return __fadd2_rn(accE, accO);
}

// Quantises the two columnwise blocks held in 16 words wc[i] (row i of the
// block; low half = column j, high half = column j+1).
template <bool F46>
__device__ __forceinline__ void quant_col_pair(const uint32_t wc[16], float E, const ScaleEnt* tbl,
                                               uint32_t cj[2], uint32_t ck[2], uint32_t& sbj,
                                               uint32_t& sbk) {
  uint32_t m = wc[0];
#pragma unroll
  for (int i = 1; i < 16; i++) m = maxabs2(m, wc[i]);
  m &= 0x7fff7fffu;
  const float2 E2 = make_float2(E, E);
  float2 a = __fmul2_rn(make_float2(lo_f(m), hi_f(m)), E2);
  float2 a6 = div6x2(a);
  float2 a4 = __fmul2_rn(a, make_float2(0.25f, 0.25f));
  uint32_t s6 = e4m3x2(a6.x, a6.y);  // byte 0: column j, byte 1: column j+1
  uint32_t s4 = e4m3x2(a4.x, a4.y);
  float2 u[16];
#pragma unroll
  for (int i = 0; i < 16; i++) u[i] = __fmul2_rn(make_float2(lo_f(wc[i]), hi_f(wc[i])), E2);
  const uint32_t s6j = s6 & 0x7fu, s6k = (s6 >> 8) & 0x7fu;
  float2 e6 = col_candidate(u, tbl[s6j], tbl[s6k], cj[0], cj[1], ck[0], ck[1]);
  sbj = s6j;
  sbk = s6k;
  if (F46) {
    const uint32_t s4j = s4 & 0x7fu, s4k = (s4 >> 8) & 0x7fu;
    uint32_t dj0, dj1, dk0, dk1;
    float2 e4 = col_candidate(u, tbl[s4j], tbl[s4k], dj0, dj1, dk0, dk1);
    if (e4.x < e6.x) {
      cj[0] = dj0;
      cj[1] = dj1;
      sbj = s4j;
    }
    if (e4.y < e6.y) {
      ck[0] = dk0;
      ck[1] = dk1;
      sbk = s4k;
    }
  }
}

// ------------------------------------------------------------ small helpers
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace nvq
