// nvq_nf4_nest.cu -- the nested (double-quantised) NF4 absmax for sm_103a.
//
// Source: "nf4moe -- QLoRA for a 743B Fused-MoE", "The fix: dequant-on-forward
// for routed experts": the NF4 state of each expert slice holds its absmax
// and a "nested code".  Read as the published double quantisation of QLoRA
// (Dettmers et al., 2023, "Double Quantization"): the slice's FP32 absmax
// values are centred on their mean and quantised again to 8-bit floats in
// blocks of 256.  The readings where that description is silent:
//   mean  = RN32(RN64(S / n)), S the FP32 pairwise-tree sum of the n values
//           (zero padded to a power of two, adjacent pairs added per level);
//   code  = E4M3(fl(fl(a - mean) * k)), k = min(fl(448 / c1), FLT_MAX), c1 the
//           block's largest |fl(a - mean)|; nearest-even, saturating, sign kept;
//   value = fma(E4M3 value of code, fl(c1 / 448), mean).
//
// The absmax arrays are 1/64 of the weights, so these kernels are small next
// to the NF4 quantisation itself; they are written to be HBM-bound anyway.
#include <cfloat>
#include <algorithm>
#include <cstdint>

#include "nvq_common.cuh"
#include "nvq_internal.h"

namespace nvq {

constexpr int kNestThreads = 512;
constexpr int kNestWarps = kNestThreads / 32;
constexpr int kNestLeaves = kNestThreads * 8;  // leaves of one chunk's subtree
constexpr int kNestMaxChunks = 8192;           // n <= 2^25 absmax values per slice

static_assert(kNestMaxChunks * kNestLeaves == (1 << 25), "chunk limit");

// E4M3 bytes of two FP32 values with the sign kept (byte 0 encodes lo).
__device__ __forceinline__ uint32_t e4m3x2_signed(float lo, float hi) {
  uint16_t s;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(s) : "f"(hi), "f"(lo));
  return (uint32_t)s;
}

// Eight leaves of one thread, zero beyond n.
__device__ __forceinline__ void load8(const float* a, int64_t i0, int64_t n, bool vec, float v[8]) {
  if (vec && i0 + 8 <= n) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(a + i0));
    const float4 y = __ldg(reinterpret_cast<const float4*>(a + i0 + 4));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; j++) v[j] = (i0 + j < n) ? __ldg(a + i0 + j) : 0.0f;
  }
}

// One CTA per slice (grid-stride over slices).  Pass 1 forms the tree sum:
// each chunk of 4096 leaves is a complete subtree -- eight leaves per thread
// added pairwise in registers, then the 32 lanes of a warp with butterfly
// shuffles at distances 1, 2, ..., 16 (lane l meets l ^ d, so every addition
// joins two adjacent subtrees; IEEE addition is commutative, so both lanes
// hold the same sum), then the 16 warps the same way.  The chunk sums,
// zero padded to a power of two, are added level by level in shared memory.
// Pass 2 quantises: one warp per block of 256, eight values per lane.
__global__ void __launch_bounds__(kNestThreads)
k_nf4_nest(const float* __restrict__ absmax, int64_t nexp, int64_t n, uint8_t* __restrict__ codes,
           float* __restrict__ c1, float* __restrict__ mean, int* status) {
  __shared__ float csum[kNestMaxChunks];
  __shared__ float ws[kNestWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nch = (n + kNestLeaves - 1) / kNestLeaves;
  int64_t P = 1;
  while (P < nch) P *= 2;
  const int64_t nb = (n + 255) / 256;
  const bool vec = (n & 3) == 0 && (reinterpret_cast<uintptr_t>(absmax) & 15) == 0;
  const bool vec_out = (n & 7) == 0 && (reinterpret_cast<uintptr_t>(codes) & 7) == 0;

  for (int64_t e = blockIdx.x; e < nexp; e += gridDim.x) {
    const float* a = absmax + e * n;
    // ---- pass 1: the pairwise tree sum
    for (int64_t ch = 0; ch < nch; ch++) {
      float v[8];
      load8(a, ch * kNestLeaves + (int64_t)tid * 8, n, vec, v);
      float s = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) s = s + __shfl_xor_sync(0xffffffffu, s, d);
      if (lane == 0) ws[warp] = s;
      __syncthreads();
      if (warp == 0) {
        float t = lane < kNestWarps ? ws[lane] : 0.0f;
#pragma unroll
        for (int d = 1; d < kNestWarps; d <<= 1) t = t + __shfl_xor_sync(0xffffffffu, t, d);
        if (lane == 0) csum[ch] = t;
      }
      __syncthreads();
    }
    for (int64_t i = nch + tid; i < P; i += kNestThreads) csum[i] = 0.0f;
    __syncthreads();
    for (int64_t len = P; len > 1; len >>= 1) {
      // read every pair of this level before any sum of it is written
      constexpr int kPer = kNestMaxChunks / 2 / kNestThreads;
      float part[kPer];
#pragma unroll
      for (int j = 0; j < kPer; j++) {
        const int64_t i = tid + j * kNestThreads;
        part[j] = i < len / 2 ? csum[2 * i] + csum[2 * i + 1] : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kPer; j++) {
        const int64_t i = tid + j * kNestThreads;
        if (i < len / 2) csum[i] = part[j];
      }
      __syncthreads();
    }
    const float S = nch > 0 ? csum[0] : 0.0f;
    const float mu = n > 0 ? __double2float_rn(__ddiv_rn((double)S, (double)n)) : 0.0f;
    if (tid == 0) {
      mean[e] = mu;
      if (status && !isfinite(mu)) atomicOr(status, kStatusNonFinite);
    }

    // ---- pass 2: E4M3 codes of the centred values, one warp per block
    for (int64_t b = warp; b < nb; b += kNestWarps) {
      const int64_t i0 = b * 256 + lane * 8;
      float v[8];
      load8(a, i0, n, vec, v);
      float m = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        v[j] = __fsub_rn(v[j], mu);
        if (i0 + j < n) m = fmaxf(m, fabsf(v[j]));
      }
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
      const float k = fminf(__fdiv_rn(448.0f, m), FLT_MAX);
      uint32_t q[4];
#pragma unroll
      for (int j = 0; j < 4; j++) q[j] = e4m3x2_signed(__fmul_rn(v[2 * j], k), __fmul_rn(v[2 * j + 1], k));
      uint8_t* dst = codes + e * n + i0;
      if (vec_out && i0 + 8 <= n) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
      } else {
#pragma unroll
        for (int j = 0; j < 8; j++)
          if (i0 + j < n) dst[j] = (uint8_t)(q[j >> 1] >> (8 * (j & 1)));
      }
      if (lane == 0) {
        c1[e * nb + b] = m;
        if (status && !isfinite(m)) atomicOr(status, kStatusNonFinite);
      }
    }
    __syncthreads();  // csum is rewritten by the next slice
  }
}

cudaError_t launch_nf4_nest(const float* absmax, int64_t nexp, int64_t n, uint8_t* codes,
                            float* c1, float* mean, int* status, cudaStream_t s) {
  if (nexp <= 0) return cudaSuccess;
  if (n > (int64_t)kNestMaxChunks * kNestLeaves) return cudaErrorInvalidValue;
  const DevInfo* di = device_info();
  const int grid = (int)std::min<int64_t>(nexp, (int64_t)di->sms * 2);
  k_nf4_nest<<<grid, kNestThreads, 0, s>>>(absmax, nexp, n, codes, c1, mean, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ decode
// Eight values per thread: grid.y walks the slices, grid.x the values.
constexpr int kUnnestThreads = 256;

__device__ __forceinline__ float e4m3_value(uint32_t byte) {
  uint32_t h;
  const uint16_t two = (uint16_t)(byte & 0xffu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

__global__ void __launch_bounds__(kUnnestThreads)
k_nf4_unnest(const uint8_t* __restrict__ codes, const float* __restrict__ c1,
             const float* __restrict__ mean, int64_t nexp, int64_t n, float* __restrict__ out,
             bool vec) {
  const int64_t nb = (n + 255) / 256;
  for (int64_t e = blockIdx.y; e < nexp; e += gridDim.y) {
    const float mu = mean[e];
    for (int64_t i0 = ((int64_t)blockIdx.x * kUnnestThreads + threadIdx.x) * 8; i0 < n;
         i0 += (int64_t)gridDim.x * kUnnestThreads * 8) {
      // eight values never straddle a block of 256 (i0 is a multiple of 8)
      const float r = __fdiv_rn(c1[e * nb + i0 / 256], 448.0f);
      const uint8_t* src = codes + e * n + i0;
      float* dst = out + e * n + i0;
      if (vec && i0 + 8 <= n) {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
          const uint32_t byte = ((j < 4 ? w.x : w.y) >> (8 * (j & 3))) & 0xffu;
          y[j] = __fmaf_rn(e4m3_value(byte), r, mu);
        }
        reinterpret_cast<float4*>(dst)[0] = make_float4(y[0], y[1], y[2], y[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(y[4], y[5], y[6], y[7]);
      } else {
        for (int j = 0; j < 8 && i0 + j < n; j++) dst[j] = __fmaf_rn(e4m3_value(src[j]), r, mu);
      }
    }
  }
}

cudaError_t launch_nf4_unnest(const uint8_t* codes, const float* c1, const float* mean,
                              int64_t nexp, int64_t n, float* out, cudaStream_t s) {
  if (nexp <= 0 || n <= 0) return cudaSuccess;
  const DevInfo* di = device_info();
  const bool vec = (n & 7) == 0 && (reinterpret_cast<uintptr_t>(codes) & 7) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  const int64_t per = (n + 8 * kUnnestThreads - 1) / (8 * kUnnestThreads);
  const int64_t target = (int64_t)di->sms * 8;  // CTAs in flight over all slices
  dim3 grid((unsigned)std::max<int64_t>(1, std::min<int64_t>(per, std::max<int64_t>(1, target / nexp))),
            (unsigned)std::min<int64_t>(nexp, 65535));
  k_nf4_unnest<<<grid, kUnnestThreads, 0, s>>>(codes, c1, mean, nexp, n, out, vec);
  return cudaGetLastError();
}

}  // namespace nvq
