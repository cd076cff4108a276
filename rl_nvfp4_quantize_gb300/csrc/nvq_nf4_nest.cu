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

// The tree sum of chunk `ch` of slice `a` (4096 leaves, a complete subtree):
// eight leaves per thread added pairwise in registers, then the 32 lanes of a
// warp with butterfly shuffles at distances 1, 2, ..., 16 (lane l meets l ^ d,
// so every addition joins two adjacent subtrees; IEEE addition is
// commutative, so both lanes hold the same sum), then the 16 warps the same
// way.  The result is valid in thread 0; `ws` is reused on return.
// Two chunks are summed together (their loads in flight at once): chunk ch0
// of slice a0 and chunk ch1 of slice a1 (a1 null: none), results in r[0], r[1].
__device__ __forceinline__ void chunk_tree_sums(const float* a0, int64_t ch0, const float* a1,
                                                int64_t ch1, int64_t n, bool vec, float* ws,
                                                float r[2]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float v[8], u[8];
  load8(a0, ch0 * kNestLeaves + (int64_t)tid * 8, n, vec, v);
  if (a1) {
    load8(a1, ch1 * kNestLeaves + (int64_t)tid * 8, n, vec, u);
  } else {
#pragma unroll
    for (int j = 0; j < 8; j++) u[j] = 0.0f;
  }
  float s = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
  float q = ((u[0] + u[1]) + (u[2] + u[3])) + ((u[4] + u[5]) + (u[6] + u[7]));
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    s = s + __shfl_xor_sync(0xffffffffu, s, d);
    q = q + __shfl_xor_sync(0xffffffffu, q, d);
  }
  if (lane == 0) {
    ws[warp] = s;
    ws[kNestWarps + warp] = q;
  }
  __syncthreads();
  if (warp == 0) {
    float t = lane < kNestWarps ? ws[lane] : 0.0f;
    float w = lane < kNestWarps ? ws[kNestWarps + lane] : 0.0f;
#pragma unroll
    for (int d = 1; d < kNestWarps; d <<= 1) {
      t = t + __shfl_xor_sync(0xffffffffu, t, d);
      w = w + __shfl_xor_sync(0xffffffffu, w, d);
    }
    r[0] = t;
    r[1] = w;
  }
  __syncthreads();
}

// Launch 1: the chunk sums of every slice, CTAs striding over the chunks of
// all slices, into the first ceil(n / 4096) entries of the slice's row of c1
// (the row has ceil(n / 256) entries; launch 3 overwrites it with the block
// maxima).
__global__ void __launch_bounds__(kNestThreads)
k_nf4_nest_chunks(const float* __restrict__ absmax, int64_t nexp, int64_t n, float* __restrict__ c1) {
  __shared__ float ws[2 * kNestWarps];
  const int64_t nch = (n + kNestLeaves - 1) / kNestLeaves, nb = (n + 255) / 256;
  const int64_t total = nexp * nch;
  const bool vec = (n & 3) == 0 && (reinterpret_cast<uintptr_t>(absmax) & 15) == 0;
  for (int64_t gc = blockIdx.x; gc < total; gc += 2 * (int64_t)gridDim.x) {
    const int64_t g1 = gc + gridDim.x;
    const int64_t e0 = gc / nch, ch0 = gc - e0 * nch;
    const int64_t e1 = g1 < total ? g1 / nch : 0, ch1 = g1 < total ? g1 - e1 * nch : 0;
    float r[2] = {0.0f, 0.0f};
    chunk_tree_sums(absmax + e0 * n, ch0, g1 < total ? absmax + e1 * n : nullptr, ch1, n, vec, ws, r);
    if (threadIdx.x == 0) {
      c1[e0 * nb + ch0] = r[0];
      if (g1 < total) c1[e1 * nb + ch1] = r[1];
    }
  }
}

// Launch 2: one CTA per slice adds the chunk sums, zero padded to a power of
// two, level by level in shared memory (each level read completely before it
// is written), and forms the mean.
__global__ void __launch_bounds__(kNestThreads)
k_nf4_nest_mean(const float* __restrict__ c1, int64_t nexp, int64_t n, float* __restrict__ mean,
                int* status) {
  __shared__ float csum[kNestMaxChunks];
  const int tid = threadIdx.x;
  const int64_t nch = (n + kNestLeaves - 1) / kNestLeaves, nb = (n + 255) / 256;
  int64_t P = 1;
  while (P < nch) P *= 2;
  for (int64_t e = blockIdx.x; e < nexp; e += gridDim.x) {
    for (int64_t i = tid; i < P; i += kNestThreads) csum[i] = i < nch ? c1[e * nb + i] : 0.0f;
    __syncthreads();
    for (int64_t len = P; len > 1; len >>= 1) {
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
    if (tid == 0) {
      const float S = nch > 0 ? csum[0] : 0.0f;
      const float mu = n > 0 ? __double2float_rn(__ddiv_rn((double)S, (double)n)) : 0.0f;
      mean[e] = mu;
      if (status && !isfinite(mu)) atomicOr(status, kStatusNonFinite);
    }
    __syncthreads();  // csum is rewritten by the next slice
  }
}

// Launch 3: E4M3 codes of the centred values, one warp per block of 256
// (eight values per lane), warps striding over the blocks of all slices.
constexpr int kNestCodeThreads = 256;

__global__ void __launch_bounds__(kNestCodeThreads)
k_nf4_nest_codes(const float* __restrict__ absmax, int64_t nexp, int64_t n,
                 uint8_t* __restrict__ codes, float* __restrict__ c1,
                 const float* __restrict__ mean, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = (n + 255) / 256, total = nexp * nb;
  const bool vec = (n & 3) == 0 && (reinterpret_cast<uintptr_t>(absmax) & 15) == 0;
  const bool vec_out = (n & 7) == 0 && (reinterpret_cast<uintptr_t>(codes) & 7) == 0;
  const int64_t warps = (int64_t)gridDim.x * (kNestCodeThreads / 32);
  // block gb of all slices (e = gb / nb): centre, block maximum, codes
  auto finish = [&](int64_t gb, float v[8]) {
    const int64_t e = gb / nb, b = gb - e * nb;
    const float mu = mean[e];
    const int64_t i0 = b * 256 + lane * 8;
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
  };
  auto load = [&](int64_t gb, float v[8]) {
    const int64_t e = gb / nb, b = gb - e * nb;
    load8(absmax + e * n, b * 256 + lane * 8, n, vec, v);
  };
  // two blocks per warp at a time, both loads in flight before either is used
  for (int64_t gb = (int64_t)blockIdx.x * (kNestCodeThreads / 32) + (threadIdx.x >> 5); gb < total;
       gb += 2 * warps) {
    const int64_t gb1 = gb + warps;
    float v0[8], v1[8];
    load(gb, v0);
    if (gb1 < total) load(gb1, v1);
    finish(gb, v0);
    if (gb1 < total) finish(gb1, v1);
  }
}

cudaError_t launch_nf4_nest(const float* absmax, int64_t nexp, int64_t n, uint8_t* codes,
                            float* c1, float* mean, int* status, cudaStream_t s) {
  if (nexp <= 0 || n <= 0) return cudaSuccess;
  if (n > (int64_t)kNestMaxChunks * kNestLeaves) return cudaErrorInvalidValue;
  const DevInfo* di = device_info();
  // launches 1 and 3 stride over all slices with as many CTAs as fit at once
  const int64_t nch = (n + kNestLeaves - 1) / kNestLeaves;
  const int g1 = (int)std::min<int64_t>(nexp * nch, (int64_t)di->sms * 4);
  k_nf4_nest_chunks<<<g1, kNestThreads, 0, s>>>(absmax, nexp, n, c1);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int gm = (int)std::min<int64_t>(nexp, (int64_t)di->sms * 2);
  k_nf4_nest_mean<<<gm, kNestThreads, 0, s>>>(c1, nexp, n, mean, status);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const int64_t blocks = nexp * ((n + 255) / 256);
  const int gc = (int)std::min<int64_t>((blocks + 7) / 8, (int64_t)di->sms * 4);
  k_nf4_nest_codes<<<gc, kNestCodeThreads, 0, s>>>(absmax, nexp, n, codes, c1, mean, status);
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
