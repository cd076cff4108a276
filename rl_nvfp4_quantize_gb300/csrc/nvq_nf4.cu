// nvq_nf4.cu -- NF4 kernels for sm_103a: blockwise quantisation with block
// size 64, dequantisation of whole expert slices, the routed-expert union
// and the routed dequant-on-forward.
//
// Source: "nf4moe -- QLoRA for a 743B Fused-MoE", "The fix: dequant-on-forward
// for routed experts" (experts stored as NF4 with one absmax per 64 elements;
// the union of top_k_index is formed once and only those experts are
// dequantised) and "Making it fast: the step tax" (the per-step dequant cost
// this path exists to shrink).
#include <cfloat>
#include <algorithm>
#include <cstdint>

#include "nvq_common.cuh"
#include "nvq_internal.h"
#include "nvq_nf4_levels.cuh"

namespace nvq {

static const float h_nf4[16] = NVQ_NF4_LEVELS;

void nf4_levels_host(float out[16]) {
  for (int i = 0; i < 16; i++) out[i] = h_nf4[i];
}

// --------------------------------------------------------------- quantise
// The nearest level is found through the cell of g = fl(16 v + 96): for every
// |v| < 2, g lies in [64, 128), where floats step by 2^-17, so bits 17..22 of
// g number 64 cells of width 1/16 in v.  g never decreases as v grows, and the
// NF4 midpoints lie more than 1/16 apart, so a cell holds at most one midpoint
// mu; the code, the number of midpoints strictly below v, is then
// lo + (v > mu), with lo the number of midpoints in lower cells and mu = +inf
// in cells without one.  Any float (a NaN or an infinity too) lands in one of
// the 64 cells.  The 64-entry table is replicated for the 32 lanes (row of
// cell c at byte 256 c, lane l at byte 8 l): every lookup of a warp touches
// each bank pair once, whatever cells its lanes hit.
struct __align__(8) Nf4Ent {
  float thr;
  int lo;
};
constexpr int kNf4Cells = 64;
constexpr int kNqThreads = 256;
constexpr int kNqSmem = kNf4Cells * 32 * 8;

// Byte offset of the table row of the cell of g.
__device__ __forceinline__ uint32_t nf4_cell_row(float g) {
  return (__float_as_uint(g) >> 9) & ((uint32_t)(kNf4Cells - 1) << 8);
}

__device__ __forceinline__ void build_nf4_cells(Nf4Ent* tbl) {
  float m[15];
  uint32_t cm[15];
#pragma unroll
  for (int j = 0; j < 15; j++) {
    m[j] = __fmul_rn(__fadd_rn(c_nf4[j], c_nf4[j + 1]), 0.5f);
    cm[j] = nf4_cell_row(__fmaf_rn(m[j], 16.0f, 96.0f)) >> 8;
  }
  for (int idx = threadIdx.x; idx < kNf4Cells * 32; idx += blockDim.x) {
    const uint32_t cell = (uint32_t)idx >> 5;
    Nf4Ent ent;
    ent.thr = __int_as_float(0x7f800000);
    ent.lo = 0;
#pragma unroll
    for (int j = 0; j < 15; j++) {
      if (cm[j] < cell) ent.lo++;
      else if (cm[j] == cell) ent.thr = m[j];
    }
    tbl[idx] = ent;
  }
}

// Code of v; g = fl(16 v + 96); `lane_tbl` is this lane's column of the table.
__device__ __forceinline__ uint32_t nf4_code(float v, float g, const unsigned char* lane_tbl) {
  const Nf4Ent e = *reinterpret_cast<const Nf4Ent*>(lane_tbl + nf4_cell_row(g));
  return (uint32_t)e.lo + (v > e.thr ? 1u : 0u);
}

// One thread per half block (32 elements = 64 bytes); the two halves of a
// block sit in adjacent lanes and exchange their maxima by shuffle.
__global__ void __launch_bounds__(kNqThreads)
    k_nf4_quant(const uint16_t* __restrict__ w, int64_t nhalf, uint8_t* __restrict__ codes,
                float* __restrict__ absmax, int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem[];
  build_nf4_cells(reinterpret_cast<Nf4Ent*>(smem));
  __syncthreads();
  const unsigned char* const lane_tbl = smem + (threadIdx.x & 31) * 8;
  const int64_t stride = (int64_t)gridDim.x * kNqThreads;
  const float2 k16 = make_float2(16.0f, 16.0f), k96 = make_float2(96.0f, 96.0f);
  const bool w32 = (reinterpret_cast<uintptr_t>(w) & 31) == 0;
  // half block h's 64 bytes as two 32-byte loads (one full sector each) when
  // the stack is 32-byte aligned, else as four 16-byte loads; zeros past the end
  auto load = [&](int64_t h, uint4 v[4]) {
    if (h < nhalf && !w32) {
#pragma unroll
      for (int u = 0; u < 4; u++) v[u] = __ldg(reinterpret_cast<const uint4*>(w + h * 32 + u * 8));
    } else if (h < nhalf) {
      uint32_t a[8], b[8];
      ldg32(w + h * 32, a);
      ldg32(w + h * 32 + 16, b);
      v[0] = make_uint4(a[0], a[1], a[2], a[3]);
      v[1] = make_uint4(a[4], a[5], a[6], a[7]);
      v[2] = make_uint4(b[0], b[1], b[2], b[3]);
      v[3] = make_uint4(b[4], b[5], b[6], b[7]);
    } else {
#pragma unroll
      for (int u = 0; u < 4; u++) v[u] = make_uint4(0, 0, 0, 0);
    }
  };
  // The loop bound is taken at the warp's first lane so that whole warps
  // stay together for the shuffle; lanes past the end only skip the stores.
  // Each thread loads its next half block before it quantises this one, so
  // two are in flight per thread.
  int64_t h = (int64_t)blockIdx.x * kNqThreads + threadIdx.x;
  uint4 v[4], vn[4];
  load(h, v);
  for (; h - (threadIdx.x & 31) < nhalf; h += stride) {
    const bool act = h < nhalf;
    load(h + stride, vn);
    uint32_t m = maxabs2_nan(v[0].x, v[0].y);
    m = maxabs2_nan(m, v[0].z);
    m = maxabs2_nan(m, v[0].w);
#pragma unroll
    for (int u = 1; u < 4; u++) {
      m = maxabs2_nan(m, v[u].x);
      m = maxabs2_nan(m, v[u].y);
      m = maxabs2_nan(m, v[u].z);
      m = maxabs2_nan(m, v[u].w);
    }
    uint32_t mm = maxabs2_nan(m, __byte_perm(m, 0, 0x1032)) & 0x7fff0000u;  // FP32 bits
    mm = max(mm, __shfl_xor_sync(0xffffffffu, mm, 1));
    const float am = __uint_as_float(mm);
    const float r = (am == 0.0f) ? 0.0f : __frcp_rn(am);
    const float2 r2 = make_float2(r, r);
    if (act) {
      uint32_t out[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const float2 x = __fmul2_rn(widen2(wv[i]), r2);
          const float2 g = __ffma2_rn(x, k16, k96);
          c[2 * i] = nf4_code(x.x, g.x, lane_tbl);
          c[2 * i + 1] = nf4_code(x.y, g.y, lane_tbl);
        }
        // nibble j of the word is code j (a shallow tree keeps the chain short)
        const uint32_t b0 = c[0] | (c[1] << 4), b1 = c[2] | (c[3] << 4);
        const uint32_t b2 = c[4] | (c[5] << 4), b3 = c[6] | (c[7] << 4);
        out[u] = (b0 | (b1 << 8)) | ((b2 | (b3 << 8)) << 16);
      }
      *reinterpret_cast<uint4*>(codes + h * 16) = make_uint4(out[0], out[1], out[2], out[3]);
      if ((h & 1) == 0) {
        absmax[h >> 1] = am;
        if (status && !isfinite(am)) atomicOr(status, kStatusNonFinite);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; u++) v[u] = vn[u];
  }
}

cudaError_t launch_nf4_quant(const uint16_t* w, int64_t n, uint8_t* codes, float* absmax,
                             int* status, cudaStream_t s) {
  static PerDeviceOnce attr;
  cudaError_t err = attr.run([] {
    return cudaFuncSetAttribute(k_nf4_quant, cudaFuncAttributeMaxDynamicSharedMemorySize, kNqSmem);
  });
  if (err != cudaSuccess) return err;
  const int64_t nhalf = n / 32;
  if (nhalf == 0) return cudaSuccess;
  const DevInfo* di = device_info();
  static PerDeviceInt occupancy;  // resident CTAs per SM (registers and shared memory permitting)
  const int per_sm = std::max(1, occupancy.get([](cudaError_t* e) {
    int b = 0;
    *e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_nf4_quant, kNqThreads, kNqSmem);
    return b;
  }, &err));
  if (err != cudaSuccess) return err;
  const int grid =
      (int)std::min<int64_t>((nhalf + kNqThreads - 1) / kNqThreads, (int64_t)di->sms * per_sm);
  k_nf4_quant<<<grid, kNqThreads, kNqSmem, s>>>(w, nhalf, codes, absmax, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- dequant
// y = bf16(level[c] * absmax).  A 256-entry table maps a code byte to the
// pair (level[low nibble], level[high nibble]); one packed multiply and one
// bf16x2 conversion finish two elements.  The table is replicated 16 times,
// entry p of copy l at (p * 16 + l) * 8 bytes, and lane l reads copy l & 15:
// the lanes of a 128-byte wavefront then never share a bank, whatever codes
// they look up.
constexpr int kNdThreads = 256;
constexpr int kNdTableBytes = 256 * 16 * 8;  // 32 KiB
constexpr int kNdSlabs = 8;                   // 8-element slabs per thread per item
constexpr int64_t kNdChunk = (int64_t)kNdThreads * kNdSlabs * 8;  // elements per item

// Work item = 16384 consecutive elements of one slice.  In slab k, thread t
// owns elements k*2048 + 8t .. +7: its 4 code bytes, its block's absmax, and
// a 16-byte output run, so every warp load and store is one contiguous run.
__global__ void __launch_bounds__(kNdThreads)
    k_nf4_dequant(const uint8_t* __restrict__ codes, const float* __restrict__ absmax,
                  int64_t nexp, int64_t per_slice, FastDiv cps,
                  const int32_t* __restrict__ hit_list, const int32_t* __restrict__ n_hit,
                  uint16_t* __restrict__ dst) {
  extern __shared__ __align__(16) float2 pairs[];  // [256][16]
  for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
    const int p = i >> 4;
    pairs[i] = make_float2(c_nf4[p & 15], c_nf4[p >> 4]);
  }
  __syncthreads();
  const float2* const mine = pairs + (threadIdx.x & 15);
  const uint32_t nslots = hit_list ? (uint32_t)max(0, min(*n_hit, (int32_t)nexp)) : (uint32_t)nexp;
  const uint32_t nitems = nslots * cps.d;
  for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x) {
    const uint32_t slot = cps.div(it);
    const int64_t e = hit_list ? (int64_t)hit_list[slot] : (int64_t)slot;
    if (e < 0 || e >= nexp) continue;
    const int64_t x0 = (int64_t)(it - slot * cps.d) * kNdChunk + threadIdx.x * 8;
    const uint8_t* cs = codes + e * (per_slice / 2);
    const float* as = absmax + e * (per_slice / 64);
    uint16_t* ds = dst + e * per_slice;
    uint32_t cw[kNdSlabs];
    float a[kNdSlabs];
#pragma unroll
    for (int k = 0; k < kNdSlabs; k++) {
      const int64_t x = x0 + k * (kNdThreads * 8);
      const bool ok = x < per_slice;
      cw[k] = ok ? __ldg(reinterpret_cast<const uint32_t*>(cs) + (x >> 3)) : 0u;
      a[k] = ok ? __ldg(as + (x >> 6)) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < kNdSlabs; k++) {
      const int64_t x = x0 + k * (kNdThreads * 8);
      if (x < per_slice) {
        const float2 a2 = make_float2(a[k], a[k]);
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const float2 y = __fmul2_rn(mine[__byte_perm(cw[k], 0, 0x4440 + j) * 16], a2);
          o[j] = bf16x2_rn(y.x, y.y);
        }
        stg_stream(ds + x, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
}

cudaError_t launch_nf4_dequant(const uint8_t* codes, const float* absmax, int64_t nexp,
                               int64_t per_slice, const int32_t* hit_list, const int32_t* n_hit,
                               uint16_t* dst, cudaStream_t s) {
  const int64_t cps = (per_slice + kNdChunk - 1) / kNdChunk;
  if (nexp == 0 || cps == 0) return cudaSuccess;
  if (nexp * cps >= (1ll << 31) - (1ll << 24)) return cudaErrorInvalidValue;
  FastDiv fd;
  fd.d = (uint32_t)cps;
  make_fastdiv(fd.d, &fd.m, &fd.s);
  const DevInfo* di = device_info();
  const int grid = (int)std::min<int64_t>(nexp * cps, (int64_t)di->sms * 6);
  static PerDeviceOnce attr;
  const cudaError_t err = attr.run([] {
    return cudaFuncSetAttribute(k_nf4_dequant, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kNdTableBytes);
  });
  if (err != cudaSuccess) return err;
  k_nf4_dequant<<<grid, kNdThreads, kNdTableBytes, s>>>(codes, absmax, nexp, per_slice, fd,
                                                        hit_list, n_hit, dst);
  return cudaGetLastError();
}

// ---------------------------------------------------------- routed union
// One CTA: mark every routed expert in a shared byte map, then compact the
// map in ascending order with a block-wide scan.  No host synchronisation:
// the hit list and its length stay on the device for the dequant kernel.
constexpr int kUnThreads = 1024;

__global__ void __launch_bounds__(kUnThreads)
    k_routed_union(const int32_t* __restrict__ topk, int64_t n_idx, int nexp,
                   int32_t* __restrict__ hit_list, int32_t* __restrict__ n_hit,
                   int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char flags[];
  __shared__ int wsum[kUnThreads / 32];
  __shared__ int bad_any;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwords = (nexp + 3) / 4;
  for (int i = tid; i < nwords; i += kUnThreads) reinterpret_cast<uint32_t*>(flags)[i] = 0;
  if (tid == 0) bad_any = 0;
  __syncthreads();
  int bad = 0;
  for (int64_t i = tid; i < n_idx; i += kUnThreads) {
    const int32_t e = topk[i];
    if (e >= 0 && e < nexp) flags[e] = 1;
    else bad = 1;
  }
  if (bad) bad_any = 1;
  __syncthreads();
  if (tid == 0 && bad_any && status) atomicOr(status, kStatusBadIndex);
  // each thread owns a contiguous run of experts
  const int per = (nexp + kUnThreads - 1) / kUnThreads;
  const int e0 = min(tid * per, nexp), e1 = min(e0 + per, nexp);
  int cnt = 0;
  for (int e = e0; e < e1; e++) cnt += flags[e];
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += u;
    }
    wsum[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  int pos = incl - cnt + (warp > 0 ? wsum[warp - 1] : 0);
  const int total = wsum[kUnThreads / 32 - 1];
  for (int e = e0; e < e1; e++)
    if (flags[e]) hit_list[pos++] = e;
  for (int i = total + tid; i < nexp; i += kUnThreads) hit_list[i] = -1;
  if (tid == 0) *n_hit = total;
}

cudaError_t launch_routed_union(const int32_t* topk, int64_t n_idx, int nexp, int32_t* hit_list,
                                int32_t* n_hit, int* status, cudaStream_t s) {
  static PerDeviceOnce attr;
  const int smem = ((nexp + 15) / 16) * 16;
  const cudaError_t err = attr.run([] {
    return cudaFuncSetAttribute(k_routed_union, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536);
  });
  if (err != cudaSuccess) return err;
  k_routed_union<<<1, kUnThreads, smem, s>>>(topk, n_idx, nexp, hit_list, n_hit, status);
  return cudaGetLastError();
}

}  // namespace nvq
