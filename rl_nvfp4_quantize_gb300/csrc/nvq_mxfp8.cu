// nvq_mxfp8.cu -- MXFP8 quantisation (OCP Microscaling: blocks of 32
// elements sharing one E8M0 scale 2^s, elements in E4M3) of an expert stack,
// rowwise and optionally columnwise from one read, and its dequantisation.
//
// Source: "The 4-bitter Lesson", "Key claims": the dequantised backward was
// validated first with MXFP8.  The pages name the format only; the
// definition is the OCP MX one: s = floor(log2 amax) - 8 (8 being the
// exponent of E4M3's largest power of two), clamped to [-127, 127] (amax = 0
// gives -127); scale byte s + 127; element E4M3(v * 2^-s), nearest-even,
// saturating at 448, sign kept.  v * 2^-s is one exact binary32 product.
#include <algorithm>
#include <cstdint>

#include "nvq_common.cuh"
#include "nvq_internal.h"

namespace nvq {

// Shared exponent of a block from the FP32 bits of its amax: the exponent
// field minus 127 is floor(log2 amax) for a normal amax; a subnormal or zero
// amax (field 0) and anything below 2^-119 give s = -127 after the clamp.
__device__ __forceinline__ int mx_shared_exp(uint32_t amax_bits) {
  const int f = (int)((amax_bits >> 23) & 0xFFu);
  return max(-127, min(127, f - 135));
}
// 2^-s as FP32 (a normal number for every s a finite bf16 amax gives:
// s <= 119, so 127 - s >= 8; s = 127 would need an infinite amax and then
// yields 0, which is out of contract anyway).
__device__ __forceinline__ float mx_inv_scale(int s) {
  return __uint_as_float((uint32_t)max(0, 127 - s) << 23);
}

// ------------------------------------------------------------ quantise tiles
// A CTA of 256 threads walks tiles of 64 rows x 256 columns of one slice
// (persistent grid-stride loop), loaded by one thread as four TMA boxes
// (64 x 64 bf16, 128-byte swizzle) into one of two stages; the copy of the
// next tile runs while the current one is quantised.
//   rowwise pass   : warp w takes block column w (32 columns), lane l rows l
//                    and l + 32: 32 codes (one 32-byte store) and one scale
//                    byte per block;
//   columnwise pass: thread t takes columns 2 (t & 127), +1 and rows
//                    32 (t >> 7) .. +31: per column 32 codes (one 32-byte
//                    store into the transposed layout) and one scale byte.
// Every code store fills one whole 32-byte L2 sector.  The scale bytes are
// staged in shared memory and leave after the tile as one 8-byte store per
// row (its 8 blocks) and one 2-byte store per column (its 2 blocks): written
// one byte at a time, each would be a separate partial-sector write, and the
// L2 write-operation rate, not DRAM bandwidth, bounded the kernel.
// Inside a swizzled box, 16-byte chunk c of row r sits at chunk c ^ (r & 7).
constexpr int kMxTR = 64, kMxTC = 256, kMxThreads = 256;
constexpr int kMxBoxC = 64;
constexpr int kMxBoxBytes = kMxTR * kMxBoxC * 2;  // 8 KiB
constexpr int kMxStage = kMxTR * kMxTC * 2;       // 32 KiB
constexpr int kMxScaleStage = kMxTR * 8 + kMxTC * 2;  // row scales [64][8], column scales [256][2]
constexpr int kMxSmem = 2 * kMxStage + kMxScaleStage + 64;
constexpr int kMxMinBlocks = 3;
constexpr uint32_t kMxWaitTries = 1u << 22;

struct MxTileArgs {
  CUtensorMap tmap;       // w as [nexp * rows, cols] bf16, 64 x 64 boxes
  uint8_t* codes_row;     // [nexp, rows, cols]
  uint8_t* scales_row;    // [nexp, rows, cols/32] (or tiled)
  uint8_t* codes_col;     // [nexp, cols, rows] or null
  uint8_t* scales_col;    // [nexp, cols, rows/32] (or tiled)
  int* status;
  int rows, cols, tiles_c;
  uint32_t ntiles;
  FastDiv per_exp, by_tiles_c;
  int tiled, ct_row, ct_col;
  int64_t sl_row, sl_col;
};

// Two FP32 -> two E4M3 bytes (RNE, satfinite, sign kept); byte 0 = lo.
__device__ __forceinline__ uint32_t e4m3x2_f32(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

template <bool DUAL>
__global__ void __launch_bounds__(kMxThreads, kMxMinBlocks) k_mx_tiles(const __grid_constant__ MxTileArgs A) {
  extern __shared__ __align__(1024) unsigned char smem[];
  uint8_t* const srow = smem + 2 * kMxStage;    // [64 rows][8 blocks]
  uint8_t* const scol = srow + kMxTR * 8;       // [256 columns][2 blocks]
  uint64_t* const bar = reinterpret_cast<uint64_t*>(scol + kMxTC * 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem) & 1023u) {
    if (tid == 0 && A.status) atomicOr(A.status, kStatusTimeout);
    return;
  }
  const int rows = A.rows, cols = A.cols;
  const int64_t nb_row = cols / 32, nb_col = rows / 32;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();

  struct Tile { uint32_t e; int r0, c0, rv, cv; };
  auto tile_of = [&](uint32_t t) {
    Tile T;
    T.e = A.per_exp.div(t);
    const uint32_t rem = t - T.e * A.per_exp.d;
    const uint32_t tr = A.by_tiles_c.div(rem);
    T.r0 = (int)tr * kMxTR;
    T.c0 = (int)(rem - tr * (uint32_t)A.tiles_c) * kMxTC;
    T.rv = min(kMxTR, rows - T.r0);
    T.cv = min(kMxTC, cols - T.c0);
    return T;
  };
  auto issue = [&](uint32_t t, int st) {
    if (tid == 0 && t < A.ntiles) {
      const Tile T = tile_of(t);
      mbar_arrive_expect_tx(&bar[st], kMxStage);
      const int y = (int)(T.e * (uint32_t)rows) + T.r0;
#pragma unroll
      for (int j = 0; j < kMxTC / kMxBoxC; j++)
        tma_load_2d(smem + st * kMxStage + j * kMxBoxBytes, &A.tmap, T.c0 + j * kMxBoxC, y, &bar[st]);
    }
  };
  issue(blockIdx.x, 0);
  issue(blockIdx.x + gridDim.x, 1);

  int st = 0;
  uint32_t it = 0;
  for (uint32_t t = blockIdx.x; t < A.ntiles; t += gridDim.x, st ^= 1, it++) {
    const bool ok = mbar_wait(&bar[st], (it >> 1) & 1, kMxWaitTries);
    if (__syncthreads_or(!ok)) {
      if (tid == 0 && A.status) atomicOr(A.status, kStatusTimeout);
      mbar_wait(&bar[st ^ 1], ((it + 1) >> 1) & 1, kMxWaitTries);
      return;
    }
    const Tile T = tile_of(t);
    const unsigned char* tile = smem + st * kMxStage;
    bool inf = false;

    // rowwise: block column b = warp, rows lane and lane + 32
    {
      const int b = warp;
      const unsigned char* box = tile + (b >> 1) * kMxBoxBytes;
      const int ch0 = 4 * (b & 1);
#pragma unroll
      for (int k = 0; k < 2; k++) {
        const int r = lane + 32 * k;
        if (r < T.rv && 32 * b < T.cv) {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 4; j++) {
            const uint4 v = *reinterpret_cast<const uint4*>(box + r * 128 + (((ch0 + j) ^ (r & 7)) << 4));
            w[4 * j] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
          }
          uint32_t m = maxabs2(w[0], w[1]);
#pragma unroll
          for (int i = 2; i < 16; i++) m = maxabs2(m, w[i]);
          m &= 0x7fff7fffu;
          const uint32_t am = max(m & 0xffffu, m >> 16) << 16;  // FP32 bits of the block amax
          inf |= am >= 0x7f800000u;
          const int s = mx_shared_exp(am);
          const float2 inv = make_float2(mx_inv_scale(s), mx_inv_scale(s));
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const float2 a = __fmul2_rn(widen2(w[2 * i]), inv);
            const float2 c = __fmul2_rn(widen2(w[2 * i + 1]), inv);
            o[i] = e4m3x2_f32(a.x, a.y) | (e4m3x2_f32(c.x, c.y) << 16);
          }
          const int64_t grow = (int64_t)T.e * rows + T.r0 + r;
          stg256(A.codes_row + grow * cols + T.c0 + 32 * b, o);
          srow[r * 8 + b] = (uint8_t)(s + 127);
        }
      }
    }

    if (DUAL) {
      // columnwise: columns 2p, 2p + 1, rows 32 rb .. 32 rb + 31
      const int p = tid & 127, rb = tid >> 7;
      if (2 * p < T.cv && 32 * rb < T.rv) {
        const unsigned char* colp = tile + ((2 * p) >> 6) * kMxBoxBytes + ((p & 3) << 2);
        const int ch = ((2 * p) & 63) >> 3;
        uint32_t wv[32];  // row i: (column 2p, column 2p + 1)
#pragma unroll
        for (int i = 0; i < 32; i++) {
          const int r = 32 * rb + i;
          wv[i] = *reinterpret_cast<const uint32_t*>(colp + r * 128 + ((ch ^ (r & 7)) << 4));
        }
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 32; i++) m = maxabs2(m, wv[i]);
        m &= 0x7fff7fffu;
        const uint32_t amj = (m & 0xffffu) << 16, amk = m & 0xffff0000u;
        inf |= amj >= 0x7f800000u || amk >= 0x7f800000u;
        const int sj = mx_shared_exp(amj), sk = mx_shared_exp(amk);
        const float2 inv = make_float2(mx_inv_scale(sj), mx_inv_scale(sk));
        uint32_t oj[8], ok[8];
#pragma unroll
        for (int q = 0; q < 8; q++) {
          // rows 4q .. 4q + 3 of both columns
          const float2 a = __fmul2_rn(widen2(wv[4 * q]), inv);
          const float2 b = __fmul2_rn(widen2(wv[4 * q + 1]), inv);
          const float2 c = __fmul2_rn(widen2(wv[4 * q + 2]), inv);
          const float2 d = __fmul2_rn(widen2(wv[4 * q + 3]), inv);
          oj[q] = e4m3x2_f32(a.x, b.x) | (e4m3x2_f32(c.x, d.x) << 16);
          ok[q] = e4m3x2_f32(a.y, b.y) | (e4m3x2_f32(c.y, d.y) << 16);
        }
        const int64_t gcol = (int64_t)T.e * cols + T.c0 + 2 * p;
        const int64_t r0 = T.r0 + 32 * rb;
        stg256(A.codes_col + gcol * rows + r0, oj);
        stg256(A.codes_col + (gcol + 1) * rows + r0, ok);
        scol[(2 * p) * 2 + rb] = (uint8_t)(sj + 127);
        scol[(2 * p + 1) * 2 + rb] = (uint8_t)(sk + 127);
      }
    }
    if (inf && A.status) atomicOr(A.status, kStatusNonFinite);
    __syncthreads();
    issue(t + 2 * gridDim.x, st);

    // scale write-out (the next iteration's barrier keeps the staging area
    // until every thread has read it)
    const int nbt = T.cv >> 5;        // blocks per row in this tile
    const int bc0 = T.c0 >> 5;
    if (tid < T.rv) {
      const int r = tid;
      const uint2 v = *reinterpret_cast<const uint2*>(srow + r * 8);
      if (A.tiled) {
        // block columns bc0 .. bc0 + 7: two runs of four bytes in two tiles
        uint8_t* base = A.scales_row + T.e * A.sl_row;
        if (nbt == 8) {
          *reinterpret_cast<uint32_t*>(base + scale_off_tiled(T.r0 + r, bc0, A.ct_row)) = v.x;
          *reinterpret_cast<uint32_t*>(base + scale_off_tiled(T.r0 + r, bc0 + 4, A.ct_row)) = v.y;
        } else {
          for (int b = 0; b < nbt; b++)
            base[scale_off_tiled(T.r0 + r, bc0 + b, A.ct_row)] = srow[r * 8 + b];
        }
      } else {
        uint8_t* d = A.scales_row + ((int64_t)T.e * rows + T.r0 + r) * nb_row + bc0;
        if (nbt == 8 && (nb_row & 7) == 0) {
          *reinterpret_cast<uint2*>(d) = v;
        } else {
          for (int b = 0; b < nbt; b++) d[b] = srow[r * 8 + b];
        }
      }
    }
    if (DUAL && tid < T.cv) {
      const int c = tid, nrb = min(2, T.rv >> 5);
      const int bc = T.r0 >> 5;     // even: tiles are 64 rows
      const uint16_t v = *reinterpret_cast<const uint16_t*>(scol + c * 2);
      if (A.tiled) {
        uint8_t* base = A.scales_col + T.e * A.sl_col;
        if (nrb == 2) {
          *reinterpret_cast<uint16_t*>(base + scale_off_tiled(T.c0 + c, bc, A.ct_col)) = v;
        } else {
          base[scale_off_tiled(T.c0 + c, bc, A.ct_col)] = scol[c * 2];
        }
      } else {
        uint8_t* d = A.scales_col + ((int64_t)T.e * cols + T.c0 + c) * nb_col + bc;
        if (nrb == 2 && (nb_col & 1) == 0) {
          *reinterpret_cast<uint16_t*>(d) = v;
        } else {
          for (int b = 0; b < nrb; b++) d[b] = scol[c * 2 + b];
        }
      }
    }
  }
}

cudaError_t launch_mx_tiles(const uint16_t* w, int64_t nexp, int rows, int cols, uint8_t* codes_row,
                            uint8_t* scales_row, uint8_t* codes_col, uint8_t* scales_col,
                            int* status, bool tiled, cudaStream_t s) {
  const DevInfo* di = device_info();
  const int tiles_r = (rows + kMxTR - 1) / kMxTR, tiles_c = (cols + kMxTC - 1) / kMxTC;
  const int64_t per = (int64_t)tiles_r * tiles_c;
  const int64_t ntiles = nexp * per;
  if (ntiles == 0) return cudaSuccess;
  if (ntiles >= (1ll << 31) - (1ll << 24) || nexp * (int64_t)rows >= (1ll << 31))
    return cudaErrorInvalidValue;
  static PerDeviceOnce attr[2];
  const bool dual = codes_col != nullptr;
  cudaError_t err = attr[dual].run([&] {
    return dual ? cudaFuncSetAttribute(k_mx_tiles<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kMxSmem)
                : cudaFuncSetAttribute(k_mx_tiles<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kMxSmem);
  });
  if (err != cudaSuccess) return err;
  MxTileArgs A;
  if (!encode_tmap_2d(&A.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, w, (uint64_t)cols,
                      (uint64_t)(nexp * rows), (uint64_t)cols * 2, kMxBoxC, kMxTR,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  A.codes_row = codes_row;
  A.scales_row = scales_row;
  A.codes_col = codes_col;
  A.scales_col = scales_col;
  A.status = status;
  A.rows = rows;
  A.cols = cols;
  A.tiles_c = tiles_c;
  A.ntiles = (uint32_t)ntiles;
  A.per_exp.d = (uint32_t)per;
  make_fastdiv((uint32_t)per, &A.per_exp.m, &A.per_exp.s);
  A.by_tiles_c.d = (uint32_t)tiles_c;
  make_fastdiv((uint32_t)tiles_c, &A.by_tiles_c.m, &A.by_tiles_c.s);
  A.tiled = tiled ? 1 : 0;
  A.ct_row = (cols / 32 + 3) / 4;
  A.ct_col = (rows / 32 + 3) / 4;
  A.sl_row = tiled_bytes(rows, cols / 32);
  A.sl_col = tiled_bytes(cols, rows / 32);
  const int grid = (int)std::min<int64_t>(ntiles, (int64_t)di->sms * kMxMinBlocks);
  if (dual) k_mx_tiles<true><<<grid, kMxThreads, kMxSmem, s>>>(A);
  else k_mx_tiles<false><<<grid, kMxThreads, kMxSmem, s>>>(A);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- dequant
// y = bf16(E4M3 value * 2^(scale - 127)): each E4M3 pair decodes exactly to
// an f16 pair, widens exactly to FP32, and one packed multiply by the power
// of two is exact; the bf16 conversion rounds to nearest even.  A thread
// takes 16 consecutive codes (half a block) per item.
constexpr int kMxDqThreads = 256;

__global__ void __launch_bounds__(kMxDqThreads)
    k_mx_dequant(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int64_t n16,
                 uint16_t* __restrict__ dst) {
  for (int64_t i = blockIdx.x * (int64_t)kMxDqThreads + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * kMxDqThreads) {
    const uint4 c = ldg_stream(codes + i * 16);
    const int sb = __ldg(scales + (i >> 1));
    // 2^(sb - 127) as FP32: normal for sb >= 1; 2^-127 (subnormal) for sb = 0
    const float X = sb > 0 ? __uint_as_float((uint32_t)sb << 23) : __uint_as_float(0x00400000u);
    const float2 X2 = make_float2(X, X);
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; k++) {
#pragma unroll
      for (int h = 0; h < 2; h++) {
        uint32_t f;
        const uint16_t pair = (uint16_t)(cw[k] >> (16 * h));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f) : "h"(pair));
        const float2 y = __fmul2_rn(cs_exact(f, 0x3C003C00u), X2);  // f16 pair * 1, widened exactly
        o[2 * k + h] = bf16x2_rn(y.x, y.y);
      }
    }
    stg256_stream(dst + i * 16, o);  // one whole sector
  }
}

cudaError_t launch_mx_dequant(const uint8_t* codes, const uint8_t* scales, int64_t n, uint16_t* dst,
                              cudaStream_t s) {
  const int64_t n16 = n / 16;
  if (n16 == 0) return cudaSuccess;
  const DevInfo* di = device_info();
  const int grid = (int)std::min<int64_t>((n16 + kMxDqThreads - 1) / kMxDqThreads,
                                          (int64_t)di->sms * 8);
  k_mx_dequant<<<grid, kMxDqThreads, 0, s>>>(codes, scales, n16, dst);
  return cudaGetLastError();
}

}  // namespace nvq
