// nvq_nvfp4.cu -- NVFP4 kernels for sm_103a: slice amax, rowwise and
// dual-layout (rowwise + columnwise from one read) quantisation with optional
// Four-Over-Six, per-token activation quantisation, and dequantisation in
// plain and transposed layouts.
//
// Sources: "Getting GLM-5.2 NVFP4 Post-Training off the ground", Part I ("Why
// can't we just transpose the one copy?", "The bottom line") and "The
// 4-bitter Lesson" ("Key claims", "Method").
#include <cfloat>
#include <algorithm>
#include <cstdint>

#include "nvq_common.cuh"
#include "nvq_internal.h"

namespace nvq {

// ------------------------------------------------------------------ amax
constexpr int kAmaxThreads = 256;
constexpr int kAmaxVec = 8;  // 16-byte vectors per thread per item
constexpr int64_t kAmaxChunk = (int64_t)kAmaxThreads * kAmaxVec * 8;  // elements per item

__global__ void k_zero_f32(float* p, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0.0f;
}

// Each work item is one chunk of one slice.  The magnitude maximum is taken
// on bf16 bit patterns (exact); the item's result is folded into amax[e]
// with an atomic max on the FP32 bit pattern (ordered like the values for
// non-negative floats, NaN above infinity).
__global__ void __launch_bounds__(kAmaxThreads)
    k_amax(const uint16_t* __restrict__ w, int64_t per_slice, FastDiv cps, uint32_t nitems,
           float* __restrict__ amax) {
  __shared__ uint32_t red[kAmaxThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x) {
    const uint32_t e = cps.div(it);
    const int64_t start = (int64_t)(it - e * cps.d) * kAmaxChunk;
    const uint16_t* base = w + (int64_t)e * per_slice;
    uint4 v[kAmaxVec];
#pragma unroll
    for (int u = 0; u < kAmaxVec; u++) {
      const int64_t idx = start + ((int64_t)u * kAmaxThreads + threadIdx.x) * 8;
      v[u] = (idx < per_slice) ? ldg_stream(base + idx) : make_uint4(0, 0, 0, 0);
    }
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < kAmaxVec; u++) {
      m = umaxmag2(m, v[u].x);
      m = umaxmag2(m, v[u].y);
      m = umaxmag2(m, v[u].z);
      m = umaxmag2(m, v[u].w);
    }
    uint32_t mm = max(m & 0xffffu, m >> 16) << 16;
    mm = __reduce_max_sync(0xffffffffu, mm);
    if (lane == 0) red[warp] = mm;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t r = red[0];
#pragma unroll
      for (int i = 1; i < kAmaxThreads / 32; i++) r = max(r, red[i]);
      atomicMax(reinterpret_cast<unsigned int*>(amax + e), r);
    }
    __syncthreads();
  }
}

// G[e] from amax[e] alone (used when the slices are empty).
__global__ void k_tensor_scales(const float* amax, float* G, int64_t n, float six_m) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float g, e;
    global_scales(amax[i], six_m, g, e);
    G[i] = g;
  }
}

cudaError_t launch_tensor_scales(const float* amax, float* G, int64_t n, bool f46, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int grid = (int)std::min<int64_t>((n + 255) / 256, 1024);
  k_tensor_scales<<<grid, 256, 0, s>>>(amax, G, n, f46 ? 1536.0f : 2688.0f);
  return cudaGetLastError();
}

cudaError_t launch_zero_f32(float* p, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int grid = (int)std::min<int64_t>((n + 255) / 256, 1024);
  k_zero_f32<<<grid, 256, 0, s>>>(p, n);
  return cudaGetLastError();
}

cudaError_t launch_amax(const uint16_t* w, int64_t nexp, int64_t per_slice, float* amax,
                        cudaStream_t s) {
  const DevInfo* di = device_info();
  const int64_t cps = (per_slice + kAmaxChunk - 1) / kAmaxChunk;
  const int64_t nitems = nexp * cps;
  if (nitems == 0) return cudaSuccess;
  if (nitems >= (1ll << 31) - (1ll << 24)) return cudaErrorInvalidValue;
  FastDiv fd;
  fd.d = (uint32_t)cps;
  make_fastdiv(fd.d, &fd.m, &fd.s);
  int grid = (int)std::min<int64_t>(nitems, (int64_t)di->sms * 8);
  k_amax<<<grid, kAmaxThreads, 0, s>>>(w, per_slice, fd, (uint32_t)nitems, amax);
  return cudaGetLastError();
}

// ----------------------------------------------------- rowwise / dual tiles
// A CTA of 256 threads walks tiles of 64 rows x 256 columns of one expert
// slice (persistent grid-stride loop).  One thread loads each tile with four
// TMA box copies (64 x 64 bf16, 128-byte swizzle) into one of two shared
// stages; the copy of the next tile runs while the current one is quantised.
// From the staged tile:
//   rowwise pass   : 1024 blocks of 1x16, four per thread, results stored
//                    straight to global (8 code bytes + 1 scale byte);
//   columnwise pass: 256 units of 16 rows x 4 columns, one per thread, each
//                    column pair processed with packed f32x2 arithmetic; the
//                    results are staged and written as contiguous runs of the
//                    transposed [in, out/2] layout.
// Inside a swizzled box, 16-byte chunk c of row r sits at chunk c ^ (r & 7).
#ifndef NVQ_QT_MINB
#define NVQ_QT_MINB 2
#endif
constexpr int kTR = 64, kTC = 256, kQT = 256;
constexpr int kBoxC = 64;                       // box columns (128 bytes)
constexpr int kBoxBytes = kTR * kBoxC * 2;      // 8 KiB
constexpr int kInStage = kTR * kTC * 2;         // 32 KiB (four boxes)
constexpr int kColCodes = 4 * kTC * 8;          // [rb][col] 8 bytes
constexpr int kColScales = 4 * kTC;             // [rb][col] 1 byte
constexpr int kQuantSmem = 2 * kInStage + kColCodes + kColScales + kScaleTableBytes + 64;
constexpr uint32_t kWaitTries = 1u << 22;

struct __align__(64) QuantTileArgs {
  CUtensorMap tmap;       // w as [nexp * rows, cols] bf16, 64 x 64 boxes
  uint8_t* codes_row;
  uint8_t* scales_row;
  uint8_t* codes_col;
  uint8_t* scales_col;
  const float* amax;
  float* tensor_scale;
  int* status;
  int rows, cols;         // per slice
  int tiles_c;            // column tiles per slice
  uint32_t ntiles;        // all slices
  FastDiv per_exp;        // tiles per slice
  FastDiv by_tiles_c;
};

template <bool F46, bool DUAL>
__global__ void __launch_bounds__(kQT, NVQ_QT_MINB) k_quant_tiles(const __grid_constant__ QuantTileArgs A) {
  // The kernel has no static shared memory, so the dynamic block starts at
  // the (1 KiB aligned) base of the CTA's window, as the swizzled TMA boxes
  // require; a misaligned base is reported instead of used.
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* const in0 = smem;
  unsigned char* const colc = smem + 2 * kInStage;
  unsigned char* const cols_s = colc + kColCodes;
  ScaleEnt* const tbl = reinterpret_cast<ScaleEnt*>(cols_s + kColScales);
  uint64_t* const bar = reinterpret_cast<uint64_t*>(cols_s + kColScales + kScaleTableBytes);
  float* const s_E = reinterpret_cast<float*>(bar + 2);
  const int tid = threadIdx.x;
  if (smem_u32(smem) & 1023u) {
    if (tid == 0 && A.status) atomicOr(A.status, kStatusTimeout);
    return;
  }
  const float six_m = F46 ? 1536.0f : 2688.0f;
  const int rows = A.rows, cols = A.cols;
  const int64_t cols_h = cols >> 1, cols_16 = cols >> 4, rows_h = rows >> 1, rows_16 = rows >> 4;

  build_scale_table(tbl);
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();

  struct Tile { uint32_t e; int r0, c0, rv, cv; bool first; };
  auto tile_of = [&](uint32_t t) {
    Tile T;
    T.e = A.per_exp.div(t);
    const uint32_t rem = t - T.e * A.per_exp.d;
    const uint32_t tr = A.by_tiles_c.div(rem);
    const uint32_t tc = rem - tr * (uint32_t)A.tiles_c;
    T.r0 = (int)tr * kTR;
    T.c0 = (int)tc * kTC;
    T.rv = min(kTR, rows - T.r0);
    T.cv = min(kTC, cols - T.c0);
    T.first = rem == 0;
    return T;
  };

  // producer: thread 0 arms the stage barrier with the tile's byte count and
  // issues the four box loads (out-of-range parts are zero-filled), then
  // forms the slice's encode factor for the consumers.
  auto issue = [&](uint32_t t, int st) {
    if (tid == 0 && t < A.ntiles) {
      const Tile T = tile_of(t);
      mbar_arrive_expect_tx(&bar[st], kInStage);
      const int y = (int)(T.e * (uint32_t)rows) + T.r0;
#pragma unroll
      for (int j = 0; j < kTC / kBoxC; j++)
        tma_load_2d(in0 + st * kInStage + j * kBoxBytes, &A.tmap, T.c0 + j * kBoxC, y, &bar[st]);
      const float am = A.amax[T.e];
      float G, E;
      global_scales(am, six_m, G, E);
      s_E[st] = E;
      if (T.first) {
        A.tensor_scale[T.e] = G;
        if (A.status && !isfinite(am)) atomicOr(A.status, kStatusNonFinite);
      }
    }
  };

  const uint32_t t0 = blockIdx.x;
  issue(t0, 0);
  issue(t0 + gridDim.x, 1);

  // rowwise geometry of this thread: 16-column block cb, rows (tid >> 4) + 16k
  const int cb = tid & 15, rb0 = tid >> 4;
  const int rbox = (cb >> 2) * kBoxBytes, rchunk = 2 * (cb & 3);
  // columnwise geometry: row block cr, columns 4q .. 4q+3
  const int warp = tid >> 5, lane = tid & 31;
  const int cr = warp >> 1, q = ((warp & 1) << 5) + lane;
  const int cbox = (q >> 4) * kBoxBytes, cchunk = (q & 15) >> 1, chalf = (q & 1) * 8;

  int st = 0;
  uint32_t it = 0;
  for (uint32_t t = t0; t < A.ntiles; t += gridDim.x, st ^= 1, it++) {
    const bool ok = mbar_wait(&bar[st], (it >> 1) & 1, kWaitTries);
    if (__syncthreads_or(!ok)) {  // a copy never landed: report and stop
      if (tid == 0 && A.status) atomicOr(A.status, kStatusTimeout);
      mbar_wait(&bar[st ^ 1], ((it + 1) >> 1) & 1, kWaitTries);
      return;
    }
    const Tile T = tile_of(t);
    const float E = s_E[st];
    const unsigned char* tile = in0 + st * kInStage;

    // rowwise blocks: four per thread, 16 rows apart
    {
      const int64_t grow0 = (int64_t)T.e * rows + T.r0 + rb0;
      uint8_t* pc = A.codes_row + grow0 * cols_h + (T.c0 >> 1) + cb * 8;
      uint8_t* ps = A.scales_row + grow0 * cols_16 + (T.c0 >> 4) + cb;
      const bool cvalid = cb * 16 < T.cv;
#pragma unroll 1
      for (int k = 0; k < 4; k++) {
        const int r = rb0 + 16 * k;
        if (cvalid && r < T.rv) {
          const unsigned char* rowp = tile + rbox + r * 128;
          const uint4 lo = *reinterpret_cast<const uint4*>(rowp + ((rchunk ^ (r & 7)) << 4));
          const uint4 hi = *reinterpret_cast<const uint4*>(rowp + (((rchunk + 1) ^ (r & 7)) << 4));
          const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          uint32_t c0w, c1w, sb;
          quant_row_block<F46>(wv, E, tbl, c0w, c1w, sb);
          *reinterpret_cast<uint2*>(pc + 16 * k * cols_h) = make_uint2(c0w, c1w);
          ps[16 * k * cols_16] = (uint8_t)sb;
        }
      }
    }

    if (DUAL) {
      if (cr * 16 < T.rv && q * 4 < T.cv) {
        const unsigned char* colp = tile + cbox + cr * 16 * 128 + chalf;
        uint32_t wa[16], wb[16];
#pragma unroll
        for (int i = 0; i < 16; i++) {
          const uint2 v =
              *reinterpret_cast<const uint2*>(colp + i * 128 + ((cchunk ^ (i & 7)) << 4));
          wa[i] = v.x;
          wb[i] = v.y;
        }
        uint32_t cj[2], ck[2], sbj, sbk, sw;
        quant_col_pair<F46>(wa, E, tbl, cj, ck, sbj, sbk);
        *reinterpret_cast<uint4*>(colc + cr * (kTC * 8) + q * 32) =
            make_uint4(cj[0], cj[1], ck[0], ck[1]);
        sw = sbj | (sbk << 8);
        quant_col_pair<F46>(wb, E, tbl, cj, ck, sbj, sbk);
        *reinterpret_cast<uint4*>(colc + cr * (kTC * 8) + q * 32 + 16) =
            make_uint4(cj[0], cj[1], ck[0], ck[1]);
        sw |= (sbj << 16) | (sbk << 24);
        *reinterpret_cast<uint32_t*>(cols_s + cr * kTC + q * 4) = sw;
      }
    }
    __syncthreads();
    issue(t + 2 * gridDim.x, st);

    if (DUAL) {
      const int c = tid;
      if (c < T.cv) {
        const int nrb = T.rv >> 4;
        const int64_t grow = (int64_t)T.e * cols + T.c0 + c;
        uint8_t* dstc = A.codes_col + grow * rows_h + (T.r0 >> 1);
        uint8_t* dsts = A.scales_col + grow * rows_16 + (T.r0 >> 4);
        if (nrb == 4 && (rows & 31) == 0) {
          const uint2 v0 = *reinterpret_cast<const uint2*>(colc + c * 8);
          const uint2 v1 = *reinterpret_cast<const uint2*>(colc + kTC * 8 + c * 8);
          const uint2 v2 = *reinterpret_cast<const uint2*>(colc + 2 * kTC * 8 + c * 8);
          const uint2 v3 = *reinterpret_cast<const uint2*>(colc + 3 * kTC * 8 + c * 8);
          reinterpret_cast<uint4*>(dstc)[0] = make_uint4(v0.x, v0.y, v1.x, v1.y);
          reinterpret_cast<uint4*>(dstc)[1] = make_uint4(v2.x, v2.y, v3.x, v3.y);
        } else {
          for (int rb = 0; rb < nrb; rb++)
            *reinterpret_cast<uint2*>(dstc + rb * 8) =
                *reinterpret_cast<const uint2*>(colc + rb * (kTC * 8) + c * 8);
        }
        if (nrb == 4 && (rows & 63) == 0) {
          const uint32_t sc = (uint32_t)cols_s[c] | ((uint32_t)cols_s[kTC + c] << 8) |
                              ((uint32_t)cols_s[2 * kTC + c] << 16) |
                              ((uint32_t)cols_s[3 * kTC + c] << 24);
          *reinterpret_cast<uint32_t*>(dsts) = sc;
        } else {
          for (int rb = 0; rb < nrb; rb++) dsts[rb] = cols_s[rb * kTC + c];
        }
      }
    }
  }
}

template <bool F46, bool DUAL>
static cudaError_t set_quant_smem() {
  static int attr_done = 0;  // per process; the attribute is per function
  if (!attr_done) {
    cudaError_t err = cudaFuncSetAttribute(k_quant_tiles<F46, DUAL>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kQuantSmem);
    if (err != cudaSuccess) return err;
    attr_done = 1;
  }
  return cudaSuccess;
}

cudaError_t launch_quant_tiles(const uint16_t* w, int64_t nexp, int rows, int cols, bool f46,
                               uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col,
                               uint8_t* scales_col, const float* amax, float* tensor_scale,
                               int* status, cudaStream_t s) {
  const DevInfo* di = device_info();
  const int tiles_r = (rows + kTR - 1) / kTR, tiles_c = (cols + kTC - 1) / kTC;
  const int64_t per = (int64_t)tiles_r * tiles_c;
  const int64_t ntiles = nexp * per;
  if (ntiles == 0) return cudaSuccess;
  if (ntiles >= (1ll << 31) - (1ll << 24) || nexp * (int64_t)rows >= (1ll << 31))
    return cudaErrorInvalidValue;
  QuantTileArgs A;
  if (!encode_tmap_2d(&A.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, w, (uint64_t)cols,
                      (uint64_t)(nexp * rows), (uint64_t)cols * 2, kBoxC, kTR,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  A.codes_row = codes_row;
  A.scales_row = scales_row;
  A.codes_col = codes_col;
  A.scales_col = scales_col;
  A.amax = amax;
  A.tensor_scale = tensor_scale;
  A.status = status;
  A.rows = rows;
  A.cols = cols;
  A.tiles_c = tiles_c;
  A.ntiles = (uint32_t)ntiles;
  A.per_exp.d = (uint32_t)per;
  make_fastdiv((uint32_t)per, &A.per_exp.m, &A.per_exp.s);
  A.by_tiles_c.d = (uint32_t)tiles_c;
  make_fastdiv((uint32_t)tiles_c, &A.by_tiles_c.m, &A.by_tiles_c.s);
  const int grid = (int)std::min<int64_t>(ntiles, (int64_t)di->sms * NVQ_QT_MINB);
  const bool dual = codes_col != nullptr;
  cudaError_t err;
  if (f46 && dual) {
    if ((err = set_quant_smem<true, true>())) return err;
    k_quant_tiles<true, true><<<grid, kQT, kQuantSmem, s>>>(A);
  } else if (f46) {
    if ((err = set_quant_smem<true, false>())) return err;
    k_quant_tiles<true, false><<<grid, kQT, kQuantSmem, s>>>(A);
  } else if (dual) {
    if ((err = set_quant_smem<false, true>())) return err;
    k_quant_tiles<false, true><<<grid, kQT, kQuantSmem, s>>>(A);
  } else {
    if ((err = set_quant_smem<false, false>())) return err;
    k_quant_tiles<false, false><<<grid, kQT, kQuantSmem, s>>>(A);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------ per-token activations
// One CTA of 128 threads per token row.  Up to kActRegBlocks blocks per
// thread stay in registers between the row-amax reduction and the
// quantisation; longer rows re-read the remaining blocks (from cache).
constexpr int kActThreads = 128;
constexpr int kActRegBlocks = 4;

template <bool F46>
__global__ void __launch_bounds__(kActThreads)
    k_act(const uint16_t* __restrict__ x, int64_t T, int H, uint8_t* __restrict__ codes,
          uint8_t* __restrict__ scales, float* __restrict__ token_scale, int* __restrict__ status) {
  __shared__ ScaleEnt tbl[128];
  __shared__ uint32_t red[kActThreads / 32];
  build_scale_table(tbl);
  __syncthreads();
  const int nb = H / 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float six_m = F46 ? 1536.0f : 2688.0f;
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const uint16_t* xr = x + row * H;
    uint32_t wr[kActRegBlocks][8];
    uint32_t bm[kActRegBlocks];
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < kActRegBlocks; k++) {
      const int b = threadIdx.x + k * kActThreads;
      bm[k] = 0;
      if (b < nb) {
        const uint4 lo = ldg_stream(xr + b * 16);
        const uint4 hi = ldg_stream(xr + b * 16 + 8);
        wr[k][0] = lo.x; wr[k][1] = lo.y; wr[k][2] = lo.z; wr[k][3] = lo.w;
        wr[k][4] = hi.x; wr[k][5] = hi.y; wr[k][6] = hi.z; wr[k][7] = hi.w;
        uint32_t mk = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) mk = umaxmag2(mk, wr[k][i]);
        bm[k] = mk;
        m = umaxmag2(m, mk);
      }
    }
    for (int b = threadIdx.x + kActRegBlocks * kActThreads; b < nb; b += kActThreads) {
      const uint4 lo = ldg_stream(xr + b * 16);
      const uint4 hi = ldg_stream(xr + b * 16 + 8);
      m = umaxmag2(m, lo.x); m = umaxmag2(m, lo.y); m = umaxmag2(m, lo.z); m = umaxmag2(m, lo.w);
      m = umaxmag2(m, hi.x); m = umaxmag2(m, hi.y); m = umaxmag2(m, hi.z); m = umaxmag2(m, hi.w);
    }
    uint32_t mm = max(m & 0xffffu, m >> 16) << 16;
    mm = __reduce_max_sync(0xffffffffu, mm);
    if (lane == 0) red[warp] = mm;
    __syncthreads();
    uint32_t rmax = red[0];
#pragma unroll
    for (int i = 1; i < kActThreads / 32; i++) rmax = max(rmax, red[i]);
    const float am = __uint_as_float(rmax);
    float G, E;
    global_scales(am, six_m, G, E);
    if (threadIdx.x == 0) {
      token_scale[row] = G;
      if (status && !isfinite(am)) atomicOr(status, kStatusNonFinite);
    }
#pragma unroll
    for (int k = 0; k < kActRegBlocks; k++) {
      const int b = threadIdx.x + k * kActThreads;
      if (b < nb) {
        uint32_t c0w, c1w, sb;
        quant_row_block_amax<F46>(wr[k], amax_of(bm[k]), E, tbl, c0w, c1w, sb);
        *reinterpret_cast<uint2*>(codes + row * (H / 2) + b * 8) = make_uint2(c0w, c1w);
        scales[row * nb + b] = (uint8_t)sb;
      }
    }
    for (int b = threadIdx.x + kActRegBlocks * kActThreads; b < nb; b += kActThreads) {
      const uint4 lo = *reinterpret_cast<const uint4*>(xr + b * 16);
      const uint4 hi = *reinterpret_cast<const uint4*>(xr + b * 16 + 8);
      const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      uint32_t c0w, c1w, sb;
      quant_row_block<F46>(wv, E, tbl, c0w, c1w, sb);
      *reinterpret_cast<uint2*>(codes + row * (H / 2) + b * 8) = make_uint2(c0w, c1w);
      scales[row * nb + b] = (uint8_t)sb;
    }
    __syncthreads();
  }
}

cudaError_t launch_act(const uint16_t* x, int64_t T, int H, bool f46, uint8_t* codes,
                       uint8_t* scales, float* token_scale, int* status, cudaStream_t s) {
  if (T == 0 || H == 0) return cudaSuccess;
  const DevInfo* di = device_info();
  const int grid = (int)std::min<int64_t>(T, (int64_t)di->sms * 16);
  if (f46)
    k_act<true><<<grid, kActThreads, 0, s>>>(x, T, H, codes, scales, token_scale, status);
  else
    k_act<false><<<grid, kActThreads, 0, s>>>(x, T, H, codes, scales, token_scale, status);
  return cudaGetLastError();
}

// --------------------------------------------------------------- dequant
// y = bf16( (c * S) * G ): c * S formed exactly as an f16 pair, widened to
// FP32, multiplied by the slice's tensor scale, rounded to bf16.
__device__ __forceinline__ uint32_t dq_pair(uint32_t byte, uint32_t S2, float2 G2) {
  const uint32_t h2 = e2m1x2_dec(byte);
  __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), *reinterpret_cast<const __half2*>(&S2));
  const float2 y = __fmul2_rn(__half22float2(v), G2);
  return bf16x2_rn(y.x, y.y);
}

constexpr int kDqThreads = 256;
constexpr int kDqPer = 4;  // blocks per thread per item
constexpr int64_t kDqChunk = (int64_t)kDqThreads * kDqPer;  // blocks per item

__global__ void __launch_bounds__(kDqThreads)
    k_dequant(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
              const float* __restrict__ Gs, int64_t blocks_per_slice, FastDiv cps,
              uint32_t nitems, uint16_t* __restrict__ dst) {
  __shared__ ScaleEnt tbl[128];
  build_scale_table(tbl);
  __syncthreads();
  for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x) {
    const uint32_t e = cps.div(it);
    const int64_t b0 = (int64_t)(it - e * cps.d) * kDqChunk;
    const float G = Gs[e];
    const float2 G2 = make_float2(G, G);
#pragma unroll
    for (int k = 0; k < kDqPer; k++) {
      const int64_t bl = b0 + k * kDqThreads + threadIdx.x;
      if (bl < blocks_per_slice) {
        const int64_t b = (int64_t)e * blocks_per_slice + bl;
        const uint2 c = *reinterpret_cast<const uint2*>(codes + b * 8);
        const uint32_t S2 = tbl[scales[b] & 0x7f].negS2 ^ 0x80008000u;
        uint4 o0, o1;
        o0.x = dq_pair(c.x & 0xff, S2, G2);
        o0.y = dq_pair((c.x >> 8) & 0xff, S2, G2);
        o0.z = dq_pair((c.x >> 16) & 0xff, S2, G2);
        o0.w = dq_pair(c.x >> 24, S2, G2);
        o1.x = dq_pair(c.y & 0xff, S2, G2);
        o1.y = dq_pair((c.y >> 8) & 0xff, S2, G2);
        o1.z = dq_pair((c.y >> 16) & 0xff, S2, G2);
        o1.w = dq_pair(c.y >> 24, S2, G2);
        uint4* out = reinterpret_cast<uint4*>(dst + b * 16);
        out[0] = o0;
        out[1] = o1;
      }
    }
  }
}

cudaError_t launch_dequant(const uint8_t* codes, const uint8_t* scales, const float* G,
                           int64_t nexp, int64_t per_slice, uint16_t* dst, cudaStream_t s) {
  const DevInfo* di = device_info();
  const int64_t bps = per_slice / 16;
  const int64_t cps = (bps + kDqChunk - 1) / kDqChunk;
  const int64_t nitems = nexp * cps;
  if (nitems == 0) return cudaSuccess;
  if (nitems >= (1ll << 31) - (1ll << 24)) return cudaErrorInvalidValue;
  FastDiv fd;
  fd.d = (uint32_t)cps;
  make_fastdiv(fd.d, &fd.m, &fd.s);
  const int grid = (int)std::min<int64_t>(nitems, (int64_t)di->sms * 8);
  k_dequant<<<grid, kDqThreads, 0, s>>>(codes, scales, G, bps, fd, (uint32_t)nitems, dst);
  return cudaGetLastError();
}

// ------------------------------------------------------- transposed dequant
// Tiles of 128 out-rows x 256 in-columns of the rowwise copy.  Each thread
// dequantises 8 consecutive out-rows of one 16-wide block column and writes
// them, transposed, as 16-byte runs into a shared [in][out] tile (chunks
// XOR-swizzled by (row >> 4) & 7 so the writes do not conflict); the tile is
// then stored as 256-byte runs of the [in, out] bf16 result.
constexpr int kTqR = 128, kTqC = 256, kTqThreads = 256;
constexpr int kTqSmem = kTqC * kTqR * 2 + kScaleTableBytes;  // 64 KiB tile + table

__global__ void __launch_bounds__(kTqThreads, 3)
    k_dequant_t(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                const float* __restrict__ Gs, int out, int in, FastDiv per_exp,
                FastDiv by_tiles_c, uint32_t ntiles, uint16_t* __restrict__ dst) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* const tile = smem;
  ScaleEnt* const tbl = reinterpret_cast<ScaleEnt*>(smem + kTqC * kTqR * 2);
  build_scale_table(tbl);
  const int tid = threadIdx.x;
  const int g = tid >> 4, b = tid & 15;
  for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    __syncthreads();  // table ready / previous tile stored
    const uint32_t e = per_exp.div(t);
    const uint32_t rem = t - e * per_exp.d;
    const int tr = (int)by_tiles_c.div(rem), tc = (int)(rem - tr * by_tiles_c.d);
    const int r0 = tr * kTqR, c0 = tc * kTqC;
    const int rv = min(kTqR, out - r0), cv = min(kTqC, in - c0);
    const float G = Gs[e];
    const float2 G2 = make_float2(G, G);
    if (g * 8 < rv && b * 16 < cv) {
      uint2 cw[8];
      uint32_t S2[8];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int64_t grow = (int64_t)e * out + r0 + g * 8 + i;
        cw[i] = *reinterpret_cast<const uint2*>(codes + grow * (in / 2) + c0 / 2 + b * 8);
        S2[i] = tbl[scales[grow * (in / 16) + c0 / 16 + b] & 0x7f].negS2 ^ 0x80008000u;
      }
#pragma unroll
      for (int kp = 0; kp < 8; kp++) {
        uint32_t ylo[8], yhi[8];  // bf16 of columns 2kp (low) and 2kp+1 (high) per row i
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const uint32_t word = kp < 4 ? cw[i].x : cw[i].y;
          const uint32_t byte = (word >> (8 * (kp & 3))) & 0xff;
          const uint32_t p = dq_pair(byte, S2[i], G2);
          ylo[i] = p & 0xffffu;
          yhi[i] = p >> 16;
        }
        const int rowA = b * 16 + 2 * kp, rowB = rowA + 1;  // in-index within the tile
        const int chA = g ^ ((rowA >> 4) & 7), chB = g ^ ((rowB >> 4) & 7);
        uint4 va = make_uint4(ylo[0] | (ylo[1] << 16), ylo[2] | (ylo[3] << 16),
                              ylo[4] | (ylo[5] << 16), ylo[6] | (ylo[7] << 16));
        uint4 vb = make_uint4(yhi[0] | (yhi[1] << 16), yhi[2] | (yhi[3] << 16),
                              yhi[4] | (yhi[5] << 16), yhi[6] | (yhi[7] << 16));
        *reinterpret_cast<uint4*>(tile + rowA * (kTqR * 2) + chA * 16) = va;
        *reinterpret_cast<uint4*>(tile + rowB * (kTqR * 2) + chB * 16) = vb;
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int it = 0; it < (kTqC * kTqR * 2 / 16) / kTqThreads; it++) {
      const int lin = it * kTqThreads + tid;
      const int row = lin >> 4, j = lin & 15;  // in-row within tile, 16-byte chunk
      if (row < cv && j * 8 < rv) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + row * (kTqR * 2) +
                                                        (j ^ ((row >> 4) & 7)) * 16);
        *reinterpret_cast<uint4*>(dst + ((int64_t)e * in + c0 + row) * out + r0 + j * 8) = v;
      }
    }
  }
}

cudaError_t launch_dequant_t(const uint8_t* codes, const uint8_t* scales, const float* G,
                             int64_t nexp, int out, int in, uint16_t* dst, cudaStream_t s) {
  static int attr_done = 0;
  if (!attr_done) {
    cudaError_t err = cudaFuncSetAttribute(k_dequant_t, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kTqSmem);
    if (err != cudaSuccess) return err;
    attr_done = 1;
  }
  const DevInfo* di = device_info();
  const int tiles_r = (out + kTqR - 1) / kTqR, tiles_c = (in + kTqC - 1) / kTqC;
  const int64_t ntiles = nexp * tiles_r * tiles_c;
  if (ntiles == 0) return cudaSuccess;
  if (ntiles >= (1ll << 31) - (1ll << 24)) return cudaErrorInvalidValue;
  FastDiv fpe, ftc;
  fpe.d = (uint32_t)(tiles_r * tiles_c);
  make_fastdiv(fpe.d, &fpe.m, &fpe.s);
  ftc.d = (uint32_t)tiles_c;
  make_fastdiv(ftc.d, &ftc.m, &ftc.s);
  const int grid = (int)std::min<int64_t>(ntiles, (int64_t)di->sms * 3);
  k_dequant_t<<<grid, kTqThreads, kTqSmem, s>>>(codes, scales, G, out, in, fpe, ftc,
                                                (uint32_t)ntiles, dst);
  return cudaGetLastError();
}

}  // namespace nvq
