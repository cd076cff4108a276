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
#include <cmath>
#include <cstdlib>

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
// CTAs per SM: the dual kernel keeps two (128 registers; at three it spills
// and runs 29 % slower), the rowwise-only kernel three (64 registers; 4 %
// faster than two).
constexpr int kQtMinbDual = 2, kQtMinbRow = 3;
constexpr int kTR = 64, kTC = 256, kQT = 256;
constexpr int kBoxC = 64;                       // box columns (128 bytes)
constexpr int kBoxBytes = kTR * kBoxC * 2;      // 8 KiB
constexpr int kInStage = kTR * kTC * 2;         // 32 KiB (four boxes)
constexpr int kColCodes = 4 * kTC * 8;          // [rb][col] 8 bytes
constexpr int kColScales = 4 * kTC;             // [rb][col] 1 byte
constexpr int kColBuf = kColCodes + kColScales; // one tile's staged columnwise results
// Shared memory of the rowwise-only (DUAL false) and dual-layout kernels.
template <bool DUAL>
constexpr int quant_smem() { return 2 * kInStage + (DUAL ? kColBuf : 0) + kScaleTableBytes + 64; }
constexpr uint32_t kWaitTries = 1u << 22;

struct QuantTileArgs {  // aligned as CUtensorMap requires
  CUtensorMap tmap;       // w as [nexp * rows, cols] bf16, 64 x 64 boxes
  uint8_t* codes_row;
  uint8_t* scales_row;
  uint8_t* codes_col;
  uint8_t* scales_col;
  const float* amax;      // complete for this launch's slices
  float* tensor_scale;
  int* status;
  int rows, cols;         // per slice
  int tiles_c;            // column tiles per slice
  uint32_t ntiles;        // tiles of this launch
  FastDiv per_exp;        // tiles per slice
  FastDiv by_tiles_c;
  uint32_t e0;            // first slice of this launch
  uint32_t nexp;          // slices in the whole stack
  uint32_t ahead;         // > 0: also reduce the amax of slice e + ahead (0: off)
  const uint16_t* w;      // the stack (for the look-ahead amax reads)
  float* amax_out;        // the look-ahead amax accumulators (same array as amax)
  int tiled;              // block scales in the tensor-core tiled layout
  int ct_row, ct_col;     // tiled layout: tiles per tile row (rowwise, columnwise)
  int64_t sl_row, sl_col; // tiled layout: bytes per slice (rowwise, columnwise)
  int col32;              // codes_col is 32-byte aligned
};

template <bool F46, bool DUAL>
__global__ void __launch_bounds__(kQT, DUAL ? kQtMinbDual : kQtMinbRow) k_quant_tiles(const __grid_constant__ QuantTileArgs A) {
  // The kernel has no static shared memory, so the dynamic block starts at
  // the (1 KiB aligned) base of the CTA's window, as the swizzled TMA boxes
  // require; a misaligned base is reported instead of used.
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* const in0 = smem;
  unsigned char* const colc = smem + 2 * kInStage;  // DUAL: kColBuf bytes
  unsigned char* const cols_s = colc + kColCodes;
  ScaleEnt* const tbl = reinterpret_cast<ScaleEnt*>(colc + (DUAL ? kColBuf : 0));
  uint64_t* const bar = reinterpret_cast<uint64_t*>(colc + (DUAL ? kColBuf : 0) + kScaleTableBytes);
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
    const uint32_t el = A.per_exp.div(t);
    const uint32_t rem = t - el * A.per_exp.d;
    T.e = A.e0 + el;
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

  // The columnwise results of a tile, staged in shared memory (codes
  // [rb][col] 8 bytes, then scales [rb][col] 1 byte), leave as contiguous
  // runs of the transposed layout: thread c writes column c.
  auto write_col = [&](const Tile& T) {
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
        if (A.col32 && (rows & 63) == 0) {
          // the run is 32-byte aligned: one full-sector store (half the
          // write requests of two 16-byte stores)
          const uint32_t v8[8] = {v0.x, v0.y, v1.x, v1.y, v2.x, v2.y, v3.x, v3.y};
          stg256(dstc, v8);
        } else {
          reinterpret_cast<uint4*>(dstc)[0] = make_uint4(v0.x, v0.y, v1.x, v1.y);
          reinterpret_cast<uint4*>(dstc)[1] = make_uint4(v2.x, v2.y, v3.x, v3.y);
        }
      } else {
        for (int rb = 0; rb < nrb; rb++)
          *reinterpret_cast<uint2*>(dstc + rb * 8) =
              *reinterpret_cast<const uint2*>(colc + rb * (kTC * 8) + c * 8);
      }
      if (A.tiled) {
        // the tile's four row blocks are block columns r0/16 .. +3, a
        // multiple of 4: four consecutive bytes of one tiled row
        uint8_t* dt = A.scales_col + T.e * A.sl_col +
                      scale_off_tiled(T.c0 + c, T.r0 >> 4, A.ct_col);
        if (nrb == 4) {
          *reinterpret_cast<uint32_t*>(dt) =
              (uint32_t)cols_s[c] | ((uint32_t)cols_s[kTC + c] << 8) |
              ((uint32_t)cols_s[2 * kTC + c] << 16) | ((uint32_t)cols_s[3 * kTC + c] << 24);
        } else {
          for (int rb = 0; rb < nrb; rb++) dt[rb] = cols_s[rb * kTC + c];
        }
      } else if (nrb == 4 && (rows & 63) == 0) {
        const uint32_t sc = (uint32_t)cols_s[c] | ((uint32_t)cols_s[kTC + c] << 8) |
                            ((uint32_t)cols_s[2 * kTC + c] << 16) |
                            ((uint32_t)cols_s[3 * kTC + c] << 24);
        *reinterpret_cast<uint32_t*>(dsts) = sc;
      } else {
        for (int rb = 0; rb < nrb; rb++) dsts[rb] = cols_s[rb * kTC + c];
      }
    }
  };

  // The rowwise-only kernel has one barrier per tile: the barrier that
  // opens tile t + 1 also frees tile t's input stage, which then takes the
  // copy two tiles ahead.  The dual kernel needs a second barrier between
  // the columnwise pass and the write-out of its staged results, and frees
  // the stage there.
  int st = 0;
  uint32_t it = 0;
  for (uint32_t t = t0; t < A.ntiles; t += gridDim.x, st ^= 1, it++) {
    const bool ok = mbar_wait(&bar[st], (it >> 1) & 1, kWaitTries);
    if (__syncthreads_or(!ok)) {  // a copy never landed: report and stop
      if (tid == 0 && A.status) atomicOr(A.status, kStatusTimeout);
      // the other stage's copy, if one is in flight
      if (DUAL || it == 0) mbar_wait(&bar[st ^ 1], ((it + 1) >> 1) & 1, kWaitTries);
      return;
    }
    if (!DUAL && it > 0) issue(t + gridDim.x, st ^ 1);
    const Tile T = tile_of(t);
    const float E = s_E[st];
    const unsigned char* tile = in0 + st * kInStage;

    // look-ahead amax: the same tile position of slice e + ahead is read now
    // and reduced after the rowwise pass, whose arithmetic covers the load
    // latency (the dual kernel is bound by instruction issue, so these reads
    // use HBM bandwidth it leaves idle).
    const bool ahead = DUAL && A.ahead != 0 && T.e + A.ahead < A.nexp;
    uint32_t sh[4][8];
    if (ahead) {
      const uint16_t* base = A.w + ((int64_t)(T.e + A.ahead) * rows + T.r0) * cols + T.c0;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int id = tid + i * kQT, r = id >> 4, c = (id & 15) * 16;
        if (r < T.rv && c < T.cv) {
          ldg32(base + (int64_t)r * cols + c, sh[i]);
        } else {
#pragma unroll
          for (int k = 0; k < 8; k++) sh[i][k] = 0;
        }
      }
    }

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
          if (A.tiled)
            A.scales_row[T.e * A.sl_row +
                         scale_off_tiled(T.r0 + r, (T.c0 >> 4) + cb, A.ct_row)] = (uint8_t)sb;
          else
            ps[16 * k * cols_16] = (uint8_t)sb;
        }
      }
    }

    if (ahead) {
      uint32_t m = maxabs2_nan(sh[0][0], sh[0][1]);
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int k = 0; k < 8; k++)
          if (i > 0 || k > 1) m = maxabs2_nan(m, sh[i][k]);
      uint32_t mm = maxabs2_nan(m, __byte_perm(m, 0, 0x1032)) & 0x7fff0000u;  // FP32 bits
      mm = __reduce_max_sync(0xffffffffu, mm);
      if ((tid & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(A.amax_out + T.e + A.ahead), mm);
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
      __syncthreads();
      issue(t + 2 * gridDim.x, st);
      write_col(T);
    }
  }
}

template <bool F46, bool DUAL>
static cudaError_t set_quant_smem() {
  static PerDeviceOnce attr;
  return attr.run([] {
    return cudaFuncSetAttribute(k_quant_tiles<F46, DUAL>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, quant_smem<DUAL>());
  });
}

cudaError_t launch_quant_tiles(const uint16_t* w, int64_t nexp, int rows, int cols, bool f46,
                               uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col,
                               uint8_t* scales_col, float* amax, float* tensor_scale,
                               int* status, bool compute_amax, bool tiled, cudaStream_t s) {
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
  A.amax_out = amax;
  A.tensor_scale = tensor_scale;
  A.status = status;
  A.rows = rows;
  A.cols = cols;
  A.tiles_c = tiles_c;
  A.per_exp.d = (uint32_t)per;
  make_fastdiv((uint32_t)per, &A.per_exp.m, &A.per_exp.s);
  A.by_tiles_c.d = (uint32_t)tiles_c;
  make_fastdiv((uint32_t)tiles_c, &A.by_tiles_c.m, &A.by_tiles_c.s);
  A.nexp = (uint32_t)nexp;
  A.w = w;
  A.tiled = tiled ? 1 : 0;
  A.ct_row = (cols / 16 + 3) / 4;
  A.ct_col = (rows / 16 + 3) / 4;
  A.sl_row = tiled_scale_bytes(rows, cols);
  A.sl_col = tiled_scale_bytes(cols, rows);
  A.col32 = (reinterpret_cast<uintptr_t>(codes_col) & 31) == 0;
  const bool dual = codes_col != nullptr;
  const int full_grid = di->sms * (dual ? kQtMinbDual : kQtMinbRow);
  // Slices per launch: with the look-ahead amax every launch quantises one
  // chunk while reducing the amax of the next, so each launch must see its
  // chunk's amax complete.  Two costs set the chunk: every launch boundary
  // (a partial last wave and the refill of the copy pipeline, about 16 us
  // measured), and the separate amax pass over the first chunk (2 bytes per
  // element at about 7 TB/s).  Their sum is smallest at
  // chunk = sqrt(nexp * 16 us / amax time of one slice)
  //       = sqrt(nexp * 5.6e7 / elements per slice),
  // and a chunk is kept at 40 waves of tiles or more.
  // The look-ahead is used by the dual-layout kernel only (the rowwise kernel
  // is close to memory bound, where a separate reduction pass is as fast);
  // its reads are 32-byte vectors, so it also needs a 32-byte aligned stack.
  // Otherwise the whole amax is reduced by one pass up front.
  const bool lookahead = compute_amax && codes_col != nullptr &&
                         (reinterpret_cast<uintptr_t>(w) & 31) == 0;
  int64_t chunk = nexp;
  if (lookahead) {
    const double balanced = std::floor(std::sqrt((double)nexp * 5.6e7 / ((double)rows * cols)) + 0.5);
    chunk = std::max<int64_t>((int64_t)balanced, (40ll * full_grid + per - 1) / per);
    chunk = std::max<int64_t>(chunk, 1);
    // NVQ_QUANT_CHUNK (slices per launch) overrides the choice; the tests use
    // it to exercise the look-ahead on small stacks.
    if (const char* env = std::getenv("NVQ_QUANT_CHUNK")) {
      const long long v = std::atoll(env);
      if (v > 0) chunk = v;
    }
    chunk = std::min<int64_t>(chunk, nexp);
  }
  if (compute_amax) {
    cudaError_t err = launch_amax(w, chunk, (int64_t)rows * cols, amax, s);
    if (err != cudaSuccess) return err;
  }
  cudaError_t err;
  if (f46 && dual) err = set_quant_smem<true, true>();
  else if (f46) err = set_quant_smem<true, false>();
  else if (dual) err = set_quant_smem<false, true>();
  else err = set_quant_smem<false, false>();
  if (err != cudaSuccess) return err;
  for (int64_t e0 = 0; e0 < nexp; e0 += chunk) {
    const int64_t n = std::min<int64_t>(chunk, nexp - e0);
    A.e0 = (uint32_t)e0;
    A.ntiles = (uint32_t)(n * per);
    A.ahead = (lookahead && e0 + chunk < nexp) ? (uint32_t)chunk : 0u;
    const int grid = (int)std::min<int64_t>(n * per, full_grid);
    if (f46 && dual) k_quant_tiles<true, true><<<grid, kQT, quant_smem<true>(), s>>>(A);
    else if (f46) k_quant_tiles<true, false><<<grid, kQT, quant_smem<false>(), s>>>(A);
    else if (dual) k_quant_tiles<false, true><<<grid, kQT, quant_smem<true>(), s>>>(A);
    else k_quant_tiles<false, false><<<grid, kQT, quant_smem<false>(), s>>>(A);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
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
          uint8_t* __restrict__ scales, float* __restrict__ token_scale, int* __restrict__ status,
          int tiled) {
  __shared__ ScaleEnt tbl[128];
  __shared__ uint32_t red[kActThreads / 32];
  build_scale_table(tbl);
  __syncthreads();
  const int nb = H / 16;
  const int ct = (nb + 3) / 4;  // tiled layout: tiles per tile row
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
        scales[tiled ? scale_off_tiled(row, b, ct) : row * nb + b] = (uint8_t)sb;
      }
    }
    for (int b = threadIdx.x + kActRegBlocks * kActThreads; b < nb; b += kActThreads) {
      const uint4 lo = *reinterpret_cast<const uint4*>(xr + b * 16);
      const uint4 hi = *reinterpret_cast<const uint4*>(xr + b * 16 + 8);
      const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      uint32_t c0w, c1w, sb;
      quant_row_block<F46>(wv, E, tbl, c0w, c1w, sb);
      *reinterpret_cast<uint2*>(codes + row * (H / 2) + b * 8) = make_uint2(c0w, c1w);
      scales[tiled ? scale_off_tiled(row, b, ct) : row * nb + b] = (uint8_t)sb;
    }
    __syncthreads();
  }
}

// Short rows (H <= 2048: at most 4 blocks per lane) take one warp per
// token: the row amax is a warp reduction with no CTA barrier, and each warp
// keeps two rows in flight (one CTA per token kept too few loads in flight
// per SM to cover the memory latency on such rows).
constexpr int kActWarpThreads = 256;
constexpr int kActWarpBlocks = 4;  // blocks per lane

template <bool F46>
__global__ void __launch_bounds__(kActWarpThreads)
    k_act_warp(const uint16_t* __restrict__ x, int64_t T, int H, uint8_t* __restrict__ codes,
               uint8_t* __restrict__ scales, float* __restrict__ token_scale,
               int* __restrict__ status, int tiled) {
  __shared__ ScaleEnt tbl[128];
  build_scale_table(tbl);
  __syncthreads();
  const int nb = H / 16;
  const int ct = (nb + 3) / 4;  // tiled layout: tiles per tile row
  const int lane = threadIdx.x & 31;
  const float six_m = F46 ? 1536.0f : 2688.0f;
  const int64_t nwarps = (int64_t)gridDim.x * (kActWarpThreads / 32);
  // the next row's blocks are loaded while this row is quantised, so each
  // warp keeps two rows in flight
  auto load = [&](int64_t row, uint32_t w[kActWarpBlocks][8]) {
#pragma unroll
    for (int k = 0; k < kActWarpBlocks; k++) {
      const int b = lane + 32 * k;
      if (row < T && b < nb) {
        const uint4 lo = ldg_stream(x + row * H + b * 16);
        const uint4 hi = ldg_stream(x + row * H + b * 16 + 8);
        w[k][0] = lo.x; w[k][1] = lo.y; w[k][2] = lo.z; w[k][3] = lo.w;
        w[k][4] = hi.x; w[k][5] = hi.y; w[k][6] = hi.z; w[k][7] = hi.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; i++) w[k][i] = 0;
      }
    }
  };
  int64_t row = blockIdx.x * (int64_t)(kActWarpThreads / 32) + (threadIdx.x >> 5);
  uint32_t wr[kActWarpBlocks][8], wn[kActWarpBlocks][8];
  load(row, wr);
  for (; row < T; row += nwarps) {
    load(row + nwarps, wn);
    uint32_t bm[kActWarpBlocks];
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < kActWarpBlocks; k++) {
      uint32_t mk = 0;
#pragma unroll
      for (int i = 0; i < 8; i++) mk = umaxmag2(mk, wr[k][i]);
      bm[k] = mk;
      m = umaxmag2(m, mk);
    }
    uint32_t mm = max(m & 0xffffu, m >> 16) << 16;
    mm = __reduce_max_sync(0xffffffffu, mm);
    const float am = __uint_as_float(mm);
    float G, E;
    global_scales(am, six_m, G, E);
    if (lane == 0) {
      token_scale[row] = G;
      if (status && !isfinite(am)) atomicOr(status, kStatusNonFinite);
    }
#pragma unroll
    for (int k = 0; k < kActWarpBlocks; k++) {
      const int b = lane + 32 * k;
      if (b < nb) {
        uint32_t c0w, c1w, sb;
        quant_row_block_amax<F46>(wr[k], amax_of(bm[k]), E, tbl, c0w, c1w, sb);
        *reinterpret_cast<uint2*>(codes + row * (H / 2) + b * 8) = make_uint2(c0w, c1w);
        scales[tiled ? scale_off_tiled(row, b, ct) : row * nb + b] = (uint8_t)sb;
      }
    }
#pragma unroll
    for (int k = 0; k < kActWarpBlocks; k++)
#pragma unroll
      for (int i = 0; i < 8; i++) wr[k][i] = wn[k][i];
  }
}

cudaError_t launch_act(const uint16_t* x, int64_t T, int H, bool f46, uint8_t* codes,
                       uint8_t* scales, float* token_scale, int* status, bool tiled,
                       cudaStream_t s) {
  if (T == 0 || H == 0) return cudaSuccess;
  const DevInfo* di = device_info();
  const int t = tiled ? 1 : 0;
  if (H / 16 <= 32 * kActWarpBlocks) {
    static PerDeviceInt occupancy[2];
    cudaError_t err = cudaSuccess;
    const int per_sm = std::max(1, occupancy[f46].get([&](cudaError_t* e) {
      int b = 0;
      *e = f46 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_act_warp<true>,
                                                               kActWarpThreads, 0)
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_act_warp<false>,
                                                               kActWarpThreads, 0);
      return b;
    }, &err));
    if (err != cudaSuccess) return err;
    const int64_t need = (T + kActWarpThreads / 32 - 1) / (kActWarpThreads / 32);
    const int g = (int)std::min<int64_t>(need, (int64_t)di->sms * per_sm);
    if (f46)
      k_act_warp<true><<<g, kActWarpThreads, 0, s>>>(x, T, H, codes, scales, token_scale, status, t);
    else
      k_act_warp<false><<<g, kActWarpThreads, 0, s>>>(x, T, H, codes, scales, token_scale, status, t);
    return cudaGetLastError();
  }
  const int grid = (int)std::min<int64_t>(T, (int64_t)di->sms * 16);
  if (f46)
    k_act<true><<<grid, kActThreads, 0, s>>>(x, T, H, codes, scales, token_scale, status, t);
  else
    k_act<false><<<grid, kActThreads, 0, s>>>(x, T, H, codes, scales, token_scale, status, t);
  return cudaGetLastError();
}

// --------------------------------------------------------------- dequant
// y = bf16( (c * S) * G ): c * S formed exactly as an f16 pair, widened to
// FP32, multiplied by the slice's tensor scale, rounded to bf16.
// Dequantises the 8 codes of a word (one scale S as an f16 pair, tensor
// scale G): four bf16 pairs, element 2j+{0,1} in word j.
__device__ __forceinline__ void dq_word(uint32_t w, uint32_t S2, float2 G2, uint32_t o[4]) {
  uint32_t h[4];
  e2m1x8_dec(w, h);
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const float2 y = __fmul2_rn(cs_exact(h[j], S2), G2);
    o[j] = bf16x2_rn(y.x, y.y);
  }
}

constexpr int kDqThreads = 256;
constexpr int kDqSlabs = 8;                                     // 8-element slabs per thread
constexpr int64_t kDqChunk = (int64_t)kDqThreads * kDqSlabs * 8;  // elements per item

// Work item = 16384 consecutive elements of one slice.  In slab k, thread t
// owns elements k*2048 + 8t .. +7 (half of a block): 4 code bytes, the
// block's scale byte and a 16-byte output run, so warp accesses are
// contiguous runs.
__global__ void __launch_bounds__(kDqThreads)
    k_dequant(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
              const float* __restrict__ Gs, int64_t per_slice, FastDiv cps, uint32_t nitems,
              uint16_t* __restrict__ dst) {
  __shared__ ScaleEnt tbl[128];
  build_scale_table(tbl);
  __syncthreads();
  for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x) {
    const uint32_t e = cps.div(it);
    const int64_t x0 = (int64_t)(it - e * cps.d) * kDqChunk + threadIdx.x * 8;
    const int64_t base = (int64_t)e * per_slice;
    const float G = Gs[e];
    const float2 G2 = make_float2(G, G);
    uint32_t cw[kDqSlabs], sbyte[kDqSlabs];
#pragma unroll
    for (int k = 0; k < kDqSlabs; k++) {
      const int64_t x = x0 + k * (kDqThreads * 8);
      const bool ok = x < per_slice;
      cw[k] = ok ? __ldg(reinterpret_cast<const uint32_t*>(codes) + ((base + x) >> 3)) : 0u;
      sbyte[k] = ok ? __ldg(scales + ((base + x) >> 4)) : 0u;
    }
#pragma unroll
    for (int k = 0; k < kDqSlabs; k++) {
      const int64_t x = x0 + k * (kDqThreads * 8);
      if (x < per_slice) {
        uint32_t o[4];
        dq_word(cw[k], pos_s2(tbl[sbyte[k] & 0x7f]), G2, o);
        stg_stream(dst + base + x, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
}

cudaError_t launch_dequant(const uint8_t* codes, const uint8_t* scales, const float* G,
                           int64_t nexp, int64_t per_slice, uint16_t* dst, cudaStream_t s) {
  const DevInfo* di = device_info();
  const int64_t cps = (per_slice + kDqChunk - 1) / kDqChunk;
  const int64_t nitems = nexp * cps;
  if (nitems == 0) return cudaSuccess;
  if (nitems >= (1ll << 31) - (1ll << 24)) return cudaErrorInvalidValue;
  FastDiv fd;
  fd.d = (uint32_t)cps;
  make_fastdiv(fd.d, &fd.m, &fd.s);
  const int grid = (int)std::min<int64_t>(nitems, (int64_t)di->sms * 8);
  k_dequant<<<grid, kDqThreads, 0, s>>>(codes, scales, G, per_slice, fd, (uint32_t)nitems, dst);
  return cudaGetLastError();
}

// ------------------------------------------------------- transposed dequant
// Tiles of 128 out-rows x 256 in-columns of the rowwise copy.  Thread
// (g = tid & 15, b = tid >> 4) dequantises out-rows 8g .. 8g+7 of 16-wide
// block column b and writes them, transposed, as 16-byte runs into a shared
// [in][out] tile laid out as two 128-byte-swizzled TMA boxes of 64 out-rows
// (chunk c of tile row r at c ^ (r & 7)): the eight lanes of each store
// phase hit eight different chunks.  One thread then stores the two boxes
// with TMA into the [nexp, in, out] result (a 3-D map, so a ragged tile never
// spills into the next slice).  The next tile's codes are loaded into
// registers while the stores drain.  Each column pair of a thread's block is
// dequantised and written to shared memory before the next, so no 8 x 8
// output block is held in registers.  Two CTAs per SM: with a third, L1
// shrinks to about a third and the row-strided code loads, whose 32-byte
// sectors other warps finish using, miss it (measured 47 % slower).
#ifndef NVQ_TQ_MINB
#define NVQ_TQ_MINB 2
#endif
constexpr int kTqR = 128, kTqC = 256, kTqThreads = 256;
constexpr int kTqBox = kTqC * 64 * 2;                                  // 32 KiB per box
constexpr int kTqSmem = 2 * kTqBox + kScaleTableBytes;                  // 64 KiB tile + table

// Column pair J (block columns 2J, 2J+1) of this thread's eight out-rows:
// dequantised and written as two 16-byte runs of the shared [in][out] tile.
template <int J>
__device__ __forceinline__ void dqt_column_pair(const uint2 cw[8], const uint32_t S2[8], float2 G2,
                                                unsigned char* box, int b, int g) {
  uint32_t v[8];  // bf16 pair (columns 2J, 2J+1) of row i
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const uint32_t h = e2m1x2_dec_byte<J & 3>(J < 4 ? cw[i].x : cw[i].y);
    const float2 y = __fmul2_rn(cs_exact(h, S2[i]), G2);
    v[i] = bf16x2_rn(y.x, y.y);
  }
  const int r = b * 16 + 2 * J;  // tile row (in-index) of column 2J
  const int off0 = r * 128 + (((g & 7) ^ (r & 7)) << 4);
  const int off1 = (r + 1) * 128 + (((g & 7) ^ ((r + 1) & 7)) << 4);
  *reinterpret_cast<uint4*>(box + off0) =
      make_uint4(__byte_perm(v[0], v[1], 0x5410), __byte_perm(v[2], v[3], 0x5410),
                 __byte_perm(v[4], v[5], 0x5410), __byte_perm(v[6], v[7], 0x5410));
  *reinterpret_cast<uint4*>(box + off1) =
      make_uint4(__byte_perm(v[0], v[1], 0x7632), __byte_perm(v[2], v[3], 0x7632),
                 __byte_perm(v[4], v[5], 0x7632), __byte_perm(v[6], v[7], 0x7632));
}

struct DequantTArgs {  // aligned as CUtensorMap requires
  CUtensorMap tmap;  // dst as [nexp][in][out] bf16, boxes of 64 x 256 x 1
  const uint8_t* codes;
  const uint8_t* scales;
  const float* G;
  int out, in;
  FastDiv per_exp, by_tiles_r;
  uint32_t ntiles;
};

__global__ void __launch_bounds__(kTqThreads, NVQ_TQ_MINB) k_dequant_t(const __grid_constant__ DequantTArgs A) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* const tile = smem;
  ScaleEnt* const tbl = reinterpret_cast<ScaleEnt*>(smem + 2 * kTqBox);
  build_scale_table(tbl);
  const int tid = threadIdx.x;
  const int g = tid & 15, b = tid >> 4;
  const int out = A.out, in = A.in;
  const int64_t in_h = in >> 1, in_16 = in >> 4;
  unsigned char* const box = tile + (g >> 3) * kTqBox;

  // Consecutive tiles step along `out` first: the CTAs running at the same
  // time then fill neighbouring 256-byte pieces of the same rows of the
  // transposed result.
  struct Tile { uint32_t e; int r0, c0, rv, cv; };
  auto tile_of = [&](uint32_t t) {
    Tile T;
    T.e = A.per_exp.div(t);
    const uint32_t rem = t - T.e * A.per_exp.d;
    const int tc = (int)A.by_tiles_r.div(rem), tr = (int)(rem - tc * A.by_tiles_r.d);
    T.r0 = tr * kTqR;
    T.c0 = tc * kTqC;
    T.rv = min(kTqR, out - T.r0);
    T.cv = min(kTqC, in - T.c0);
    return T;
  };
  uint2 cw[8];
  uint32_t sb[8];
  auto load = [&](uint32_t t) {
    const Tile T = tile_of(t);
    const bool ok = g * 8 < T.rv && b * 16 < T.cv;
    const int64_t grow = (int64_t)T.e * out + T.r0 + g * 8;
    const uint8_t* pc = A.codes + grow * in_h + (T.c0 >> 1) + b * 8;
    const uint8_t* ps = A.scales + grow * in_16 + (T.c0 >> 4) + b;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      cw[i] = ok ? __ldg(reinterpret_cast<const uint2*>(pc + i * in_h)) : make_uint2(0, 0);
      sb[i] = ok ? __ldg(ps + i * in_16) : 0u;
    }
  };

  if (smem_u32(smem) & 1023u) return;  // the swizzled boxes need a 1 KiB aligned base
  if (blockIdx.x < A.ntiles) load(blockIdx.x);
  for (uint32_t t = blockIdx.x; t < A.ntiles; t += gridDim.x) {
    if (tid == 0) bulk_wait_read<0>();  // the previous tile's stores have read the tile
    __syncthreads();
    const Tile T = tile_of(t);
    const float Gv = A.G[T.e];
    const float2 G2 = make_float2(Gv, Gv);
    if (g * 8 < T.rv && b * 16 < T.cv) {
      uint32_t S2[8];
#pragma unroll
      for (int i = 0; i < 8; i++) S2[i] = pos_s2(tbl[sb[i] & 0x7f]);
      dqt_column_pair<0>(cw, S2, G2, box, b, g);
      dqt_column_pair<1>(cw, S2, G2, box, b, g);
      dqt_column_pair<2>(cw, S2, G2, box, b, g);
      dqt_column_pair<3>(cw, S2, G2, box, b, g);
      dqt_column_pair<4>(cw, S2, G2, box, b, g);
      dqt_column_pair<5>(cw, S2, G2, box, b, g);
      dqt_column_pair<6>(cw, S2, G2, box, b, g);
      dqt_column_pair<7>(cw, S2, G2, box, b, g);
    }
    fence_proxy_async_smem();  // make this thread's tile writes visible to the TMA unit
    __syncthreads();
    if (tid == 0) {
      tma_store_3d(&A.tmap, T.r0, T.c0, (int)T.e, tile);
      if (T.rv > 64) tma_store_3d(&A.tmap, T.r0 + 64, T.c0, (int)T.e, tile + kTqBox);
      bulk_commit();
    }
    if (t + gridDim.x < A.ntiles) load(t + gridDim.x);
  }
  if (tid == 0) bulk_wait<0>();
}

cudaError_t launch_dequant_t(const uint8_t* codes, const uint8_t* scales, const float* G,
                             int64_t nexp, int out, int in, uint16_t* dst, cudaStream_t s) {
  static PerDeviceOnce attr;
  const cudaError_t err0 = attr.run([] {
    return cudaFuncSetAttribute(k_dequant_t, cudaFuncAttributeMaxDynamicSharedMemorySize, kTqSmem);
  });
  if (err0 != cudaSuccess) return err0;
  const DevInfo* di = device_info();
  const int tiles_r = (out + kTqR - 1) / kTqR, tiles_c = (in + kTqC - 1) / kTqC;
  const int64_t ntiles = nexp * tiles_r * tiles_c;
  if (ntiles == 0) return cudaSuccess;
  if (ntiles >= (1ll << 31) - (1ll << 24) || nexp >= (1ll << 31)) return cudaErrorInvalidValue;
  DequantTArgs A;
  if (!encode_tmap_3d(&A.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, dst, (uint64_t)out, (uint64_t)in,
                      (uint64_t)nexp, (uint64_t)out * 2, (uint64_t)out * in * 2, 64, kTqC, 1,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  A.codes = codes;
  A.scales = scales;
  A.G = G;
  A.out = out;
  A.in = in;
  A.per_exp.d = (uint32_t)(tiles_r * tiles_c);
  make_fastdiv(A.per_exp.d, &A.per_exp.m, &A.per_exp.s);
  A.by_tiles_r.d = (uint32_t)tiles_r;
  make_fastdiv(A.by_tiles_r.d, &A.by_tiles_r.m, &A.by_tiles_r.s);
  A.ntiles = (uint32_t)ntiles;
  const int grid = (int)std::min<int64_t>(ntiles, (int64_t)di->sms * NVQ_TQ_MINB);
  k_dequant_t<<<grid, kTqThreads, kTqSmem, s>>>(A);
  return cudaGetLastError();
}

}  // namespace nvq
