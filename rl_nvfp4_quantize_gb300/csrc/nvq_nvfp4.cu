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
#include <atomic>

#include "nvq_common.cuh"
#include "nvq_internal.h"

namespace nvq {

// ------------------------------------------------------- per-slice scales
// Zeroes p[0, n) and, when q is given, q[0, n).
__global__ void k_zero_f32(float* p, float* q, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    p[i] = 0.0f;
    if (q) q[i] = 0.0f;
  }
}

// G[e] = amax[e] / (6 M) for every slice, the last step of a quantisation
// call (it also replaces the look-ahead counts kept in G), and status bit 0
// for a non-finite amax.
__global__ void k_tensor_scales(const float* amax, float* G, int64_t n, float six_m, int* status) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float g, e;
    const float am = amax[i];
    global_scales(am, six_m, g, e);
    G[i] = g;
    if (status && !isfinite(am)) atomicOr(status, kStatusNonFinite);
  }
}

cudaError_t launch_tensor_scales(const float* amax, float* G, int64_t n, bool f46, int* status,
                                 cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int grid = (int)std::min<int64_t>((n + 255) / 256, 1024);
  k_tensor_scales<<<grid, 256, 0, s>>>(amax, G, n, f46 ? 1536.0f : 2688.0f, status);
  return cudaGetLastError();
}

// Lead of the quantisers' look-ahead beyond one slice, in waves of the grid
// (see k_quant_tiles).  Process-wide; nvq_debug_set_quant_lead changes it.
std::atomic<int> g_quant_lead_waves{2};

cudaError_t launch_zero_f32(float* p, int64_t n, cudaStream_t s, float* q) {
  if (n <= 0) return cudaSuccess;
  int grid = (int)std::min<int64_t>((n + 255) / 256, 1024);
  k_zero_f32<<<grid, 256, 0, s>>>(p, q, n);
  return cudaGetLastError();
}

// ----------------------------------------------------- rowwise / dual tiles
// One co-resident grid (cooperative launch), one CTA per SM, walks the
// tiles of the whole stack -- 64 rows x 256 columns of one slice each --
// in one global order g = slice * P + tile (P tiles per slice).  Each CTA
// has two compute groups of eight warps, one control warp per group and a
// look-ahead stream of two warps:
//   * compute group k of CTA b (group index q = 2b + k of Gq = 2 * grid)
//     quantises tiles q, q + Gq, q + 2Gq, ... from a two-stage ring.  It
//     waits only on the stage's `full` barrier, which completes when the
//     copy has landed and its control warp has placed the tile's slice
//     encode factor E beside it, and releases the stage on its `empty`
//     barrier.  It never waits on the rest of the grid.
//   * control warp k issues group k's copies in order, each once its stage
//     is released, and gives each tile its E once the slice is finished.
//     It spends its time blocked in barrier waits, not polling, so the
//     compute warps keep the issue slots.
//   * the look-ahead stream computes the slice amax in the same pass over
//     the stack: it streams this CTA's look-ahead tiles (the same tile
//     indices as its two groups, up to L tiles ahead of them) through a
//     small ring, reduces each to its magnitude maximum, and keeps the
//     per-slice results described below.
// The look-ahead copies use the L2 evict-last policy and the quantising
// copies (the same bytes, later) evict-first: the look-ahead read is the
// HBM read, the second read hits L2, which holds the window of about L
// tiles (32 KiB each); L = P + lead waves of Gq tiles.
//
// Per slice s, word ts[s] (the tensor_scale output, zeroed first) counts
// the look-ahead tiles reduced so far, until it holds the slice's result.
// The look-ahead stream folds each tile's maximum into amax[s] with an atomic
// max at once and adds its CTA's tile count for a slice to ts[s] in one
// release add when its look-ahead moves on to the next slice (by then its
// earlier atomics have completed, so the release costs little).  The CTA
// whose add completes the count acquires, reads the complete amax[s] and
// replaces ts[s] by DONE | bits(G_s) (the sign bit marks it: a count never
// has it, and G_s >= 0).  E for a tile comes from that word alone.
//
// Every wait ends.  The look-ahead stream waits only for its own ring and
// for its window, la <= (the least tile its groups still need E for) + L.
// A group waiting for slice s holds that least tile inside slice s, so the
// window admits every look-ahead tile below (s + 1) P + lead Gq; with
// lead >= 1 that includes the CTA's first look-ahead tile in slice s + 1,
// whose arrival publishes the CTA's slice-s count.  By induction over the
// slices every count is published, and all CTAs are resident (cooperative
// launch).  The waits are bounded all the same.  With the amax given
// (L = 0) there is no look-ahead.
//
// Per tile, from the staged input (four TMA boxes of 64 x 64 bf16, 128-byte
// swizzle):
//   rowwise pass   : 1024 blocks of 1x16, four per thread, results stored
//                    straight to global (8 code bytes + 1 scale byte);
//   columnwise pass: 256 units of 16 rows x 4 columns, one per thread, each
//                    column widened into the pair layout of a rowwise block
//                    and quantised as one; the results are staged and written
//                    as contiguous runs of the transposed [in, out/2] layout.
// Inside a swizzled box, 16-byte chunk c of row r sits at chunk c ^ (r & 7).
constexpr int kTR = 64, kTC = 256;
constexpr int kBoxC = 64;                       // box columns (128 bytes)
constexpr int kBoxBytes = kTR * kBoxC * 2;      // 8 KiB
constexpr int kInStage = kTR * kTC * 2;         // 32 KiB (four boxes)
constexpr int kColCodes = 4 * kTC * 8;          // [rb][col] 8 bytes
constexpr int kColScales = 4 * kTC;             // [rb][col] 1 byte
constexpr int kColBuf = kColCodes + kColScales; // one tile's staged columnwise results
constexpr int kQGroups = 2;                     // compute groups per CTA
constexpr int kQGT = 256;                       // threads per compute group
// Four compute warpgroups and one warpgroup of two control warps and the
// two look-ahead warps (96 registers per thread: the compute path fits them
// unspilled).
constexpr int kQThreads = kQGroups * kQGT + 128;
template <bool DUAL>
__host__ __device__ constexpr int group_bytes() { return 2 * kInStage + (DUAL ? kColBuf : 0); }
// look-ahead stages: as many as fit beside the groups' buffers
template <bool DUAL>
__host__ __device__ constexpr int la_stages() { return DUAL ? 2 : 3; }
// the groups' stages (and staging), the look-ahead stages, the E4M3 table,
// the barriers, the E slots and a few words
template <bool DUAL>
constexpr int quant_smem() {
  return kQGroups * group_bytes<DUAL>() + la_stages<DUAL>() * kInStage + kScaleTableBytes + 256;
}
constexpr uint32_t kWaitTries = 1u << 22;

struct QuantTileArgs {  // aligned as CUtensorMap requires
  CUtensorMap tmap;       // w as [nexp * rows, cols] bf16, 64 x 64 boxes
  uint8_t* codes_row;
  uint8_t* scales_row;
  uint8_t* codes_col;
  uint8_t* scales_col;
  float* amax;            // L > 0: accumulated here (zeroed first); L = 0: given
  uint32_t* ts;           // L > 0: the per-slice words described above (zeroed first)
  int* status;
  int rows, cols;         // per slice
  int tiles_c;            // column tiles per slice
  int ntiles;             // tiles of the stack
  int la;                 // look-ahead distance L in tiles (0: amax given)
  FastDiv per_exp;        // tiles per slice (P)
  FastDiv by_tiles_c;
  int tiled;              // block scales in the tensor-core tiled layout
  int ct_row, ct_col;     // tiled layout: tiles per tile row (rowwise, columnwise)
  int64_t sl_row, sl_col; // tiled layout: bytes per slice (rowwise, columnwise)
  int col32;              // codes_col is 32-byte aligned
};

struct QTile { uint32_t e; int r0, c0, rv, cv; };

__device__ __forceinline__ QTile qtile_of(const QuantTileArgs& A, int t) {
  QTile T;
  const uint32_t e = A.per_exp.div((uint32_t)t);
  const uint32_t rem = (uint32_t)t - e * A.per_exp.d;
  const uint32_t tr = A.by_tiles_c.div(rem);
  const uint32_t tc = rem - tr * (uint32_t)A.tiles_c;
  T.e = e;
  T.r0 = (int)tr * kTR;
  T.c0 = (int)tc * kTC;
  T.rv = min(kTR, A.rows - T.r0);
  T.cv = min(kTC, A.cols - T.c0);
  return T;
}

// Thread `lane 0` of the control warp: the four box loads of tile t into
// `dst`, completing on `b` (parts out of range are zero-filled).
__device__ __forceinline__ void qload_tile(const QuantTileArgs& A, const QTile& T,
                                           unsigned char* dst, uint64_t* b, uint64_t pol) {
  mbar_arrive_expect_tx(b, kInStage);
  const int y = (int)(T.e * (uint32_t)A.rows) + T.r0;
#pragma unroll
  for (int j = 0; j < kTC / kBoxC; j++)
    tma_load_2d_hint(dst + j * kBoxBytes, &A.tmap, T.c0 + j * kBoxC, y, b, pol);
}
__device__ __forceinline__ void qload_tile(const QuantTileArgs& A, int t, unsigned char* dst,
                                           uint64_t* b, uint64_t pol) {
  qload_tile(A, qtile_of(A, t), dst, b, pol);
}

// A tile's place, as the control warp hands it to the group beside E.
__device__ __forceinline__ uint4 qtile_pack(const QTile& T) {
  return make_uint4(T.e, (uint32_t)T.r0, (uint32_t)T.c0, ((uint32_t)T.rv << 16) | (uint32_t)T.cv);
}
__device__ __forceinline__ QTile qtile_unpack(const uint4 p) {
  QTile T;
  T.e = p.x;
  T.r0 = (int)p.y;
  T.c0 = (int)p.z;
  T.rv = (int)(p.w >> 16);
  T.cv = (int)(p.w & 0xffffu);
  return T;
}

// Two columnwise blocks side by side: wc[i] holds row i of the block, low
// half column j, high half column j + 1.  One magnitude-max tree over the 16
// words gives both column maxima; each value is widened and scaled into the
// pair layout of a rowwise block, (row 2k, row 2k + 1), and each column is
// quantised as one rowwise block; cj / ck receive the codes of column j /
// j + 1.  (The pairs come straight from the widening, so no byte regroup is
// needed; processing the two columns side by side in packed pairs instead
// would need the pairs transposed for the error chains.)
template <bool F46>
__device__ __forceinline__ void quant_col_pair(const uint32_t wc[16], float E, const ScaleEnt* tbl,
                                               uint32_t cj[2], uint32_t ck[2], uint32_t& sbj,
                                               uint32_t& sbk) {
  uint32_t m = maxabs2(wc[0], wc[1]);
#pragma unroll
  for (int i = 2; i < 16; i++) m = maxabs2(m, wc[i]);
  m &= 0x7fff7fffu;
  const float2 E2 = make_float2(E, E);
  float2 tj[8], tk[8];
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const float2 r0 = widen2(wc[2 * k]), r1 = widen2(wc[2 * k + 1]);
    tj[k] = __fmul2_rn(make_float2(r0.x, r1.x), E2);
    tk[k] = __fmul2_rn(make_float2(r0.y, r1.y), E2);
  }
  quant_block_t2<F46>(tj, __fmul_rn(lo_f(m), E), tbl, cj[0], cj[1], sbj);
  quant_block_t2<F46>(tk, __fmul_rn(hi_f(m), E), tbl, ck[0], ck[1], sbk);
}

// ---- compute group k (threads tg = 0 .. 255 of the group)
template <bool F46, bool DUAL>
__device__ __forceinline__ void quant_group(const QuantTileArgs& A, unsigned char* gbase,
                                            const ScaleEnt* tbl, uint64_t* full, uint64_t* empty,
                                            const float* s_E, const uint4* s_T, int k, int tg) {
  const int rows = A.rows, cols = A.cols, N = A.ntiles;
  const int Gq = kQGroups * gridDim.x;
  const int64_t cols_h = cols >> 1, cols_16 = cols >> 4, rows_h = rows >> 1, rows_16 = rows >> 4;
  unsigned char* const colc = gbase + 2 * kInStage;  // DUAL: kColBuf bytes
  unsigned char* const cols_s = colc + kColCodes;
  const int warp = tg >> 5, lane = tg & 31;
  // rowwise geometry: 16-column block cb of rows rb0 + 16k.  In each
  // quarter warp the lanes of odd boxes take the other row of the row pair,
  // so their 16-byte loads fall in the other half of the banks.
  const int cb = tg & 15;
  const int rb0 = 2 * warp + (((tg >> 4) ^ (tg >> 2)) & 1);
  const int rbox = (cb >> 2) * kBoxBytes, rchunk = 2 * (cb & 3);
  const int row_lo = (rchunk ^ (rb0 & 7)) << 4, row_hi = ((rchunk + 1) ^ (rb0 & 7)) << 4;
  // columnwise geometry: row block cr, columns 4q .. 4q+3
  const int cr = warp >> 1, q = ((warp & 1) << 5) + lane;
  const int cbox = (q >> 4) * kBoxBytes, cchunk = (q & 15) >> 1, chalf = (q & 1) * 8;
  // columnwise staging: columns 4q..4q+1 and 4q+2..4q+3 fill the two
  // 16-byte halves of a 32-byte group, in swapped order for odd q >> 2, so
  // a quarter warp's 16-byte stores cover all banks.
  const int hsw = (q >> 2) & 1;

  // The columnwise results of a tile, staged in shared memory (codes
  // [rb][col] 8 bytes, the two halves of each 32-byte group swapped as
  // above, then scales [rb][col] 1 byte), leave as contiguous runs of the
  // transposed layout: thread c writes column c.
  // write-out constants of this thread's column c = tg: its staged code
  // offset, and whether whole tiles take the one-store paths (rows a
  // multiple of 64, 32-byte aligned columnwise codes, linear scales)
  const int soff = (tg >> 2) * 32 + ((((tg >> 1) & 1) ^ ((tg >> 4) & 1)) << 4) + (tg & 1) * 8;
  const bool col_fast = (rows & 63) == 0 && A.col32 && !A.tiled;
  auto write_col = [&](const QTile& T) {
    const int c = tg;
    if (col_fast && T.rv == kTR && c < T.cv) {
      const int64_t grow = (int64_t)T.e * cols + T.c0 + c;
      const uint2 v0 = *reinterpret_cast<const uint2*>(colc + soff);
      const uint2 v1 = *reinterpret_cast<const uint2*>(colc + kTC * 8 + soff);
      const uint2 v2 = *reinterpret_cast<const uint2*>(colc + 2 * kTC * 8 + soff);
      const uint2 v3 = *reinterpret_cast<const uint2*>(colc + 3 * kTC * 8 + soff);
      const uint32_t v8[8] = {v0.x, v0.y, v1.x, v1.y, v2.x, v2.y, v3.x, v3.y};
      stg256_stream(A.codes_col + grow * rows_h + (T.r0 >> 1), v8);
      const uint32_t b01 = __byte_perm(cols_s[c], cols_s[kTC + c], 0x0040);
      const uint32_t b23 = __byte_perm(cols_s[2 * kTC + c], cols_s[3 * kTC + c], 0x0040);
      stg_stream_u32(A.scales_col + grow * rows_16 + (T.r0 >> 4), __byte_perm(b01, b23, 0x5410));
    } else if (c < T.cv) {
      const int nrb = T.rv >> 4;
      const int64_t grow = (int64_t)T.e * cols + T.c0 + c;
      uint8_t* dstc = A.codes_col + grow * rows_h + (T.r0 >> 1);
      uint8_t* dsts = A.scales_col + grow * rows_16 + (T.r0 >> 4);
      if (nrb == 4 && (rows & 31) == 0) {
        const uint2 v0 = *reinterpret_cast<const uint2*>(colc + soff);
        const uint2 v1 = *reinterpret_cast<const uint2*>(colc + kTC * 8 + soff);
        const uint2 v2 = *reinterpret_cast<const uint2*>(colc + 2 * kTC * 8 + soff);
        const uint2 v3 = *reinterpret_cast<const uint2*>(colc + 3 * kTC * 8 + soff);
        if (A.col32 && (rows & 63) == 0) {
          // the run is 32-byte aligned: one full-sector store (half the
          // write requests of two 16-byte stores)
          const uint32_t v8[8] = {v0.x, v0.y, v1.x, v1.y, v2.x, v2.y, v3.x, v3.y};
          stg256_stream(dstc, v8);
        } else {
          stg_stream(dstc, make_uint4(v0.x, v0.y, v1.x, v1.y));
          stg_stream(dstc + 16, make_uint4(v2.x, v2.y, v3.x, v3.y));
        }
      } else {
        for (int rb = 0; rb < nrb; rb++) {
          const uint2 v = *reinterpret_cast<const uint2*>(colc + rb * (kTC * 8) + soff);
          stg_stream_v2(dstc + rb * 8, v.x, v.y);
        }
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
        stg_stream_u32(dsts, sc);
      } else {
        for (int rb = 0; rb < nrb; rb++) stg_stream_u8(dsts + rb, cols_s[rb * kTC + c]);
      }
    }
  };

  const int bar_id = 1 + k;
  int j = 0;
  for (int g = kQGroups * (int)blockIdx.x + k; g < N; g += Gq, j++) {
    const int st = j & 1;
    const bool ok = mbar_wait(&full[2 * k + st], (j >> 1) & 1, kWaitTries);
    // The whole group agrees to go on, and the previous tile's staged
    // results have been written out by every thread.
    if (named_barrier_or(bar_id, kQGT, !ok)) {
      if (tg == 0 && A.status) atomicOr(A.status, kStatusTimeout);
      return;
    }
    const float E = s_E[2 * k + st];
    const unsigned char* tile = gbase + st * kInStage;
    const QTile T = qtile_unpack(s_T[2 * k + st]);

    // rowwise blocks: four per thread, 16 rows apart (rows r = rb0 + 16 kk
    // share r & 7, so the swizzled chunk offsets are fixed per thread and the
    // pointers step by a constant)
    {
      const int64_t grow0 = (int64_t)T.e * rows + T.r0 + rb0;
      uint8_t* pc = A.codes_row + grow0 * cols_h + (T.c0 >> 1) + cb * 8;
      uint8_t* ps = A.scales_row + grow0 * cols_16 + (T.c0 >> 4) + cb;
      const unsigned char* rowp = tile + rbox + rb0 * 128;
      const int nkk = cb * 16 < T.cv ? min(4, (T.rv - rb0 + 15) >> 4) : 0;
#pragma unroll 1
      for (int kk = 0; kk < nkk; kk++) {
        const uint4 lo = *reinterpret_cast<const uint4*>(rowp + row_lo);
        const uint4 hi = *reinterpret_cast<const uint4*>(rowp + row_hi);
        const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        uint32_t c0w, c1w, sb;
        quant_row_block<F46>(wv, E, tbl, c0w, c1w, sb);
        stg_stream_v2(pc, c0w, c1w);
        if (A.tiled)
          A.scales_row[T.e * A.sl_row +
                       scale_off_tiled(T.r0 + rb0 + 16 * kk, (T.c0 >> 4) + cb, A.ct_row)] =
              (uint8_t)sb;
        else
          stg_stream_u8(ps, sb);
        rowp += 16 * 128;
        pc += 16 * cols_h;
        ps += 16 * cols_16;
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
        unsigned char* const cq = colc + cr * (kTC * 8) + q * 32;
        uint32_t cj[2], ck[2], sbj, sbk, sw;
        quant_col_pair<F46>(wa, E, tbl, cj, ck, sbj, sbk);
        *reinterpret_cast<uint4*>(cq + hsw * 16) = make_uint4(cj[0], cj[1], ck[0], ck[1]);
        sw = sbj | (sbk << 8);
        quant_col_pair<F46>(wb, E, tbl, cj, ck, sbj, sbk);
        *reinterpret_cast<uint4*>(cq + (hsw ^ 1) * 16) = make_uint4(cj[0], cj[1], ck[0], ck[1]);
        sw |= (sbj << 16) | (sbk << 24);
        *reinterpret_cast<uint32_t*>(cols_s + cr * kTC + q * 4) = sw;
      }
    }
    named_barrier(bar_id, kQGT);  // the stage is read; the staged results are complete
    if (tg == 0) mbar_arrive(&empty[2 * k + st]);
    if (DUAL) write_col(T);
  }
}

// ---- control warp k: group k's copies, and E beside each
template <bool F46>
__device__ __forceinline__ void quant_control(const QuantTileArgs& A, unsigned char* gbase,
                                              uint64_t* full, uint64_t* empty, float* s_E, uint4* s_T,
                                              volatile int* s_least, int k) {
  const float six_m = F46 ? 1536.0f : 2688.0f;
  const int lane = threadIdx.x & 31, N = A.ntiles;
  const int Gq = kQGroups * gridDim.x;
  uint64_t pol = 0;
  if (lane == 0) pol = l2_policy_evict_first();
  int e_s = -1;  // the slice whose E is cached
  float e_E = 0.0f;
  bool failed = false;
  int j = 0;  // the group's tile count so far
  for (int g = kQGroups * (int)blockIdx.x + k; g < N; g += Gq, j++) {
    const int st = j & 1;
    // the stage holds the group's tile j - 2 until the group releases it
    int ok = 1;
    if (j >= 2 && lane == 0) ok = mbar_wait(&empty[2 * k + st], ((j - 2) >> 1) & 1, kWaitTries);
    if (!__shfl_sync(0xffffffffu, ok, 0)) {
      failed = true;
      break;
    }
    const QTile T = qtile_of(A, g);
    if (lane == 0) qload_tile(A, T, gbase + st * kInStage, &full[2 * k + st], pol);
    const int s = (int)A.per_exp.div((uint32_t)g);
    float E = 0.0f;
    if (A.la == 0) {
      float Gs;
      global_scales(A.amax[s], six_m, Gs, E);
    } else if (s == e_s) {
      E = e_E;
    } else {
      // the slice's word, once it holds the result (bounded wait)
      uint32_t w = 0;
      if (lane == 0) wait_done(A.ts + s, w);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w & kSliceDone) {
        E = fminf(__frcp_rn(__uint_as_float(w & ~kSliceDone)), FLT_MAX);
        e_s = s;
        e_E = E;
      } else {
        failed = true;  // the tile still gets its arrival (E = 0) below
      }
    }
    if (lane == 0) {
      s_E[2 * k + st] = E;
      s_T[2 * k + st] = qtile_pack(T);
      mbar_arrive(&full[2 * k + st]);
      *s_least = g + Gq;  // the next tile this group needs E for
    }
    if (failed) {
      j++;
      break;
    }
  }
  if (failed && lane == 0) {
    // A stage was never released or a slice never finished: report, and
    // wait (bounded) for this warp's copies still in flight; the group
    // stops on its own at its next bounded wait.
    if (A.status) atomicOr(A.status, kStatusTimeout);
    for (int i = max(0, j - 2); i < j; i++) mbar_wait(&full[2 * k + (i & 1)], (i >> 1) & 1, kWaitTries);
  }
}

// ---- the look-ahead stream (kLaThreads threads, two warps): this CTA's
// look-ahead tiles in increasing order, n -> q0 + n % 2 + (n / 2) Gq, each
// copied into a ring of S stages, reduced to its magnitude maximum (bf16 bit
// patterns, exact; NaN propagates) and counted into the per-slice words.
// Rows past the slice (a ragged last row tile) belong to the next slice and
// are left out; columns past the slice are zero-filled by the copy.
constexpr int kLaThreads = 64;
template <bool F46, int S>
__device__ __forceinline__ void quant_lookahead(const QuantTileArgs& A, unsigned char* lab,
                                                uint64_t* lafull, uint32_t* s_lamax,
                                                const volatile int* s_least) {
  const float six_m = F46 ? 1536.0f : 2688.0f;
  const int lt = threadIdx.x - (kQGroups * kQGT + 32 * kQGroups), lane = lt & 31, lw = lt >> 5;
  const int N = A.ntiles, L = A.la;
  const int Gq = kQGroups * gridDim.x;
  const int q0 = kQGroups * (int)blockIdx.x;
  const uint32_t P = A.per_exp.d;
  int la_count = 0;
  for (int k = 0; k < kQGroups; k++)
    if (q0 + k < N) la_count += (N - 1 - (q0 + k)) / Gq + 1;
  auto la_tile = [&](int n) { return q0 + (n % kQGroups) + (n / kQGroups) * Gq; };
  uint64_t pol = 0;
  if (lt == 0) pol = l2_policy_evict_last();
  // thread 0 of the stream: this CTA's unpublished count, and the last add
  int pend_s = -1, chk_s = -1;
  uint32_t pend_n = 0, chk_old = 0, chk_n = 0;
  auto finish_if_last = [&]() {
    if (chk_s >= 0 && chk_old + chk_n == P) {
      fence_acq_rel_gpu();
      float Gs, Es;
      global_scales(ld_relaxed_f32(A.amax + chk_s), six_m, Gs, Es);
      st_relaxed_u32(A.ts + chk_s, kSliceDone | __float_as_uint(Gs));
    }
    chk_s = -1;
  };
  auto publish = [&]() {
    finish_if_last();
    if (pend_s >= 0) {
      chk_old = atom_add_release(A.ts + pend_s, pend_n);
      chk_s = pend_s;
      chk_n = pend_n;
    }
    pend_s = -1;
    pend_n = 0;
  };
  // thread 0: copy look-ahead tile n once the window admits it (bounded)
  auto issue = [&](int n) -> bool {
    const int t = la_tile(n);
    uint64_t t0 = 0;
    for (uint32_t i = 0; t > min(s_least[0], s_least[1]) + L; i++) {
      finish_if_last();  // nothing of ours may be held while we wait
      const uint64_t now = globaltimer_ns();
      if (i == 0) t0 = now;
      else if (now - t0 > kMaxWaitNs) return false;
      __nanosleep(64);
    }
    qload_tile(A, t, lab + (n % S) * kInStage, &lafull[n % S], pol);
    return true;
  };
  int issued = 0;
  bool ok = true;
  if (lt == 0)
    for (; issued < S && issued < la_count && ok; issued++) ok = issue(issued);
  for (int n = 0; n < la_count; n++) {
    const int st = n % S;
    bool landed = __shfl_sync(0xffffffffu, (int)ok, 0) && mbar_wait(&lafull[st], (n / S) & 1, kWaitTries);
    uint32_t m[4] = {0, 0, 0, 0};
    if (landed) {
      const int rv = (A.rows & (kTR - 1)) == 0
                         ? kTR
                         : min(kTR, A.rows - (int)A.by_tiles_c.div(
                                                 (uint32_t)la_tile(n) -
                                                 A.per_exp.div((uint32_t)la_tile(n)) * P) *
                                                 kTR);
      // thread lt reads 16-byte chunks lt + 64 i: row (lt >> 3) + 8 (i & 7) of its box
      const unsigned char* p = lab + st * kInStage + lt * 16;
      if (rv == kTR) {
#pragma unroll 8
        for (int i = 0; i < kInStage / (16 * kLaThreads); i++) {
          const uint4 v = *reinterpret_cast<const uint4*>(p + i * 16 * kLaThreads);
          m[i & 3] = maxabs2_nan(m[i & 3], maxabs2_nan(maxabs2_nan(v.x, v.y), maxabs2_nan(v.z, v.w)));
        }
      } else {
#pragma unroll 8
        for (int i = 0; i < kInStage / (16 * kLaThreads); i++) {
          if ((lt >> 3) + 8 * (i & 7) < rv) {
            const uint4 v = *reinterpret_cast<const uint4*>(p + i * 16 * kLaThreads);
            m[i & 3] = maxabs2_nan(m[i & 3], maxabs2_nan(maxabs2_nan(v.x, v.y), maxabs2_nan(v.z, v.w)));
          }
        }
      }
    }
    uint32_t mm = maxabs2_nan(maxabs2_nan(m[0], m[1]), maxabs2_nan(m[2], m[3]));
    mm = maxabs2_nan(mm, __byte_perm(mm, 0, 0x1032)) & 0x7fff0000u;  // FP32 bits
    mm = __reduce_max_sync(0xffffffffu, mm);
    if (lane == 0) s_lamax[2 * (n & 1) + lw] = mm;
    if (named_barrier_or(3, kLaThreads, !landed)) {
      // a look-ahead copy never landed: report and stop, after the copies
      // still in flight
      if (lt == 0) {
        if (A.status) atomicOr(A.status, kStatusTimeout);
        for (int i = n + 1; i < issued; i++) mbar_wait(&lafull[i % S], (i / S) & 1, kWaitTries);
      }
      return;
    }
    if (lt == 0) {
      const uint32_t mx = max(s_lamax[2 * (n & 1)], s_lamax[2 * (n & 1) + 1]);
      finish_if_last();  // the add published earlier has returned by now
      const int s = (int)A.per_exp.div((uint32_t)la_tile(n));
      if (s != pend_s) publish();  // before this tile's atomic: nothing left in flight
      atomicMax(reinterpret_cast<unsigned int*>(A.amax + s), mx);
      pend_s = s;
      pend_n++;
      if (n + 1 == la_count) {  // this CTA's last look-ahead tile
        publish();
        finish_if_last();
      }
      if (ok && issued < la_count) {  // the stage just read takes tile n + S
        ok = issue(issued);
        issued++;
        if (!ok && A.status) atomicOr(A.status, kStatusTimeout);
      }
    }
  }
}

template <bool F46, bool DUAL>
__global__ void __launch_bounds__(kQThreads, 1) k_quant_tiles(const __grid_constant__ QuantTileArgs A) {
  // The kernel has no static shared memory, so the dynamic block starts at
  // the (1 KiB aligned) base of the CTA's window, as the swizzled TMA boxes
  // require; a misaligned base is reported instead of used.
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int kG = group_bytes<DUAL>();
  constexpr int kS = la_stages<DUAL>();
  unsigned char* const lab = smem + kQGroups * kG;
  ScaleEnt* const tbl = reinterpret_cast<ScaleEnt*>(lab + kS * kInStage);
  uint4* const s_T = reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(tbl) +
                                               kScaleTableBytes);          // [group][stage]
  uint64_t* const full = reinterpret_cast<uint64_t*>(s_T + 2 * kQGroups);  // [group][stage]
  uint64_t* const empty = full + 2 * kQGroups;                           // [group][stage]
  uint64_t* const lafull = empty + 2 * kQGroups;                         // [look-ahead stage]
  float* const s_E = reinterpret_cast<float*>(lafull + kS);              // [group][stage]
  uint32_t* const s_lamax = reinterpret_cast<uint32_t*>(s_E + 2 * kQGroups);  // [2][warp]
  int* const s_least = reinterpret_cast<int*>(s_lamax + 4);  // [group]
  const int tid = threadIdx.x;
  const bool misaligned = (smem_u32(smem) & 1023u) != 0;
  if (!misaligned) {
    build_scale_table(tbl);
    if (tid == 0) {
      for (int i = 0; i < 2 * kQGroups; i++) {
        mbar_init(&full[i], 2);   // the copy's arrival with its bytes, and E's
        mbar_init(&empty[i], 1);  // the group's release
      }
      for (int i = 0; i < kS; i++) mbar_init(&lafull[i], 1);
      for (int k = 0; k < kQGroups; k++) s_least[k] = kQGroups * (int)blockIdx.x + k;
      fence_barrier_init();
    }
  } else if (tid == 0 && A.status) {
    atomicOr(A.status, kStatusTimeout);
  }
  __syncthreads();
  constexpr int kCtl = kQGroups * kQGT;  // the control warps, then the look-ahead warps
  if (misaligned) return;
  if (tid >= kCtl + 32 * kQGroups) {
    if (A.la > 0) quant_lookahead<F46, kS>(A, lab, lafull, s_lamax, s_least);
  } else if (tid >= kCtl) {
    const int k = (tid - kCtl) >> 5;
    quant_control<F46>(A, smem + k * kG, full, empty, s_E, s_T, s_least + k, k);
  } else {
    quant_group<F46, DUAL>(A, smem + (tid / kQGT) * kG, tbl, full, empty, s_E, s_T, tid / kQGT,
                           tid % kQGT);
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

// CTAs of k_quant_tiles<F46, DUAL> resident per SM (the cooperative grid's
// limit), once per device.
template <bool F46, bool DUAL>
static int quant_occupancy(cudaError_t* err) {
  static PerDeviceInt occ;
  return occ.get(
      [](cudaError_t* e) {
        int b = 0;
        *e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_quant_tiles<F46, DUAL>, kQThreads,
                                                           quant_smem<DUAL>());
        return b;
      },
      err);
}

template <bool F46, bool DUAL>
static cudaError_t launch_quant_kernel(const QuantTileArgs& A, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = quant_smem<DUAL>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_quant_tiles<F46, DUAL>, A);
}

template <bool F46, bool DUAL>
static cudaError_t run_quant(QuantTileArgs& A, int64_t per, cudaStream_t s) {
  const DevInfo* di = device_info();
  cudaError_t err = set_quant_smem<F46, DUAL>();
  if (err != cudaSuccess) return err;
  const int occ = quant_occupancy<F46, DUAL>(&err);
  if (err != cudaSuccess) return err;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  // one CTA per compute-group pair of tiles; no more CTAs than resident
  const int grid = (int)std::min<int64_t>(((int64_t)A.ntiles + kQGroups - 1) / kQGroups,
                                          (int64_t)occ * di->sms);
  // Look-ahead distance: one slice of tiles plus a lead of a few waves of
  // the grid's compute groups (see above); 0 when the amax is given.
  if (A.la) {
    const int64_t la =
        per + (int64_t)g_quant_lead_waves.load(std::memory_order_relaxed) * kQGroups * grid;
    if (la + A.ntiles >= (1ll << 31)) return cudaErrorInvalidValue;
    A.la = (int)la;
  }
  return launch_quant_kernel<F46, DUAL>(A, grid, s);
}

cudaError_t launch_quant_tiles(const uint16_t* w, int64_t nexp, int rows, int cols, bool f46,
                               uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col,
                               uint8_t* scales_col, float* amax, float* tensor_scale,
                               int* status, bool compute_amax, bool tiled, cudaStream_t s) {
  const int tiles_r = (rows + kTR - 1) / kTR, tiles_c = (cols + kTC - 1) / kTC;
  const int64_t per = (int64_t)tiles_r * tiles_c;
  const int64_t ntiles = nexp * per;
  if (ntiles == 0) return cudaSuccess;
  if (ntiles >= (1ll << 30) || nexp * (int64_t)rows >= (1ll << 31))
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
  // The per-slice words live in tensor_scale until the final pass below
  // overwrites them with the tensor scales.
  A.ts = reinterpret_cast<uint32_t*>(tensor_scale);
  A.status = status;
  A.rows = rows;
  A.cols = cols;
  A.tiles_c = tiles_c;
  A.ntiles = (int)ntiles;
  A.la = compute_amax ? 1 : 0;
  A.per_exp.d = (uint32_t)per;
  make_fastdiv((uint32_t)per, &A.per_exp.m, &A.per_exp.s);
  A.by_tiles_c.d = (uint32_t)tiles_c;
  make_fastdiv((uint32_t)tiles_c, &A.by_tiles_c.m, &A.by_tiles_c.s);
  A.tiled = tiled ? 1 : 0;
  A.ct_row = (cols / 16 + 3) / 4;
  A.ct_col = (rows / 16 + 3) / 4;
  A.sl_row = tiled_scale_bytes(rows, cols);
  A.sl_col = tiled_scale_bytes(cols, rows);
  A.col32 = (reinterpret_cast<uintptr_t>(codes_col) & 31) == 0;
  cudaError_t err;
  if (compute_amax) {
    // amax accumulators and arrival counters start at zero
    if ((err = launch_zero_f32(amax, nexp, s, tensor_scale)) != cudaSuccess) return err;
  }
  const bool dual = codes_col != nullptr;
  if (f46 && dual) err = run_quant<true, true>(A, per, s);
  else if (f46) err = run_quant<true, false>(A, per, s);
  else if (dual) err = run_quant<false, true>(A, per, s);
  else err = run_quant<false, false>(A, per, s);
  if (err != cudaSuccess) return err;
  return launch_tensor_scales(amax, tensor_scale, nexp, f46, status, s);
}

// ------------------------------------------------------ per-token activations
// Three kernels by row length H: rows of at most 2048 values take one warp
// per token with the row in registers (k_act_warp); rows up to
// kActStreamMaxH values one warp per token streaming rows through shared
// memory (k_act_stream); longer rows one CTA per token (k_act).
//
// k_act: one CTA of 128 threads per token row.  Up to kActRegBlocks blocks
// per thread stay in registers between the row-amax reduction and the
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
        uint32_t mk = maxabs2_nan(wr[k][0], wr[k][1]);
#pragma unroll
        for (int i = 2; i < 8; i++) mk = maxabs2_nan(mk, wr[k][i]);
        bm[k] = mk;
        m = maxabs2_nan(m, mk);
      }
    }
    for (int b = threadIdx.x + kActRegBlocks * kActThreads; b < nb; b += kActThreads) {
      const uint4 lo = ldg_stream(xr + b * 16);
      const uint4 hi = ldg_stream(xr + b * 16 + 8);
      m = maxabs2_nan(m, maxabs2_nan(maxabs2_nan(lo.x, lo.y), maxabs2_nan(lo.z, lo.w)));
      m = maxabs2_nan(m, maxabs2_nan(maxabs2_nan(hi.x, hi.y), maxabs2_nan(hi.z, hi.w)));
    }
    m &= 0x7fff7fffu;  // magnitudes: NaN patterns order above infinity as integers
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
      uint32_t mk = maxabs2_nan(wr[k][0], wr[k][1]);
#pragma unroll
      for (int i = 2; i < 8; i++) mk = maxabs2_nan(mk, wr[k][i]);
      bm[k] = mk;
      m = maxabs2_nan(m, mk);
    }
    m &= 0x7fff7fffu;  // magnitudes: NaN patterns order above infinity as integers
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

// Longer rows of up to kActStreamMaxH values take one warp per token row, and
// each warp streams its rows (w, w + W, w + 2W, ... of the grid's W warps)
// through its own ring of S shared-memory row buffers filled by 1-D bulk
// copies (L2 evict-first), so many rows are in flight per SM without
// holding them in registers.  From a staged row the warp takes the row
// amax (any chunk order, one pass), then quantises block b = lane + 32k
// from its 32 bytes in a second pass.  16 warps per CTA, one CTA per SM;
// S = as many buffers as fit 200 KiB.
constexpr int kActStreamThreads = 512;
constexpr int kActStreamWarps = kActStreamThreads / 32;
constexpr int kActStreamBytes = 200 * 1024;
constexpr int kActStreamMaxH = kActStreamBytes / (kActStreamWarps * 2);  // S >= 1
constexpr int kActStreamMaxS = 8;

__host__ __device__ constexpr int act_stream_stages(int H) {
  return (kActStreamBytes / (kActStreamWarps * 2 * H)) < kActStreamMaxS
             ? kActStreamBytes / (kActStreamWarps * 2 * H)
             : kActStreamMaxS;
}
__host__ __device__ constexpr int act_stream_smem(int H) {
  return kActStreamWarps * act_stream_stages(H) * 2 * H + kActStreamWarps * kActStreamMaxS * 8 +
         kScaleTableBytes;
}

template <bool F46>
__global__ void __launch_bounds__(kActStreamThreads, 1)
    k_act_stream(const uint16_t* __restrict__ x, int64_t T, int H, uint8_t* __restrict__ codes,
                 uint8_t* __restrict__ scales, float* __restrict__ token_scale,
                 int* __restrict__ status, int tiled) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int S = act_stream_stages(H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rowbytes = 2u * (uint32_t)H;
  unsigned char* const ring = smem + (size_t)warp * S * rowbytes;
  uint64_t* const bar = reinterpret_cast<uint64_t*>(smem + (size_t)kActStreamWarps * S * rowbytes) +
                        warp * kActStreamMaxS;
  ScaleEnt* const tbl = reinterpret_cast<ScaleEnt*>(
      smem + (size_t)kActStreamWarps * S * rowbytes + kActStreamWarps * kActStreamMaxS * 8);
  build_scale_table(tbl);
  if (lane == 0) {
    for (int i = 0; i < S; i++) mbar_init(&bar[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int nb = H / 16;
  const int ct = (nb + 3) / 4;  // tiled layout: tiles per tile row
  const float six_m = F46 ? 1536.0f : 2688.0f;
  const int64_t W = (int64_t)gridDim.x * kActStreamWarps;
  const int64_t w0 = (int64_t)blockIdx.x * kActStreamWarps + warp;
  uint64_t pol = 0;
  if (lane == 0) pol = l2_policy_evict_first();
  auto issue = [&](int64_t j) {  // lane 0: the warp's j-th row into stage j % S
    const int64_t row = w0 + j * W;
    if (row < T) {
      uint64_t* b = &bar[j % S];
      mbar_arrive_expect_tx(b, rowbytes);
      bulk_load_hint(ring + (j % S) * rowbytes, x + row * H, rowbytes, b, pol);
    }
  };
  if (lane == 0)
    for (int j = 0; j < S; j++) issue(j);
  for (int64_t j = 0; w0 + j * W < T; j++) {
    const int64_t row = w0 + j * W;
    const unsigned char* buf = ring + (j % S) * rowbytes;
    if (!__all_sync(0xffffffffu, mbar_wait(&bar[j % S], (uint32_t)(j / S) & 1, 1u << 22))) {
      // a copy never landed: report and stop, after the copies in flight
      if (lane == 0) {
        if (status) atomicOr(status, kStatusTimeout);
        for (int64_t i = j + 1; i < j + S && w0 + i * W < T; i++)
          mbar_wait(&bar[i % S], (uint32_t)(i / S) & 1, 1u << 22);
      }
      return;
    }
    // row amax: magnitude maximum of bf16 pairs (a selection, hence exact;
    // a NaN propagates), four independent chains
    uint32_t m4[4] = {0, 0, 0, 0};
#pragma unroll 4
    for (int c = lane; c < (int)(rowbytes >> 4); c += 32) {
      const uint4 v = *reinterpret_cast<const uint4*>(buf + c * 16);
      m4[0] = maxabs2_nan(m4[0], v.x);
      m4[1] = maxabs2_nan(m4[1], v.y);
      m4[2] = maxabs2_nan(m4[2], v.z);
      m4[3] = maxabs2_nan(m4[3], v.w);
    }
    // magnitudes: NaN patterns order above infinity as integers
    const uint32_t m =
        maxabs2_nan(maxabs2_nan(m4[0], m4[1]), maxabs2_nan(m4[2], m4[3])) & 0x7fff7fffu;
    uint32_t mm = max(m & 0xffffu, m >> 16) << 16;
    mm = __reduce_max_sync(0xffffffffu, mm);
    const float am = __uint_as_float(mm);
    float G, E;
    global_scales(am, six_m, G, E);
    if (lane == 0) {
      token_scale[row] = G;
      if (status && !isfinite(am)) atomicOr(status, kStatusNonFinite);
    }
    // blocks lane + 32k, four at a time so that their chains interleave
    for (int b0 = lane; b0 < nb; b0 += 128) {
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int b = b0 + 32 * k;
        if (b < nb) {
          const uint4 lo = *reinterpret_cast<const uint4*>(buf + b * 32);
          const uint4 hi = *reinterpret_cast<const uint4*>(buf + b * 32 + 16);
          const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          uint32_t c0w, c1w, sb;
          quant_row_block<F46>(wv, E, tbl, c0w, c1w, sb);
          stg_stream_v2(codes + row * (H / 2) + b * 8, c0w, c1w);
          if (tiled) scales[scale_off_tiled(row, b, ct)] = (uint8_t)sb;
          else stg_stream_u8(scales + row * nb + b, sb);
        }
      }
    }
    __syncwarp();  // every lane is done with the buffer before it is refilled
    if (lane == 0) issue(j + S);
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
  if (H <= kActStreamMaxH) {
    const int smem = act_stream_smem(H);
    static PerDeviceOnce attr[2];
    cudaError_t err = attr[f46].run([] {
      cudaError_t e = cudaFuncSetAttribute(k_act_stream<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kActStreamBytes + kActStreamWarps * kActStreamMaxS * 8 +
                                               kScaleTableBytes);
      if (e != cudaSuccess) return e;
      return cudaFuncSetAttribute(k_act_stream<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kActStreamBytes + kActStreamWarps * kActStreamMaxS * 8 +
                                      kScaleTableBytes);
    });
    if (err != cudaSuccess) return err;
    const int64_t need = (T + kActStreamWarps - 1) / kActStreamWarps;
    const int g = (int)std::min<int64_t>(need, (int64_t)di->sms);
    if (f46)
      k_act_stream<true><<<g, kActStreamThreads, smem, s>>>(x, T, H, codes, scales, token_scale,
                                                            status, t);
    else
      k_act_stream<false><<<g, kActStreamThreads, smem, s>>>(x, T, H, codes, scales, token_scale,
                                                             status, t);
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
// Tiles of 128 out-rows x 256 NB in-columns of the rowwise copy.  Thread
// (g = tid & 15, b = tid >> 4) dequantises out-rows 8g .. 8g+7 of the NB
// 16-wide block columns NB b .. NB b + NB - 1 and writes each of its 16 NB
// in-columns straight to global memory as one 16-byte run of an output row:
// the 16 lanes of a warp that share b write 16 x 16 contiguous bytes of one
// row, so a warp store is two full 256-byte runs and no shared staging,
// fence, barrier or TMA store is needed.  Consecutive tiles step along `out`
// first, so the CTAs running together fill neighbouring pieces of the same
// output rows.  NB = 2 when `in` is a multiple of 32: a warp's code load then
// takes 32 contiguous bytes of each of 16 rows (whole sectors when the rows
// are 32-byte aligned) and each thread has twice the bytes in flight; with
// NB = 1 a warp takes 16 bytes of each row and the neighbouring warp the
// other half of the sector.  Measured alternatives: staging the tile in
// shared memory and storing it with TMA boxes was the same speed (2 % slower
// on the down stack); taller tiles (256 or 512 out-rows, longer contiguous
// output per row) and one block column per warp (512-byte stores) were
// 15-35 % slower, as were three or four CTAs per SM.
constexpr int kTqThreads = 256;

template <int NB>
__global__ void __launch_bounds__(kTqThreads, 2)
    k_dequant_t(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                const float* __restrict__ G, int out, int in, FastDiv per_exp, FastDiv by_tiles_r,
                uint32_t ntiles, uint16_t* __restrict__ dst) {
  __shared__ ScaleEnt tbl[128];
  build_scale_table(tbl);
  __syncthreads();
  constexpr int kTC = 256 * NB;  // in-columns per tile
  const int tid = threadIdx.x;
  const int g = tid & 15, b = tid >> 4;
  const int64_t in_h = in >> 1, in_16 = in >> 4;
  for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const uint32_t e = per_exp.div(t);
    const uint32_t rem = t - e * per_exp.d;
    const int tc = (int)by_tiles_r.div(rem), tr = (int)(rem - tc * by_tiles_r.d);
    const int r0 = tr * 128, c0 = tc * kTC;
    if (g * 8 >= min(128, out - r0) || b * 16 * NB >= min(kTC, in - c0)) continue;
    const int64_t grow = (int64_t)e * out + r0 + g * 8;
    const uint8_t* pc = codes + grow * in_h + (c0 >> 1) + b * 8 * NB;
    const uint8_t* ps = scales + grow * in_16 + (c0 >> 4) + b * NB;
    // code words of out-row i: cw[i][2h], cw[i][2h + 1] hold block column h;
    // sc[i] the row's NB scale bytes (block column h in byte h)
    uint32_t cw[8][2 * NB], sc[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      if constexpr (NB == 2) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(pc + i * in_h));
        cw[i][0] = v.x; cw[i][1] = v.y; cw[i][2] = v.z; cw[i][3] = v.w;
        sc[i] = __ldg(reinterpret_cast<const uint16_t*>(ps + i * in_16));
      } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(pc + i * in_h));
        cw[i][0] = v.x; cw[i][1] = v.y;
        sc[i] = __ldg(ps + i * in_16);
      }
    }
    const float Gv = G[e];
    const float2 G2 = make_float2(Gv, Gv);
#pragma unroll
    for (int h = 0; h < NB; h++) {
      uint32_t S2[8];
#pragma unroll
      for (int i = 0; i < 8; i++) S2[i] = pos_s2(tbl[(sc[i] >> (8 * h)) & 0x7f]);
      // output row (in-index) c0 + 16 (NB b + h) + j, out-columns r0 + 8g .. +7
      uint16_t* const d0 = dst + ((int64_t)e * in + c0 + 16 * (NB * b + h)) * out + r0 + 8 * g;
#pragma unroll
      for (int J = 0; J < 8; J++) {
        uint32_t v[8];  // bf16 pair (in-columns 2J, 2J+1) of out-row i
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const uint32_t word = cw[i][2 * h + (J >> 2)];
          const uint32_t hh = e2m1x2_dec(__byte_perm(word, 0, 0x4440 + (J & 3)));
          const float2 y = __fmul2_rn(cs_exact(hh, S2[i]), G2);
          v[i] = bf16x2_rn(y.x, y.y);
        }
        stg_stream(d0 + (int64_t)(2 * J) * out,
                   make_uint4(__byte_perm(v[0], v[1], 0x5410), __byte_perm(v[2], v[3], 0x5410),
                              __byte_perm(v[4], v[5], 0x5410), __byte_perm(v[6], v[7], 0x5410)));
        stg_stream(d0 + (int64_t)(2 * J + 1) * out,
                   make_uint4(__byte_perm(v[0], v[1], 0x7632), __byte_perm(v[2], v[3], 0x7632),
                              __byte_perm(v[4], v[5], 0x7632), __byte_perm(v[6], v[7], 0x7632)));
      }
    }
  }
}

cudaError_t launch_dequant_t(const uint8_t* codes, const uint8_t* scales, const float* G,
                             int64_t nexp, int out, int in, uint16_t* dst, cudaStream_t s) {
  const DevInfo* di = device_info();
  // two block columns per thread when every row holds an even number of
  // blocks (its codes then start on a 16-byte boundary, its scales on a
  // 2-byte one)
  const bool two = (in % 32) == 0;
  const int tiles_r = (out + 127) / 128, tiles_c = two ? (in + 511) / 512 : (in + 255) / 256;
  const int64_t ntiles = nexp * tiles_r * tiles_c;
  if (ntiles == 0) return cudaSuccess;
  if (ntiles >= (1ll << 31) - (1ll << 24)) return cudaErrorInvalidValue;
  FastDiv pe, br;
  pe.d = (uint32_t)(tiles_r * tiles_c);
  make_fastdiv(pe.d, &pe.m, &pe.s);
  br.d = (uint32_t)tiles_r;
  make_fastdiv(br.d, &br.m, &br.s);
  const int grid = (int)std::min<int64_t>(ntiles, (int64_t)di->sms * 2);
  if (two)
    k_dequant_t<2><<<grid, kTqThreads, 0, s>>>(codes, scales, G, out, in, pe, br,
                                                (uint32_t)ntiles, dst);
  else
    k_dequant_t<1><<<grid, kTqThreads, 0, s>>>(codes, scales, G, out, in, pe, br,
                                                (uint32_t)ntiles, dst);
  return cudaGetLastError();
}

}  // namespace nvq
