// nvq_gemm.cuh -- grouped (routed-expert) GEMM on the fifth-generation tensor
// cores with the weight dequantised on the fly: Y = X . B_e^T for the token
// rows of each expert e, where B_e is the bf16 value of a 4-bit weight that a
// "producer" forms tile by tile in shared memory, so the bf16 weight never
// goes to HBM.
//
//   X  bf16 [T][K], the rows of expert e following those of expert e-1
//   B_e bf16 values, N x K per expert (the producer decides how they are
//       read and where they sit in shared memory: K-major or MN-major)
//   Y  [T][N], FP32 or bf16 (round to nearest even of the FP32 sum)
//
// Tile: 256 token rows (two M = 128 halves) x 256 columns of N, K in steps of
// 64; the B slice of a K step serves both halves.  One CTA per tile, 18
// warps:
//   warps 0-15: producers -- form the 256 x 64 B slice of each K step in one
//               of SB shared stages from the packed weight data of that step
//               (codes and scales, staged by TMA in one of SC shared stages);
//               afterwards the epilogue: tensor memory -> registers -> Y rows
//               (warp w: accumulator rows 32 (w & 3) .. +31 of half
//               (w >> 2) & 1, columns 128 (w >> 3) .. +127);
//   warp 16   : lane 0: TMA loads of the two X tiles [128 rows][64 K]
//               (128-byte swizzle) into one of SA shared stages; lane 1: TMA
//               loads of the packed weight data of each K step;
//   warp 17   : allocates all 512 columns of tensor memory (two 128 x 256
//               FP32 accumulators), issues tcgen05.mma (M 128, N 256, K 16,
//               bf16 x bf16 -> FP32) -- four per K step and half, the second
//               half only when the expert has rows there -- commits them to
//               the stages' "empty" barriers, and frees the tensor memory.
// X, the packed weight data and B have stage rings of their own, so each runs
// as far ahead as its own buffers allow; the producers issue no global loads
// of their own (only shared-memory reads at fixed offsets).
// Every wait is bounded; a wait that gives up sets the status word's timeout
// bit, and every path still reaches the tensor-memory release.
#pragma once

#include <cuda.h>
#include <cstdint>
#include <algorithm>

#include "nvq_common.cuh"
#include "nvq_internal.h"
#include "nvq_tc.cuh"

namespace nvq {

constexpr int kGM = 128, kGN = 256, kGK = 64;
constexpr int kGHalves = 2;                    // M halves per CTA tile
constexpr int kGA = kGHalves * kGM * kGK * 2;  // 32 KiB of X per stage (two 16 KiB halves)
constexpr int kGB = kGN * kGK * 2;             // 32 KiB of B per stage
constexpr int kGProducerWarps = 16;
constexpr int kGProducers = kGProducerWarps * 32;
constexpr int kGTmaWarp = kGProducerWarps, kGMmaWarp = kGProducerWarps + 1;
constexpr int kGThreads = kGProducers + 64;
constexpr uint32_t kGTmemCols = 512;           // two FP32 accumulators of 128 x 256
constexpr uint32_t kGWaitTries = 1u << 22;

template <class WP>
struct GroupedGemmArgs {  // aligned as CUtensorMap requires
  CUtensorMap tmap_a;   // X as [T][K] bf16, boxes of 64 x 128, 128-byte swizzle
  WP w;                 // the producer's weight operand
  void* y;              // [T][N]
  int* status;
  int K, N, nexp, tiles_n;
  int tok_off[kGroupedMaxExperts + 1];   // first row of each expert
  int tile_off[kGroupedMaxExperts + 1];  // first tile of each expert
};

// Shared-memory descriptor of an MN-major bf16 tile with the 128-byte
// swizzle: blocks of 64 N values (128 bytes) x 8 K rows, rows 128 bytes apart;
// `lbo` bytes between consecutive 64-value blocks along N, 1024 bytes between
// consecutive 8-row groups along K.
__device__ __forceinline__ uint64_t umma_desc_mn_sw128(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Producer P provides:
//   P::Params                 the weight operand (tensor maps, pointers)
//   P::kSC, P::kCBytes        stages of packed weight data and bytes per stage
//   P::kCExtra                bytes of further staged data (kept across steps)
//   P::kExtraSmem             bytes of shared memory of its own (tables)
//   P::kMnMajor               true: B slices are MN-major (blocks of 64 N
//                             values x 64 K rows, 8 KiB apart); false:
//                             K-major (256 rows of 64 K values)
//   static build_extra(extra) fills its tables (all threads)
//   static stage(params, e, n0, K, N, ks, cst, cextra, bar)
//                             arms `bar` and issues the TMA loads of K step ks
//                             (one thread)
//   setup(params, e, n0, K, N, p, extra)
//   produce(ks, cst, cextra, tile)
//                             forms the slice of K step ks into `tile` from
//                             its staged data
template <class P, int SA, int SB, bool OUT_BF16>
struct GroupedGemm {
  static constexpr int kSC = P::kSC;
  static constexpr int kSmem =
      SA * kGA + SB * kGB + kSC * P::kCBytes + P::kCExtra + P::kExtraSmem + 256;
  static constexpr uint32_t kIdesc =
      idesc_bf16_f32(kGM, kGN) | (P::kMnMajor ? (1u << 16) : 0u);  // bit 16: B is MN-major
};

template <class P, int SA, int SB, bool OUT_BF16>
__global__ void __launch_bounds__(kGThreads, 1)
    k_grouped_gemm(const __grid_constant__ GroupedGemmArgs<typename P::Params> A) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int SC = P::kSC;
  unsigned char* const sa = smem;
  unsigned char* const sb = smem + SA * kGA;
  unsigned char* const sc = sb + SB * kGB;
  unsigned char* const cextra = sc + SC * P::kCBytes;
  unsigned char* const extra = cextra + P::kCExtra;
  uint64_t* const full_a = reinterpret_cast<uint64_t*>(extra + P::kExtraSmem);
  uint64_t* const empty_a = full_a + SA;
  uint64_t* const full_b = empty_a + SA;
  uint64_t* const empty_b = full_b + SB;
  uint64_t* const full_c = empty_b + SB;
  uint64_t* const empty_c = full_c + SC;
  uint64_t* const acc_bar = empty_c + SC;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  constexpr uint32_t kIdesc = GroupedGemm<P, SA, SB, OUT_BF16>::kIdesc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {  // the swizzled tiles need a 1 KiB aligned base
    if (threadIdx.x == 0 && A.status) atomicOr(A.status, kStatusTimeout);
    return;
  }

  // this CTA's tile: expert e (largest e with tile_off[e] <= tile), then
  // token tile mt and column tile nt within it
  const int tile = blockIdx.x;
  int lo = 0, hi = A.nexp;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (A.tile_off[mid] <= tile) lo = mid;
    else hi = mid;
  }
  const int e = lo;
  const int local = tile - A.tile_off[e];
  const int mt = local / A.tiles_n, nt = local - mt * A.tiles_n;
  const int tok0 = A.tok_off[e] + mt * (kGHalves * kGM), tok_end = A.tok_off[e + 1];
  const bool two = tok0 + kGM < tok_end;  // the second half has rows of this expert
  const int n0 = nt * kGN;
  const int nk = A.K / kGK;

  P::build_extra(extra);
  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; s++) {
      mbar_init(&full_a[s], 1);
      mbar_init(&empty_a[s], 1);
    }
    for (int s = 0; s < SB; s++) {
      mbar_init(&full_b[s], kGProducers / 32);
      mbar_init(&empty_b[s], 1);
    }
    for (int s = 0; s < SC; s++) {
      mbar_init(&full_c[s], 1);
      mbar_init(&empty_c[s], kGProducers / 32);
    }
    mbar_init(acc_bar, 1);
    fence_barrier_init();
  }
  if (warp == kGMmaWarp) tmem_alloc(tmem_slot, kGTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  if (warp < kGProducerWarps) {
    // ---- B producers
    P prod;
    prod.setup(A.w, e, n0, A.K, A.N, threadIdx.x, extra);
    for (int ks = 0; ks < nk; ks++) {
      const int c = ks % SC, s = ks % SB;
      // the whole warp agrees on each wait, so the warp-wide steps below are
      // reached by all of its lanes or by none
      if (!__all_sync(0xffffffffu, mbar_wait(&full_c[c], (ks / SC) & 1, kGWaitTries)) ||
          (ks >= SB &&
           !__all_sync(0xffffffffu, mbar_wait(&empty_b[s], (ks / SB - 1) & 1, kGWaitTries)))) {
        ok = false;
        break;
      }
      prod.produce(ks, sc + c * P::kCBytes, cextra, sb + s * kGB);
      fence_proxy_async_smem();  // the tensor cores read the slice through the async proxy
      __syncwarp();              // then one arrival per warp on each barrier
      if (lane == 0) {
        mbar_arrive(&full_b[s]);
        mbar_arrive(&empty_c[c]);  // the staged data of step ks has been read
      }
    }
  } else if (warp == kGTmaWarp) {
    if (lane == 0) {
      // ---- X tiles by TMA
      int issued = 0;
      for (int ks = 0; ks < nk; ks++) {
        const int s = ks % SA, u = ks / SA;
        if (ks >= SA && !mbar_wait(&empty_a[s], (u - 1) & 1, kGWaitTries)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full_a[s], kGA);
        tma_load_2d(sa + s * kGA, &A.tmap_a, ks * kGK, tok0, &full_a[s]);
        tma_load_2d(sa + s * kGA + kGA / 2, &A.tmap_a, ks * kGK, tok0 + kGM, &full_a[s]);
        issued = ks + 1;
      }
      if (!ok) {  // let the copies already issued land before the CTA leaves
        for (int ks = max(0, issued - SA); ks < issued; ks++)
          mbar_wait(&full_a[ks % SA], (ks / SA) & 1, kGWaitTries);
      }
    } else if (lane == 1) {
      // ---- packed weight data by TMA
      int issued = 0;
      for (int ks = 0; ks < nk; ks++) {
        const int c = ks % SC, u = ks / SC;
        if (ks >= SC && !mbar_wait(&empty_c[c], (u - 1) & 1, kGWaitTries)) {
          ok = false;
          break;
        }
        P::stage(A.w, e, n0, A.K, A.N, ks, sc + c * P::kCBytes, cextra, &full_c[c]);
        issued = ks + 1;
      }
      if (!ok) {
        for (int ks = max(0, issued - SC); ks < issued; ks++)
          mbar_wait(&full_c[ks % SC], (ks / SC) & 1, kGWaitTries);
      }
    }
  } else if (warp == kGMmaWarp) {
    // ---- tensor-core issue
    if (lane == 0) {
      for (int ks = 0; ks < nk; ks++) {
        const int s = ks % SA, u = ks / SA, t = ks % SB, v = ks / SB;
        if (!mbar_wait(&full_a[s], u & 1, kGWaitTries) ||
            !mbar_wait(&full_b[t], v & 1, kGWaitTries)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sa + s * kGA), b0 = smem_u32(sb + t * kGB);
#pragma unroll
        for (int kk = 0; kk < kGK / 16; kk++) {
          // K slice kk: 32 bytes further along the K-major rows, or two
          // 8-row groups further down the MN-major blocks
          const uint64_t bd = P::kMnMajor ? umma_desc_mn_sw128(b0 + kk * 2048, kGB / 4)
                                          : umma_desc_k_sw128(b0 + kk * 32);
          umma_bf16(tmem, umma_desc_k_sw128(a0 + kk * 32), bd, kIdesc, (ks | kk) != 0);
          if (two)
            umma_bf16(tmem + kGN, umma_desc_k_sw128(a0 + kGA / 2 + kk * 32), bd, kIdesc,
                      (ks | kk) != 0);
        }
        umma_commit(&empty_a[s]);
        umma_commit(&empty_b[t]);
      }
      umma_commit(acc_bar);  // also after a failed wait: covers what was issued
    }
  }

  // ---- epilogue
  __syncwarp();
  if (warp < kGProducerWarps) {
    // warp w reads lanes 32 (w & 3) .. +31 of accumulator (w >> 2) & 1,
    // columns 128 (w >> 3) .. +127
    const int q = warp & 3, half = (warp >> 2) & 1, part = warp >> 3;
    // tcgen05.ld is executed by whole warps, so the warp agrees on the wait
    if (!__all_sync(0xffffffffu, mbar_wait(acc_bar, 0, kGWaitTries))) {
      ok = false;
    } else if (half == 0 || two) {
      tc_fence_after();
      const int row = tok0 + half * kGM + q * 32 + lane;
      const bool store = ok && row < tok_end;
#pragma unroll 1
      for (int c = part * 4; c < part * 4 + 4; c++) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + half * kGN + c * 32, v);
        if (store) {
          if (OUT_BF16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(A.y) +
                                                  (int64_t)row * A.N + n0 + c * 32);
#pragma unroll
            for (int j = 0; j < 4; j++)
              dst[j] = make_uint4(
                  bf16x2_rn(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                  bf16x2_rn(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                  bf16x2_rn(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                  bf16x2_rn(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(A.y) +
                                                  (int64_t)row * A.N + n0 + c * 32);
#pragma unroll
            for (int j = 0; j < 8; j++)
              dst[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
        }
      }
    }
  } else if (warp == kGMmaWarp && lane == 0) {
    // the tensor memory is released only after every issued MMA has finished
    if (!mbar_wait(acc_bar, 0, kGWaitTries)) ok = false;
  }
  if (!ok && A.status) atomicOr(A.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == kGMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kGTmemCols);
  }
}

// Host side: builds the tile schedule (experts in order; per expert its
// 256-row token tiles, each split into N / 256 column tiles) and launches
// one CTA per tile.  K % 64 == 0 and N % 256 == 0 are the caller's to check.
template <class P, int SA, int SB, bool OUT_BF16>
cudaError_t launch_grouped_gemm(const uint16_t* x, const int64_t* counts, int64_t nexp, int K,
                                int N, const typename P::Params& w, void* y, int* status,
                                cudaStream_t s) {
  using G = GroupedGemm<P, SA, SB, OUT_BF16>;
  static_assert(G::kSmem <= 232448, "shared memory per CTA");
  static PerDeviceOnce attr;
  cudaError_t err = attr.run([] {
    return cudaFuncSetAttribute(k_grouped_gemm<P, SA, SB, OUT_BF16>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem);
  });
  if (err != cudaSuccess) return err;
  GroupedGemmArgs<typename P::Params> A;
  int64_t tok = 0, tiles = 0;
  const int tiles_n = N / kGN;
  for (int64_t e = 0; e < nexp; e++) {
    A.tok_off[e] = (int)tok;
    A.tile_off[e] = (int)tiles;
    tok += counts[e];
    tiles += (counts[e] + kGHalves * kGM - 1) / (kGHalves * kGM) * tiles_n;
  }
  A.tok_off[nexp] = (int)tok;
  A.tile_off[nexp] = (int)tiles;
  if (tiles == 0) return cudaSuccess;
  if (!encode_tmap_2d(&A.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, (uint64_t)K, (uint64_t)tok,
                      (uint64_t)K * 2, kGK, kGM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  A.w = w;
  A.y = y;
  A.status = status;
  A.K = K;
  A.N = N;
  A.nexp = (int)nexp;
  A.tiles_n = tiles_n;
  k_grouped_gemm<P, SA, SB, OUT_BF16><<<(unsigned)tiles, kGThreads, G::kSmem, s>>>(A);
  return cudaGetLastError();
}

}  // namespace nvq
