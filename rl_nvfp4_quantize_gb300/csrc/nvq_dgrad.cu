// nvq_dgrad.cu -- the dgrad GEMM of a routed expert read straight from its
// NVFP4 rowwise copy: dX = dY . DQ(Q(W)) on the fifth-generation tensor cores
// (tcgen05.mma, accumulator in tensor memory), with the dequantisation fused
// into the B-operand load so the bf16 weight never goes to HBM.
//
// Sources: "The 4-bitter Lesson", "Key claims" (dequantised backward: the
// backward uses x . DQ(Q(w))) and "Getting GLM-5.2 NVFP4 Post-Training off
// the ground", "The bottom line" (the rowwise copy is dequantised to bf16 for
// the dgrad GEMM instead of keeping a columnwise copy).
//
// Tile: 256 tokens (two M = 128 halves) x 256 in-columns (N), K = out in
// steps of 64; the dequantised B slice of a K step serves both halves.  One
// CTA per tile, ten warps:
//   warps 0-7 : B producers -- dequantise the 64 x 256 slice of the rowwise
//               copy (codes, scales, G) into a K-major, 128-byte-swizzled bf16
//               tile [256 in][64 out] in shared memory; afterwards the
//               epilogue (warps 0-3: tokens 0-127, warps 4-7: tokens
//               128-255): tensor memory -> registers -> FP32 dX rows;
//   warp 8    : TMA loads of the two dY tiles [128 tokens][64 out] (same
//               swizzle);
//   warp 9    : allocates all 512 columns of tensor memory (two 128 x 256
//               FP32 accumulators), issues the tcgen05.mma (M 128, N 256,
//               K 16, bf16 x bf16 -> FP32) -- four per K step and half, the
//               second half only when the expert has tokens there -- commits
//               them to the stage's "empty" barrier, and frees the tensor
//               memory at the end.
// Every wait is bounded; a wait that gives up sets the status word's timeout
// bit, and every path still reaches the tensor-memory release.
#include <cuda.h>
#include <cstdint>
#include <algorithm>

#include "nvq_common.cuh"
#include "nvq_internal.h"

namespace nvq {

constexpr int kGM = 128, kGN = 256, kGK = 64;
constexpr int kGHalves = 2;                // M halves per CTA tile
constexpr int kGStages = 3;
constexpr int kGAhead = 3;                     // K steps of codes in flight per producer
constexpr int kGA = kGHalves * kGM * kGK * 2;  // 32 KiB of dY per stage (two 16 KiB halves)
constexpr int kGB = kGN * kGK * 2;             // 32 KiB of dequantised W per stage
constexpr int kGThreads = 320;
constexpr int kGProducers = 256;
constexpr uint32_t kGTmemCols = 512;           // two FP32 accumulators of 128 x 256
constexpr int kGSmem = kGStages * (kGA + kGB) + 128;
constexpr uint32_t kGWaitTries = 1u << 22;

struct __align__(64) DgradArgs {
  CUtensorMap tmap_a;       // dY as [T][out] bf16, boxes of 64 x 128, 128-byte swizzle
  const uint8_t* codes;     // [nexp, out, in/2]
  const uint8_t* scales;    // [nexp, out, in/16]
  const float* G;           // [nexp]
  float* dx;                // [T, in]
  int* status;
  int out, in, nexp, tiles_n;
  int tok_off[kDgradMaxExperts + 1];   // first token row of each expert
  int tile_off[kDgradMaxExperts + 1];  // first tile of each expert
};

// ------------------------------------------------------ tcgen05 wrappers
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor of a K-major operand tile stored as 8-row
// groups of 128-byte rows with the 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B): start address, stride between 8-row
// groups 1024 bytes, descriptor version 1, layout "128-byte swizzle".
__device__ __forceinline__ uint64_t umma_desc_k_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor: FP32 accumulator, bf16 A and B, both K-major,
// N = kGN, M = kGM.
constexpr uint32_t kGIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kGN >> 3) << 17) |
                             ((uint32_t)(kGM >> 4) << 24);
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kGIdesc), "r"(accumulate)
      : "memory");
}
// Arrives (once) on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 consecutive FP32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t v[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------- the kernel
// B tile of one K step: out-rows k0 .. k0+63 x in-columns n0 .. n0+255 of the
// expert's rowwise copy, written transposed ([in][out]) as 256 rows of 128
// bytes, 16-byte chunk c of row r at chunk c ^ (r & 7).  Producer thread
// p: out-rows 8g .. 8g+7 (g = p & 7) of 16-wide block column b = (p >> 3) & 15.
// Producer p takes word wh = p >> 7 (columns 8 wh .. 8 wh + 7) of that block
// column; column pair J of the word covers block columns 8 wh + 2J, +1.
template <int J>
__device__ __forceinline__ void dgrad_column_pair(const uint32_t cw[8], const uint32_t S2[8],
                                                  float2 G2, unsigned char* tile, int c0, int g) {
  uint32_t v[8];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const uint32_t h = e2m1x2_dec_byte<J>(cw[i]);
    const float2 y = __fmul2_rn(cs_exact(h, S2[i]), G2);
    v[i] = bf16x2_rn(y.x, y.y);
  }
  const int r = c0 + 2 * J;
  *reinterpret_cast<uint4*>(tile + r * 128 + ((g ^ (r & 7)) << 4)) =
      make_uint4(__byte_perm(v[0], v[1], 0x5410), __byte_perm(v[2], v[3], 0x5410),
                 __byte_perm(v[4], v[5], 0x5410), __byte_perm(v[6], v[7], 0x5410));
  *reinterpret_cast<uint4*>(tile + (r + 1) * 128 + ((g ^ ((r + 1) & 7)) << 4)) =
      make_uint4(__byte_perm(v[0], v[1], 0x7632), __byte_perm(v[2], v[3], 0x7632),
                 __byte_perm(v[4], v[5], 0x7632), __byte_perm(v[6], v[7], 0x7632));
}

__global__ void __launch_bounds__(kGThreads, 1) k_dgrad(const __grid_constant__ DgradArgs A) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* const sa = smem;
  unsigned char* const sb = smem + kGStages * kGA;
  uint64_t* const full_a = reinterpret_cast<uint64_t*>(smem + kGStages * (kGA + kGB));
  uint64_t* const full_b = full_a + kGStages;
  uint64_t* const empty = full_b + kGStages;
  uint64_t* const acc_bar = empty + kGStages;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
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
  const bool two = tok0 + kGM < tok_end;  // the second half has tokens of this expert
  const int n0 = nt * kGN;
  const int nk = A.out / kGK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; s++) {
      mbar_init(&full_a[s], 1);
      mbar_init(&full_b[s], kGProducers / 32);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_bar, 1);
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(tmem_slot, kGTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  if (warp < 8) {
    // ---- B producers
    const int p = threadIdx.x, g = p & 7, b = (p >> 3) & 15, wh = p >> 7;
    const int64_t in_h = A.in >> 1, in_16 = A.in >> 4;
    const uint8_t* pc0 = A.codes + (int64_t)e * A.out * in_h + (n0 >> 1) + b * 8 + wh * 4;
    const uint8_t* ps0 = A.scales + (int64_t)e * A.out * in_16 + (n0 >> 4) + b;
    const float Gv = A.G[e];
    const float2 G2 = make_float2(Gv, Gv);
    const int c0 = b * 16 + wh * 8;  // first tile row (in-index) of this thread
    // codes and scale bytes of K step ks, loaded kGAhead steps before use
    // into one of kGAhead register buffers (the loop is unrolled by kGAhead
    // so every buffer index is a constant)
    uint32_t cw[kGAhead][8], sbyte[kGAhead][8];
    auto load = [&](int ks, uint32_t* c, uint32_t* sbv) {
      const int64_t row = (int64_t)ks * kGK + g * 8;
#pragma unroll
      for (int i = 0; i < 8; i++) {
        c[i] = __ldg(reinterpret_cast<const uint32_t*>(pc0 + (row + i) * in_h));
        sbv[i] = __ldg(ps0 + (row + i) * in_16);
      }
    };
#pragma unroll
    for (int j = 0; j < kGAhead; j++)
      if (j < nk) load(j, cw[j], sbyte[j]);
    auto step = [&](int ks, uint32_t* c, uint32_t* sbv) -> bool {
      const int s = ks % kGStages, u = ks / kGStages;
      if (ks >= kGStages && !mbar_wait(&empty[s], (u - 1) & 1, kGWaitTries)) return false;
      uint32_t S2[8], cur[8];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        S2[i] = e4m3_to_f16x2(sbv[i] & 0x7f);
        cur[i] = c[i];
      }
      if (ks + kGAhead < nk) load(ks + kGAhead, c, sbv);
      unsigned char* tileb = sb + s * kGB;
      dgrad_column_pair<0>(cur, S2, G2, tileb, c0, g);
      dgrad_column_pair<1>(cur, S2, G2, tileb, c0, g);
      dgrad_column_pair<2>(cur, S2, G2, tileb, c0, g);
      dgrad_column_pair<3>(cur, S2, G2, tileb, c0, g);
      fence_proxy_async_smem();  // the tensor cores read the tile through the async proxy
      __syncwarp();              // then one arrival per warp
      if (lane == 0) mbar_arrive(&full_b[s]);
      return true;
    };
    for (int k0 = 0; k0 < nk && ok; k0 += kGAhead) {
#pragma unroll
      for (int j = 0; j < kGAhead; j++)
        if (ok && k0 + j < nk) ok = step(k0 + j, cw[j], sbyte[j]);
    }
  } else if (warp == 8) {
    // ---- dY tiles by TMA
    if (lane == 0) {
      int issued = 0;
      for (int ks = 0; ks < nk; ks++) {
        const int s = ks % kGStages, u = ks / kGStages;
        if (ks >= kGStages && !mbar_wait(&empty[s], (u - 1) & 1, kGWaitTries)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full_a[s], kGA);
        tma_load_2d(sa + s * kGA, &A.tmap_a, ks * kGK, tok0, &full_a[s]);
        tma_load_2d(sa + s * kGA + kGA / 2, &A.tmap_a, ks * kGK, tok0 + kGM, &full_a[s]);
        issued = ks + 1;
      }
      if (!ok) {  // let the copies already issued land before the CTA leaves
        for (int ks = max(0, issued - kGStages); ks < issued; ks++)
          mbar_wait(&full_a[ks % kGStages], (ks / kGStages) & 1, kGWaitTries);
      }
    }
  } else if (warp == 9) {
    // ---- tensor-core issue
    if (lane == 0) {
      for (int ks = 0; ks < nk; ks++) {
        const int s = ks % kGStages, u = ks / kGStages;
        if (!mbar_wait(&full_a[s], u & 1, kGWaitTries) ||
            !mbar_wait(&full_b[s], u & 1, kGWaitTries)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sa + s * kGA), b0 = smem_u32(sb + s * kGB);
#pragma unroll
        for (int kk = 0; kk < kGK / 16; kk++) {
          const uint64_t bd = umma_desc_k_sw128(b0 + kk * 32);
          umma_bf16(tmem, umma_desc_k_sw128(a0 + kk * 32), bd, (ks | kk) != 0);
          if (two)
            umma_bf16(tmem + kGN, umma_desc_k_sw128(a0 + kGA / 2 + kk * 32), bd, (ks | kk) != 0);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(acc_bar);  // also after a failed wait: covers what was issued
    }
  }

  // ---- epilogue: warp w reads lanes 32 (w & 3) .. +31 of accumulator w >> 2
  __syncwarp();
  if (warp < 8) {
    const int half = warp >> 2, q = warp & 3;
    // tcgen05.ld is executed by whole warps, so the warp agrees on the wait
    if (!__all_sync(0xffffffffu, mbar_wait(acc_bar, 0, kGWaitTries))) {
      ok = false;
    } else if (half == 0 || two) {
      tc_fence_after();
      const int row = tok0 + half * kGM + q * 32 + lane;
      float* dst = A.dx + (int64_t)row * A.in + n0;
      const bool store = ok && row < tok_end;
#pragma unroll 1
      for (int c = 0; c < kGN / 32; c++) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + half * kGN + c * 32, v);
        if (store) {
#pragma unroll
          for (int j = 0; j < 8; j++)
            reinterpret_cast<uint4*>(dst + c * 32)[j] =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
    }
  } else if (warp == 9 && lane == 0) {
    // the tensor memory is released only after every issued MMA has finished
    if (!mbar_wait(acc_bar, 0, kGWaitTries)) ok = false;
  }
  if (!ok && A.status) atomicOr(A.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kGTmemCols);
  }
}

cudaError_t launch_dgrad(const uint16_t* dy, const int64_t* counts, int64_t nexp, int out, int in,
                         const uint8_t* codes, const uint8_t* scales, const float* G, float* dx,
                         int* status, cudaStream_t s) {
  static int attr_done = 0;
  if (!attr_done) {
    cudaError_t err =
        cudaFuncSetAttribute(k_dgrad, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
    if (err != cudaSuccess) return err;
    attr_done = 1;
  }
  DgradArgs A;
  int64_t tok = 0, tiles = 0;
  const int tiles_n = in / kGN;
  for (int64_t e = 0; e < nexp; e++) {
    A.tok_off[e] = (int)tok;
    A.tile_off[e] = (int)tiles;
    tok += counts[e];
    tiles += (counts[e] + kGHalves * kGM - 1) / (kGHalves * kGM) * tiles_n;
  }
  A.tok_off[nexp] = (int)tok;
  A.tile_off[nexp] = (int)tiles;
  if (tiles == 0) return cudaSuccess;
  if (!encode_tmap_2d(&A.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT16, dy, (uint64_t)out, (uint64_t)tok,
                      (uint64_t)out * 2, kGK, kGM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  A.codes = codes;
  A.scales = scales;
  A.G = G;
  A.dx = dx;
  A.status = status;
  A.out = out;
  A.in = in;
  A.nexp = (int)nexp;
  A.tiles_n = tiles_n;
  k_dgrad<<<(unsigned)tiles, kGThreads, kGSmem, s>>>(A);
  return cudaGetLastError();
}

}  // namespace nvq
