// nvq_dgrad.cu -- the dgrad GEMM of a routed expert read straight from its
// NVFP4 rowwise copy: dX = dY . DQ(Q(W)) on the fifth-generation tensor cores,
// with the dequantisation fused into the B-operand load so the bf16 weight
// never goes to HBM (the grouped GEMM of nvq_gemm.cuh with K = out, N = in).
//
// Sources: "The 4-bitter Lesson", "Key claims" (dequantised backward: the
// backward uses x . DQ(Q(w))) and "Getting GLM-5.2 NVFP4 Post-Training off
// the ground", "The bottom line" (the rowwise copy is dequantised to bf16 for
// the dgrad GEMM instead of keeping a columnwise copy).
//
// B is the weight slice itself, W_e [out][in] = [K][N]: N-contiguous, so the
// producers write it MN-major, in the orientation it is stored in -- no
// transposition.  The codes and scales of each K step (64 rows x 256 columns)
// are staged in shared memory by TMA; producer warp w (of 16) forms K rows
// 4w .. 4w+3 of the step, lane l the eight N values 8l .. 8l+7 (one code
// word, half a scale block), so a warp reads one contiguous 128-byte row of
// codes.
#include <cuda.h>
#include <cstdint>

#include "nvq_common.cuh"
#include "nvq_gemm.cuh"
#include "nvq_internal.h"

namespace nvq {

struct Nvfp4DgradProducer {
  struct Params {
    CUtensorMap codes;      // [nexp * out][in/2] u8, boxes of 128 bytes x 64 rows
    CUtensorMap scales;     // [nexp * out][in/16] u8, boxes of 16 bytes x 64 rows
    const float* G;         // [nexp]
  };
  // staged per K step: the codes of 64 rows x 256 columns (64 x 128 bytes),
  // then their scales (64 x 16 bytes)
  static constexpr int kSC = 3;
  static constexpr int kCBytes = kGK * 128 + kGK * 16;
  static constexpr int kCExtra = 0;
  static constexpr int kExtraSmem = 0;
  static constexpr bool kMnMajor = true;

  float2 G2;
  int coff;   // this lane's code word in K row 4w of a staged step
  int soff;   // its scale byte
  int toff;   // its 16-byte chunk in K row 4w of the slice (unswizzled)
  int chunk;  // that chunk's index within the 128-byte row
  int phase;  // swizzle phase of K row 4w (4w & 7)

  __device__ static void build_extra(unsigned char*) {}

  __device__ static void stage(const Params& P, int e, int n0, int K, int, int ks,
                               unsigned char* cst, unsigned char*, uint64_t* bar) {
    const int y = e * K + ks * kGK;
    mbar_arrive_expect_tx(bar, kCBytes);
    tma_load_2d(cst, &P.codes, n0 >> 1, y, bar);
    tma_load_2d(cst + kGK * 128, &P.scales, n0 >> 4, y, bar);
  }

  __device__ __forceinline__ void setup(const Params& P, int e, int, int, int, int p,
                                        const unsigned char*) {
    const int w = p >> 5, l = p & 31;
    const float g = P.G[e];
    G2 = make_float2(g, g);
    coff = 4 * w * 128 + 4 * l;
    soff = kGK * 128 + 4 * w * 16 + (l >> 1);
    // block of 64 N values l >> 3 (8 KiB apart), K row 4w
    toff = (l >> 3) * (kGB / 4) + 4 * w * 128;
    chunk = l & 7;
    phase = (4 * w) & 7;
  }

  // One code word: the eight values 8l .. 8l+7 of one K row, as four bf16
  // pairs in N order.
  template <int B>
  __device__ __forceinline__ uint32_t pair(uint32_t c, uint32_t S2) const {
    const float2 y = __fmul2_rn(cs_exact(e2m1x2_dec_byte<B>(c), S2), G2);
    return bf16x2_rn(y.x, y.y);
  }

  __device__ __forceinline__ void produce(int, const unsigned char* cst, const unsigned char*,
                                          unsigned char* tile) const {
    // K row 4w + i: code word at row * 128, scale byte at row * 16; in the
    // slice it sits at (4w + i) * 128 in its block, swizzle phase
    // (4w + i) & 7 = phase + i
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint32_t c = *reinterpret_cast<const uint32_t*>(cst + coff + i * 128);
      const uint32_t S2 = e4m3_to_f16x2(cst[soff + i * 16] & 0x7f);
      *reinterpret_cast<uint4*>(tile + toff + i * 128 + ((chunk ^ (phase + i)) << 4)) =
          make_uint4(pair<0>(c, S2), pair<1>(c, S2), pair<2>(c, S2), pair<3>(c, S2));
    }
  }
};

cudaError_t launch_dgrad(const uint16_t* dy, const int64_t* counts, int64_t nexp, int out, int in,
                         const uint8_t* codes, const uint8_t* scales, const float* G, float* dx,
                         int* status, cudaStream_t s) {
  Nvfp4DgradProducer::Params w;
  const uint64_t rows = (uint64_t)nexp * out;
  if (!encode_tmap_2d(&w.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, (uint64_t)in / 2, rows,
                      (uint64_t)in / 2, 128, kGK, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tmap_2d(&w.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, scales, (uint64_t)in / 16, rows,
                      (uint64_t)in / 16, 16, kGK, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  w.G = G;
  return launch_grouped_gemm<Nvfp4DgradProducer, 4, 2, false>(dy, counts, nexp, out, in, w, dx,
                                                                status, s);
}

}  // namespace nvq
