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
// transposition.  Producer warp w forms K rows 8w .. 8w+7 of each K step;
// lane l the eight N values 8l .. 8l+7 (one code word, half a scale block), so
// a warp's code loads cover one contiguous 128-byte run of a row.
#include <cuda.h>
#include <cstdint>

#include "nvq_common.cuh"
#include "nvq_gemm.cuh"
#include "nvq_internal.h"

namespace nvq {

struct Nvfp4DgradProducer {
  struct Params {
    const uint8_t* codes;   // [nexp, out, in/2]
    const uint8_t* scales;  // [nexp, out, in/16]
    const float* G;         // [nexp]
  };
  static constexpr int kAhead = 3;
  static constexpr int kExtraSmem = 0;
  static constexpr bool kMnMajor = true;

  const uint8_t* pc;  // this lane's code word in K row 8w of K step 0
  const uint8_t* ps;  // its scale byte
  int64_t in_h, in_16;
  float2 G2;
  int soff;           // byte offset of this lane's chunk in row 8w of the slice (unswizzled)
  int chunk;          // its 16-byte chunk within the 128-byte row
  uint32_t cw[kAhead][8], sbyte[kAhead][8];

  __device__ static void build_extra(unsigned char*) {}

  __device__ __forceinline__ void setup(const Params& P, int e, int n0, int K, int N, int p,
                                        const unsigned char*) {
    const int w = p >> 5, l = p & 31;
    in_h = N >> 1;
    in_16 = N >> 4;
    const int64_t row0 = (int64_t)e * K + 8 * w;
    pc = P.codes + row0 * in_h + (n0 >> 1) + 4 * l;
    ps = P.scales + row0 * in_16 + (n0 >> 4) + (l >> 1);
    const float g = P.G[e];
    G2 = make_float2(g, g);
    // block of 64 N values l >> 3 (8 KiB apart), K row 8w
    soff = (l >> 3) * (kGB / 4) + 8 * w * 128;
    chunk = l & 7;
  }

  __device__ __forceinline__ void load(int ks, int j) {
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const int64_t r = (int64_t)ks * kGK + i;
      cw[j][i] = __ldg(reinterpret_cast<const uint32_t*>(pc + r * in_h));
      sbyte[j][i] = __ldg(ps + r * in_16);
    }
  }

  // One code word: the eight values 8l .. 8l+7 of one K row, as four bf16
  // pairs in N order.
  template <int B>
  __device__ __forceinline__ uint32_t pair(uint32_t c, uint32_t S2) const {
    const float2 y = __fmul2_rn(cs_exact(e2m1x2_dec_byte<B>(c), S2), G2);
    return bf16x2_rn(y.x, y.y);
  }

  __device__ __forceinline__ void produce(int j, int next, unsigned char* tile) {
    uint32_t cur[8], S2[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      S2[i] = e4m3_to_f16x2(sbyte[j][i] & 0x7f);
      cur[i] = cw[j][i];
    }
    if (next >= 0) load(next, j);
    // K row 8w + i sits at (8w + i) * 128 in its block; its swizzle phase is
    // (8w + i) & 7 = i
#pragma unroll
    for (int i = 0; i < 8; i++)
      *reinterpret_cast<uint4*>(tile + soff + i * 128 + ((chunk ^ i) << 4)) =
          make_uint4(pair<0>(cur[i], S2[i]), pair<1>(cur[i], S2[i]), pair<2>(cur[i], S2[i]),
                     pair<3>(cur[i], S2[i]));
  }
};

cudaError_t launch_dgrad(const uint16_t* dy, const int64_t* counts, int64_t nexp, int out, int in,
                         const uint8_t* codes, const uint8_t* scales, const float* G, float* dx,
                         int* status, cudaStream_t s) {
  const Nvfp4DgradProducer::Params w{codes, scales, G};
  return launch_grouped_gemm<Nvfp4DgradProducer, 4, 2, false>(dy, counts, nexp, out, in, w, dx,
                                                                status, s);
}

}  // namespace nvq
