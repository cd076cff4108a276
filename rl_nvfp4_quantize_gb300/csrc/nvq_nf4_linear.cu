// nvq_nf4_linear.cu -- the forward product of routed experts stored as NF4:
// Y = X . DQ(W_e)^T for the token rows routed to each expert e, on the
// fifth-generation tensor cores, with the NF4 dequantisation fused into the
// B-operand load (the grouped GEMM of nvq_gemm.cuh with K = in, N = out).
//
// Source: "nf4moe -- QLoRA for a 743B Fused-MoE", "The fix: dequant-on-forward
// for routed experts" (each routed expert's weight is dequantised to bf16 and
// applied as F.linear(x, W[e]) to the tokens sent to it) and "Making it fast:
// the step tax" (the dequantised bf16 copies are the per-step cost; here they
// are formed tile by tile in shared memory and never written to HBM).
//
// B is W_e [out][in] = [N][K]: K-contiguous, one absmax per 64 K values, so one
// NF4 block is exactly one row of a K step.  The codes (and absmax) of each K
// step are staged in shared memory by TMA; producer thread p (of 512) forms
// half p >> 8 of row p & 255 of the slice from 16 of its code bytes and its
// absmax.  The dequantised value of
// each code is bf16(level[c] * absmax), the same value nf4_dequant writes; a
// 256-entry table maps a code byte to its two levels.
#include <cuda.h>
#include <cstdint>

#include "nvq_common.cuh"
#include "nvq_gemm.cuh"
#include "nvq_internal.h"
#include "nvq_nf4_levels.cuh"

namespace nvq {

struct Nf4LinearProducer {
  struct Params {
    CUtensorMap codes;   // [nexp * out][in/2] u8, boxes of 32 bytes x 256 rows, 32-byte swizzle
    CUtensorMap absmax;  // [nexp * out][in/64] f32, boxes of 4 values x 256 rows
  };
  // staged per K step: the codes of 256 rows x 64 K values (256 x 32 bytes);
  // every fourth step also the absmax of the next four steps (256 x 16 bytes)
  // into one of two slots kept across steps
  static constexpr int kSC = 3;
  static constexpr int kCBytes = kGN * 32;
  static constexpr int kCExtra = 2 * kGN * 16;
  // the byte -> (level[low nibble], level[high nibble]) table, replicated 16
  // times: entry b of copy l at (16 b + l) * 8 bytes; lane l reads copy l & 15,
  // so a half warp never shares a bank whatever bytes it looks up
  static constexpr int kExtraSmem = 256 * 16 * 8;
  static constexpr bool kMnMajor = false;

  const float2* tbl;
  int p;     // this thread's row of the slice
  int h;     // its half of the row: K values 32 h .. 32 h + 31
  int roff;  // byte offset of that row in the slice
  int phase; // its swizzle phase (row & 7)
  float4 am; // the row's absmax for the four K steps of the current slot

  __device__ static void build_extra(unsigned char* extra) {
    float2* t = reinterpret_cast<float2*>(extra);
    for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
      const int b = i >> 4;
      t[i] = make_float2(c_nf4[b & 15], c_nf4[b >> 4]);
    }
  }

  __device__ static void stage(const Params& P, int e, int n0, int, int N, int ks,
                               unsigned char* cst, unsigned char* cextra, uint64_t* bar) {
    const int y = e * N + n0;
    const bool am = (ks & 3) == 0;
    mbar_arrive_expect_tx(bar, kCBytes + (am ? kGN * 16 : 0));
    tma_load_2d(cst, &P.codes, ks * 32, y, bar);
    if (am) tma_load_2d(cextra + ((ks >> 2) & 1) * (kGN * 16), &P.absmax, ks, y, bar);
  }

  __device__ __forceinline__ void setup(const Params&, int, int, int, int, int pp,
                                        const unsigned char* extra) {
    p = pp & (kGN - 1);
    h = pp >> 8;
    tbl = reinterpret_cast<const float2*>(extra) + (pp & 15);
    roff = p * 128;
    phase = p & 7;
  }

  __device__ __forceinline__ uint32_t pair(uint32_t byte, float2 a2) const {
    const float2 y = __fmul2_rn(tbl[byte * 16], a2);
    return bf16x2_rn(y.x, y.y);
  }

  __device__ __forceinline__ void produce(int ks, const unsigned char* cst,
                                          const unsigned char* cextra, unsigned char* tile) {
    // half h of row p's 32 code bytes: 16-byte chunk h, swapped with the
    // other one on rows with bit 2 set (the 32-byte swizzle)
    const uint4 cv = *reinterpret_cast<const uint4*>(cst + p * 32 + ((h ^ ((p >> 2) & 1)) << 4));
    // the absmax of this step is value ks & 3 of the row's 16 bytes in the
    // slot; the four are read once per slot (one 16-byte read: a warp's 32
    // rows are contiguous, so the read is conflict-free)
    if ((ks & 3) == 0)
      am = *reinterpret_cast<const float4*>(cextra + ((ks >> 2) & 1) * (kGN * 16) + p * 16);
    const int k4 = ks & 3;
    const float a = k4 == 0 ? am.x : k4 == 1 ? am.y : k4 == 2 ? am.z : am.w;
    const float2 a2 = make_float2(a, a);
    const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
    // word j holds the codes of K values 32 h + 8 j .. +7 (code 2b in the
    // low nibble of byte b): 16-byte chunk 4 h + j of the row, swizzled by phase
#pragma unroll
    for (int j = 0; j < 4; j++)
      *reinterpret_cast<uint4*>(tile + roff + (((4 * h + j) ^ phase) << 4)) =
          make_uint4(pair(cw[j] & 0xffu, a2), pair((cw[j] >> 8) & 0xffu, a2),
                     pair((cw[j] >> 16) & 0xffu, a2), pair(cw[j] >> 24, a2));
  }
};

cudaError_t launch_nf4_linear(const uint16_t* x, const int64_t* counts, int64_t nexp, int out,
                              int in, const uint8_t* codes, const float* absmax, uint16_t* y,
                              int* status, cudaStream_t s) {
  Nf4LinearProducer::Params w;
  const uint64_t rows = (uint64_t)nexp * out;
  if (!encode_tmap_2d(&w.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, (uint64_t)in / 2, rows,
                      (uint64_t)in / 2, 32, kGN, CU_TENSOR_MAP_SWIZZLE_32B) ||
      !encode_tmap_2d(&w.absmax, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, absmax, (uint64_t)in / 64, rows,
                      (uint64_t)in / 16, 4, kGN, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  return launch_grouped_gemm<Nf4LinearProducer, 3, 2, true>(x, counts, nexp, in, out, w, y,
                                                             status, s);
}

}  // namespace nvq
