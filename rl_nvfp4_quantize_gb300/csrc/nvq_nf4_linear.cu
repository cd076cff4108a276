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
// NF4 block is exactly one row of a K step.  Producer thread p forms row p of
// the slice: 32 code bytes (one 32-byte load) and one absmax per K step.  The
// dequantised value of each code is bf16(level[c] * absmax), the same value
// nf4_dequant writes; a 256-entry table maps a code byte to its two levels.
#include <cuda.h>
#include <cstdint>

#include "nvq_common.cuh"
#include "nvq_gemm.cuh"
#include "nvq_internal.h"
#include "nvq_nf4_levels.cuh"

namespace nvq {

struct Nf4LinearProducer {
  struct Params {
    const uint8_t* codes;  // [nexp, out, in/2]
    const float* absmax;   // [nexp, out, in/64]
  };
  static constexpr int kAhead = 3;
  // the byte -> (level[low nibble], level[high nibble]) table, replicated 16
  // times: entry b of copy l at (16 b + l) * 8 bytes; lane l reads copy l & 15,
  // so a half warp never shares a bank whatever bytes it looks up
  static constexpr int kExtraSmem = 256 * 16 * 8;
  static constexpr bool kMnMajor = false;

  const uint8_t* pc;
  const float* pa;
  const float2* tbl;
  int roff;  // byte offset of this thread's row in the slice
  int phase; // its swizzle phase (row & 7)
  uint32_t cw[kAhead][8];
  float am[kAhead];

  __device__ static void build_extra(unsigned char* extra) {
    float2* t = reinterpret_cast<float2*>(extra);
    for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
      const int b = i >> 4;
      t[i] = make_float2(c_nf4[b & 15], c_nf4[b >> 4]);
    }
  }

  __device__ __forceinline__ void setup(const Params& P, int e, int n0, int K, int N, int p,
                                        const unsigned char* extra) {
    const int64_t row = (int64_t)e * N + n0 + p;
    pc = P.codes + row * (K >> 1);
    pa = P.absmax + row * (K >> 6);
    tbl = reinterpret_cast<const float2*>(extra) + (p & 15);
    roff = p * 128;
    phase = p & 7;
  }

  __device__ __forceinline__ void load(int ks, int j) {
    ldg32(pc + (int64_t)ks * 32, cw[j]);
    am[j] = __ldg(pa + ks);
  }

  __device__ __forceinline__ uint32_t pair(uint32_t byte, float2 a2) const {
    const float2 y = __fmul2_rn(tbl[byte * 16], a2);
    return bf16x2_rn(y.x, y.y);
  }

  __device__ __forceinline__ void produce(int j, int next, unsigned char* tile) {
    uint32_t cur[8];
#pragma unroll
    for (int c = 0; c < 8; c++) cur[c] = cw[j][c];
    const float2 a2 = make_float2(am[j], am[j]);
    if (next >= 0) load(next, j);
    // word c holds the codes of K values 8c .. 8c+7 (code 2b in the low
    // nibble of byte b): one 16-byte chunk of the row, swizzled by phase
#pragma unroll
    for (int c = 0; c < 8; c++)
      *reinterpret_cast<uint4*>(tile + roff + ((c ^ phase) << 4)) =
          make_uint4(pair(cur[c] & 0xffu, a2), pair((cur[c] >> 8) & 0xffu, a2),
                     pair((cur[c] >> 16) & 0xffu, a2), pair(cur[c] >> 24, a2));
  }
};

cudaError_t launch_nf4_linear(const uint16_t* x, const int64_t* counts, int64_t nexp, int out,
                              int in, const uint8_t* codes, const float* absmax, uint16_t* y,
                              int* status, cudaStream_t s) {
  const Nf4LinearProducer::Params w{codes, absmax};
  return launch_grouped_gemm<Nf4LinearProducer, 3, 2, true>(x, counts, nexp, in, out, w, y,
                                                             status, s);
}

}  // namespace nvq
