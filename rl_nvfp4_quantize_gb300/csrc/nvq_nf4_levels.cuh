// nvq_nf4_levels.cuh -- the 16 levels of the NF4 data type (QLoRA's 4-bit
// NormalFloat, "4-bit NormalFloat Quantization" and the value list in the
// QLoRA paper's appendix), ascending, as binary32: standard-normal quantiles
// at probabilities spaced evenly between the outer probability 0.9677083 and
// 1/2 (seven levels below zero, eight above, zero exact), normalised so the
// outermost levels are -1 and +1.  Each translation unit that includes this
// header gets its own constant-memory copy (the library is built without
// relocatable device code).
#pragma once

#define NVQ_NF4_LEVELS                                                  \
  {-0x1.000000p+0f, -0x1.647362p-1f, -0x1.0cd660p-1f, -0x1.946540p-2f, \
   -0x1.23449ap-2f, -0x1.7a6a7ep-3f, -0x1.74f0e2p-4f, 0x0.0p+0f,       \
   0x1.45f5fep-4f,  0x1.4995c6p-3f,  0x1.f809bap-3f,  0x1.5a0674p-2f,  \
   0x1.c34970p-2f,  0x1.200f56p-1f,  0x1.722766p-1f,  0x1.000000p+0f}

namespace nvq {
static __constant__ float c_nf4[16] = NVQ_NF4_LEVELS;
}  // namespace nvq
