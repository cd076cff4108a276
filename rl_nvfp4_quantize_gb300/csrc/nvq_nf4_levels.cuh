// nvq_nf4_levels.cuh -- the 16 NF4 levels, ascending: standard-normal
// quantiles at probabilities evenly spaced from 1/2 to 31/32 (7 steps below
// zero, 8 above), divided by the quantile at 31/32 so the outermost levels are
// -1 and +1, zero exact.  Each translation unit that includes this header gets
// its own constant-memory copy (the library is built without relocatable
// device code).
#pragma once

#define NVQ_NF4_LEVELS                                                  \
  {-0x1.000000p+0f, -0x1.6311acp-1f, -0x1.0b8d60p-1f, -0x1.924c0ap-2f, \
   -0x1.21b102p-2f, -0x1.7851c6p-3f, -0x1.72d976p-4f, 0x0.0p+0f,       \
   0x1.4421acp-4f,  0x1.47c076p-3f,  0x1.f54804p-3f,  0x1.582f80p-2f,  \
   0x1.c1002ap-2f,  0x1.1eba52p-1f,  0x1.70ca9ap-1f,  0x1.000000p+0f}

namespace nvq {
static __constant__ float c_nf4[16] = NVQ_NF4_LEVELS;
}  // namespace nvq
