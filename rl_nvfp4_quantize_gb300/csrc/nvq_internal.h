// nvq_internal.h -- host-side launchers behind the C ABI (not exported).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvq {

// Host-side setup done once per kernel and device (the dynamic shared-memory
// limit is a property of a function on each device).  Safe to call from
// several host threads: a race at most repeats the setup, which is harmless.
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};  // bit d: device d
  template <class F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    const cudaError_t err = setup();
    if (err == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return err;
  }
};

// A positive per-device value (an occupancy figure) computed once per device.
struct PerDeviceInt {
  std::atomic<int> v[64];
  PerDeviceInt() {
    for (auto& x : v) x.store(0, std::memory_order_relaxed);
  }
  // compute() returns the value (> 0) or a CUDA error through *err.
  template <class F>
  int get(F&& compute, cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
      const int x = v[dev].load(std::memory_order_acquire);
      if (x > 0) return x;
    }
    const int x = compute(err);
    if (*err == cudaSuccess && x > 0 && dev >= 0 && dev < 64) v[dev].store(x, std::memory_order_release);
    return x;
  }
};

struct FastDiv;

// Host construction of a FastDiv for 1 <= d < 2^31.
inline void make_fastdiv(uint32_t d, uint32_t* m, uint32_t* s) {
  uint32_t l = 0;
  while ((1ull << l) < d) l++;
  *s = l;
  *m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
}

// Encodes a 2-D tiled tensor map (row-major [dim1][dim0] of `elem_bytes`
// elements, row pitch `stride_bytes`) with the given box and swizzle.
// Returns false when the driver entry point is unavailable or rejects it.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t dim0, uint64_t dim1, uint64_t stride_bytes, uint32_t box0,
                    uint32_t box1, CUtensorMapSwizzle swizzle);

struct DevInfo {
  int sms;
  int ok;  // 1 when the device is compute capability 10.3
};

// Current device's properties, or nullptr when there is no usable device.
const DevInfo* device_info();

// Zeroes n floats at p (and at q, when given) on the stream.
cudaError_t launch_zero_f32(float* p, int64_t n, cudaStream_t s, float* q = nullptr);

// tensor_scale[e] = amax[e] / (6 M) for every slice; status bit 0 for a
// non-finite amax.
cudaError_t launch_tensor_scales(const float* amax, float* G, int64_t n, bool f46, int* status,
                                 cudaStream_t s);

// Lead of the quantisers' look-ahead beyond one slice, in waves of the grid
// (default 1; a debug hook sets it).
extern std::atomic<int> g_quant_lead_waves;


// Bytes of a [rows, nblocks] matrix of block scales in the tensor-core tiled
// layout: rows padded to a multiple of 128, blocks per row to a multiple of 4.
inline int64_t tiled_bytes(int64_t rows, int64_t nblocks) {
  return (rows + 127) / 128 * 128 * ((nblocks + 3) / 4 * 4);
}
// The same for the NVFP4 scales of a [rows, cols] slice (16-element blocks).
inline int64_t tiled_scale_bytes(int64_t rows, int64_t cols) { return tiled_bytes(rows, cols / 16); }

// Rowwise (and, with codes_col != nullptr, columnwise) NVFP4 of a stack,
// then tensor_scale from amax.  With compute_amax the per-slice amax is
// reduced inside the same single pass over the stack (tensor_scale serves
// as the look-ahead counters until it is written); otherwise amax is given.
// With tiled, the block scales are written in the tensor-core tiled layout
// (padding entries are the caller's to zero).
cudaError_t launch_quant_tiles(const uint16_t* w, int64_t nexp, int rows, int cols, bool f46,
                               uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col,
                               uint8_t* scales_col, float* amax, float* tensor_scale,
                               int* status, bool compute_amax, bool tiled, cudaStream_t s);

cudaError_t launch_act(const uint16_t* x, int64_t T, int H, bool f46, uint8_t* codes,
                       uint8_t* scales, float* token_scale, int* status, bool tiled,
                       cudaStream_t s);

cudaError_t launch_dequant(const uint8_t* codes, const uint8_t* scales, const float* G,
                           int64_t nexp, int64_t per_slice, uint16_t* dst, cudaStream_t s);

cudaError_t launch_dequant_t(const uint8_t* codes, const uint8_t* scales, const float* G,
                             int64_t nexp, int out, int in, uint16_t* dst, cudaStream_t s);

cudaError_t launch_nf4_quant(const uint16_t* w, int64_t n, uint8_t* codes, float* absmax,
                             int* status, cudaStream_t s);

// Dequantises whole expert slices.  With hit_list == nullptr every slice
// 0..nexp-1 is written; otherwise the first *n_hit entries of hit_list
// (device) name the slices.
cudaError_t launch_nf4_dequant(const uint8_t* codes, const float* absmax, int64_t nexp,
                               int64_t per_slice, const int32_t* hit_list, const int32_t* n_hit,
                               uint16_t* dst, cudaStream_t s);

cudaError_t launch_routed_union(const int32_t* topk, int64_t n_idx, int nexp, int32_t* hit_list,
                                int32_t* n_hit, int* status, cudaStream_t s);

// MXFP8 of a stack: rowwise (1x32 blocks) and, with codes_col != nullptr,
// columnwise (32x1 blocks, stored transposed) from one read.
cudaError_t launch_mx_tiles(const uint16_t* w, int64_t nexp, int rows, int cols, uint8_t* codes_row,
                            uint8_t* scales_row, uint8_t* codes_col, uint8_t* scales_col,
                            int* status, bool tiled, cudaStream_t s);
// bf16 of n MXFP8 codes (n % 32 == 0) with one scale byte per 32.
cudaError_t launch_mx_dequant(const uint8_t* codes, const uint8_t* scales, int64_t n, uint16_t* dst,
                              cudaStream_t s);

cudaError_t launch_debug_convert(int kind, const void* in, void* out, int64_t n, cudaStream_t s);
cudaError_t launch_debug_wait_timeout(uint32_t max_tries, int* status, cudaStream_t s);
cudaError_t launch_debug_count_timeout(uint32_t max_polls, const uint32_t* counter, int* status,
                                       cudaStream_t s);
// Experts per grouped-GEMM call (nvfp4_dgrad, nf4_routed_linear): their
// token and tile offsets travel in the kernel's parameter block.
constexpr int kGroupedMaxExperts = 256;
cudaError_t launch_dgrad(const uint16_t* dy, const int64_t* counts, int64_t nexp, int out, int in,
                         const uint8_t* codes, const uint8_t* scales, const float* G, float* dx,
                         int* status, cudaStream_t s);
cudaError_t launch_nf4_linear(const uint16_t* x, const int64_t* counts, int64_t nexp, int out,
                              int in, const uint8_t* codes, const float* absmax, uint16_t* y,
                              int* status, cudaStream_t s);

// The 16 NF4 levels used by the kernels (host copy).
void nf4_levels_host(float out[16]);
cudaError_t launch_nf4_nest(const float* absmax, int64_t nexp, int64_t n, uint8_t* codes,
                            float* c1, float* mean, int* status, cudaStream_t s);
cudaError_t launch_nf4_unnest(const uint8_t* codes, const float* c1, const float* mean,
                              int64_t nexp, int64_t n, float* out, cudaStream_t s);

}  // namespace nvq
