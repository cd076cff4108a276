// nvq_api.cu -- the C ABI of libnvq: argument validation on the host, then
// kernel launches on the caller's stream.  See include/nvq.h for the
// contract of every entry point.
#include <climits>
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "nvq.h"
#include "nvq_common.cuh"
#include "nvq_internal.h"

namespace nvq {

namespace {
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
int g_dev_state[kMaxDevices];  // 0 unknown, 1 known
std::mutex g_dev_mu;
}  // namespace

const DevInfo* device_info() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev_state[dev]) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_dev[dev].sms = sms;
    g_dev[dev].ok = (major == 10 && minor == 3) ? 1 : 0;
    g_dev_state[dev] = 1;
  }
  return &g_dev[dev];
}

// ----------------------------------------------------------- tensor maps
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

static bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    cudaGetLastError();
  });
  return g_encode != nullptr;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t dim0, uint64_t dim1, uint64_t stride_bytes, uint32_t box0,
                    uint32_t box1, CUtensorMapSwizzle swizzle) {
  if (!get_encode()) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ debug kernels
__global__ void k_debug_convert(int kind, const void* in, void* out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    switch (kind) {
      case 0: {  // f32 -> E4M3
        const float x = static_cast<const float*>(in)[i];
        static_cast<uint8_t*>(out)[i] = (uint8_t)(e4m3x2(x, 0.0f) & 0xff);
        break;
      }
      case 1: {  // f32 pair -> E2M1x2 byte
        const float* f = static_cast<const float*>(in);
        uint32_t h2;
        static_cast<uint8_t*>(out)[i] = (uint8_t)e2m1x2_enc_dec(f[2 * i], f[2 * i + 1], h2);
        break;
      }
      case 2: {  // f32 -> bf16
        const float x = static_cast<const float*>(in)[i];
        static_cast<uint16_t*>(out)[i] = (uint16_t)(bf16x2_rn(x, 0.0f) & 0xffff);
        break;
      }
      case 3: {  // a -> E4M3(a/6) via the block-scale path
        const float a = static_cast<const float*>(in)[i];
        static_cast<uint8_t*>(out)[i] = (uint8_t)(block_scale_bytes(a) & 0xff);
        break;
      }
      case 4: {  // E4M3 byte -> f32
        const uint8_t b = static_cast<const uint8_t*>(in)[i];
        static_cast<float*>(out)[i] = e4m3_decode(b & 0x7f) * ((b & 0x80) ? -1.0f : 1.0f);
        break;
      }
      case 5: {  // E2M1x2 byte -> two f32
        const uint8_t b = static_cast<const uint8_t*>(in)[i];
        const uint32_t h2 = e2m1x2_dec(b);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
        static_cast<float*>(out)[2 * i] = f.x;
        static_cast<float*>(out)[2 * i + 1] = f.y;
        break;
      }
      case 6: {  // a -> E4M3(a/4) via the block-scale path
        const float a = static_cast<const float*>(in)[i];
        static_cast<uint8_t*>(out)[i] = (uint8_t)((block_scale_bytes(a) >> 8) & 0xff);
        break;
      }
      default:
        break;
    }
  }
}

cudaError_t launch_debug_convert(int kind, const void* in, void* out, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const DevInfo* di = device_info();
  const int grid = (int)std::min<int64_t>((n + 255) / 256, (int64_t)di->sms * 8);
  k_debug_convert<<<grid, 256, 0, s>>>(kind, in, out, n);
  return cudaGetLastError();
}

// One CTA waits on a barrier that expects one arrival and never gets it.
__global__ void k_debug_wait_timeout(uint32_t max_tries, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0, max_tries);
  if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicOr(status, kStatusTimeout);
}

cudaError_t launch_debug_wait_timeout(uint32_t max_tries, int* status, cudaStream_t s) {
  k_debug_wait_timeout<<<1, 32, 0, s>>>(max_tries, status);
  return cudaGetLastError();
}

// The quantisers' wait for a slice's finished word, on a word that the
// caller left without the finished bit and nothing writes.
__global__ void k_debug_count_timeout(uint32_t max_polls, const uint32_t* counter, int* status) {
  uint32_t w;
  if (threadIdx.x == 0 && !wait_done(counter, w, max_polls)) atomicOr(status, kStatusTimeout);
}

cudaError_t launch_debug_count_timeout(uint32_t max_polls, const uint32_t* counter, int* status,
                                       cudaStream_t s) {
  k_debug_count_timeout<<<1, 32, 0, s>>>(max_polls, counter, status);
  return cudaGetLastError();
}

}  // namespace nvq

// ---------------------------------------------------------------- the C ABI
namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// a * b * c without int64 overflow (all non-negative)
bool mul_ok(int64_t a, int64_t b, int64_t c, int64_t* out) {
  __int128 p = (__int128)a * b * c;
  if (p > (__int128)(INT64_MAX / 4)) return false;
  *out = (int64_t)p;
  return true;
}

int device_check() {
  const nvq::DevInfo* di = nvq::device_info();
  if (!di || !di->ok) return NVQ_ERR_DEVICE;
  return NVQ_OK;
}

int launch_result(cudaError_t e) {
  if (e == cudaSuccess) return NVQ_OK;
  cudaGetLastError();
  return NVQ_ERR_CUDA;
}

cudaStream_t cs(nvq_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Shape checks shared by the NVFP4 quantisers: non-negative sizes, per-slice
// dimensions that fit in int, and total sizes that fit in int64.
int check_stack(int64_t nexp, int64_t rows, int64_t cols, int64_t* total) {
  if (nexp < 0 || rows < 0 || cols < 0) return NVQ_ERR_SHAPE;
  if (rows > INT_MAX || cols > INT_MAX) return NVQ_ERR_SHAPE;
  if (!mul_ok(nexp, rows, cols, total)) return NVQ_ERR_SHAPE;
  return NVQ_OK;
}

}  // namespace

extern "C" {

int nvq_version(void) { return (1 << 16) | 0; }

const char* nvq_status_string(int code) {
  switch (code) {
    case NVQ_OK: return "ok";
    case NVQ_ERR_NULL: return "a required pointer is NULL";
    case NVQ_ERR_ALIGN: return "a pointer violates its alignment rule";
    case NVQ_ERR_SHAPE: return "invalid shape (negative, not divisible, or too large)";
    case NVQ_ERR_FLAGS: return "unknown flag bit";
    case NVQ_ERR_DEVICE: return "no CUDA device of compute capability 10.3 is current";
    case NVQ_ERR_CUDA: return "a CUDA launch failed";
    default: return "unknown status code";
  }
}

// The tiled layout pads rows to a multiple of 128 and blocks per row to a
// multiple of 4; the kernels write only the real entries, so a ragged shape
// first zeroes the whole buffer (the common, unpadded shapes skip this).
static int zero_tiled_padding(uint8_t* scales, int64_t nexp, int64_t rows, int64_t cols,
                              cudaStream_t s) {
  if (rows % 128 == 0 && (cols / 16) % 4 == 0) return NVQ_OK;
  return launch_result(cudaMemsetAsync(
      scales, 0, (size_t)(nexp * nvq::tiled_scale_bytes(rows, cols)), s));
}

int64_t nvq_scale_bytes(int64_t rows, int64_t cols, unsigned flags) {
  if (rows < 0 || cols < 0 || cols % 16 || (flags & ~(unsigned)NVQ_SCALES_SWIZZLED)) return -1;
  if (rows > (1ll << 40) || cols > (1ll << 40)) return -1;
  return (flags & NVQ_SCALES_SWIZZLED) ? nvq::tiled_scale_bytes(rows, cols) : rows * (cols / 16);
}

int nvfp4_quantize(const uint16_t* w, int64_t nexp, int64_t rows, int64_t cols, unsigned flags,
                   uint8_t* codes, uint8_t* scales, float* amax, float* tensor_scale, int* status,
                   nvq_stream_t stream) {
  if (flags & ~(unsigned)(NVQ_4OVER6 | NVQ_AMAX_GIVEN | NVQ_SCALES_SWIZZLED)) return NVQ_ERR_FLAGS;
  int64_t total;
  int rc = check_stack(nexp, rows, cols, &total);
  if (rc) return rc;
  if (cols % 16) return NVQ_ERR_SHAPE;
  if (nexp == 0) return NVQ_OK;
  if (!amax || !tensor_scale) return NVQ_ERR_NULL;
  if (!aligned(amax, 4) || !aligned(tensor_scale, 4) || (status && !aligned(status, 4)))
    return NVQ_ERR_ALIGN;
  if (total > 0) {
    if (!w || !codes || !scales) return NVQ_ERR_NULL;
    if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 16)) return NVQ_ERR_ALIGN;
  }
  if ((rc = device_check())) return rc;
  cudaStream_t s = cs(stream);
  const bool f46 = flags & NVQ_4OVER6;
  const bool given = flags & NVQ_AMAX_GIVEN;
  const bool tiled = flags & NVQ_SCALES_SWIZZLED;
  if (total == 0) {
    if (!given && (rc = launch_result(nvq::launch_zero_f32(amax, nexp, s)))) return rc;
    return launch_result(nvq::launch_tensor_scales(amax, tensor_scale, nexp, f46, status, s));
  }
  if (tiled && (rc = zero_tiled_padding(scales, nexp, rows, cols, s))) return rc;
  return launch_result(nvq::launch_quant_tiles(w, nexp, (int)rows, (int)cols, f46, codes, scales,
                                               nullptr, nullptr, amax, tensor_scale, status,
                                               !given, tiled, s));
}

int nvfp4_quantize_dual(const uint16_t* w, int64_t nexp, int64_t out, int64_t in, unsigned flags,
                        uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col,
                        uint8_t* scales_col, float* amax, float* tensor_scale, int* status,
                        nvq_stream_t stream) {
  if (flags & ~(unsigned)(NVQ_4OVER6 | NVQ_AMAX_GIVEN | NVQ_SCALES_SWIZZLED)) return NVQ_ERR_FLAGS;
  int64_t total;
  int rc = check_stack(nexp, out, in, &total);
  if (rc) return rc;
  if (out % 16 || in % 16) return NVQ_ERR_SHAPE;
  if (nexp == 0) return NVQ_OK;
  if (!amax || !tensor_scale) return NVQ_ERR_NULL;
  if (!aligned(amax, 4) || !aligned(tensor_scale, 4) || (status && !aligned(status, 4)))
    return NVQ_ERR_ALIGN;
  if (total > 0) {
    if (!w || !codes_row || !scales_row || !codes_col || !scales_col) return NVQ_ERR_NULL;
    if (!aligned(w, 16) || !aligned(codes_row, 16) || !aligned(scales_row, 16) ||
        !aligned(codes_col, 16) || !aligned(scales_col, 16))
      return NVQ_ERR_ALIGN;
  }
  if ((rc = device_check())) return rc;
  cudaStream_t s = cs(stream);
  const bool f46 = flags & NVQ_4OVER6;
  const bool given = flags & NVQ_AMAX_GIVEN;
  const bool tiled = flags & NVQ_SCALES_SWIZZLED;
  if (total == 0) {
    if (!given && (rc = launch_result(nvq::launch_zero_f32(amax, nexp, s)))) return rc;
    return launch_result(nvq::launch_tensor_scales(amax, tensor_scale, nexp, f46, status, s));
  }
  if (tiled && ((rc = zero_tiled_padding(scales_row, nexp, out, in, s)) ||
                (rc = zero_tiled_padding(scales_col, nexp, in, out, s))))
    return rc;
  return launch_result(nvq::launch_quant_tiles(w, nexp, (int)out, (int)in, f46, codes_row,
                                               scales_row, codes_col, scales_col, amax,
                                               tensor_scale, status, !given, tiled, s));
}

int nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                  int64_t nexp, int64_t rows, int64_t cols, uint16_t* dst, nvq_stream_t stream) {
  int64_t total;
  int rc = check_stack(nexp, rows, cols, &total);
  if (rc) return rc;
  if (cols % 16) return NVQ_ERR_SHAPE;
  if (total == 0) return NVQ_OK;
  if (!codes || !scales || !tensor_scale || !dst) return NVQ_ERR_NULL;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(dst, 16) || !aligned(tensor_scale, 4))
    return NVQ_ERR_ALIGN;
  if ((rc = device_check())) return rc;
  return launch_result(
      nvq::launch_dequant(codes, scales, tensor_scale, nexp, rows * cols, dst, cs(stream)));
}

int nvfp4_dequant_t(const uint8_t* codes_row, const uint8_t* scales_row, const float* tensor_scale,
                    int64_t nexp, int64_t out, int64_t in, uint16_t* dst, nvq_stream_t stream) {
  int64_t total;
  int rc = check_stack(nexp, out, in, &total);
  if (rc) return rc;
  if (out % 16 || in % 16) return NVQ_ERR_SHAPE;
  if (total == 0) return NVQ_OK;
  if (!codes_row || !scales_row || !tensor_scale || !dst) return NVQ_ERR_NULL;
  if (!aligned(codes_row, 16) || !aligned(scales_row, 16) || !aligned(dst, 16) ||
      !aligned(tensor_scale, 4))
    return NVQ_ERR_ALIGN;
  if ((rc = device_check())) return rc;
  return launch_result(nvq::launch_dequant_t(codes_row, scales_row, tensor_scale, nexp, (int)out,
                                             (int)in, dst, cs(stream)));
}

int act_quantize_per_token(const uint16_t* x, int64_t T, int64_t H, unsigned flags,
                           uint8_t* codes, uint8_t* scales, float* token_scale, int* status,
                           nvq_stream_t stream) {
  if (flags & ~(unsigned)(NVQ_4OVER6 | NVQ_SCALES_SWIZZLED)) return NVQ_ERR_FLAGS;
  int64_t total;
  int rc = check_stack(1, T, H, &total);
  if (rc) return rc;
  if (H % 16) return NVQ_ERR_SHAPE;
  if (T == 0) return NVQ_OK;
  if (!token_scale) return NVQ_ERR_NULL;
  if (!aligned(token_scale, 4) || (status && !aligned(status, 4))) return NVQ_ERR_ALIGN;
  if (H > 0) {
    if (!x || !codes || !scales) return NVQ_ERR_NULL;
    if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 16)) return NVQ_ERR_ALIGN;
  }
  if ((rc = device_check())) return rc;
  cudaStream_t s = cs(stream);
  if (H == 0) return launch_result(nvq::launch_zero_f32(token_scale, T, s));
  const bool tiled = flags & NVQ_SCALES_SWIZZLED;
  if (tiled && (rc = zero_tiled_padding(scales, 1, T, H, s))) return rc;
  return launch_result(nvq::launch_act(x, T, (int)H, (flags & NVQ_4OVER6) != 0, codes, scales,
                                       token_scale, status, tiled, s));
}

int nf4_quantize(const uint16_t* w, int64_t nexp, int64_t rows, int64_t cols, uint8_t* codes,
                 float* absmax, int* status, nvq_stream_t stream) {
  int64_t total;
  int rc = check_stack(nexp, rows, cols, &total);
  if (rc) return rc;
  if (cols % 64) return NVQ_ERR_SHAPE;
  if (total == 0) return NVQ_OK;
  if (!w || !codes || !absmax) return NVQ_ERR_NULL;
  if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(absmax, 16) ||
      (status && !aligned(status, 4)))
    return NVQ_ERR_ALIGN;
  if ((rc = device_check())) return rc;
  return launch_result(nvq::launch_nf4_quant(w, total, codes, absmax, status, cs(stream)));
}

int nf4_absmax_nest(const float* absmax, int64_t nexp, int64_t nblocks, uint8_t* codes, float* c1,
                    float* mean, int* status, nvq_stream_t stream) {
  int64_t total;
  if (nexp < 0 || nblocks < 0 || !mul_ok(nexp, nblocks, 1, &total)) return NVQ_ERR_SHAPE;
  if (nblocks > ((int64_t)1 << 25)) return NVQ_ERR_SHAPE;
  if (nexp == 0) return NVQ_OK;
  if (!mean) return NVQ_ERR_NULL;
  if (total > 0 && (!absmax || !codes || !c1)) return NVQ_ERR_NULL;
  if (!aligned(mean, 4) || (absmax && !aligned(absmax, 4)) || (c1 && !aligned(c1, 4)) ||
      (status && !aligned(status, 4)))
    return NVQ_ERR_ALIGN;
  int rc;
  if ((rc = device_check())) return rc;
  if (nblocks == 0) return launch_result(cudaMemsetAsync(mean, 0, (size_t)nexp * 4, cs(stream)));
  return launch_result(
      nvq::launch_nf4_nest(absmax, nexp, nblocks, codes, c1, mean, status, cs(stream)));
}

int nf4_absmax_unnest(const uint8_t* codes, const float* c1, const float* mean, int64_t nexp,
                      int64_t nblocks, float* absmax, nvq_stream_t stream) {
  int64_t total;
  if (nexp < 0 || nblocks < 0 || !mul_ok(nexp, nblocks, 4, &total)) return NVQ_ERR_SHAPE;
  if (total == 0) return NVQ_OK;
  if (!codes || !c1 || !mean || !absmax) return NVQ_ERR_NULL;
  if (!aligned(c1, 4) || !aligned(mean, 4) || !aligned(absmax, 4)) return NVQ_ERR_ALIGN;
  int rc;
  if ((rc = device_check())) return rc;
  return launch_result(
      nvq::launch_nf4_unnest(codes, c1, mean, nexp, nblocks, absmax, cs(stream)));
}

int nf4_dequant(const uint8_t* codes, const float* absmax, int64_t nexp, int64_t rows,
                int64_t cols, uint16_t* dst, nvq_stream_t stream) {
  int64_t total;
  int rc = check_stack(nexp, rows, cols, &total);
  if (rc) return rc;
  if (cols % 64) return NVQ_ERR_SHAPE;
  if (total == 0) return NVQ_OK;
  if (!codes || !absmax || !dst) return NVQ_ERR_NULL;
  if (!aligned(codes, 16) || !aligned(absmax, 16) || !aligned(dst, 16)) return NVQ_ERR_ALIGN;
  if ((rc = device_check())) return rc;
  return launch_result(nvq::launch_nf4_dequant(codes, absmax, nexp, rows * cols, nullptr, nullptr,
                                               dst, cs(stream)));
}

int nf4_dequant_routed(const uint8_t* codes, const float* absmax, int64_t nexp, int64_t rows,
                       int64_t cols, const int32_t* topk_idx, int64_t T, int64_t k, uint16_t* dst,
                       int32_t* hit_list, int32_t* n_hit, int* status, nvq_stream_t stream) {
  int64_t total;
  int rc = check_stack(nexp, rows, cols, &total);
  if (rc) return rc;
  if (cols % 64 || T < 0 || k < 0) return NVQ_ERR_SHAPE;
  if (nexp > 65536) return NVQ_ERR_SHAPE;
  int64_t n_idx;
  if (!mul_ok(T, k, 1, &n_idx)) return NVQ_ERR_SHAPE;
  if (!n_hit) return NVQ_ERR_NULL;
  if (nexp > 0 && !hit_list) return NVQ_ERR_NULL;
  if (n_idx > 0 && !topk_idx) return NVQ_ERR_NULL;
  if (total > 0 && (!codes || !absmax || !dst)) return NVQ_ERR_NULL;
  if (!aligned(n_hit, 4) || (hit_list && !aligned(hit_list, 4)) ||
      (topk_idx && !aligned(topk_idx, 4)) || (status && !aligned(status, 4)))
    return NVQ_ERR_ALIGN;
  if (total > 0 && (!aligned(codes, 16) || !aligned(absmax, 16) || !aligned(dst, 16)))
    return NVQ_ERR_ALIGN;
  if ((rc = device_check())) return rc;
  cudaStream_t s = cs(stream);
  if ((rc = launch_result(
           nvq::launch_routed_union(topk_idx, n_idx, (int)nexp, hit_list, n_hit, status, s))))
    return rc;
  if (total == 0) return NVQ_OK;
  return launch_result(
      nvq::launch_nf4_dequant(codes, absmax, nexp, rows * cols, hit_list, n_hit, dst, s));
}

int nvq_nf4_codebook(float* out) {
  if (!out) return NVQ_ERR_NULL;
  nvq::nf4_levels_host(out);
  return NVQ_OK;
}

int nvq_debug_convert(int kind, const void* in, void* out, int64_t n, nvq_stream_t stream) {
  if (kind < 0 || kind > 6) return NVQ_ERR_FLAGS;
  if (n < 0) return NVQ_ERR_SHAPE;
  if (n == 0) return NVQ_OK;
  if (!in || !out) return NVQ_ERR_NULL;
  int rc = device_check();
  if (rc) return rc;
  return launch_result(nvq::launch_debug_convert(kind, in, out, n, cs(stream)));
}

int nvfp4_dgrad(const uint16_t* dy, const int64_t* counts, int64_t nexp, int64_t out, int64_t in,
                const uint8_t* codes, const uint8_t* scales, const float* tensor_scale, float* dx,
                int* status, nvq_stream_t stream) {
  if (nexp < 1 || nexp > nvq::kGroupedMaxExperts || out < 0 || in < 0) return NVQ_ERR_SHAPE;
  if (out % 64 || in % 256 || nexp * out >= (1ll << 31)) return NVQ_ERR_SHAPE;
  if (!counts) return NVQ_ERR_NULL;
  int64_t T = 0;
  for (int64_t e = 0; e < nexp; e++) {
    if (counts[e] < 0) return NVQ_ERR_SHAPE;
    T += counts[e];
    if (T >= (1ll << 31)) return NVQ_ERR_SHAPE;
  }
  int64_t total;
  if (!mul_ok(nexp, out, in, &total) || T * in >= (1ll << 40) || T * out >= (1ll << 40))
    return NVQ_ERR_SHAPE;
  if (T == 0 || in == 0) return NVQ_OK;
  const bool contract = out > 0;  // out == 0: an empty contraction, dX = 0
  if (!dx || (contract && (!dy || !codes || !scales || !tensor_scale))) return NVQ_ERR_NULL;
  if (!aligned(dx, 16) || (status && !aligned(status, 4)) ||
      (contract && (!aligned(dy, 16) || !aligned(codes, 16) || !aligned(scales, 16) ||
                    !aligned(tensor_scale, 4))))
    return NVQ_ERR_ALIGN;
  int rc = device_check();
  if (rc) return rc;
  if (!contract)
    return launch_result(cudaMemsetAsync(dx, 0, (size_t)(T * in) * sizeof(float), cs(stream)));
  return launch_result(nvq::launch_dgrad(dy, counts, nexp, (int)out, (int)in, codes, scales,
                                         tensor_scale, dx, status, cs(stream)));
}

int nf4_routed_linear(const uint16_t* x, const int64_t* counts, int64_t nexp, int64_t out,
                      int64_t in, const uint8_t* codes, const float* absmax, uint16_t* y,
                      int* status, nvq_stream_t stream) {
  if (nexp < 1 || nexp > nvq::kGroupedMaxExperts || out < 0 || in < 0) return NVQ_ERR_SHAPE;
  if (out % 256 || in % 256) return NVQ_ERR_SHAPE;
  if (!counts) return NVQ_ERR_NULL;
  int64_t T = 0;
  for (int64_t e = 0; e < nexp; e++) {
    if (counts[e] < 0) return NVQ_ERR_SHAPE;
    T += counts[e];
    if (T >= (1ll << 31)) return NVQ_ERR_SHAPE;
  }
  int64_t total;
  if (!mul_ok(nexp, out, in, &total) || T * in >= (1ll << 40) || T * out >= (1ll << 40) ||
      nexp * out >= (1ll << 31))
    return NVQ_ERR_SHAPE;
  if (T == 0 || out == 0) return NVQ_OK;
  const bool contract = in > 0;  // in == 0: an empty contraction, Y = 0
  if (!y || (contract && (!x || !codes || !absmax))) return NVQ_ERR_NULL;
  if (!aligned(y, 16) || (status && !aligned(status, 4)) ||
      (contract && (!aligned(x, 16) || !aligned(codes, 32) || !aligned(absmax, 16))))
    return NVQ_ERR_ALIGN;
  int rc = device_check();
  if (rc) return rc;
  if (!contract)
    return launch_result(cudaMemsetAsync(y, 0, (size_t)(T * out) * sizeof(uint16_t), cs(stream)));
  return launch_result(nvq::launch_nf4_linear(x, counts, nexp, (int)out, (int)in, codes, absmax,
                                              y, status, cs(stream)));
}

int64_t nvq_mx_scale_bytes(int64_t rows, int64_t cols, unsigned flags) {
  if (rows < 0 || cols < 0 || cols % 32 || (flags & ~(unsigned)NVQ_SCALES_SWIZZLED)) return -1;
  if (rows > (1ll << 40) || cols > (1ll << 40)) return -1;
  return (flags & NVQ_SCALES_SWIZZLED) ? nvq::tiled_bytes(rows, cols / 32) : rows * (cols / 32);
}

int mxfp8_quantize(const uint16_t* w, int64_t nexp, int64_t rows, int64_t cols, unsigned flags,
                   uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col, uint8_t* scales_col,
                   int* status, nvq_stream_t stream) {
  if (flags & ~(unsigned)NVQ_SCALES_SWIZZLED) return NVQ_ERR_FLAGS;
  int64_t total;
  int rc = check_stack(nexp, rows, cols, &total);
  if (rc) return rc;
  const bool dual = codes_col != nullptr || scales_col != nullptr;
  if (cols % 32 || (dual && rows % 32)) return NVQ_ERR_SHAPE;
  if (total == 0) return NVQ_OK;
  if (!w || !codes_row || !scales_row || (dual && (!codes_col || !scales_col))) return NVQ_ERR_NULL;
  if (!aligned(w, 16) || !aligned(codes_row, 32) || !aligned(scales_row, 16) ||
      (dual && (!aligned(codes_col, 32) || !aligned(scales_col, 16))) ||
      (status && !aligned(status, 4)))
    return NVQ_ERR_ALIGN;
  if ((rc = device_check())) return rc;
  cudaStream_t s = cs(stream);
  const bool tiled = flags & NVQ_SCALES_SWIZZLED;
  if (tiled) {
    // the kernel writes only the real entries of the padded tiled layout
    if ((rows % 128 || (cols / 32) % 4) &&
        (rc = launch_result(cudaMemsetAsync(
             scales_row, 0, (size_t)(nexp * nvq::tiled_bytes(rows, cols / 32)), s))))
      return rc;
    if (dual && (cols % 128 || (rows / 32) % 4) &&
        (rc = launch_result(cudaMemsetAsync(
             scales_col, 0, (size_t)(nexp * nvq::tiled_bytes(cols, rows / 32)), s))))
      return rc;
  }
  return launch_result(nvq::launch_mx_tiles(w, nexp, (int)rows, (int)cols, codes_row, scales_row,
                                            dual ? codes_col : nullptr, scales_col, status, tiled,
                                            s));
}

int mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int64_t n, uint16_t* dst,
                  nvq_stream_t stream) {
  if (n < 0 || n % 32 || n >= (1ll << 46)) return NVQ_ERR_SHAPE;
  if (n == 0) return NVQ_OK;
  if (!codes || !scales || !dst) return NVQ_ERR_NULL;
  if (!aligned(codes, 16) || !aligned(dst, 32)) return NVQ_ERR_ALIGN;
  int rc = device_check();
  if (rc) return rc;
  return launch_result(nvq::launch_mx_dequant(codes, scales, n, dst, cs(stream)));
}

int nvq_debug_wait_timeout(uint32_t max_tries, int* status, nvq_stream_t stream) {
  if (max_tries == 0 || max_tries > 65536u) return NVQ_ERR_SHAPE;
  if (!status) return NVQ_ERR_NULL;
  if (!aligned(status, 4)) return NVQ_ERR_ALIGN;
  int rc = device_check();
  if (rc) return rc;
  return launch_result(nvq::launch_debug_wait_timeout(max_tries, status, cs(stream)));
}

int nvq_debug_count_timeout(uint32_t max_polls, const uint32_t* counter, int* status,
                            nvq_stream_t stream) {
  if (max_polls == 0 || max_polls > 65536u) return NVQ_ERR_SHAPE;
  if (!status || !counter) return NVQ_ERR_NULL;
  if (!aligned(status, 4) || !aligned(counter, 4)) return NVQ_ERR_ALIGN;
  int rc = device_check();
  if (rc) return rc;
  return launch_result(nvq::launch_debug_count_timeout(max_polls, counter, status, cs(stream)));
}

int nvq_debug_set_quant_lead(int waves) {
  if (waves < 2 || waves > 8) return NVQ_ERR_SHAPE;
  nvq::g_quant_lead_waves.store(waves, std::memory_order_relaxed);
  return NVQ_OK;
}

}  // extern "C"
