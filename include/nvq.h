/*
 * nvq.h -- C ABI of libnvq: block-scaled 4-bit quantisation of routed
 * mixture-of-experts weights and activations on one GB300 (sm_103a).
 *
 * Sources the operations restate (cited by page title and section):
 *   [P1] "Getting GLM-5.2 NVFP4 Post-Training off the ground", Part I,
 *        "Why can't we just transpose the one copy?" and "The bottom line".
 *   [P4] "The 4-bitter Lesson: Balancing Stability and Performance in NVFP4
 *        RL", "Key claims" and "Method".
 *   [P5] "nf4moe -- QLoRA for a 743B Fused-MoE", "Why every quantizer misses
 *        95% of the model" and "The fix: dequant-on-forward for routed experts".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers.  Every tensor argument is a DEVICE pointer on the current
 *    CUDA device, except where a comment says "host".  The caller owns and
 *    allocates every buffer; the library allocates nothing, keeps no data
 *    between calls (only per-device setup flags of its kernels, set once,
 *    atomically) and never synchronises the host.  Bulk buffers (bf16
 *    inputs and outputs, codes, scales, absmax) must be 16-byte aligned
 *    (32-byte, or only 4-byte, where a call says so); FP32 and int32 arrays
 *    4-byte aligned.
 *  - bf16 tensors are passed as uint16_t bit patterns.  Shapes are int64.
 *    An expert stack is row-major [nexp, rows, cols] with cols contiguous;
 *    for an expert weight used as F.linear(x, W[e]) rows = out, cols = in
 *    ([P5] "Why every quantizer misses 95% of the model").
 *  - Packing.  Two 4-bit codes per byte, element 2j in the low nibble and
 *    element 2j+1 in the high nibble.  Block scales are one byte per block,
 *    stored linearly (row-major over blocks), unless NVQ_SCALES_SWIZZLED
 *    selects the tensor-core tiled layout.
 *  - Asynchrony.  A call validates its arguments on the host, enqueues its
 *    kernels on `stream` and returns.  The return value reports only what is
 *    known at that point: a validation error (no work is enqueued) or a
 *    launch error (NVQ_ERR_CUDA).  A zero-sized problem returns NVQ_OK and
 *    enqueues only what still has to be written (per-slice amax and tensor
 *    scales of empty slices, n_hit of an empty routing).
 *  - Device status word.  `status` (nullable, device int) receives, by
 *    atomic OR, data-dependent conditions found while the kernels run:
 *    NVQ_STATUS_NONFINITE when an amax / absmax is NaN or infinite (those
 *    outputs are then unspecified), NVQ_STATUS_BAD_INDEX when a router
 *    index lies outside [0, nexp) (the index is ignored) and
 *    NVQ_STATUS_TIMEOUT when a bounded internal wait gave up.  Kernels never
 *    trap and never spin without a bound.
 *  - Calls on different streams that write the same buffers race; the
 *    library is otherwise thread-safe (its only global state is the
 *    per-device setup flags, updated atomically), and each call works on
 *    whichever device is current.
 */
#ifndef NVQ_H
#define NVQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define NVQ_API __attribute__((visibility("default")))
#else
#define NVQ_API
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* nvq_stream_t;

/* Return codes. */
enum nvq_status_code {
  NVQ_OK = 0,
  NVQ_ERR_NULL = 1,   /* a required pointer is NULL                          */
  NVQ_ERR_ALIGN = 2,  /* a pointer violates its alignment rule               */
  NVQ_ERR_SHAPE = 3,  /* negative size, divisibility rule broken, overflow   */
  NVQ_ERR_FLAGS = 4,  /* unknown flag bit                                    */
  NVQ_ERR_DEVICE = 5, /* no CUDA device, or the current device is not sm_103 */
  NVQ_ERR_CUDA = 6    /* a CUDA launch failed                                */
};

/* Flag bits of the quantising calls. */
enum nvq_flags {
  /* Four-Over-Six ([P4] "Method"): each block tries its amax mapped to 6 and
     to 4 and keeps the scale with the lower FP32 block squared error; a tie
     keeps 6.  Also sets the largest target block scale M to 256 instead of
     448 (see nvfp4_quantize).                                              */
  NVQ_4OVER6 = 1u << 0,
  /* amax[] is an input (the caller's per-slice absolute maximum) instead of
     being computed; lets a caller skip the reduction pass.                 */
  NVQ_AMAX_GIVEN = 1u << 1,
  /* Block scales are written in the tensor-core tiled layout the
     block-scaled FP4 GEMM reads ([P1] "Why can't we just transpose the one
     copy?": the scales are "swizzled" for the tensor-core tile) instead of
     linearly.  For a [R, C] matrix of block scales (R quantised rows, C =
     blocks per row): R is padded to a multiple of 128, C to a multiple of 4;
     tiles of 128 rows x 4 block columns (512 bytes) follow one another
     row-major (ceil(C/4) tiles per tile row); inside a tile, scale (r, c)
     sits at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4.  Padding
     entries are 0.  Each expert slice occupies nvq_scale_bytes(R, 16 C,
     NVQ_SCALES_SWIZZLED) bytes.  Codes are unchanged.  Accepted by
     nvfp4_quantize, nvfp4_quantize_dual (both copies) and
     act_quantize_per_token; the dequantising and GEMM calls of this library
     read the linear layout.                                                */
  NVQ_SCALES_SWIZZLED = 1u << 2
};

/* Bits of the device status word. */
enum nvq_device_status {
  NVQ_STATUS_NONFINITE = 1, /* an amax / absmax is NaN or infinite           */
  NVQ_STATUS_BAD_INDEX = 2, /* a router index outside [0, nexp) was ignored  */
  /* An internal wait (a bulk tile copy that did not arrive within a fixed
     number of polls, or a shared-memory layout the kernel could not align)
     was abandoned: the CTA stopped early and some outputs of the call were
     not written.  Never expected in normal operation; the call's outputs are
     then unspecified and the device stays usable. */
  NVQ_STATUS_TIMEOUT = 4
};

/* Bytes of the block scales of one [rows, cols] slice (cols % 16 == 0) in
   the layout `flags` selects: rows * cols / 16 linearly, or the padded size
   of the tiled layout with NVQ_SCALES_SWIZZLED.  -1 for invalid arguments.
   Host only; needs no device. */
NVQ_API int64_t nvq_scale_bytes(int64_t rows, int64_t cols, unsigned flags);

/* Library version, (major << 16) | minor. */
NVQ_API int nvq_version(void);

/* Static text for a return code (never NULL). */
NVQ_API const char* nvq_status_string(int code);

/*
 * nvfp4_quantize -- rowwise NVFP4 quantisation of an expert stack.
 * [P1] "Why can't we just transpose the one copy?": 4-bit E2M1 values, one
 * FP8 E4M3 scale per 16-element block along one axis, one FP32 global scale;
 * rowwise blocks are 1x16 along `in` (= cols).  [P4] "Key claims": round to
 * nearest even, no stochastic rounding.
 *
 * Per expert slice e: amax_e = max|w| (or given), G_e = amax_e / (6*M) with
 * M = 448, or 256 under NVQ_4OVER6; E_e = min(1/G_e, FLT_MAX).  Per block of
 * 16: t_i = w_i*E_e, a = max|t_i|, S = E4M3(a/6) (or the Four-Over-Six
 * choice between E4M3(a/6) and E4M3(a/4)), code_i = E2M1(t_i * (1/S)); E4M3
 * and E2M1 round to nearest even and saturate (448, 6); S = 0 gives
 * sign-only codes.
 *
 *   w        in   bf16 [nexp, rows, cols]; cols % 16 == 0
 *   codes    out  u8   [nexp, rows, cols/2]
 *   scales   out  u8   [nexp, rows, cols/16]  E4M3 bytes (with
 *            NVQ_SCALES_SWIZZLED: nexp slices of nvq_scale_bytes(rows, cols,
 *            NVQ_SCALES_SWIZZLED) bytes in the tiled layout)
 *   amax     in/out f32 [nexp]  (input iff NVQ_AMAX_GIVEN; empty slices give 0)
 *   tensor_scale out f32 [nexp] G_e.  Until the call's last kernel writes
 *            G_e, the call uses this buffer as its per-slice work counters,
 *            so it must not be read before the call completes.
 *   status   out  device int, nullable (with NVQ_AMAX_GIVEN the input is not
 *            scanned, so only a non-finite given amax is reported)
 *
 * One pass over the stack: the kernel reduces each slice's amax from tiles
 * it loads a little more than one slice ahead of the tiles it quantises,
 * and reads those tiles again to quantise them.  The second read hits L2
 * while that window (one slice plus two waves of tiles, and the outputs
 * written meanwhile) fits in it, as for [256, 6144, 2048] slices; slices as
 * large as 4096 x 6144 go back to HBM for most of it.  The quantising
 * kernel is a cooperative launch (all its CTAs resident at once), because a
 * CTA that starts a slice waits, bounded, for the amax of that slice; if a
 * wait gives up, NVQ_STATUS_TIMEOUT is set in *status and the outputs are
 * unspecified.
 */
NVQ_API int nvfp4_quantize(const uint16_t* w, int64_t nexp, int64_t rows, int64_t cols,
                   unsigned flags, uint8_t* codes, uint8_t* scales, float* amax,
                   float* tensor_scale, int* status, nvq_stream_t stream);

/*
 * nvfp4_quantize_dual -- rowwise AND columnwise NVFP4 from one read of w.
 * [P1] "Why can't we just transpose the one copy?": the two copies are two
 * independent quantisations of the same weight, rowwise blocks 1x16 along
 * `in` and columnwise blocks 16x1 along `out`, each with its own scales; the
 * columnwise copy is K-major for dgrad, i.e. stored as the transpose.  Both
 * use the same per-expert G_e.  Same arithmetic and flags as nvfp4_quantize.
 *
 *   w           in   bf16 [nexp, out, in]; out % 16 == 0, in % 16 == 0
 *   codes_row   out  u8 [nexp, out, in/2]     scales_row out u8 [nexp, out, in/16]
 *   codes_col   out  u8 [nexp, in, out/2]     scales_col out u8 [nexp, in, out/16]
 *   (with NVQ_SCALES_SWIZZLED each scale buffer holds nexp tiled slices of
 *   nvq_scale_bytes(out, in, .) resp. nvq_scale_bytes(in, out, .) bytes)
 *   amax, tensor_scale, status as in nvfp4_quantize
 */
NVQ_API int nvfp4_quantize_dual(const uint16_t* w, int64_t nexp, int64_t out, int64_t in,
                        unsigned flags, uint8_t* codes_row, uint8_t* scales_row,
                        uint8_t* codes_col, uint8_t* scales_col, float* amax,
                        float* tensor_scale, int* status, nvq_stream_t stream);

/*
 * nvfp4_dequant -- DQ(Q(w)) in the layout of the codes.
 * [P1] "The bottom line" and [P4] "Method" (dequantised backward):
 * y = bf16( (|c| * S) * G_e ) with the sign of the code; |c|*S is exact,
 * the product with G_e is one FP32 rounding, the bf16 conversion rounds to
 * nearest even.
 *
 *   codes in u8 [nexp, rows, cols/2]; scales in u8 [nexp, rows, cols/16];
 *   tensor_scale in f32 [nexp]; dst out bf16 [nexp, rows, cols]; cols % 16 == 0
 */
NVQ_API int nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                  int64_t nexp, int64_t rows, int64_t cols, uint16_t* dst,
                  nvq_stream_t stream);

/*
 * nvfp4_dequant_t -- DQ(Q(w)) of the ROWWISE copy written transposed, the
 * bf16 operand of the dgrad product dX = dY*W ([P1] "The bottom line": keep
 * only the rowwise copy, dequantise it to bf16 and run dgrad in bf16, where
 * the transposed view is free).  Values as in nvfp4_dequant.
 *
 *   codes_row in u8 [nexp, out, in/2]; scales_row in u8 [nexp, out, in/16];
 *   tensor_scale in f32 [nexp]; dst out bf16 [nexp, in, out];
 *   out % 16 == 0, in % 16 == 0
 */
NVQ_API int nvfp4_dequant_t(const uint8_t* codes_row, const uint8_t* scales_row,
                    const float* tensor_scale, int64_t nexp, int64_t out, int64_t in,
                    uint16_t* dst, nvq_stream_t stream);

/*
 * act_quantize_per_token -- NVFP4 activations with one FP32 scale per token.
 * [P4] "Key claims" and "Method": the scale of each token is computed over
 * the hidden dimension inside the quantising kernel, which emits the packed
 * codes, the per-16 E4M3 scales and the per-token FP32 scale in one pass; no
 * state is shared across tokens.  Per row: the nvfp4_quantize arithmetic with
 * the row as the slice.
 *
 *   x in bf16 [T, H], H % 16 == 0; codes out u8 [T, H/2];
 *   scales out u8 [T, H/16] (with NVQ_SCALES_SWIZZLED: nvq_scale_bytes(T,
 *   H, .) bytes in the tiled layout); token_scale out f32 [T];
 *   flags: NVQ_4OVER6, NVQ_SCALES_SWIZZLED
 */
NVQ_API int act_quantize_per_token(const uint16_t* x, int64_t T, int64_t H, unsigned flags,
                           uint8_t* codes, uint8_t* scales, float* token_scale,
                           int* status, nvq_stream_t stream);

/*
 * nf4_quantize -- NF4 blockwise quantisation, blocksize 64
 * ([P5] "The fix": each expert slice stored as NF4 with one absmax per 64
 * elements).  Per block: absmax = max|x| (FP32), v = x * (1/absmax) (0 when
 * absmax = 0), code = nearest of the 16 NF4 levels (see nvq_nf4_codebook),
 * an exact midpoint going to the lower level.
 *
 *   w in bf16 [nexp, rows, cols], cols % 64 == 0;
 *   codes out u8 [nexp, rows, cols/2]; absmax out f32 [nexp, rows, cols/64]
 */
NVQ_API int nf4_quantize(const uint16_t* w, int64_t nexp, int64_t rows, int64_t cols,
                 uint8_t* codes, float* absmax, int* status, nvq_stream_t stream);

/*
 * nf4_dequant -- full-stack NF4 dequantisation, y = bf16(level[c] * absmax).
 *   codes in [nexp, rows, cols/2]; absmax in [nexp, rows, cols/64];
 *   dst out bf16 [nexp, rows, cols]
 */
NVQ_API int nf4_dequant(const uint8_t* codes, const float* absmax, int64_t nexp, int64_t rows,
                int64_t cols, uint16_t* dst, nvq_stream_t stream);

/*
 * nf4_absmax_nest -- the nested ("double-quantised") form of NF4 absmax
 * values ([P5] "The fix": the NF4 state holds the absmax and a "nested
 * code"), read as QLoRA's double quantisation (Dettmers et al., 2023,
 * "Double Quantization"), per expert slice of n = nblocks absmax values:
 *   mean    = RN32(RN64(S / n)), S = the FP32 pairwise-tree sum of the n
 *             values (zero padded to a power of two, adjacent pairs added
 *             level by level; the result does not depend on the launch);
 *   v_i     = fl(absmax_i - mean);
 *   c1_b    = max |v_i| over block b of 256 consecutive values (the last
 *             block of a slice may be shorter);
 *   code_i  = E4M3(fl(v_i * k_b)), k_b = min(fl(448 / c1_b), FLT_MAX),
 *             nearest-even, saturating at 448, sign kept.
 * Decoding (nf4_absmax_unnest): absmax'_i = fma(value(code_i), fl(c1_b/448),
 * mean).  1 byte + 4/256 bytes per NF4 block instead of 4.
 *
 *   absmax  in   f32 [nexp, nblocks] (4-byte aligned; e.g. nf4_quantize's
 *                absmax with nblocks = rows * cols / 64)
 *   codes   out  u8 [nexp, nblocks] (E4M3 bytes)
 *   c1      out  f32 [nexp, ceil(nblocks / 256)] (during the call it also
 *                holds the slice's partial sums; the final values are the
 *                block maxima)
 *   mean    out  f32 [nexp]
 *   status  out  nullable; NVQ_STATUS_NONFINITE for a non-finite mean or c1
 * nblocks <= 2^25 (NVQ_ERR_SHAPE otherwise).  nblocks == 0 writes mean = 0.
 */
NVQ_API int nf4_absmax_nest(const float* absmax, int64_t nexp, int64_t nblocks, uint8_t* codes,
                            float* c1, float* mean, int* status, nvq_stream_t stream);

/*
 * nf4_absmax_unnest -- FP32 absmax decoded from the nested form (above):
 * absmax[e, i] = fma(E4M3 value of codes[e, i], fl(c1[e, i / 256] / 448),
 * mean[e]).  The result feeds nf4_dequant, nf4_dequant_routed and
 * nf4_routed_linear as their absmax.
 *
 *   codes, c1, mean  in   as written by nf4_absmax_nest
 *   absmax           out  f32 [nexp, nblocks] (4-byte aligned)
 */
NVQ_API int nf4_absmax_unnest(const uint8_t* codes, const float* c1, const float* mean,
                              int64_t nexp, int64_t nblocks, float* absmax, nvq_stream_t stream);

/*
 * nf4_dequant_routed -- dequant-on-forward of only the experts the router hit
 * ([P5] "The fix": the union of top_k_index is formed once, and only those
 * experts are dequantised).  The union is computed on the device and consumed
 * there: no host synchronisation at all.
 *
 *   codes, absmax  in   as nf4_dequant
 *   topk_idx       in   int32 [T, k] router choices (may be NULL when T*k == 0)
 *   dst            out  bf16 [nexp, rows, cols]; only hit slices are written
 *   hit_list       out  int32 [nexp]: hit experts ascending, then -1
 *   n_hit          out  int32 [1]: number of hit experts
 *   status         out  nullable; NVQ_STATUS_BAD_INDEX for ignored indices
 */
NVQ_API int nf4_dequant_routed(const uint8_t* codes, const float* absmax, int64_t nexp, int64_t rows,
                       int64_t cols, const int32_t* topk_idx, int64_t T, int64_t k,
                       uint16_t* dst, int32_t* hit_list, int32_t* n_hit, int* status,
                       nvq_stream_t stream);

/*
 * nvq_nf4_codebook -- copies the 16 NF4 levels the kernels use (ascending,
 * level 7 = 0, levels 0 and 15 = -1 and +1) into `out` (HOST, 16 floats).
 * They are the binary32 values of QLoRA's NF4 data type (the type behind
 * quant_type "nf4" in [P5] "The fix"): standard-normal quantiles, 7
 * negative, zero, 8 positive, at probabilities spaced evenly between the
 * outer probability 0.9677083 and 1/2, normalised to [-1, 1].
 */
NVQ_API int nvq_nf4_codebook(float* out);

/*
 * nvfp4_dgrad -- the dgrad GEMM of routed experts read straight from their
 * rowwise NVFP4 copy: dX = dY . DQ(Q(W_e)) for the tokens of each expert.
 * [P4] "Key claims": the backward uses the dequantised weight
 * x . DQ(Q(w)); [P1] "The bottom line": the rowwise copy is dequantised to
 * bf16 for dgrad.  DQ(Q(W_e)) is the bf16 tensor nvfp4_dequant produces; it
 * is formed in shared memory, tile by tile, and never written to HBM.  The
 * products run on the tensor cores with FP32 accumulation, so dX matches an
 * exact evaluation of the same sums to within FP32 rounding of the sums
 * (|error| <= out * 2^-23 * sum |dY| |DQ|), not bit for bit.
 *   dy           bf16 [T, out], T = sum(counts); rows of expert e follow
 *                those of expert e-1
 *   counts       HOST int64 [nexp]: tokens routed to each expert (>= 0)
 *   nexp         1 .. 256
 *   out, in      the weight slice is [out, in]; out % 64 == 0, in % 256 == 0
 *   codes, scales, tensor_scale   the rowwise copy as nvfp4_quantize writes it
 *   dx           FP32 [T, in], written (zeros when out == 0)
 *   status       device int, nullable: NVQ_STATUS_TIMEOUT if a bounded wait
 *                gave up (dx is then unspecified)
 */
NVQ_API int nvfp4_dgrad(const uint16_t* dy, const int64_t* counts, int64_t nexp, int64_t out,
                        int64_t in, const uint8_t* codes, const uint8_t* scales,
                        const float* tensor_scale, float* dx, int* status, nvq_stream_t stream);

/*
 * nf4_routed_linear -- the forward product of routed experts stored as NF4:
 * Y = X . DQ(W_e)^T for the tokens routed to each expert e.  [P5] "The fix:
 * dequant-on-forward for routed experts": each routed expert's weight is
 * dequantised to bf16 and applied as F.linear(x, W[e]) to the tokens sent to
 * it; "Making it fast: the step tax": the dequantised copies are the per-step
 * cost.  DQ(W_e) is the bf16 tensor nf4_dequant produces; it is formed in
 * shared memory, tile by tile, and never written to HBM.  The products run on
 * the tensor cores with FP32 accumulation and Y is the bf16 round to nearest
 * even of the FP32 sum, so |Y - exact| <= 2^-8 (|exact| + d) + d with
 * d = in * 2^-23 * sum |X| |DQ| (not bit for bit).
 *   x            bf16 [T, in], T = sum(counts); rows of expert e follow those
 *                of expert e-1 (the caller sorts tokens by expert)
 *   counts       HOST int64 [nexp]: tokens routed to each expert (>= 0)
 *   nexp         1 .. 256
 *   out, in      the weight slice is [out, in]; out % 256 == 0, in % 256 == 0
 *   codes        u8 [nexp, out, in/2] as nf4_quantize writes them (32-byte
 *                aligned); absmax f32 [nexp, out, in/64] (16-byte aligned)
 *   y            bf16 [T, out], written (zeros when in == 0)
 *   status       device int, nullable: NVQ_STATUS_TIMEOUT if a bounded wait
 *                gave up (y is then unspecified)
 */
NVQ_API int nf4_routed_linear(const uint16_t* x, const int64_t* counts, int64_t nexp, int64_t out,
                              int64_t in, const uint8_t* codes, const float* absmax, uint16_t* y,
                              int* status, nvq_stream_t stream);

/*
 * mxfp8_quantize -- MXFP8 of an expert stack, rowwise and optionally
 * columnwise from one read.  [P4] "Key claims": the dequantised backward was
 * validated first with MXFP8.  The pages name the format only; this is the
 * OCP Microscaling definition: blocks of 32 elements along one axis share a
 * scale 2^s stored as an E8M0 byte s + 127, with s = floor(log2 amax) - 8
 * clamped to [-127, 127] (amax = 0 gives -127); each element is the E4M3 value
 * of v * 2^-s (an exact product), rounded to nearest even, saturating at 448
 * (so the top of a binade can clamp), sign kept.  No global scale.
 *
 *   w           in   bf16 [nexp, rows, cols]; cols % 32 == 0
 *   codes_row   out  u8 [nexp, rows, cols] (E4M3, 32-byte aligned)
 *   scales_row  out  u8 [nexp, rows, cols/32]
 *   codes_col   out  u8 [nexp, cols, rows] (32-byte aligned), nullable: the columnwise copy (32x1 blocks along
 *                    rows, stored transposed, K-major for the transposed product);
 *                    rows % 32 == 0 when given
 *   scales_col  out  u8 [nexp, cols, rows/32] (null iff codes_col is)
 *   flags       0 or NVQ_SCALES_SWIZZLED (tiled layout as for NVFP4, with 32-element
 *               blocks; sizes from nvq_mx_scale_bytes)
 *   status      device int, nullable: NVQ_STATUS_NONFINITE if a block amax is infinite
 *               (NaN inputs are out of contract)
 */
NVQ_API int mxfp8_quantize(const uint16_t* w, int64_t nexp, int64_t rows, int64_t cols,
                           unsigned flags, uint8_t* codes_row, uint8_t* scales_row,
                           uint8_t* codes_col, uint8_t* scales_col, int* status,
                           nvq_stream_t stream);

/*
 * mxfp8_dequant -- y = bf16(E4M3 value * 2^(byte - 127)) for n codes in any
 * layout whose blocks of 32 are contiguous (either copy of mxfp8_quantize):
 * the product is exact, the bf16 conversion rounds to nearest even.
 *   codes in u8 [n]; scales in u8 [n/32] (linear); dst out bf16 [n] (32-byte
 *   aligned); n % 32 == 0
 */
NVQ_API int mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int64_t n, uint16_t* dst,
                          nvq_stream_t stream);

/* Bytes of the MXFP8 block scales of one [rows, cols] slice (cols % 32 == 0):
   rows * cols / 32 linearly, or the padded tiled size with
   NVQ_SCALES_SWIZZLED.  -1 for invalid arguments.  Host only. */
NVQ_API int64_t nvq_mx_scale_bytes(int64_t rows, int64_t cols, unsigned flags);

/*
 * nvq_debug_convert -- runs one device rounding primitive elementwise, for
 * conversion sweeps against an independent implementation.
 *   kind 0: f32 -> E4M3 byte (RNE, satfinite); in f32[n], out u8[n]
 *   kind 1: f32 pair -> byte of two E2M1 codes (RNE, satfinite, sign in bit 3);
 *           in f32[2n], out u8[n]
 *   kind 2: f32 -> bf16 (RNE); in f32[n], out u16[n]
 *   kind 3: f32 a -> E4M3(a/6) byte via the block-scale path; in f32[n], out u8[n]
 *   kind 4: E4M3 byte -> f32 value; in u8[n], out f32[n]
 *   kind 5: byte of two E2M1 codes -> two f32 (low nibble first); in u8[n], out f32[2n]
 *   kind 6: f32 a -> E4M3(a/4) byte via the block-scale path; in f32[n], out u8[n]
 * kind 1 reads n PAIRS of f32 (element 2i goes to the low nibble of byte i).
 */
NVQ_API int nvq_debug_convert(int kind, const void* in, void* out, int64_t n, nvq_stream_t stream);

/*
 * nvq_debug_wait_timeout -- exercises the bounded wait that every kernel of
 * the library uses for its shared-memory copy barriers: one CTA waits, for
 * at most `max_tries` polls, on a barrier that nothing ever completes, then
 * ORs NVQ_STATUS_TIMEOUT into *status and returns.  No copy is in flight and
 * nothing is left running, so the device stays usable.
 *   max_tries  1 .. 65536 (larger values return NVQ_ERR_SHAPE)
 *   status     device int, required
 */
NVQ_API int nvq_debug_wait_timeout(uint32_t max_tries, int* status, nvq_stream_t stream);

/*
 * nvq_debug_count_timeout -- exercises the bounded wait of nvfp4_quantize
 * and nvfp4_quantize_dual for a slice's amax: one thread polls the word at
 * `counter` (device u32, which the caller leaves with bit 31 clear and
 * nothing writes) for the finished mark, bit 31, for at most `max_polls`
 * polls, then ORs NVQ_STATUS_TIMEOUT into *status and returns.  Nothing is
 * left running, so the device stays usable.
 *   max_polls  1 .. 65536 (larger values return NVQ_ERR_SHAPE)
 *   counter    device u32, 4-byte aligned, required
 *   status     device int, required
 */
NVQ_API int nvq_debug_count_timeout(uint32_t max_polls, const uint32_t* counter, int* status,
                                    nvq_stream_t stream);

/*
 * nvq_debug_set_quant_lead -- how far beyond one slice the single-pass amax
 * of nvfp4_quantize and nvfp4_quantize_dual reads ahead of the tiles being
 * quantised, in waves of the kernel's grid (default 2; the kernel's waits
 * stay acyclic for any lead of one wave or more).  Outputs do not depend on
 * it; at 2 the slices' amax complete shortly before they are needed.
 * Process-wide setting for tests and tuning, read at each call.
 *   waves   2 .. 8 (other values return NVQ_ERR_SHAPE and change nothing)
 * Host only; returns NVQ_OK.
 */
NVQ_API int nvq_debug_set_quant_lead(int waves);

#ifdef __cplusplus
}
#endif

#endif /* NVQ_H */
