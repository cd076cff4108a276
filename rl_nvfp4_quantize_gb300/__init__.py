"""Block-scaled 4-bit quantisation of routed-MoE weights and activations on GB300.

Thin Python binding over the C ABI of ``libnvq.so`` (declared in
``include/nvq.h``).  Every function here only marshals arguments: it checks
dtypes and shapes, allocates outputs with PyTorch when the caller passes
none, and calls the C entry point of the same name on the current CUDA
stream.  All arithmetic runs in the library's CUDA kernels; there is no CPU
fallback -- importing this package fails if the library is missing or cannot
be loaded.

Sources restated by the kernels: "Getting GLM-5.2 NVFP4 Post-Training off the
ground" (NVFP4 rowwise/columnwise copies, dequantised bf16 backward), "The
4-bitter Lesson" (round-to-nearest, Four-Over-Six, per-token FP32 activation
scales) and "nf4moe -- QLoRA for a 743B Fused-MoE" (NF4 blocksize 64,
dequant-on-forward of the routed experts).
"""
from __future__ import annotations

import ctypes as C
import os

import torch

__all__ = [
    "NvqError", "FLAG_4OVER6", "FLAG_AMAX_GIVEN", "FLAG_SCALES_SWIZZLED", "STATUS_NONFINITE", "STATUS_BAD_INDEX", "STATUS_TIMEOUT",
    "nvfp4_quantize", "nvfp4_quantize_dual", "nvfp4_dequant", "nvfp4_dequant_t", "nvfp4_dgrad",
    "act_quantize_per_token", "nf4_quantize", "nf4_dequant", "nf4_dequant_routed", "nf4_routed_linear",
    "nf4_absmax_nest", "nf4_absmax_unnest",
    "mxfp8_quantize", "mxfp8_dequant", "mx_scale_bytes",
    "nf4_codebook", "scale_bytes", "debug_convert", "debug_wait_timeout", "debug_set_quant_lead",
    "debug_count_timeout", "lib", "library_path",
]

FLAG_4OVER6 = 1
FLAG_AMAX_GIVEN = 2
FLAG_SCALES_SWIZZLED = 4
STATUS_NONFINITE = 1
STATUS_BAD_INDEX = 2
STATUS_TIMEOUT = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libnvq.so")


class NvqError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = lib.nvq_status_string(code).decode() if lib else str(code)
        super().__init__("%s failed: %s (code %d)" % (fn, msg, code))
        self.code = code


def _load():
    if not os.path.exists(library_path):
        raise ImportError("libnvq.so is not built (run __graft_entry__.build() or "
                          "python rl_nvfp4_quantize_gb300/build.py)")
    L = C.CDLL(library_path)
    P, i64, u32, i32 = C.c_void_p, C.c_int64, C.c_uint, C.c_int
    sig = {
        "nvq_version": ([], i32),
        "nvq_status_string": ([i32], C.c_char_p),
        "nvq_scale_bytes": ([i64, i64, u32], i64),
        "nvfp4_quantize": ([P, i64, i64, i64, u32, P, P, P, P, P, P], i32),
        "nvfp4_quantize_dual": ([P, i64, i64, i64, u32, P, P, P, P, P, P, P, P], i32),
        "nvfp4_dequant": ([P, P, P, i64, i64, i64, P, P], i32),
        "nvfp4_dequant_t": ([P, P, P, i64, i64, i64, P, P], i32),
        "act_quantize_per_token": ([P, i64, i64, u32, P, P, P, P, P], i32),
        "nf4_quantize": ([P, i64, i64, i64, P, P, P, P], i32),
        "nf4_dequant": ([P, P, i64, i64, i64, P, P], i32),
        "nf4_dequant_routed": ([P, P, i64, i64, i64, P, i64, i64, P, P, P, P, P], i32),
        "nvq_nf4_codebook": ([P], i32),
        "nvq_debug_convert": ([i32, P, P, i64, P], i32),
        "nvq_debug_wait_timeout": ([u32, P, P], i32),
        "nvq_debug_set_quant_lead": ([i32], i32),
        "nvq_debug_count_timeout": ([u32, P, P, P], i32),
        "nvfp4_dgrad": ([P, P, i64, i64, i64, P, P, P, P, P, P], i32),
        "nf4_routed_linear": ([P, P, i64, i64, i64, P, P, P, P, P], i32),
        "mxfp8_quantize": ([P, i64, i64, i64, u32, P, P, P, P, P, P], i32),
        "mxfp8_dequant": ([P, P, i64, P, P], i32),
        "nvq_mx_scale_bytes": ([i64, i64, u32], i64),
        "nf4_absmax_nest": ([P, i64, i64, P, P, P, P, P], i32),
        "nf4_absmax_unnest": ([P, P, P, i64, i64, P, P], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    return L


lib = None
lib = _load()


# ---------------------------------------------------------------- helpers

def _ptr(t):
    """Address of a contiguous tensor on the current CUDA device (None: NULL).
    Host tensors are refused here: the kernels would dereference a host
    address."""
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise TypeError("expected a contiguous CUDA tensor, got %s (%s, contiguous=%s)"
                        % (tuple(t.shape), t.device, t.is_contiguous()))
    if t.device.index != torch.cuda.current_device():
        raise ValueError("tensor on %s, but the current device is cuda:%d"
                         % (t.device, torch.cuda.current_device()))
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise NvqError(fn, rc)


def _bf16(t, name):
    """A bf16 input; its device is checked by _ptr, after the size checks."""
    if t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise TypeError("%s must be a contiguous bfloat16 tensor" % name)
    return t


def _as3d(w):
    if w.dim() == 2:
        return w.unsqueeze(0)
    if w.dim() != 3:
        raise ValueError("expected [nexp, rows, cols] or [rows, cols]")
    return w


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def _need(t, name, dtype, numel=None, shape=None, at_least=False):
    """Refuses, before any call, a tensor the library would read or write
    past its end or reinterpret: the C ABI sees only an address, so its size
    and element type are checked here.  `numel` is the exact element count
    the call touches (`at_least`: a lower bound); `shape`, when given, must
    match exactly.  Returns t."""
    if t is None:
        return t
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if numel is not None:
        n = t.numel()
        if (n < numel) if at_least else (n != numel):
            raise ValueError("%s must hold %s%d elements, got %d"
                             % (name, "at least " if at_least else "", numel, n))
    return t


def _status(status):
    return _need(status, "status", torch.int32, 1, at_least=True)


def _scale_numel(E, R, K, swizzled):
    return E * scale_bytes(R, K, True) if swizzled else E * R * (K // 16)


# ---------------------------------------------------------------- NVFP4

def scale_bytes(rows, cols, swizzled=False):
    """Bytes of the block scales of one [rows, cols] slice (see
    nvq_scale_bytes in nvq.h)."""
    n = lib.nvq_scale_bytes(rows, cols, FLAG_SCALES_SWIZZLED if swizzled else 0)
    if n < 0:
        raise ValueError("invalid scale shape [%d, %d]" % (rows, cols))
    return n


def _scales(E, R, K, swizzled, like):
    """Block-scale buffer: [E, R, K/16] linear, or [E, bytes] tiled."""
    if swizzled:
        return _empty((E, scale_bytes(R, K, True)), torch.uint8, like)
    return _empty((E, R, K // 16), torch.uint8, like)


def nvfp4_quantize(w, four_over_six=False, amax=None, status=None, stream=None, out=None,
                   swizzled_scales=False):
    """Rowwise NVFP4 of w [nexp, rows, cols] (bf16).  Returns a dict with
    codes [nexp, rows, cols/2] u8, scales [nexp, rows, cols/16] u8 (E4M3; with
    swizzled_scales [nexp, scale_bytes(rows, cols, True)] in the tensor-core
    tiled layout), amax [nexp] f32 and tensor_scale [nexp] f32."""
    w = _as3d(_bf16(w, "w"))
    E, R, K = w.shape
    o = out or {}
    codes = o.get("codes", _empty((E, R, K // 2), torch.uint8, w))
    scales = o.get("scales") if "scales" in o else _scales(E, R, K, swizzled_scales, w)
    am = amax if amax is not None else o.get("amax", _empty((E,), torch.float32, w))
    G = o.get("tensor_scale", _empty((E,), torch.float32, w))
    if K % 16 == 0:
        _need(codes, "codes", torch.uint8, E * R * (K // 2))
        _need(scales, "scales", torch.uint8, _scale_numel(E, R, K, swizzled_scales))
    _need(am, "amax", torch.float32, E)
    _need(G, "tensor_scale", torch.float32, E)
    flags = ((FLAG_4OVER6 if four_over_six else 0) | (FLAG_AMAX_GIVEN if amax is not None else 0)
             | (FLAG_SCALES_SWIZZLED if swizzled_scales else 0))
    _status(status)
    _check("nvfp4_quantize", lib.nvfp4_quantize(_ptr(w), E, R, K, flags, _ptr(codes), _ptr(scales),
                                                _ptr(am), _ptr(G), _ptr(status), _stream(stream)))
    return dict(codes=codes, scales=scales, amax=am, tensor_scale=G)


def nvfp4_quantize_dual(w, four_over_six=True, amax=None, status=None, stream=None, out=None,
                        swizzled_scales=False):
    """Rowwise and columnwise NVFP4 of w [nexp, out, in] from one read.
    Columnwise outputs are K-major for dgrad: [nexp, in, out/2] / [nexp, in, out/16]
    (scales [nexp, scale_bytes(in, out, True)] with swizzled_scales)."""
    w = _as3d(_bf16(w, "w"))
    E, R, K = w.shape
    o = out or {}
    cr = o.get("codes_row", _empty((E, R, K // 2), torch.uint8, w))
    sr = o.get("scales_row") if "scales_row" in o else _scales(E, R, K, swizzled_scales, w)
    cc = o.get("codes_col", _empty((E, K, R // 2), torch.uint8, w))
    sc = o.get("scales_col") if "scales_col" in o else _scales(E, K, R, swizzled_scales, w)
    am = amax if amax is not None else o.get("amax", _empty((E,), torch.float32, w))
    G = o.get("tensor_scale", _empty((E,), torch.float32, w))
    if K % 16 == 0 and R % 16 == 0:
        _need(cr, "codes_row", torch.uint8, E * R * (K // 2))
        _need(sr, "scales_row", torch.uint8, _scale_numel(E, R, K, swizzled_scales))
        _need(cc, "codes_col", torch.uint8, E * K * (R // 2))
        _need(sc, "scales_col", torch.uint8, _scale_numel(E, K, R, swizzled_scales))
    _need(am, "amax", torch.float32, E)
    _need(G, "tensor_scale", torch.float32, E)
    flags = ((FLAG_4OVER6 if four_over_six else 0) | (FLAG_AMAX_GIVEN if amax is not None else 0)
             | (FLAG_SCALES_SWIZZLED if swizzled_scales else 0))
    _status(status)
    _check("nvfp4_quantize_dual",
           lib.nvfp4_quantize_dual(_ptr(w), E, R, K, flags, _ptr(cr), _ptr(sr), _ptr(cc), _ptr(sc),
                                   _ptr(am), _ptr(G), _ptr(status), _stream(stream)))
    return dict(codes_row=cr, scales_row=sr, codes_col=cc, scales_col=sc, amax=am, tensor_scale=G)


def _dequant_inputs(codes, scales, tensor_scale):
    """Shapes of the rowwise copy a dequant call reads.  The scales must be
    in the linear layout [nexp, rows, cols/16]: a tiled (swizzled_scales)
    buffer is refused rather than decoded as linear."""
    _need(codes, "codes", torch.uint8)
    if codes.dim() != 3:
        raise ValueError("codes must be [nexp, rows, cols/2]")
    E, R, K2 = codes.shape
    K = K2 * 2
    if K % 16 == 0:
        _need(scales, "scales", torch.uint8, shape=(E, R, K // 16))
    _need(tensor_scale, "tensor_scale", torch.float32, E)
    return E, R, K


def nvfp4_dequant(codes, scales, tensor_scale, stream=None, out=None):
    """DQ(Q(w)) in the layout of the codes: bf16 [nexp, rows, cols]."""
    E, R, K = _dequant_inputs(codes, scales, tensor_scale)
    dst = out if out is not None else _empty((E, R, K), torch.bfloat16, codes)
    _need(dst, "out", torch.bfloat16, E * R * K)
    _check("nvfp4_dequant", lib.nvfp4_dequant(_ptr(codes), _ptr(scales), _ptr(tensor_scale), E, R, K,
                                              _ptr(dst), _stream(stream)))
    return dst


def nvfp4_dequant_t(codes_row, scales_row, tensor_scale, stream=None, out=None):
    """DQ(Q(w)) of the rowwise copy, transposed: bf16 [nexp, in, out]."""
    E, R, K = _dequant_inputs(codes_row, scales_row, tensor_scale)
    dst = out if out is not None else _empty((E, K, R), torch.bfloat16, codes_row)
    _need(dst, "out", torch.bfloat16, E * K * R)
    _check("nvfp4_dequant_t",
           lib.nvfp4_dequant_t(_ptr(codes_row), _ptr(scales_row), _ptr(tensor_scale), E, R, K,
                               _ptr(dst), _stream(stream)))
    return dst


def act_quantize_per_token(x, four_over_six=True, status=None, stream=None, out=None,
                           swizzled_scales=False):
    """NVFP4 activations [T, H] with one FP32 scale per token (scales
    [scale_bytes(T, H, True)] in the tiled layout with swizzled_scales)."""
    x = _bf16(x, "x")
    if x.dim() != 2:
        raise ValueError("expected x [T, H]")
    T, H = x.shape
    o = out or {}
    codes = o.get("codes", _empty((T, H // 2), torch.uint8, x))
    if "scales" in o:
        scales = o["scales"]
    elif swizzled_scales:
        scales = _empty((scale_bytes(T, H, True),), torch.uint8, x)
    else:
        scales = _empty((T, H // 16), torch.uint8, x)
    ts = o.get("token_scale", _empty((T,), torch.float32, x))
    if H % 16 == 0:
        _need(codes, "codes", torch.uint8, T * (H // 2))
        _need(scales, "scales", torch.uint8, _scale_numel(1, T, H, swizzled_scales))
    _need(ts, "token_scale", torch.float32, T)
    _status(status)
    flags = (FLAG_4OVER6 if four_over_six else 0) | (FLAG_SCALES_SWIZZLED if swizzled_scales else 0)
    _check("act_quantize_per_token",
           lib.act_quantize_per_token(_ptr(x), T, H, flags, _ptr(codes), _ptr(scales), _ptr(ts),
                                      _ptr(status), _stream(stream)))
    return dict(codes=codes, scales=scales, token_scale=ts)


# ---------------------------------------------------------------- NF4

def nf4_quantize(w, status=None, stream=None, out=None):
    """NF4 with blocksize 64: codes [nexp, rows, cols/2], absmax [nexp, rows, cols/64]."""
    w = _as3d(_bf16(w, "w"))
    E, R, K = w.shape
    o = out or {}
    codes = o.get("codes", _empty((E, R, K // 2), torch.uint8, w))
    absmax = o.get("absmax", _empty((E, R, K // 64), torch.float32, w))
    if K % 64 == 0:
        _need(codes, "codes", torch.uint8, E * R * (K // 2))
        _need(absmax, "absmax", torch.float32, E * R * (K // 64))
    _status(status)
    _check("nf4_quantize", lib.nf4_quantize(_ptr(w), E, R, K, _ptr(codes), _ptr(absmax),
                                            _ptr(status), _stream(stream)))
    return dict(codes=codes, absmax=absmax)


def _nf4_inputs(codes, absmax):
    _need(codes, "codes", torch.uint8)
    if codes.dim() != 3:
        raise ValueError("codes must be [nexp, rows, cols/2]")
    E, R, K2 = codes.shape
    K = K2 * 2
    if K % 64 == 0:
        _need(absmax, "absmax", torch.float32, E * R * (K // 64))
    return E, R, K


def nf4_dequant(codes, absmax, stream=None, out=None):
    E, R, K = _nf4_inputs(codes, absmax)
    dst = out if out is not None else _empty((E, R, K), torch.bfloat16, codes)
    _need(dst, "out", torch.bfloat16, E * R * K)
    _check("nf4_dequant", lib.nf4_dequant(_ptr(codes), _ptr(absmax), E, R, K, _ptr(dst),
                                          _stream(stream)))
    return dst


def nf4_absmax_nest(absmax, status=None, stream=None, out=None):
    """Nested (double-quantised) form of NF4 absmax [nexp, ...] (FP32):
    codes u8 [nexp, n], c1 f32 [nexp, ceil(n/256)], mean f32 [nexp]."""
    if absmax.dtype != torch.float32:
        raise TypeError("absmax must be float32")
    a = absmax.contiguous()
    E = a.shape[0]
    n = a.numel() // E if E else 0
    o = out or {}
    codes = o.get("codes", _empty((E, n), torch.uint8, a))
    c1 = o.get("c1", _empty((E, (n + 255) // 256), torch.float32, a))
    mean = o.get("mean", _empty((E,), torch.float32, a))
    _need(codes, "codes", torch.uint8, E * n)
    _need(c1, "c1", torch.float32, E * ((n + 255) // 256))
    _need(mean, "mean", torch.float32, E)
    _status(status)
    _check("nf4_absmax_nest", lib.nf4_absmax_nest(_ptr(a), E, n, _ptr(codes), _ptr(c1), _ptr(mean),
                                                  _ptr(status), _stream(stream)))
    return dict(codes=codes, c1=c1, mean=mean)


def nf4_absmax_unnest(codes, c1, mean, shape=None, stream=None, out=None):
    """FP32 absmax decoded from the nested form, [nexp, n] (or `shape`)."""
    _need(codes, "codes", torch.uint8)
    E = codes.shape[0]
    n = codes.numel() // E if E else 0
    _need(c1, "c1", torch.float32, E * ((n + 255) // 256))
    _need(mean, "mean", torch.float32, E)
    dst = out if out is not None else _empty((E, n), torch.float32, codes)
    _need(dst, "out", torch.float32, E * n)
    _check("nf4_absmax_unnest", lib.nf4_absmax_unnest(_ptr(codes), _ptr(c1), _ptr(mean), E, n,
                                                      _ptr(dst), _stream(stream)))
    return dst.view(shape) if shape is not None else dst


def nf4_dequant_routed(codes, absmax, topk_idx, dst=None, status=None, stream=None,
                       hit_list=None, n_hit=None):
    """Dequantises only the experts present in topk_idx [T, k] (int32) into
    dst [nexp, rows, cols]; returns (dst, hit_list, n_hit), both device
    tensors -- nothing is synchronised to the host."""
    E, R, K = _nf4_inputs(codes, absmax)
    if topk_idx.dtype != torch.int32 or not topk_idx.is_contiguous() or topk_idx.dim() != 2:
        raise TypeError("topk_idx must be a contiguous int32 tensor [T, k]")
    T, k = topk_idx.shape
    if dst is None:
        dst = _empty((E, R, K), torch.bfloat16, codes)
    hl = hit_list if hit_list is not None else _empty((E,), torch.int32, codes)
    nh = n_hit if n_hit is not None else _empty((1,), torch.int32, codes)
    _need(dst, "dst", torch.bfloat16, E * R * K)
    _need(hl, "hit_list", torch.int32, E)
    _need(nh, "n_hit", torch.int32, 1, at_least=True)
    _status(status)
    _check("nf4_dequant_routed",
           lib.nf4_dequant_routed(_ptr(codes), _ptr(absmax), E, R, K, _ptr(topk_idx), T, k,
                                  _ptr(dst), _ptr(hl), _ptr(nh), _ptr(status), _stream(stream)))
    return dst, hl, nh


def nf4_codebook():
    """The 16 NF4 levels used by the kernels (host float32 tensor)."""
    out = (C.c_float * 16)()
    _check("nvq_nf4_codebook", lib.nvq_nf4_codebook(out))
    return torch.tensor(list(out), dtype=torch.float32)


_DEBUG_OUT = {0: (torch.uint8, 1), 1: (torch.uint8, 1), 2: (torch.int16, 1), 3: (torch.uint8, 1),
              4: (torch.float32, 1), 5: (torch.float32, 2), 6: (torch.uint8, 1)}


def debug_convert(kind: int, x, stream=None):
    """Runs one device rounding primitive elementwise (see nvq_debug_convert)."""
    n = x.numel() // 2 if kind == 1 else x.numel()
    dt, mult = _DEBUG_OUT[kind]
    out = torch.empty(n * mult, dtype=dt, device=x.device)
    _check("nvq_debug_convert", lib.nvq_debug_convert(kind, _ptr(x), _ptr(out), n, _stream(stream)))
    return out


def debug_wait_timeout(max_tries: int, status, stream=None):
    """Runs the bounded-wait probe (see nvq_debug_wait_timeout): ORs
    STATUS_TIMEOUT into the device int `status`."""
    _check("nvq_debug_wait_timeout", lib.nvq_debug_wait_timeout(max_tries, _ptr(status), _stream(stream)))


def debug_count_timeout(max_polls: int, counter, status, stream=None):
    """Runs the quantisers' slice-amax wait on `counter` (a device int32 the
    caller leaves non-negative; see nvq_debug_count_timeout): ORs
    STATUS_TIMEOUT into the device int `status`."""
    _need(counter, "counter", torch.int32, 1, at_least=True)
    _need(status, "status", torch.int32, 1, at_least=True)
    _check("nvq_debug_count_timeout",
           lib.nvq_debug_count_timeout(max_polls, _ptr(counter), _ptr(status), _stream(stream)))


def debug_set_quant_lead(waves: int):
    """Sets the quantisers' look-ahead lead beyond one slice, in grid waves
    (see nvq_debug_set_quant_lead); outputs do not depend on it."""
    _check("nvq_debug_set_quant_lead", lib.nvq_debug_set_quant_lead(int(waves)))


def nvfp4_dgrad(dy, counts, codes, scales, tensor_scale, status=None, stream=None, out=None):
    """dX = dY . DQ(Q(W_e)) for the tokens routed to each expert (see
    nvfp4_dgrad in nvq.h).  dy bf16 [T, out_dim] grouped by expert; counts:
    tokens per expert (host sequence); codes/scales/tensor_scale: the
    rowwise NVFP4 copy of the [nexp, out_dim, in_dim] stack.  Returns FP32
    dX [T, in_dim]."""
    E, R, K = _dequant_inputs(codes, scales, tensor_scale)
    if len(counts) != E:
        raise ValueError("counts must give one token count per expert (%d)" % E)
    cnt = (C.c_int64 * E)(*[int(c) for c in counts])
    T = sum(int(c) for c in counts)
    _need(dy, "dy", torch.bfloat16, shape=(T, R))
    dst = out if out is not None else _empty((T, K), torch.float32, codes)
    _need(dst, "out", torch.float32, shape=(T, K))
    _status(status)
    _check("nvfp4_dgrad", lib.nvfp4_dgrad(_ptr(_bf16(dy, "dy")), C.cast(cnt, C.c_void_p), E, R, K,
                                          _ptr(codes),
                                          _ptr(scales), _ptr(tensor_scale), _ptr(dst),
                                          _ptr(status), _stream(stream)))
    return dst


def nf4_routed_linear(x, counts, codes, absmax, status=None, stream=None, out=None):
    """Y = X . DQ(W_e)^T for the tokens routed to each expert (see
    nf4_routed_linear in nvq.h).  x bf16 [T, in_dim] grouped by expert;
    counts: tokens per expert (host sequence); codes/absmax: the NF4 copy of
    the [nexp, out_dim, in_dim] stack.  Returns bf16 Y [T, out_dim]."""
    E, R, K = _nf4_inputs(codes, absmax)
    if len(counts) != E:
        raise ValueError("counts must give one token count per expert (%d)" % E)
    cnt = (C.c_int64 * E)(*[int(c) for c in counts])
    T = sum(int(c) for c in counts)
    _need(x, "x", torch.bfloat16, shape=(T, K))
    dst = out if out is not None else _empty((T, R), torch.bfloat16, codes)
    _need(dst, "out", torch.bfloat16, shape=(T, R))
    _status(status)
    _check("nf4_routed_linear", lib.nf4_routed_linear(_ptr(_bf16(x, "x")), C.cast(cnt, C.c_void_p),
                                                      E, R, K, _ptr(codes), _ptr(absmax), _ptr(dst),
                                                      _ptr(status), _stream(stream)))
    return dst


# ---------------------------------------------------------------- MXFP8

def mx_scale_bytes(rows, cols, swizzled=False):
    """Bytes of the MXFP8 block scales of one [rows, cols] slice (see
    nvq_mx_scale_bytes in nvq.h)."""
    n = lib.nvq_mx_scale_bytes(rows, cols, FLAG_SCALES_SWIZZLED if swizzled else 0)
    if n < 0:
        raise ValueError("invalid MXFP8 scale shape [%d, %d]" % (rows, cols))
    return n


def mxfp8_quantize(w, columnwise=False, swizzled_scales=False, status=None, stream=None, out=None):
    """MXFP8 of w [nexp, rows, cols] (bf16): codes_row [nexp, rows, cols] u8
    (E4M3), scales_row [nexp, rows, cols/32] u8 (E8M0) and, with columnwise,
    codes_col [nexp, cols, rows] / scales_col [nexp, cols, rows/32] from the
    same read.  With swizzled_scales the scales are [nexp, bytes] in the
    tensor-core tiled layout."""
    w = _as3d(_bf16(w, "w"))
    E, R, K = w.shape
    o = out or {}

    def sc(rows, cols):
        if swizzled_scales:
            return _empty((E, mx_scale_bytes(rows, cols, True)), torch.uint8, w)
        return _empty((E, rows, cols // 32), torch.uint8, w)
    cr = o.get("codes_row", _empty((E, R, K), torch.uint8, w))
    sr = o.get("scales_row") if "scales_row" in o else sc(R, K)
    cc = sco = None
    if columnwise:
        cc = o.get("codes_col", _empty((E, K, R), torch.uint8, w))
        sco = o.get("scales_col") if "scales_col" in o else sc(K, R)
    if K % 32 == 0:
        def sc_numel(rows, cols):
            return E * (mx_scale_bytes(rows, cols, True) if swizzled_scales else rows * (cols // 32))
        _need(cr, "codes_row", torch.uint8, E * R * K)
        _need(sr, "scales_row", torch.uint8, sc_numel(R, K))
        if columnwise and R % 32 == 0:
            _need(cc, "codes_col", torch.uint8, E * K * R)
            _need(sco, "scales_col", torch.uint8, sc_numel(K, R))
    _status(status)
    flags = FLAG_SCALES_SWIZZLED if swizzled_scales else 0
    _check("mxfp8_quantize", lib.mxfp8_quantize(_ptr(w), E, R, K, flags, _ptr(cr), _ptr(sr), _ptr(cc),
                                                _ptr(sco), _ptr(status), _stream(stream)))
    r = dict(codes_row=cr, scales_row=sr)
    if columnwise:
        r.update(codes_col=cc, scales_col=sco)
    return r


def mxfp8_dequant(codes, scales, stream=None, out=None):
    """bf16 of MXFP8 codes (any shape whose last dimension holds whole blocks
    of 32) with their linear scales."""
    _need(codes, "codes", torch.uint8)
    _need(scales, "scales", torch.uint8, codes.numel() // 32)
    dst = out if out is not None else _empty(tuple(codes.shape), torch.bfloat16, codes)
    _need(dst, "out", torch.bfloat16, codes.numel())
    _check("mxfp8_dequant", lib.mxfp8_dequant(_ptr(codes), _ptr(scales), codes.numel(), _ptr(dst),
                                              _stream(stream)))
    return dst
