"""CPU oracle for block-scaled 4-bit quantisation -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library never
imports it; it shares no code with the CUDA path.

The arithmetic lives in ``nvq_oracle.c`` (plain C, one thread, binary32 with
contraction off).  This module compiles it with gcc and wraps it for numpy
arrays.  Every function cites the source passage it restates in the C file.

Parity status: all functions are pinned by host tests; the NF4 level table
is pinned to the NF4 values printed in the QLoRA paper.  The nested absmax
follows the
published double quantisation with the readings stated in the C file; its
equality with any third-party nested code (whose 8-bit table differs) is not
claimed.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvq_oracle.c")
_LIB = os.path.join(_HERE, "libnvq_oracle.so")
_lock = threading.Lock()
_lib = None

FLAG_4OVER6 = 1
FLAG_AMAX_GIVEN = 2
STATUS_NONFINITE = 1
STATUS_BAD_INDEX = 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = C.CDLL(_LIB)
            P = C.c_void_p
            i64 = C.c_int64
            u32 = C.c_uint32
            lib.oracle_bf16_to_f32.restype = C.c_float
            lib.oracle_bf16_to_f32.argtypes = [C.c_uint16]
            lib.oracle_f32_to_bf16.restype = C.c_uint16
            lib.oracle_f32_to_bf16.argtypes = [C.c_float]
            lib.oracle_e4m3_value.restype = C.c_float
            lib.oracle_e4m3_value.argtypes = [C.c_uint8]
            lib.oracle_e4m3_encode.restype = C.c_uint8
            lib.oracle_e4m3_encode.argtypes = [C.c_float]
            lib.oracle_e2m1_value.restype = C.c_float
            lib.oracle_e2m1_value.argtypes = [C.c_uint8]
            lib.oracle_e2m1_encode.restype = C.c_uint8
            lib.oracle_e2m1_encode.argtypes = [C.c_float]
            lib.oracle_tensor_scales.restype = None
            lib.oracle_tensor_scales.argtypes = [C.c_float, C.c_int, P, P]
            lib.oracle_nvfp4_block.restype = None
            lib.oracle_nvfp4_block.argtypes = [P, i64, C.c_float, C.c_int, P, P, P, P]
            lib.oracle_amax_bf16.restype = C.c_float
            lib.oracle_amax_bf16.argtypes = [P, i64]
            for name in ("oracle_nvfp4_quantize", "oracle_nvfp4_quantize_colwise"):
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = [P, i64, i64, i64, u32, P, P, P, P, P]
            for name in ("oracle_nvfp4_dequant", "oracle_nvfp4_dequant_t"):
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = [P, P, P, i64, i64, i64, P]
            lib.oracle_act_quantize_per_token.restype = None
            lib.oracle_act_quantize_per_token.argtypes = [P, i64, i64, u32, P, P, P, P]
            for name in ("oracle_e4m3_encode_n", "oracle_e2m1_encode_n", "oracle_f32_to_bf16_n"):
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = [P, P, i64]
            lib.oracle_nf4_codebook.restype = None
            lib.oracle_nf4_codebook.argtypes = [P]
            lib.oracle_nf4_quantize.restype = None
            lib.oracle_nf4_quantize.argtypes = [P, i64, i64, i64, P, P, P]
            lib.oracle_nf4_dequant.restype = None
            lib.oracle_nf4_dequant.argtypes = [P, P, i64, i64, i64, P]
            lib.oracle_routed_union.restype = None
            lib.oracle_routed_union.argtypes = [P, i64, i64, i64, P, P, P]
            lib.oracle_mxfp8_block.restype = C.c_uint8
            lib.oracle_mxfp8_block.argtypes = [P, i64, P]
            for name in ("oracle_mxfp8_quantize", "oracle_mxfp8_quantize_colwise"):
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = [P, i64, i64, i64, P, P]
            lib.oracle_mxfp8_dequant.restype = None
            lib.oracle_mxfp8_dequant.argtypes = [P, P, i64, P]
            lib.oracle_tree_sum.restype = C.c_float
            lib.oracle_tree_sum.argtypes = [P, i64]
            lib.oracle_absmax_mean.restype = C.c_float
            lib.oracle_absmax_mean.argtypes = [P, i64]
            lib.oracle_nf4_absmax_nest.restype = None
            lib.oracle_nf4_absmax_nest.argtypes = [P, i64, i64, P, P, P]
            lib.oracle_nf4_absmax_unnest.restype = None
            lib.oracle_nf4_absmax_unnest.argtypes = [P, P, P, i64, i64, P]
            lib.oracle_nf4_dequant_routed.restype = None
            lib.oracle_nf4_dequant_routed.argtypes = [P, P, i64, i64, i64, P, i64, i64, P, P, P, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


def _u16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return x


# --- scalar formats --------------------------------------------------------

def bf16_to_f32(h: int) -> float:
    return _load().oracle_bf16_to_f32(int(h))


def f32_to_bf16(x: float) -> int:
    return int(_load().oracle_f32_to_bf16(float(x)))


def e4m3_value(c: int) -> float:
    return _load().oracle_e4m3_value(int(c))


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def e2m1_value(c: int) -> float:
    return _load().oracle_e2m1_value(int(c))


def e2m1_encode(x: float) -> int:
    return int(_load().oracle_e2m1_encode(float(x)))


def f32_to_bf16_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.zeros(x.size, np.uint16)
    _load().oracle_f32_to_bf16_n(_p(x), _p(out), x.size)
    return out


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.zeros(x.size, np.uint8)
    _load().oracle_e4m3_encode_n(_p(x), _p(out), x.size)
    return out


def e2m1_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.zeros(x.size, np.uint8)
    _load().oracle_e2m1_encode_n(_p(x), _p(out), x.size)
    return out


def tensor_scales(amax: float, four_over_six: bool):
    G = C.c_float()
    E = C.c_float()
    _load().oracle_tensor_scales(float(amax), int(bool(four_over_six)), C.byref(G), C.byref(E))
    return G.value, E.value


def nvfp4_block(x16: np.ndarray, E: float, four_over_six: bool, stride: int = 1):
    """One block: returns (scale_byte, codes[16], sse6, sse4)."""
    x16 = _u16(x16)
    s = C.c_uint8()
    codes = np.zeros(16, dtype=np.uint8)
    e6 = C.c_float()
    e4 = C.c_float()
    _load().oracle_nvfp4_block(_p(x16), int(stride), float(E), int(bool(four_over_six)),
                               C.byref(s), _p(codes), C.byref(e6), C.byref(e4))
    return int(s.value), codes, e6.value, e4.value


def amax_bf16(x: np.ndarray) -> float:
    x = _u16(x)
    return _load().oracle_amax_bf16(_p(x), x.size)


# --- tensor-level NVFP4 -----------------------------------------------------

def _flags(four_over_six: bool, amax_given: bool) -> int:
    return (FLAG_4OVER6 if four_over_six else 0) | (FLAG_AMAX_GIVEN if amax_given else 0)


def nvfp4_quantize(w: np.ndarray, four_over_six: bool = False, amax: np.ndarray | None = None):
    """Rowwise NVFP4 of w [nexp, rows, cols] (uint16 bf16 bits).

    Returns dict(codes, scales, amax, G, status)."""
    w = _u16(w)
    nexp, rows, cols = w.shape
    codes = np.zeros((nexp, rows, cols // 2), np.uint8)
    scales = np.zeros((nexp, rows, cols // 16), np.uint8)
    am = np.zeros(nexp, np.float32) if amax is None else np.array(amax, np.float32).copy()
    G = np.zeros(nexp, np.float32)
    st = C.c_int(0)
    _load().oracle_nvfp4_quantize(_p(w), nexp, rows, cols, _flags(four_over_six, amax is not None),
                                  _p(codes), _p(scales), _p(am), _p(G), C.byref(st))
    return dict(codes=codes, scales=scales, amax=am, G=G, status=st.value)


def nvfp4_quantize_colwise(w: np.ndarray, four_over_six: bool = False,
                           amax: np.ndarray | None = None):
    """Columnwise NVFP4 of w [nexp, rows, cols]; outputs are [nexp, cols, rows/2|rows/16]."""
    w = _u16(w)
    nexp, rows, cols = w.shape
    codes = np.zeros((nexp, cols, rows // 2), np.uint8)
    scales = np.zeros((nexp, cols, rows // 16), np.uint8)
    am = np.zeros(nexp, np.float32) if amax is None else np.array(amax, np.float32).copy()
    G = np.zeros(nexp, np.float32)
    st = C.c_int(0)
    _load().oracle_nvfp4_quantize_colwise(_p(w), nexp, rows, cols,
                                          _flags(four_over_six, amax is not None),
                                          _p(codes), _p(scales), _p(am), _p(G), C.byref(st))
    return dict(codes=codes, scales=scales, amax=am, G=G, status=st.value)


def nvfp4_dequant(codes: np.ndarray, scales: np.ndarray, G: np.ndarray, rows: int, cols: int):
    nexp = G.size
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    G = np.ascontiguousarray(G, np.float32)
    dst = np.zeros((nexp, rows, cols), np.uint16)
    _load().oracle_nvfp4_dequant(_p(codes), _p(scales), _p(G), nexp, rows, cols, _p(dst))
    return dst


def nvfp4_dequant_t(codes: np.ndarray, scales: np.ndarray, G: np.ndarray, rows: int, cols: int):
    nexp = G.size
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    G = np.ascontiguousarray(G, np.float32)
    dst = np.zeros((nexp, cols, rows), np.uint16)
    _load().oracle_nvfp4_dequant_t(_p(codes), _p(scales), _p(G), nexp, rows, cols, _p(dst))
    return dst


def act_quantize_per_token(x: np.ndarray, four_over_six: bool = True):
    x = _u16(x)
    T, H = x.shape
    codes = np.zeros((T, H // 2), np.uint8)
    scales = np.zeros((T, H // 16), np.uint8)
    ts = np.zeros(T, np.float32)
    st = C.c_int(0)
    _load().oracle_act_quantize_per_token(_p(x), T, H, _flags(four_over_six, False),
                                          _p(codes), _p(scales), _p(ts), C.byref(st))
    return dict(codes=codes, scales=scales, token_scale=ts, status=st.value)


# --- NF4 ----------------------------------------------------------------------

def nf4_codebook() -> np.ndarray:
    cb = np.zeros(16, np.float32)
    _load().oracle_nf4_codebook(_p(cb))
    return cb


def nf4_quantize(w: np.ndarray):
    w = _u16(w)
    nexp, rows, cols = w.shape
    codes = np.zeros((nexp, rows, cols // 2), np.uint8)
    absmax = np.zeros((nexp, rows, cols // 64), np.float32)
    st = C.c_int(0)
    _load().oracle_nf4_quantize(_p(w), nexp, rows, cols, _p(codes), _p(absmax), C.byref(st))
    return dict(codes=codes, absmax=absmax, status=st.value)


def nf4_dequant(codes: np.ndarray, absmax: np.ndarray, nexp: int, rows: int, cols: int):
    codes = np.ascontiguousarray(codes, np.uint8)
    absmax = np.ascontiguousarray(absmax, np.float32)
    dst = np.zeros((nexp, rows, cols), np.uint16)
    _load().oracle_nf4_dequant(_p(codes), _p(absmax), nexp, rows, cols, _p(dst))
    return dst


def routed_union(topk: np.ndarray, nexp: int):
    topk = np.ascontiguousarray(topk, np.int32)
    T, k = topk.shape
    hit = np.zeros(nexp, np.int32)
    n = C.c_int32(0)
    st = C.c_int(0)
    _load().oracle_routed_union(_p(topk), T, k, nexp, _p(hit), C.byref(n), C.byref(st))
    return hit, n.value, st.value


def nf4_dequant_routed(codes: np.ndarray, absmax: np.ndarray, nexp: int, rows: int, cols: int,
                       topk: np.ndarray, dst: np.ndarray):
    """Dequantises the routed experts into dst (modified in place)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    absmax = np.ascontiguousarray(absmax, np.float32)
    topk = np.ascontiguousarray(topk, np.int32)
    assert dst.dtype == np.uint16 and dst.flags.c_contiguous and dst.shape == (nexp, rows, cols)
    T, k = topk.shape
    hit = np.zeros(nexp, np.int32)
    n = C.c_int32(0)
    st = C.c_int(0)
    _load().oracle_nf4_dequant_routed(_p(codes), _p(absmax), nexp, rows, cols, _p(topk), T, k,
                                      _p(dst), _p(hit), C.byref(n), C.byref(st))
    return hit, n.value, st.value


# --- dgrad through the dequantised weight ------------------------------------

def _bf16_to_f64(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: a bf16 is the top half of an f32)."""
    h = np.ascontiguousarray(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def nvfp4_dgrad(dy: np.ndarray, counts, codes: np.ndarray, scales: np.ndarray, G: np.ndarray,
                out: int, inn: int):
    """dX = dY . DQ(Q(W_e)) for each expert e, in float64.

    The backward of y = x . DQ(Q(w)) reads the weight through its dequantised
    bf16 values ("The 4-bitter Lesson", "Key claims": dequantised backward;
    "Getting GLM-5.2 NVFP4 Post-Training off the ground", "The bottom line":
    the rowwise copy dequantised to bf16 for dgrad).  dy: bf16 bits
    [sum(counts), out], token rows grouped by expert in expert order; codes /
    scales / G: the rowwise NVFP4 copy of the [nexp, out, in] stack.  The
    weight values are the oracle's own bf16 dequantisation; the contraction
    is one float64 matrix product per expert (a library primitive).  Returns
    (dx, bound): dx [T, in] float64 and bound = |dY| . |DQ(Q(W))|, the scale
    of the rounding error of any float32 evaluation of the same sums."""
    dy = np.ascontiguousarray(dy, np.uint16)
    counts = [int(c) for c in counts]
    dx = np.zeros((dy.shape[0], inn), np.float64)
    bound = np.zeros_like(dx)
    t0 = 0
    for e, c in enumerate(counts):
        if c:
            w = _bf16_to_f64(nvfp4_dequant(codes[e:e + 1], scales[e:e + 1], G[e:e + 1], out, inn)[0])
            a = _bf16_to_f64(dy[t0:t0 + c])
            dx[t0:t0 + c] = a @ w
            bound[t0:t0 + c] = np.abs(a) @ np.abs(w)
        t0 += c
    return dx, bound


def nf4_routed_linear(x: np.ndarray, counts, codes: np.ndarray, absmax: np.ndarray, out: int,
                      inn: int):
    """Y = X . DQ(W_e)^T for each expert e, in float64.

    The forward of a routed expert stored as NF4 dequantises its weight to
    bf16 and applies it to the tokens sent to it ("nf4moe -- QLoRA for a 743B
    Fused-MoE", "The fix: dequant-on-forward for routed experts": F.linear(x,
    W[e]) on the dequantised W[e]).  x: bf16 bits [sum(counts), in], token
    rows grouped by expert in expert order; codes / absmax: the NF4 copy of
    the [nexp, out, in] stack.  The weight values are the oracle's own bf16
    dequantisation; the contraction is one float64 matrix product per expert
    (a library primitive).  Returns (y, bound): y [T, out] float64, exact up
    to float64 rounding, and bound = |X| . |DQ(W)|^T, the scale of the
    rounding error of any float32 evaluation of the same sums."""
    x = np.ascontiguousarray(x, np.uint16)
    counts = [int(c) for c in counts]
    y = np.zeros((x.shape[0], out), np.float64)
    bound = np.zeros_like(y)
    t0 = 0
    for e, c in enumerate(counts):
        if c:
            w = _bf16_to_f64(nf4_dequant(codes[e:e + 1], absmax[e:e + 1], 1, out, inn)[0])
            a = _bf16_to_f64(x[t0:t0 + c])
            y[t0:t0 + c] = a @ w.T
            bound[t0:t0 + c] = np.abs(a) @ np.abs(w).T
        t0 += c
    return y, bound


def scales_tiled(scales: np.ndarray) -> np.ndarray:
    """Block scales [..., R, C] (linear: row r, block column c) -> [..., Rp * Cp]
    in the tensor-core tiled layout the block-scaled FP4 GEMM reads ("Getting
    GLM-5.2 NVFP4 Post-Training off the ground", "Why can't we just transpose
    the one copy?": the scales are swizzled for the tensor-core tile; the
    pages do not spell the layout out, so this is the published layout of
    the FP4 GEMM's scale operand).  Rp = R rounded up to 128, Cp = C rounded
    up to 4; tiles of 128 rows x 4 block columns, 512 bytes each, row-major
    over tiles; inside a tile scale (r, c) at byte (r % 32) * 16 +
    ((r // 32) % 4) * 4 + c % 4; padding 0.  Parity: pinned on the GPU by
    the FP4 GEMM that consumes the layout; on the host only its bijection,
    tile grouping and padding are checked."""
    scales = np.ascontiguousarray(scales, np.uint8)
    *lead, R, C = scales.shape
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    off = ((r // 128) * (Cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
    out = np.zeros(tuple(lead) + (Rp * Cp,), np.uint8)
    out[..., off] = scales
    return out


def nvfp4_block_values(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """c * S of every element, float64 and exact (an E2M1 value times an E4M3
    value has at most six significant bits): the operand values of a
    block-scaled FP4 product before any FP32 tensor or token scale.
    codes [..., R, K/2] (element 2j in the low nibble of byte j), scales
    [..., R, K/16] linear."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    e2 = np.array([e2m1_value(c) for c in range(16)], np.float64)
    e4 = np.array([e4m3_value(c) for c in range(256)], np.float64)
    nib = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    nib[..., 0::2] = codes & 0xF
    nib[..., 1::2] = codes >> 4
    return e2[nib] * np.repeat(e4[scales], 16, axis=-1)


def nvfp4_scaled_product(a_codes, a_scales, b_codes, b_scales):
    """Y[m, n] = sum_k (c S)_a[m, k] (c S)_b[n, k] in float64 -- the product a
    block-scaled FP4 GEMM forms from two NVFP4 operands with K-major codes --
    and bound = sum_k |(c S)_a (c S)_b|."""
    va = nvfp4_block_values(a_codes, a_scales)
    vb = nvfp4_block_values(b_codes, b_scales)
    return va @ vb.T, np.abs(va) @ np.abs(vb).T


def mxfp8_block(x32: np.ndarray):
    """One MXFP8 block of 32 bf16 values: (scale byte, codes [32])."""
    x = np.ascontiguousarray(x32, np.uint16)
    codes = np.zeros(32, np.uint8)
    s = _load().oracle_mxfp8_block(_p(x), 1, _p(codes))
    return int(s), codes


def mxfp8_quantize(w: np.ndarray):
    """MXFP8 of w [nexp, rows, cols] with 1x32 blocks along cols (OCP MX:
    E8M0 scale per block, E4M3 elements; "The 4-bitter Lesson", "Key
    claims": the MXFP8 validation of the dequantised backward).  Returns
    codes [nexp, rows, cols] and scales [nexp, rows, cols/32]."""
    w = _u16(w)
    nexp, rows, cols = w.shape
    codes = np.zeros((nexp, rows, cols), np.uint8)
    scales = np.zeros((nexp, rows, cols // 32), np.uint8)
    _load().oracle_mxfp8_quantize(_p(w), nexp, rows, cols, _p(codes), _p(scales))
    return dict(codes=codes, scales=scales)


def mxfp8_quantize_colwise(w: np.ndarray):
    """MXFP8 with 32x1 blocks along rows, stored transposed: codes
    [nexp, cols, rows], scales [nexp, cols, rows/32]."""
    w = _u16(w)
    nexp, rows, cols = w.shape
    codes = np.zeros((nexp, cols, rows), np.uint8)
    scales = np.zeros((nexp, cols, rows // 32), np.uint8)
    _load().oracle_mxfp8_quantize_colwise(_p(w), nexp, rows, cols, _p(codes), _p(scales))
    return dict(codes=codes, scales=scales)


def mxfp8_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """bf16 bits of E4M3 value x 2^(scale - 127), in the layout of the codes."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    dst = np.zeros(codes.shape, np.uint16)
    _load().oracle_mxfp8_dequant(_p(codes), _p(scales), codes.size, _p(dst))
    return dst


def mxfp8_values(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E4M3 value x 2^(scale - 127) of every element, float64 and exact;
    codes [..., K] with linear scales [..., K/32]."""
    e4 = np.array([e4m3_value(c) for c in range(256)], np.float64)
    sc = np.ldexp(1.0, np.asarray(scales, np.int64) - 127)
    return e4[np.asarray(codes, np.uint8)] * np.repeat(sc, 32, axis=-1)


def tree_sum(a: np.ndarray) -> np.float32:
    """Pairwise tree sum in binary32, zero padded to a power of two."""
    a = np.ascontiguousarray(a, dtype=np.float32).ravel()
    return np.float32(_load().oracle_tree_sum(_p(a), a.size))


def absmax_mean(a: np.ndarray) -> np.float32:
    a = np.ascontiguousarray(a, dtype=np.float32).ravel()
    return np.float32(_load().oracle_absmax_mean(_p(a), a.size))


def nf4_absmax_nest(absmax: np.ndarray):
    """Nested (double-quantised) absmax of each expert slice: absmax [nexp, ...]
    (FP32) -> codes [nexp, n] (E4M3 bytes), c1 [nexp, ceil(n/256)], mean [nexp]."""
    a = np.ascontiguousarray(absmax, dtype=np.float32)
    E = a.shape[0]
    n = a.size // E if E else 0
    nb = (n + 255) // 256
    codes = np.zeros((E, n), np.uint8)
    c1 = np.zeros((E, nb), np.float32)
    mean = np.zeros(E, np.float32)
    _load().oracle_nf4_absmax_nest(_p(a), E, n, _p(codes), _p(c1), _p(mean))
    return dict(codes=codes, c1=c1, mean=mean)


def nf4_absmax_unnest(codes: np.ndarray, c1: np.ndarray, mean: np.ndarray) -> np.ndarray:
    """FP32 absmax [nexp, n] decoded from the nested form."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    c1 = np.ascontiguousarray(c1, dtype=np.float32)
    mean = np.ascontiguousarray(mean, dtype=np.float32)
    E = codes.shape[0]
    n = codes.size // E if E else 0
    out = np.zeros((E, n), np.float32)
    _load().oracle_nf4_absmax_unnest(_p(codes), _p(c1), _p(mean), E, n, _p(out))
    return out
