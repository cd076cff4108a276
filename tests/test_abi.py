"""Host-side checks of the C ABI: the library loads, exports every function
include/nvq.h declares, validates arguments before touching the GPU, and
carries the same NF4 level table as the oracle.  No kernel is launched."""
import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvq.h")


@pytest.fixture(scope="module")
def nvq():
    import __graft_entry__
    __graft_entry__.build()
    import rl_nvfp4_quantize_gb300 as m
    return m


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^NVQ_API\s+[\w\s\*]+?\b(\w+)\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("nvfp4_quantize", "nvfp4_quantize_dual", "nvfp4_dequant_t", "act_quantize_per_token",
              "nf4_quantize", "nf4_dequant_routed"):
        assert n in names


def test_library_exports_every_declared_symbol(nvq):
    lib = C.CDLL(nvq.library_path)
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_version_and_strings(nvq):
    assert nvq.lib.nvq_version() >> 16 == 1
    for code in range(7):
        assert nvq.lib.nvq_status_string(code)
    assert b"unknown" in nvq.lib.nvq_status_string(99)


def test_nf4_table_matches_oracle(nvq, oracle_mod):
    got = nvq.nf4_codebook().numpy()
    ref = oracle_mod.nf4_codebook()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_nf4_cell_design_holds_for_the_table(oracle_mod):
    """The kernel's one-comparison NF4 encoder puts v in the cell numbered by
    bits 17..22 of g = fl(16 v + 96); it needs every midpoint of the level
    table in a cell of its own (g never decreases with v, so cells are
    ordered intervals)."""
    cb = oracle_mod.nf4_codebook()
    m = ((cb[:-1] + cb[1:]) * np.float32(0.5)).astype(np.float32)
    g = (m * np.float32(16.0) + np.float32(96.0)).astype(np.float32)  # 16 m exact, one rounding
    cells = (g.view(np.uint32) >> 17) & 63
    assert len(set(cells.tolist())) == 15
    assert np.all(np.diff(cells.astype(np.int64)) > 0)
    # the cell index is an ordered function of v over [-1, 1]
    v = np.linspace(-1.0, 1.0, 200001).astype(np.float32)
    gv = (v * np.float32(16.0) + np.float32(96.0)).astype(np.float32)
    cv = (gv.view(np.uint32) >> 17) & 63
    assert np.all(np.diff(cv.astype(np.int64)) >= 0)


P = None


def _vp(v):
    return C.c_void_p(v)


FAKE = 0x10000  # an aligned, never dereferenced address


def test_validation_before_any_device_work(nvq):
    L = nvq.lib
    ok16 = _vp(FAKE)
    # unknown flag bits
    assert L.nvfp4_quantize(ok16, 1, 16, 16, 0x80, ok16, ok16, ok16, ok16, P, P) == 4
    # shape rules
    assert L.nvfp4_quantize(ok16, 1, 16, 24, 0, ok16, ok16, ok16, ok16, P, P) == 3
    assert L.nvfp4_quantize_dual(ok16, 1, 24, 16, 0, ok16, ok16, ok16, ok16, ok16, ok16, P, P) == 3
    assert L.nvfp4_quantize(ok16, -1, 16, 16, 0, ok16, ok16, ok16, ok16, P, P) == 3
    assert L.nf4_quantize(ok16, 1, 4, 32, ok16, ok16, P, P) == 3
    assert L.nvfp4_quantize(ok16, 1 << 40, 1 << 20, 1 << 20, 0, ok16, ok16, ok16, ok16, P, P) == 3
    assert L.act_quantize_per_token(ok16, 4, 24, 0, ok16, ok16, ok16, P, P) == 3
    assert L.act_quantize_per_token(ok16, 4, 32, 2, ok16, ok16, ok16, P, P) == 4  # amax-given not allowed
    assert L.nf4_dequant_routed(ok16, ok16, 70000, 4, 64, ok16, 1, 1, ok16, ok16, ok16, P, P) == 3
    # null pointers
    assert L.nvfp4_quantize(P, 1, 16, 16, 0, ok16, ok16, ok16, ok16, P, P) == 1
    assert L.nvfp4_quantize_dual(ok16, 1, 16, 16, 0, ok16, ok16, P, ok16, ok16, ok16, P, P) == 1
    assert L.nvfp4_dequant_t(ok16, ok16, ok16, 1, 16, 16, P, P) == 1
    assert L.nf4_dequant_routed(ok16, ok16, 4, 4, 64, P, 2, 2, ok16, ok16, ok16, P, P) == 1
    assert L.nf4_dequant_routed(ok16, ok16, 4, 4, 64, ok16, 2, 2, ok16, ok16, P, P, P) == 1
    assert L.nvq_nf4_codebook(P) == 1
    # alignment
    mis = _vp(FAKE + 8)
    assert L.nvfp4_quantize(mis, 1, 16, 16, 0, ok16, ok16, ok16, ok16, P, P) == 2
    assert L.nvfp4_dequant(ok16, ok16, _vp(FAKE + 2), 1, 16, 16, ok16, P) == 2
    assert L.nf4_quantize(ok16, 1, 4, 64, ok16, mis, P, P) == 2
    # empty problems succeed without a device
    assert L.nvfp4_quantize(P, 0, 16, 16, 0, P, P, P, P, P, P) == 0
    assert L.nvfp4_dequant(P, P, P, 3, 0, 16, P, P) == 0
    assert L.nf4_quantize(P, 2, 0, 64, P, P, P, P) == 0
    assert L.nvq_debug_convert(9, ok16, ok16, 4, P) == 4
    cnt = (C.c_int64 * 2)(3, 4)
    cntp = C.cast(cnt, C.c_void_p)
    assert L.nvfp4_dgrad(ok16, cntp, 2, 64, 200, ok16, ok16, ok16, ok16, P, P) == 3   # in % 256
    assert L.nvfp4_dgrad(ok16, cntp, 2, 96, 256, ok16, ok16, ok16, ok16, P, P) == 3   # out % 64
    assert L.nvfp4_dgrad(ok16, cntp, 300, 64, 256, ok16, ok16, ok16, ok16, P, P) == 3  # > 256 experts
    assert L.nvfp4_dgrad(ok16, P, 2, 64, 256, ok16, ok16, ok16, ok16, P, P) == 1
    assert L.nvfp4_dgrad(ok16, cntp, 2, 64, 256, ok16, ok16, ok16, P, P, P) == 1
    assert L.nvfp4_dgrad(mis, cntp, 2, 64, 256, ok16, ok16, ok16, ok16, P, P) == 2
    neg = (C.c_int64 * 2)(3, -1)
    assert L.nvfp4_dgrad(ok16, C.cast(neg, C.c_void_p), 2, 64, 256, ok16, ok16, ok16, ok16, P, P) == 3
    zero = (C.c_int64 * 2)(0, 0)
    assert L.nvfp4_dgrad(P, C.cast(zero, C.c_void_p), 2, 64, 256, P, P, P, P, P, P) == 0
    assert L.nf4_routed_linear(ok16, cntp, 2, 200, 64, ok16, ok16, ok16, P, P) == 3   # out % 256
    assert L.nf4_routed_linear(ok16, cntp, 2, 256, 192, ok16, ok16, ok16, P, P) == 3  # in % 256
    assert L.nf4_routed_linear(ok16, cntp, 300, 256, 256, ok16, ok16, ok16, P, P) == 3  # > 256 experts
    assert L.nf4_routed_linear(ok16, C.cast(neg, C.c_void_p), 2, 256, 256, ok16, ok16, ok16, P, P) == 3
    assert L.nf4_routed_linear(ok16, P, 2, 256, 256, ok16, ok16, ok16, P, P) == 1
    assert L.nf4_routed_linear(ok16, cntp, 2, 256, 256, ok16, ok16, P, P, P) == 1
    assert L.nf4_routed_linear(ok16, cntp, 2, 256, 256, P, ok16, ok16, P, P) == 1
    assert L.nf4_routed_linear(mis, cntp, 2, 256, 256, ok16, ok16, ok16, P, P) == 2
    assert L.nf4_routed_linear(ok16, cntp, 2, 256, 256, _vp(FAKE + 16), ok16, ok16, P, P) == 2  # codes % 32
    assert L.nf4_routed_linear(P, C.cast(zero, C.c_void_p), 2, 256, 256, P, P, P, P, P) == 0
    assert L.nvfp4_dgrad(P, cntp, 2, 0, 256, P, P, P, P, P, P) == 1   # out == 0 still needs dX
    L.nvq_scale_bytes.restype = C.c_int64
    L.nvq_scale_bytes.argtypes = [C.c_int64, C.c_int64, C.c_uint]
    assert L.nvq_scale_bytes(200, 80, 0) == 1000
    assert L.nvq_scale_bytes(200, 80, 4) == 256 * 8
    assert L.nvq_scale_bytes(4096, 6144, 4) == 4096 * 384
    assert L.nvq_scale_bytes(200, 72, 4) == -1 and L.nvq_scale_bytes(-1, 16, 0) == -1
    assert L.nvq_scale_bytes(16, 16, 8) == -1
    assert L.nvfp4_quantize(ok16, 1, 16, 16, 8, ok16, ok16, ok16, ok16, P, P) == 4
    assert L.act_quantize_per_token(ok16, 4, 16, 2, ok16, ok16, ok16, P, P) == 4   # amax-given: rowwise only
    L.nvq_mx_scale_bytes.restype = C.c_int64
    L.nvq_mx_scale_bytes.argtypes = [C.c_int64, C.c_int64, C.c_uint]
    assert L.nvq_mx_scale_bytes(200, 160, 0) == 1000
    assert L.nvq_mx_scale_bytes(200, 160, 4) == 256 * 8
    assert L.nvq_mx_scale_bytes(200, 48, 0) == -1
    assert L.mxfp8_quantize(ok16, 1, 32, 48, 0, ok16, ok16, P, P, P, P) == 3        # cols % 32
    assert L.mxfp8_quantize(ok16, 1, 48, 64, 0, ok16, ok16, ok16, ok16, P, P) == 3  # rows % 32 (dual)
    assert L.mxfp8_quantize(ok16, 1, 48, 64, 0, ok16, ok16, P, P, P, P) == 5 or \
        L.mxfp8_quantize(ok16, 1, 48, 64, 0, ok16, ok16, P, P, P, P) == 0          # rowwise: any rows
    assert L.mxfp8_quantize(ok16, 1, 32, 64, 8, ok16, ok16, P, P, P, P) == 4        # unknown flag
    assert L.mxfp8_quantize(ok16, 1, 32, 64, 0, ok16, ok16, ok16, P, P, P) == 1     # half a column copy
    assert L.mxfp8_quantize(mis, 1, 32, 64, 0, ok16, ok16, P, P, P, P) == 2
    assert L.mxfp8_quantize(P, 0, 32, 64, 0, P, P, P, P, P, P) == 0
    assert L.mxfp8_dequant(ok16, ok16, 48, ok16, P) == 3
    assert L.mxfp8_dequant(ok16, P, 64, ok16, P) == 1
    assert L.mxfp8_dequant(P, P, 0, P, P) == 0
    assert L.nvq_debug_wait_timeout(0, ok16, P) == 3
    assert L.nvq_debug_wait_timeout(1 << 20, ok16, P) == 3
    assert L.nvq_debug_wait_timeout(16, P, P) == 1
    assert L.nvq_debug_wait_timeout(16, _vp(FAKE + 2), P) == 2
    assert L.nvq_debug_count_timeout(0, ok16, ok16, P) == 3
    assert L.nvq_debug_count_timeout(1 << 20, ok16, ok16, P) == 3
    assert L.nvq_debug_count_timeout(16, P, ok16, P) == 1
    assert L.nvq_debug_count_timeout(16, ok16, P, P) == 1
    assert L.nvq_debug_count_timeout(16, _vp(FAKE + 2), ok16, P) == 2
    assert L.nvq_debug_set_quant_lead(1) == 3 and L.nvq_debug_set_quant_lead(9) == 3
    assert L.nvq_debug_set_quant_lead(2) == 0
    # nested NF4 absmax
    assert L.nf4_absmax_nest(ok16, 1, (1 << 25) + 1, ok16, ok16, ok16, P, P) == 3
    assert L.nf4_absmax_nest(ok16, -1, 8, ok16, ok16, ok16, P, P) == 3
    assert L.nf4_absmax_nest(ok16, 2, 8, ok16, ok16, P, P, P) == 1
    assert L.nf4_absmax_nest(P, 2, 8, ok16, ok16, ok16, P, P) == 1
    assert L.nf4_absmax_nest(ok16, 2, 8, ok16, _vp(FAKE + 2), ok16, P, P) == 2
    assert L.nf4_absmax_nest(P, 0, 8, P, P, P, P, P) == 0
    assert L.nf4_absmax_unnest(ok16, ok16, ok16, 2, 8, P, P) == 1
    assert L.nf4_absmax_unnest(ok16, ok16, _vp(FAKE + 1), 2, 8, ok16, P) == 2
    assert L.nf4_absmax_unnest(ok16, ok16, ok16, 2, -8, ok16, P) == 3
    assert L.nf4_absmax_unnest(P, P, P, 2, 0, P, P) == 0


def test_valid_call_without_gpu_reports_device(nvq):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ok16 = _vp(FAKE)
    assert nvq.lib.nvfp4_quantize(ok16, 1, 16, 16, 0, ok16, ok16, ok16, ok16, P, P) == 5
    assert nvq.lib.nf4_dequant_routed(ok16, ok16, 4, 4, 64, ok16, 2, 2, ok16, ok16, ok16, P, P) == 5
    assert nvq.lib.nf4_absmax_nest(ok16, 2, 8, ok16, ok16, ok16, P, P) == 5
    assert nvq.lib.nf4_absmax_unnest(ok16, ok16, ok16, 2, 8, ok16, P) == 5


_C_CONSUMER = r"""
#include <stddef.h>
#include "nvq.h"
int main(void) {
  /* validation paths only: no device work */
  if (nvq_version() >> 16 != 1) return 1;
  if (nvq_scale_bytes(128, 64, 0) != 128 * 4) return 2;
  if (nf4_absmax_unnest(NULL, NULL, NULL, 2, 0, NULL, NULL) != NVQ_OK) return 3;
  if (nvfp4_quantize(NULL, 1, 16, 24, 0, NULL, NULL, NULL, NULL, NULL, NULL) != NVQ_ERR_SHAPE)
    return 4;
  return 0;
}
"""


def test_header_is_plain_c_and_links(nvq, tmp_path):
    """include/nvq.h compiles as C99 (-pedantic) and a C program links and
    calls the library through it."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consumer.c"
    src.write_text(_C_CONSUMER)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(nvq.library_path)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-l:libnvq.so", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, "C consumer failed with %d" % r.returncode


def test_binding_refuses_host_tensors(nvq):
    """Every tensor the binding hands to the library must be a contiguous CUDA
    tensor; host tensors are refused before any call (no device needed)."""
    import torch
    codes = torch.zeros((2, 8), dtype=torch.uint8)
    c1 = torch.zeros((2, 1), dtype=torch.float32)
    mean = torch.zeros(2, dtype=torch.float32)
    with pytest.raises(TypeError):
        nvq.nf4_absmax_unnest(codes, c1, mean)
    with pytest.raises(TypeError):
        nvq.nf4_absmax_nest(torch.ones((2, 8), dtype=torch.float32))
    with pytest.raises(TypeError):
        nvq.nvfp4_dequant(torch.zeros((1, 16, 8), dtype=torch.uint8),
                          torch.zeros((1, 16, 1), dtype=torch.uint8), torch.ones(1))
    with pytest.raises(TypeError):
        nvq.nvfp4_quantize(torch.zeros((1, 16, 16), dtype=torch.bfloat16))


def test_binding_refuses_mis_sized_buffers(nvq):
    """The C ABI sees addresses only, so the binding checks the element type
    and size of every buffer a call touches and raises before the call: a
    short or mistyped out= buffer, scales, tensor_scale or absmax would
    otherwise be read or written past its end on the GPU.  Host tensors of
    the right size reach the host-tensor check instead (TypeError)."""
    import torch
    u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
    w = torch.zeros((2, 32, 64), dtype=bf)
    # nvfp4_quantize(_dual): short codes / scales / amax / tensor_scale
    for bad in (dict(codes=torch.zeros((2, 32, 31), dtype=u8)),
                dict(scales=torch.zeros((2, 32, 3), dtype=u8)),
                dict(tensor_scale=torch.zeros(1, dtype=f32)),
                dict(amax=torch.zeros(2, dtype=torch.float64))):
        with pytest.raises((ValueError, TypeError)) as ei:
            nvq.nvfp4_quantize(w, out=bad)
        assert "expected a contiguous CUDA tensor" not in str(ei.value)
    with pytest.raises(ValueError):
        nvq.nvfp4_quantize_dual(w, out=dict(codes_col=torch.zeros((2, 64, 15), dtype=u8)))
    with pytest.raises(ValueError):
        nvq.nvfp4_quantize_dual(w, out=dict(scales_col=torch.zeros((2, 64, 1), dtype=u8)))
    with pytest.raises(ValueError):  # tiled scales need nvq_scale_bytes bytes per slice
        nvq.nvfp4_quantize(w, swizzled_scales=True, out=dict(scales=torch.zeros((2, 32, 4), dtype=u8)))
    # dequant calls: undersized scales / tensor_scale / out, and tiled scales
    codes = torch.zeros((2, 32, 32), dtype=u8)
    scales = torch.zeros((2, 32, 4), dtype=u8)
    G = torch.ones(2, dtype=f32)
    with pytest.raises(ValueError):
        nvq.nvfp4_dequant(codes, scales[:, :16], G)
    with pytest.raises(ValueError):
        nvq.nvfp4_dequant(codes, scales, G[:1])
    with pytest.raises(ValueError):
        nvq.nvfp4_dequant_t(codes, scales, G, out=torch.zeros((2, 64, 31), dtype=bf))
    with pytest.raises(ValueError):
        nvq.nvfp4_dequant(codes, torch.zeros((2, nvq.scale_bytes(32, 64, True)), dtype=u8), G)
    with pytest.raises(TypeError):  # right sizes: stopped by the host-tensor check
        nvq.nvfp4_dequant(codes, scales, G)
    # activations
    x = torch.zeros((8, 64), dtype=bf)
    with pytest.raises(ValueError):
        nvq.act_quantize_per_token(x, out=dict(token_scale=torch.zeros(7, dtype=f32)))
    # NF4: absmax and out
    c4 = torch.zeros((2, 4, 64), dtype=u8)
    with pytest.raises(ValueError):
        nvq.nf4_dequant(c4, torch.zeros((2, 4, 1), dtype=f32))
    with pytest.raises(ValueError):
        nvq.nf4_quantize(torch.zeros((2, 4, 128), dtype=bf),
                         out=dict(absmax=torch.zeros((2, 4, 1), dtype=f32)))
    with pytest.raises(ValueError):
        nvq.nf4_dequant_routed(c4, torch.zeros((2, 4, 2), dtype=f32),
                               torch.zeros((3, 2), dtype=torch.int32),
                               hit_list=torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError):
        nvq.nf4_absmax_unnest(torch.zeros((2, 300), dtype=u8), torch.zeros((2, 1), dtype=f32),
                              torch.zeros(2, dtype=f32))
    # status words are int32
    with pytest.raises(TypeError):
        nvq.nvfp4_quantize(w, status=torch.zeros(1, dtype=torch.int64))
    # GEMMs: dy / x must match the token counts and the stack
    with pytest.raises(ValueError):
        nvq.nvfp4_dgrad(torch.zeros((5, 32), dtype=bf), [2, 2], codes, scales, G)
    with pytest.raises(ValueError):
        nvq.nf4_routed_linear(torch.zeros((4, 100), dtype=bf), [2, 2], c4,
                              torch.zeros((2, 4, 2), dtype=f32))
    # MXFP8
    with pytest.raises(ValueError):
        nvq.mxfp8_dequant(torch.zeros((4, 64), dtype=u8), torch.zeros(7, dtype=u8))
