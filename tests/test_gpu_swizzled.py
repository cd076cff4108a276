"""Block scales in the tensor-core tiled layout ("Getting GLM-5.2 NVFP4
Post-Training off the ground", "Why can't we just transpose the one copy?":
the NVFP4 copies carry scales swizzled for the tensor-core tile).

1. The quantisers with swizzled scales write exactly the oracle's tiled
   layout of the oracle's scales (padding zero) and the same codes as the
   linear layout, for the rowwise, dual and per-token calls, on shapes with
   and without padding.
2. The layout is the one the block-scaled FP4 GEMM reads: cuBLASLt's NVFP4
   GEMM (through torch._scaled_mm), fed our activation and weight codes with
   their swizzled scales, returns the oracle's exact block-scaled product
   sum_k (c S)_x (c S)_w to within FP32 accumulation and the bf16 output
   rounding: |y - exact| <= 2^-8 (|exact| + d) + d, d = K 2^-23 sum |..|.
   A wrong byte order would pair codes with other blocks' scales.
"""
import numpy as np
import pytest
import torch

from nvq_testutil import u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def _np(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("E,R,K", [(2, 256, 512), (1, 200, 80), (3, 64, 48)])
def test_rowwise_swizzled_scales(nvq, oracle_mod, E, R, K):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(E, R, K, seed=R + K, device="cuda")
    q = nvq.nvfp4_quantize(w, four_over_six=True, swizzled_scales=True)
    o = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    assert np.array_equal(_np(q["codes"]), o["codes"])
    assert np.array_equal(_np(q["scales"]), oracle_mod.scales_tiled(o["scales"]))


@pytest.mark.parametrize("E,R,K", [(2, 256, 512), (1, 96, 320), (2, 400, 48)])
def test_dual_swizzled_scales(nvq, oracle_mod, E, R, K):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(E, R, K, seed=R * 3 + K, device="cuda")
    # a buffer full of garbage: the call must also write the padding
    sr = torch.full((E, nvq.scale_bytes(R, K, True)), 0x5A, dtype=torch.uint8, device="cuda")
    sc = torch.full((E, nvq.scale_bytes(K, R, True)), 0x5A, dtype=torch.uint8, device="cuda")
    q = nvq.nvfp4_quantize_dual(w, four_over_six=True, swizzled_scales=True,
                                out={"scales_row": sr, "scales_col": sc})
    orow = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    ocol = oracle_mod.nvfp4_quantize_colwise(u16(w), four_over_six=True)
    assert np.array_equal(_np(q["codes_row"]), orow["codes"])
    assert np.array_equal(_np(q["codes_col"]), ocol["codes"])
    assert np.array_equal(_np(sr), oracle_mod.scales_tiled(orow["scales"]))
    assert np.array_equal(_np(sc), oracle_mod.scales_tiled(ocol["scales"]))


@pytest.mark.parametrize("T,H", [(256, 512), (37, 208), (300, 6144), (129, 3216)])
def test_act_swizzled_scales(nvq, oracle_mod, T, H):
    from rl_nvfp4_quantize_gb300 import synth
    x = synth.activations(T, H, seed=T + H, device="cuda")
    s = torch.full((nvq.scale_bytes(T, H, True),), 0x5A, dtype=torch.uint8, device="cuda")
    q = nvq.act_quantize_per_token(x, four_over_six=True, swizzled_scales=True, out={"scales": s})
    o = oracle_mod.act_quantize_per_token(u16(x), four_over_six=True)
    assert np.array_equal(_np(q["codes"]), o["codes"])
    assert np.array_equal(_np(s), oracle_mod.scales_tiled(o["scales"]))


def test_fp4_gemm_reads_the_swizzled_scales(nvq, oracle_mod):
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this PyTorch has no FP4 dtype for its block-scaled GEMM")
    from rl_nvfp4_quantize_gb300 import synth
    T, N, K = 256, 384, 1024
    x = synth.activations(T, K, seed=3, device="cuda")
    w = synth.expert_weights(1, N, K, seed=4, device="cuda")
    qx = nvq.act_quantize_per_token(x, four_over_six=True, swizzled_scales=True)
    qw = nvq.nvfp4_quantize(w, four_over_six=True, swizzled_scales=True)
    fp4, fp8 = torch.float4_e2m1fn_x2, torch.float8_e4m3fn
    try:
        y = torch._scaled_mm(qx["codes"].view(fp4), qw["codes"][0].view(fp4).t(),
                             qx["scales"].view(fp8), qw["scales"][0].view(fp8),
                             out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError) as e:  # a torch without the block-scaled NVFP4 GEMM
        pytest.skip("torch._scaled_mm has no NVFP4 path here: %s" % str(e).splitlines()[0])
    torch.cuda.synchronize()
    ox = oracle_mod.act_quantize_per_token(u16(x), four_over_six=True)
    ow = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    ref, bound = oracle_mod.nvfp4_scaled_product(ox["codes"], ox["scales"], ow["codes"][0],
                                                 ow["scales"][0])
    got = y.float().cpu().numpy().astype(np.float64)
    d = K * 2.0 ** -23 * bound
    err = np.abs(got - ref)
    tol = 2.0 ** -8 * (np.abs(ref) + d) + d
    assert np.all(err <= tol), "max excess %g" % (err - tol).max()
    # the same codes with the LINEAR scales viewed as if tiled give a wrong
    # product: the check above does discriminate the layout
    lin = nvq.nvfp4_quantize(w, four_over_six=True)
    yb = torch._scaled_mm(qx["codes"].view(fp4), lin["codes"][0].view(fp4).t(),
                          qx["scales"].view(fp8), lin["scales"][0].reshape(-1).view(fp8),
                          out_dtype=torch.bfloat16)
    errb = np.abs(yb.float().cpu().numpy().astype(np.float64) - ref)
    assert np.any(errb > tol)
