"""MXFP8 quantisation and dequantisation on the GPU against the oracle,
bit for bit (OCP MX definition; "The 4-bitter Lesson", "Key claims": the
MXFP8 validation of the dequantised backward).

Inputs span every exponent a block scale can take, signed zeros, bf16
subnormals and values that saturate at 448 X; shapes include ragged tiles.
The columnwise copy, the tiled scale layout and the dequantisation (fed the
oracle's codes) are checked the same way, and at full size [32, 4096, 6144]
on sampled blocks.
"""
import numpy as np
import pytest
import torch

from nvq_testutil import bf16_from_u16, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def _hard_weights(E, R, K, seed):
    from test_oracle_nvfp4 import bf16
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((E, R, K)) * np.exp(rng.uniform(-60, 60, (E, R, K // 32, 1))).repeat(32, -1).reshape(E, R, K)
    x[..., :3, :32] = 0.0
    x[..., 3, :16] = -0.0
    x[..., 4, 0] = 2.0 ** -133                       # smallest bf16 subnormal
    x[..., 5, :32] = 2.0 ** -130 * rng.standard_normal(32)
    x[..., 6, 0] = 500.0                             # amax in [256, 512): saturates at 448 X
    x[..., 6, 1:32] = rng.uniform(-480, 480, 31)
    return bf16(x)


@pytest.mark.parametrize("E,R,K", [(2, 64, 256), (1, 96, 320), (3, 128, 96), (1, 32, 32)])
def test_mxfp8_dual_bit_exact(nvq, oracle_mod, E, R, K):
    wh = _hard_weights(E, R, K, seed=R + K)
    w = bf16_from_u16(wh)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = nvq.mxfp8_quantize(w, columnwise=True, status=st)
    orow = oracle_mod.mxfp8_quantize(wh)
    ocol = oracle_mod.mxfp8_quantize_colwise(wh)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(q["codes_row"].cpu().numpy(), orow["codes"])
    assert np.array_equal(q["scales_row"].cpu().numpy(), orow["scales"])
    assert np.array_equal(q["codes_col"].cpu().numpy(), ocol["codes"])
    assert np.array_equal(q["scales_col"].cpu().numpy(), ocol["scales"])


@pytest.mark.parametrize("E,R,K", [(2, 64, 256), (1, 100, 160)])
def test_mxfp8_rowwise_and_tiled_scales(nvq, oracle_mod, E, R, K):
    wh = _hard_weights(E, R, K, seed=7 * R + K)
    w = bf16_from_u16(wh)
    q = nvq.mxfp8_quantize(w)
    sr = torch.full((E, nvq.mx_scale_bytes(R, K, True)), 0x5A, dtype=torch.uint8, device="cuda")
    qt = nvq.mxfp8_quantize(w, swizzled_scales=True, out={"scales_row": sr})
    o = oracle_mod.mxfp8_quantize(wh)
    assert np.array_equal(q["codes_row"].cpu().numpy(), o["codes"])
    assert np.array_equal(q["scales_row"].cpu().numpy(), o["scales"])
    assert np.array_equal(qt["codes_row"].cpu().numpy(), o["codes"])
    assert np.array_equal(sr.cpu().numpy(), oracle_mod.scales_tiled(o["scales"]))


def test_mxfp8_dequant_bit_exact(nvq, oracle_mod):
    wh = _hard_weights(2, 64, 512, seed=3)
    o = oracle_mod.mxfp8_quantize(wh)
    d = nvq.mxfp8_dequant(torch.from_numpy(o["codes"]).cuda(), torch.from_numpy(o["scales"]).cuda())
    ref = oracle_mod.mxfp8_dequant(o["codes"], o["scales"])
    assert np.array_equal(u16(d), ref)
    # every code and every scale byte the format allows (NaN codes excluded)
    codes = np.arange(256, dtype=np.uint8).repeat(32 * 4).reshape(-1, 32)
    codes[(codes & 0x7F) == 0x7F] = 0
    scales = np.tile(np.array([0, 1, 64, 127, 200, 254], np.uint8), codes.shape[0] // 6 + 1)[:codes.shape[0]]
    d2 = nvq.mxfp8_dequant(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    assert np.array_equal(u16(d2), oracle_mod.mxfp8_dequant(codes, scales))


def test_mxfp8_full_size_sampled(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 32, 4096, 6144
    w = synth.expert_weights(E, R, K, seed=21, device="cuda")
    q = nvq.mxfp8_quantize(w, columnwise=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(88)
    for _ in range(96):
        e, i, b = int(rng.integers(E)), int(rng.integers(R)), int(rng.integers(K // 32))
        s, c = oracle_mod.mxfp8_block(u16(w[e, i, 32 * b:32 * b + 32]))
        assert int(q["scales_row"][e, i, b].item()) == s
        assert np.array_equal(q["codes_row"][e, i, 32 * b:32 * b + 32].cpu().numpy(), c)
        j, rb = int(rng.integers(K)), int(rng.integers(R // 32))
        s, c = oracle_mod.mxfp8_block(np.ascontiguousarray(u16(w[e, 32 * rb:32 * rb + 32, j])))
        assert int(q["scales_col"][e, j, rb].item()) == s
        assert np.array_equal(q["codes_col"][e, j, 32 * rb:32 * rb + 32].cpu().numpy(), c)
    del w, q
    torch.cuda.empty_cache()


def test_mx_gemm_reads_the_tiled_scales(nvq, oracle_mod):
    """cuBLASLt's MXFP8 GEMM (torch._scaled_mm with E8M0 block scales) fed our
    codes and tiled scales returns the oracle's exact block-scaled product
    within FP32 accumulation and bf16 rounding."""
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this PyTorch has no E8M0 dtype")
    from rl_nvfp4_quantize_gb300 import synth
    M, N, K = 256, 384, 1024
    x = synth.activations(M, K, seed=31, device="cuda")
    w = synth.expert_weights(1, N, K, seed=32, device="cuda")
    qx = nvq.mxfp8_quantize(x.unsqueeze(0), swizzled_scales=True)
    qw = nvq.mxfp8_quantize(w, swizzled_scales=True)
    f8, e8 = torch.float8_e4m3fn, torch.float8_e8m0fnu
    try:
        y = torch._scaled_mm(qx["codes_row"][0].view(f8), qw["codes_row"][0].view(f8).t(),
                             qx["scales_row"][0].view(e8), qw["scales_row"][0].view(e8),
                             out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, ValueError) as e:
        pytest.skip("torch._scaled_mm has no MXFP8 path here: %s" % str(e).splitlines()[0])
    torch.cuda.synchronize()
    ox = oracle_mod.mxfp8_quantize(u16(x).reshape(1, M, K))
    ow = oracle_mod.mxfp8_quantize(u16(w))
    va = oracle_mod.mxfp8_values(ox["codes"][0], ox["scales"][0])
    vb = oracle_mod.mxfp8_values(ow["codes"][0], ow["scales"][0])
    ref, bound = va @ vb.T, np.abs(va) @ np.abs(vb).T
    got = y.float().cpu().numpy().astype(np.float64)
    d = K * 2.0 ** -23 * bound
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * (np.abs(ref) + d) + d)
