"""Randomised shapes: every quantising and dequantising call on seeded random
shapes within its divisibility rules (ragged tiles in every dimension,
single rows and blocks, several expert slices), bit for bit against the
oracle.  The shapes are drawn once from a fixed seed, so the set is the same
on every run."""
import numpy as np
import pytest
import torch

from nvq_testutil import u16

pytestmark = pytest.mark.gpu

_RNG = np.random.default_rng(2024)


def _shapes(n, row_mult, col_mult, max_rows=300, max_cols=1100, max_e=3):
    out = []
    for _ in range(n):
        e = int(_RNG.integers(1, max_e + 1))
        r = int(_RNG.integers(1, max_rows // row_mult + 1)) * row_mult
        c = int(_RNG.integers(1, max_cols // col_mult + 1)) * col_mult
        out.append((e, r, c))
    return out + [(1, row_mult, col_mult)]


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def _w(E, R, K, seed):
    from rl_nvfp4_quantize_gb300 import synth
    return synth.expert_weights(E, R, K, seed=seed, device="cuda")


@pytest.mark.parametrize("E,R,K", _shapes(6, 1, 16))
@pytest.mark.parametrize("f46", [False, True])
def test_rowwise_and_dequant(nvq, oracle_mod, E, R, K, f46):
    w = _w(E, R, K, seed=E * 1000 + R + K)
    q = nvq.nvfp4_quantize(w, four_over_six=f46)
    d = nvq.nvfp4_dequant(q["codes"], q["scales"], q["tensor_scale"])
    o = oracle_mod.nvfp4_quantize(u16(w), four_over_six=f46)
    assert np.array_equal(q["codes"].cpu().numpy(), o["codes"])
    assert np.array_equal(q["scales"].cpu().numpy(), o["scales"])
    assert np.array_equal(q["tensor_scale"].cpu().numpy().view(np.uint32), o["G"].view(np.uint32))
    assert np.array_equal(u16(d), oracle_mod.nvfp4_dequant(o["codes"], o["scales"], o["G"], R, K))


@pytest.mark.parametrize("E,R,K", _shapes(6, 16, 16))
def test_dual_and_dequant_t(nvq, oracle_mod, E, R, K):
    w = _w(E, R, K, seed=E * 2000 + R + K)
    q = nvq.nvfp4_quantize_dual(w, four_over_six=True)
    dt = nvq.nvfp4_dequant_t(q["codes_row"], q["scales_row"], q["tensor_scale"])
    orow = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    ocol = oracle_mod.nvfp4_quantize_colwise(u16(w), four_over_six=True)
    assert np.array_equal(q["codes_row"].cpu().numpy(), orow["codes"])
    assert np.array_equal(q["scales_row"].cpu().numpy(), orow["scales"])
    assert np.array_equal(q["codes_col"].cpu().numpy(), ocol["codes"])
    assert np.array_equal(q["scales_col"].cpu().numpy(), ocol["scales"])
    assert np.array_equal(u16(dt), oracle_mod.nvfp4_dequant_t(orow["codes"], orow["scales"], orow["G"], R, K))


@pytest.mark.parametrize("T,H", [(t, h) for _, t, h in _shapes(6, 1, 16, max_rows=700, max_cols=3000)])
def test_act(nvq, oracle_mod, T, H):
    from rl_nvfp4_quantize_gb300 import synth
    x = synth.activations(T, H, seed=T + H, device="cuda")
    q = nvq.act_quantize_per_token(x, four_over_six=True)
    o = oracle_mod.act_quantize_per_token(u16(x), four_over_six=True)
    assert np.array_equal(q["codes"].cpu().numpy(), o["codes"])
    assert np.array_equal(q["scales"].cpu().numpy(), o["scales"])
    assert np.array_equal(q["token_scale"].cpu().numpy().view(np.uint32), o["token_scale"].view(np.uint32))


@pytest.mark.parametrize("E,R,K", _shapes(6, 1, 64))
def test_nf4(nvq, oracle_mod, E, R, K):
    w = _w(E, R, K, seed=E * 3000 + R + K)
    q = nvq.nf4_quantize(w)
    d = nvq.nf4_dequant(q["codes"], q["absmax"])
    o = oracle_mod.nf4_quantize(u16(w))
    assert np.array_equal(q["codes"].cpu().numpy(), o["codes"])
    assert np.array_equal(q["absmax"].cpu().numpy().view(np.uint32), o["absmax"].view(np.uint32))
    assert np.array_equal(u16(d), oracle_mod.nf4_dequant(o["codes"], o["absmax"], E, R, K))


@pytest.mark.parametrize("E,R,K", _shapes(6, 32, 32))
def test_mxfp8(nvq, oracle_mod, E, R, K):
    w = _w(E, R, K, seed=E * 4000 + R + K)
    q = nvq.mxfp8_quantize(w, columnwise=True)
    d = nvq.mxfp8_dequant(q["codes_row"], q["scales_row"])
    orow = oracle_mod.mxfp8_quantize(u16(w))
    ocol = oracle_mod.mxfp8_quantize_colwise(u16(w))
    assert np.array_equal(q["codes_row"].cpu().numpy(), orow["codes"])
    assert np.array_equal(q["scales_row"].cpu().numpy(), orow["scales"])
    assert np.array_equal(q["codes_col"].cpu().numpy(), ocol["codes"])
    assert np.array_equal(q["scales_col"].cpu().numpy(), ocol["scales"])
    assert np.array_equal(u16(d), oracle_mod.mxfp8_dequant(orow["codes"], orow["scales"]))


@pytest.mark.parametrize("E,R,K", _shapes(4, 16, 16))
def test_swizzled_scales(nvq, oracle_mod, E, R, K):
    w = _w(E, R, K, seed=E * 5000 + R + K)
    q = nvq.nvfp4_quantize_dual(w, four_over_six=True, swizzled_scales=True)
    orow = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    ocol = oracle_mod.nvfp4_quantize_colwise(u16(w), four_over_six=True)
    assert np.array_equal(q["scales_row"].cpu().numpy(), oracle_mod.scales_tiled(orow["scales"]))
    assert np.array_equal(q["scales_col"].cpu().numpy(), oracle_mod.scales_tiled(ocol["scales"]))
