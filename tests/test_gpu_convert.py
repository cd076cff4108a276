"""Conversion sweeps: the device rounding primitives against the oracle.

Each kind of nvq_debug_convert runs the same device code the kernels use
(E4M3 and E2M1 conversion instructions, the division-by-6 block-scale path,
bf16 rounding and the decodes) over structured sweeps that cover every
exponent of interest, the patterns on and next to every rounding midpoint,
and random patterns; the oracle gives the expected bytes."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def _structured(exp_lo, exp_hi, rng, n_random=400000):
    """float32 values with every exponent in [exp_lo, exp_hi], every top-8
    mantissa pattern and the low-bit patterns that decide rounding."""
    exps = np.arange(exp_lo, exp_hi + 1) + 127
    tops = np.arange(256, dtype=np.uint32) << 15
    lows = np.array([0, 1, 0x3FFF, 0x4000, 0x4001, 0x7FFF], np.uint32)
    bits = (exps[:, None, None].astype(np.uint32) << 23) | tops[None, :, None] | lows[None, None, :]
    bits = bits.ravel()
    rnd = rng.integers((exp_lo + 127) << 23, (exp_hi + 128) << 23, n_random, dtype=np.int64).astype(np.uint32)
    return np.concatenate([bits, rnd]).view(np.float32)


def test_e4m3_encode_sweep(nvq, oracle_mod):
    rng = np.random.default_rng(0)
    x = np.concatenate([_structured(-14, 9, rng), np.array([0.0, 448.0, 464.0, 1e5, 3e38], np.float32)])
    got = nvq.debug_convert(0, torch.from_numpy(x).cuda()).cpu().numpy()
    ref = oracle_mod.e4m3_encode_array(x)
    assert np.array_equal(got, ref), (x[got != ref][:8], got[got != ref][:8], ref[got != ref][:8])


def test_e4m3_of_a_over_6_and_4(nvq, oracle_mod):
    rng = np.random.default_rng(1)
    a = np.concatenate([_structured(-20, 11, rng), np.float32([0, 6, 1536, 2688, 2687.9998])])
    ga = torch.from_numpy(a).cuda()
    got6 = nvq.debug_convert(3, ga).cpu().numpy()
    got4 = nvq.debug_convert(6, ga).cpu().numpy()
    ref6 = oracle_mod.e4m3_encode_array(a / np.float32(6))
    ref4 = oracle_mod.e4m3_encode_array(a / np.float32(4))
    assert np.array_equal(got6, ref6), (a[got6 != ref6][:8], got6[got6 != ref6][:8])
    assert np.array_equal(got4, ref4)


def test_e4m3_decode_all_codes(nvq, oracle_mod):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    got = nvq.debug_convert(4, torch.from_numpy(codes).cuda()).cpu().numpy()
    ref = np.array([oracle_mod.e4m3_value(int(c)) for c in codes], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_e2m1_encode_sweep_and_nibble_order(nvq, oracle_mod):
    rng = np.random.default_rng(2)
    q = _structured(-6, 4, rng)
    q = np.concatenate([q, -q, np.float32([0.0, -0.0, 6.0, 7.0, -1e30, 0.25, 0.75, 5.0])])
    if q.size % 2:
        q = q[:-1]
    perm = rng.permutation(q.size)
    q = q[perm]
    got = nvq.debug_convert(1, torch.from_numpy(q).cuda()).cpu().numpy()
    codes = oracle_mod.e2m1_encode_array(q)
    ref = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    assert np.array_equal(got, ref), (q.reshape(-1, 2)[got != ref][:5], got[got != ref][:5], ref[got != ref][:5])


def test_e2m1_decode_all_bytes(nvq, oracle_mod):
    b = np.arange(256, dtype=np.uint8)
    got = nvq.debug_convert(5, torch.from_numpy(b).cuda()).cpu().numpy().reshape(256, 2)
    ref = np.array([[oracle_mod.e2m1_value(int(x) & 15), oracle_mod.e2m1_value(int(x) >> 4)] for x in b],
                   np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_bf16_rounding_sweep(nvq, oracle_mod):
    rng = np.random.default_rng(3)
    raw = rng.integers(0, 2**32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    ties = (raw[:200000] & 0xFFFF0000) | 0x8000
    x = np.concatenate([raw, ties]).view(np.float32)
    x = x[np.isfinite(x)]
    got = nvq.debug_convert(2, torch.from_numpy(x).cuda()).cpu().numpy().view(np.uint16)
    ref = oracle_mod.f32_to_bf16_array(x)
    assert np.array_equal(got, ref)
