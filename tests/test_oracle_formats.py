"""Pins of the oracle's scalar rounding primitives against independent routines.

bf16 widening/narrowing and E4M3 are checked against PyTorch's own dtype
conversions (library routines, round-to-nearest-even); E2M1 against an
integer-rint formulation (numpy's rint is round-half-even) and against the
hand values that follow from the E2M1 value set {0, 0.5, 1, 1.5, 2, 3, 4, 6}
and the round-to-nearest-even rule of "The 4-bitter Lesson", "Key claims".
"""
import numpy as np
import pytest
import torch


def _bits_f32(x):
    return np.asarray(x, np.float32).view(np.uint32)


def test_bf16_widen_matches_torch_all_patterns(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([oracle_mod.bf16_to_f32(int(p)) for p in pats], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(_bits_f32(got[~nan]), _bits_f32(ref[~nan]))


def _bf16_cases():
    rng = np.random.default_rng(1234)
    raw = rng.integers(0, 2**32, size=40000, dtype=np.uint64).astype(np.uint32)
    # ties: low half exactly 0x8000 with even and odd upper halves
    ties = (rng.integers(0, 2**16, size=4000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    near = (rng.integers(0, 2**16, size=4000, dtype=np.uint64).astype(np.uint32) << 16) | \
        rng.choice(np.array([0x7FFF, 0x8001, 0x0001, 0xFFFF], np.uint32), size=4000)
    special = np.array([0, 0x80000000, 0x7F7FFFFF, 0x7F7F7FFF, 0x7F7F8000, 0xFF7F8000,
                        0x00000001, 0x00008000, 0x00018000, 0x3F808000, 0x3F818000], np.uint32)
    allp = np.concatenate([raw, ties, near, special])
    f = allp.view(np.float32)
    f = f[np.isfinite(f)]
    return f


def test_f32_to_bf16_rne_matches_torch(oracle_mod):
    f = _bf16_cases()
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.f32_to_bf16_array(f)
    assert np.array_equal(got, ref), np.nonzero(got != ref)[0][:10]


def test_e4m3_values_match_torch_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle_mod.e4m3_value(int(c)) for c in codes], np.float32)
    ok = ~np.isnan(ref)
    assert ok.sum() == 254  # 0x7F and 0xFF are the two NaN patterns
    assert np.array_equal(_bits_f32(got[ok]), _bits_f32(ref[ok]))
    assert oracle_mod.e4m3_value(0x7E) == 448.0
    assert oracle_mod.e4m3_value(0x01) == 2.0 ** -9


def _e4m3_sweep():
    vals = torch.arange(0, 127, dtype=torch.int16).to(torch.uint8).view(torch.float8_e4m3fn).float()
    v = vals.numpy().astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2
    pts = [v, mids]
    for d in (1, -1):
        pts.append(np.nextafter(mids.astype(np.float32), np.float32(d * np.inf)).astype(np.float64))
    rng = np.random.default_rng(7)
    pts.append(rng.uniform(0, 470, 20000))
    pts.append(np.exp2(rng.uniform(-14, 9, 20000)))
    x = np.concatenate(pts).astype(np.float32)
    x = x[(x >= 0) & (x < 464)]
    return x


def test_e4m3_encode_rne_matches_torch(oracle_mod):
    x = _e4m3_sweep()
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_mod.e4m3_encode_array(x)
    assert np.array_equal(got, ref), (x[got != ref][:5], got[got != ref][:5], ref[got != ref][:5])


def test_e4m3_encode_saturates_and_underflows(oracle_mod):
    for x in (448.0, 463.9, 464.0, 1e6, 3.0e38, float("inf")):
        assert oracle_mod.e4m3_encode(x) == 0x7E
    assert oracle_mod.e4m3_encode(2.0 ** -10) == 0x00          # tie 0 | 2^-9 -> even (0)
    assert oracle_mod.e4m3_encode(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01
    assert oracle_mod.e4m3_encode(3 * 2.0 ** -10) == 0x02      # tie 1 | 2 (x2^-9) -> even
    assert oracle_mod.e4m3_encode(0.0) == 0 and oracle_mod.e4m3_encode(-0.0) == 0


E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_value_set(oracle_mod):
    assert [oracle_mod.e2m1_value(c) for c in range(8)] == E2M1_VALUES
    assert [oracle_mod.e2m1_value(c | 8) for c in range(8)] == [-v for v in E2M1_VALUES]


def _e2m1_by_rint(q):
    """Independent E2M1 rounding: rint at the three spacings of the format."""
    a = np.abs(q.astype(np.float64))
    r = np.where(a < 2, np.rint(2 * a) / 2, np.where(a < 4, np.rint(a), 2 * np.rint(a / 2)))
    r = np.minimum(r, 6.0)
    lut = {v: i for i, v in enumerate(E2M1_VALUES)}
    mag = np.array([lut[float(v)] for v in r], np.uint8)
    return mag | np.where(np.signbit(q), 8, 0).astype(np.uint8)


def test_e2m1_encode_matches_rint_formulation(oracle_mod):
    rng = np.random.default_rng(3)
    vals = np.array(E2M1_VALUES)
    mids = (vals[:-1] + vals[1:]) / 2
    pts = [vals, mids, rng.uniform(-8, 8, 30000)]
    for d in (1, -1):
        pts.append(np.nextafter(mids.astype(np.float32), np.float32(d * np.inf)))
    x = np.concatenate(pts).astype(np.float32)
    x = np.concatenate([x, -x])
    got = oracle_mod.e2m1_encode_array(x)
    ref = _e2m1_by_rint(x)
    assert np.array_equal(got, ref), (x[got != ref][:5], got[got != ref][:5], ref[got != ref][:5])


@pytest.mark.parametrize("q,code", [
    (0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6),
    (5.0, 0x6), (6.5, 0x7), (100.0, 0x7), (0.30078125, 0x1), (-0.25, 0x8),
    (-0.0, 0x8), (0.0, 0x0), (-3.0, 0xD), (-7.0, 0xF),
])
def test_e2m1_hand_values(oracle_mod, q, code):
    assert oracle_mod.e2m1_encode(q) == code
