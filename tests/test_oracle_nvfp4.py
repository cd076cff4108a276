"""Pins of the oracle's NVFP4 / Four-Over-Six path.

Each test checks the oracle against something it does not compute itself:
hand-derived blocks, the worked example printed in "Getting GLM-5.2 NVFP4
Post-Training off the ground" ("The bottom line"), closed forms, invariants
of the format, and identities between the rowwise, columnwise, transposed and
per-token entry points.  E4M3 expectations are produced with PyTorch's
float8_e4m3fn conversion, bf16 expectations with PyTorch's bfloat16 cast.
"""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(vals):
    """float values -> bf16 bit patterns (uint16), via torch's RNE cast."""
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_to_float(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16).copy()) \
        .view(torch.bfloat16).float().numpy()


def e4m3_torch(x):
    """E4M3 byte of a non-negative value: torch's RNE cast, saturated at 448."""
    x = min(np.float32(x), np.float32(448))
    return int(torch.tensor([np.float32(x)]).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def unpack(codes):
    codes = np.asarray(codes, np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


# --- hand blocks -------------------------------------------------------------

def test_hand_block_without_4over6(oracle_mod):
    # Block 0 holds 2688 = 6*448 so G = 1 and E = 1; block 1 then quantises
    # its values unscaled: a = 6, S = E4M3(1) = 0x38, q = x.
    b1 = [6, -3, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, 0.30078125, -0.25, 0, -0.0, 4, 1, 0.5]
    w = bf16([[2688] + [0] * 15 + b1]).reshape(1, 1, 32)
    r = oracle_mod.nvfp4_quantize(w, four_over_six=False)
    assert r["G"][0] == 1.0 and r["amax"][0] == 2688.0
    codes = unpack(r["codes"])[0, 0]
    assert list(r["scales"][0, 0]) == [0x7E, 0x38]
    assert codes[0] == 0x7
    assert list(codes[16:]) == [0x7, 0xD, 0x0, 0x2, 0x2, 0x4, 0x4, 0x6,
                                0x6, 0x1, 0x8, 0x0, 0x8, 0x6, 0x2, 0x1]


def _fos(oracle_mod, block):
    """Quantise [1536, 0...] + block with 4/6: G = 1536/(6*256) = 1, E = 1."""
    w = bf16([[1536] + [0] * 15 + list(block) + [0] * (16 - len(block))]).reshape(1, 1, 32)
    r = oracle_mod.nvfp4_quantize(w, four_over_six=True)
    assert r["G"][0] == 1.0
    return r["scales"][0, 0], unpack(r["codes"])[0, 0]


def test_hand_block_4over6_picks_four(oracle_mod):
    # [6, 4.5]: candidate 6 (S=1) rounds 4.5 to 4 (tie to even), SSE 0.25;
    # candidate 4 (S=1.5) gives 4*1.5=6 and 3*1.5=4.5, SSE 0 -> 4 wins.
    s, c = _fos(oracle_mod, [6, 4.5])
    assert s[1] == 0x3C and c[16] == 0x6 and c[17] == 0x5
    # the tensor-amax block: S6 = 256 (0x78) and S4 = 384 both exact -> tie -> 6
    assert s[0] == 0x78 and c[0] == 0x7


def test_hand_block_4over6_keeps_six(oracle_mod):
    s, c = _fos(oracle_mod, [6, 4])          # SSE6 = 0 < SSE4 = 0.25
    assert s[1] == 0x38 and c[16] == 0x7 and c[17] == 0x6


def test_hand_block_4over6_tie_keeps_six(oracle_mod):
    s, c = _fos(oracle_mod, [6, 3, 1.5])     # both candidates exact
    assert s[1] == 0x38 and list(c[16:19]) == [0x7, 0x5, 0x3]


def test_block_sse_against_float64(oracle_mod):
    rng = np.random.default_rng(11)
    for trial in range(300):
        x = bf16(rng.standard_normal(16) * rng.uniform(0.01, 3))
        E = float(np.float32(rng.uniform(10, 500)))
        s, codes, e6, e4 = oracle_mod.nvfp4_block(x, E, True)
        t = bf16_to_float(x).astype(np.float32) * np.float32(E)
        a = np.abs(t).max()
        for S_byte, e_f32 in ((e4m3_torch(a / np.float32(6)), e6), (e4m3_torch(a / np.float32(4)), e4)):
            S = float(torch.tensor([S_byte], dtype=torch.uint8).view(torch.float8_e4m3fn).float())
            q = t.astype(np.float64) * (np.float32(1) / np.float32(S) if S else 0.0)
            mag = np.where(np.abs(q) < 2, np.rint(2 * np.abs(q)) / 2,
                           np.where(np.abs(q) < 4, np.rint(np.abs(q)), 2 * np.rint(np.abs(q) / 2)))
            v = np.minimum(mag, 6) * S
            sse64 = float(np.sum((np.abs(t.astype(np.float64)) - v) ** 2))
            assert abs(sse64 - e_f32) <= 1e-5 * max(sse64, 1e-30) + 1e-30
        # the choice follows the errors: strictly lower SSE4 picks 4, else 6
        s6 = e4m3_torch(a / np.float32(6))
        s4 = e4m3_torch(a / np.float32(4))
        assert s == (s4 if e4 < e6 else s6)


# --- the worked example of the pages ------------------------------------------

def test_worked_example_rowwise_and_columnwise_scales(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "worked_example_transpose.json")))
    W = np.zeros((16, 16), np.float32)
    W[:2, :3] = np.array(g["weight"], np.float32)
    w = bf16(W).reshape(1, 16, 16)
    row = oracle_mod.nvfp4_quantize(w)
    col = oracle_mod.nvfp4_quantize_colwise(w)
    amax = 6.0
    assert row["amax"][0] == amax and col["G"][0] == row["G"][0]
    G = np.float32(amax) / np.float32(6 * 448)
    E = np.float32(1) / G
    for r, am in enumerate(g["row_block_amax"]):
        assert row["scales"][0, r, 0] == e4m3_torch(np.float32(am) * E / np.float32(6))
    for c, am in enumerate(g["col_block_amax"]):
        assert col["scales"][0, c, 0] == e4m3_torch(np.float32(am) * E / np.float32(6))
    # the column block {1,4} needs a scale that neither row scale provides
    assert col["scales"][0, 0, 0] not in (row["scales"][0, 0, 0], row["scales"][0, 1, 0])


# --- closed forms ---------------------------------------------------------------

@pytest.mark.parametrize("f46", [False, True])
def test_all_zero_block(oracle_mod, f46):
    w = bf16([[3.0] + [0] * 15 + [0.0] * 8 + [-0.0] * 8]).reshape(1, 1, 32)
    r = oracle_mod.nvfp4_quantize(w, four_over_six=f46)
    c = unpack(r["codes"])[0, 0]
    assert r["scales"][0, 0, 1] == 0
    assert list(c[16:24]) == [0] * 8 and list(c[24:]) == [8] * 8
    dq = oracle_mod.nvfp4_dequant(r["codes"], r["scales"], r["G"], 1, 32)
    assert np.all(bf16_to_float(dq[0, 0, 16:]) == 0)


@pytest.mark.parametrize("f46,M_byte", [(False, 0x7E), (True, 0x78)])
def test_all_equal_tensor(oracle_mod, f46, M_byte):
    for v in (0.02, 1.0, 3.25, 1000.0):
        w = bf16(np.full((1, 2, 32), v))
        r = oracle_mod.nvfp4_quantize(w, four_over_six=f46)
        assert np.all(r["scales"] == M_byte)
        assert np.all(unpack(r["codes"]) == 0x7)
        dq = oracle_mod.nvfp4_dequant(r["codes"], r["scales"], r["G"], 2, 32)
        assert np.array_equal(dq, w)


def test_max_element_decodes_to_amax(oracle_mod):
    rng = np.random.default_rng(5)
    for f46 in (False, True):
        for _ in range(20):
            x = rng.standard_normal((1, 16, 64)) * rng.uniform(1e-3, 1e3)
            w = bf16(x)
            r = oracle_mod.nvfp4_quantize(w, four_over_six=f46)
            dq = oracle_mod.nvfp4_dequant(r["codes"], r["scales"], r["G"], 16, 64)
            xf, df = bf16_to_float(w), bf16_to_float(dq)
            i = np.argmax(np.abs(xf))
            assert np.abs(df.ravel()[i]) == np.abs(xf.ravel()[i]) == r["amax"][0]


def test_tensor_scales_closed_form(oracle_mod):
    rng = np.random.default_rng(9)
    for am in list(np.float32(rng.uniform(1e-6, 1e6, 200))) + [np.float32(0.0)]:
        for f46, M in ((False, 448), (True, 256)):
            G, E = oracle_mod.tensor_scales(float(am), f46)
            assert np.float32(G) == np.float32(np.float64(am) / (6 * M))
            if am == 0:
                assert E == np.finfo(np.float32).max
            else:
                assert np.float32(E) == np.float32(1.0 / np.float64(np.float32(G)))


# --- invariants ----------------------------------------------------------------

def _random_weight(rng, nexp, rows, cols, outliers=True):
    x = rng.standard_normal((nexp, rows, cols)) * 0.02 * rng.uniform(0.5, 2, (nexp, 1, 1))
    if outliers:
        m = rng.random(x.shape) < 0.002
        x[m] *= 30
    return bf16(x)


@pytest.mark.parametrize("f46", [False, True])
def test_dequant_bounded_by_amax_and_block_error(oracle_mod, f46):
    rng = np.random.default_rng(21 + f46)
    w = _random_weight(rng, 3, 32, 64)
    r = oracle_mod.nvfp4_quantize(w, four_over_six=f46)
    dq = bf16_to_float(oracle_mod.nvfp4_dequant(r["codes"], r["scales"], r["G"], 32, 64))
    x = bf16_to_float(w)
    for e in range(3):
        assert np.all(np.abs(dq[e]) <= r["amax"][e] * (1 + 2.0 ** -8))
    # per-element error: at most half the local E2M1 gap times S*G (plus bf16 and
    # E4M3 rounding of the scale), or the element saturated at 6*S*G
    S = torch.from_numpy(r["scales"].copy()).view(torch.float8_e4m3fn).float().numpy()
    S = np.repeat(S, 16, axis=-1) * r["G"][:, None, None]
    err = np.abs(dq - x)
    assert np.all(err <= 1.0 * S + np.abs(x) * 2.0 ** -7 + 1e-30)


def test_idempotent_without_4over6(oracle_mod):
    rng = np.random.default_rng(33)
    w = _random_weight(rng, 2, 48, 80)
    r1 = oracle_mod.nvfp4_quantize(w)
    dq = oracle_mod.nvfp4_dequant(r1["codes"], r1["scales"], r1["G"], 48, 80)
    r2 = oracle_mod.nvfp4_quantize(dq)
    assert np.array_equal(r1["codes"], r2["codes"])
    assert np.array_equal(r1["scales"], r2["scales"])


def test_idempotent_dequant_with_4over6(oracle_mod):
    rng = np.random.default_rng(34)
    w = _random_weight(rng, 2, 48, 80)
    r1 = oracle_mod.nvfp4_quantize(w, four_over_six=True)
    d1 = oracle_mod.nvfp4_dequant(r1["codes"], r1["scales"], r1["G"], 48, 80)
    r2 = oracle_mod.nvfp4_quantize(d1, four_over_six=True)
    d2 = oracle_mod.nvfp4_dequant(r2["codes"], r2["scales"], r2["G"], 48, 80)
    assert np.array_equal(d1, d2)


# --- identities between entry points -------------------------------------------

@pytest.mark.parametrize("f46", [False, True])
def test_colwise_is_rowwise_of_transpose(oracle_mod, f46):
    rng = np.random.default_rng(40 + f46)
    w = _random_weight(rng, 2, 48, 32)
    col = oracle_mod.nvfp4_quantize_colwise(w, four_over_six=f46)
    wt = np.ascontiguousarray(np.swapaxes(w, 1, 2))
    row_t = oracle_mod.nvfp4_quantize(wt, four_over_six=f46)
    assert np.array_equal(col["codes"], row_t["codes"])
    assert np.array_equal(col["scales"], row_t["scales"])
    assert np.array_equal(col["G"], row_t["G"])


def test_dequant_t_is_transpose_of_dequant(oracle_mod):
    rng = np.random.default_rng(50)
    w = _random_weight(rng, 3, 32, 48)
    r = oracle_mod.nvfp4_quantize(w, four_over_six=True)
    d = oracle_mod.nvfp4_dequant(r["codes"], r["scales"], r["G"], 32, 48)
    dt = oracle_mod.nvfp4_dequant_t(r["codes"], r["scales"], r["G"], 32, 48)
    assert np.array_equal(dt, np.swapaxes(d, 1, 2))


def test_dequant_matches_torch_products(oracle_mod):
    rng = np.random.default_rng(51)
    w = _random_weight(rng, 2, 16, 64)
    r = oracle_mod.nvfp4_quantize(w, four_over_six=True)
    d = oracle_mod.nvfp4_dequant(r["codes"], r["scales"], r["G"], 16, 64)
    c = unpack(r["codes"])
    mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)[c & 7]
    S = torch.from_numpy(r["scales"].copy()).view(torch.float8_e4m3fn).float().numpy()
    v = (mag * np.repeat(S, 16, axis=-1)).astype(np.float32)
    y = (v * r["G"][:, None, None]).astype(np.float32)
    y = np.where(c & 8, -y, y)
    assert np.array_equal(d, bf16(y))


def test_per_token_equals_one_row_slices(oracle_mod):
    rng = np.random.default_rng(60)
    x = rng.standard_t(3, (24, 96)) * 0.5
    x[:, [3, 40]] *= 50
    xb = bf16(x)
    a = oracle_mod.act_quantize_per_token(xb, four_over_six=True)
    s = oracle_mod.nvfp4_quantize(xb.reshape(24, 1, 96), four_over_six=True)
    assert np.array_equal(a["codes"], s["codes"].reshape(24, 48))
    assert np.array_equal(a["scales"], s["scales"].reshape(24, 6))
    assert np.array_equal(a["token_scale"], s["G"])
    # no cross-token state: a sub-batch quantises to the same rows
    b = oracle_mod.act_quantize_per_token(np.ascontiguousarray(xb[5:9]), four_over_six=True)
    assert np.array_equal(b["codes"], a["codes"][5:9])
    assert np.array_equal(b["token_scale"], a["token_scale"][5:9])


def test_amax_given_and_status(oracle_mod):
    rng = np.random.default_rng(70)
    w = _random_weight(rng, 2, 16, 32)
    r = oracle_mod.nvfp4_quantize(w, four_over_six=True)
    r2 = oracle_mod.nvfp4_quantize(w, four_over_six=True, amax=r["amax"])
    assert np.array_equal(r["codes"], r2["codes"]) and np.array_equal(r["G"], r2["G"])
    assert r["status"] == 0
    bad = w.copy()
    bad[1, 3, 5] = 0x7FC0  # NaN
    assert oracle_mod.nvfp4_quantize(bad)["status"] & oracle_mod.STATUS_NONFINITE
