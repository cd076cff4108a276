"""Pins of the oracle's MXFP8 quantisation (host only).

MXFP8 is the format "The 4-bitter Lesson" ("Key claims") validated the
dequantised backward with; the pages name it only, and its definition is the
OCP Microscaling one: 32-element blocks, an E8M0 scale 2^s with
s = floor(log2 amax) - 8, E4M3 elements of v / 2^s (round to nearest even,
saturating).  The pins:
  * an independent restatement: s from the FP32 exponent bits (or float64
    log2 for subnormals), the elements from torch's float8_e4m3fn cast;
  * closed forms: all-ones, a saturating block, the zero block, the smallest
    subnormal block (scale clamped at 2^-127), signed zeros;
  * invariants: every element within half an E4M3 step (or clamped to
    448 X where the scale choice lets the top of the binade saturate),
    Q(DQ(Q(x))) = Q(x), and the
    columnwise copy equals the rowwise copy of the transpose.
"""
import numpy as np
import pytest
import torch

from test_oracle_nvfp4 import bf16, bf16_to_float


def _ref_block(xf32):
    """Independent MXFP8 of one block of 32 float32 values."""
    a = float(np.max(np.abs(xf32)))
    if a == 0.0:
        s = -127
    elif a >= 2.0 ** -126:
        s = int((np.float32(a).view(np.uint32) >> 23) & 0xFF) - 127 - 8
    else:
        s = int(np.floor(np.log2(a))) - 8
    s = max(-127, min(127, s))
    v = torch.from_numpy(np.asarray(xf32, np.float64) * 2.0 ** -s).clamp(-448.0, 448.0)
    codes = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return s + 127, codes


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_blocks_against_independent_restatement(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((64, 32)) * np.exp(rng.uniform(-20, 20, (64, 1)))
    x[3] = 0.0
    x[5, :7] = -0.0
    x[7, 0] = 470.0          # within a block of amax in [256, 512): saturates at 448
    xb = bf16(x)
    xf = bf16_to_float(xb)
    for i in range(64):
        s, c = oracle_mod.mxfp8_block(xb[i])
        rs, rc = _ref_block(xf[i])
        assert s == rs, i
        assert np.array_equal(c, rc), (i, c, rc)


def test_closed_forms(oracle_mod):
    s, c = oracle_mod.mxfp8_block(bf16(np.ones(32)))
    assert s == 127 - 8 and np.all(c == 0x78)              # 1 = 256 * 2^-8
    x = np.zeros(32)
    x[0] = 480.0
    s, c = oracle_mod.mxfp8_block(bf16(x))
    assert s == 127 and c[0] == 0x7E and np.all(c[1:] == 0)  # 480 > 448 saturates
    s, c = oracle_mod.mxfp8_block(bf16(np.zeros(32)))
    assert s == 0 and np.all(c == 0)
    s, c = oracle_mod.mxfp8_block(bf16(-np.zeros(32)))
    assert s == 0 and np.all(c == 0x80)
    tiny = np.full(32, 2.0 ** -133)                          # smallest bf16 subnormal
    s, c = oracle_mod.mxfp8_block(bf16(tiny))
    assert s == 0 and np.all(c == 0x08)                      # 2^-133 / 2^-127 = 2^-6
    x = np.full(32, 3.0)
    x[1] = -1e-6                                             # rounds to -0 at scale 2^-7
    s, c = oracle_mod.mxfp8_block(bf16(x))
    assert s == 127 - 7 and c[1] == 0x80 and c[0] == 0x7C    # 3 * 2^7 = 384 = 1.5 * 2^8


def test_dequant_invariants(oracle_mod):
    rng = np.random.default_rng(4)
    w = bf16(rng.standard_normal((2, 16, 96)) * 0.05)
    q = oracle_mod.mxfp8_quantize(w)
    d = oracle_mod.mxfp8_dequant(q["codes"], q["scales"])
    wf, df = bf16_to_float(w), bf16_to_float(d)
    # per block: the dequantised value is within half an E4M3 step of the input
    blocks_w = wf.reshape(-1, 32)
    blocks_d = df.reshape(-1, 32)
    sc = q["scales"].reshape(-1).astype(np.int64) - 127
    for bw, bd, s in zip(blocks_w, blocks_d, sc):
        X = 2.0 ** s
        sat = np.abs(bw) >= 448.0 * X          # the OCP scale lets the top of the binade clamp
        assert np.all(bd[sat] == np.sign(bw[sat]) * 448.0 * X)
        ok = np.abs(bd - bw) <= 0.0625 * np.maximum(np.abs(bw), 2.0 ** -6 * X) + 1e-45
        assert np.all(ok | sat)
    # Q(DQ(Q(x))) = Q(x)
    q2 = oracle_mod.mxfp8_quantize(d)
    assert np.array_equal(q2["codes"], q["codes"]) and np.array_equal(q2["scales"], q["scales"])


def test_colwise_is_rowwise_of_transpose(oracle_mod):
    rng = np.random.default_rng(5)
    w = bf16(rng.standard_normal((2, 64, 96)))
    qc = oracle_mod.mxfp8_quantize_colwise(w)
    qt = oracle_mod.mxfp8_quantize(np.ascontiguousarray(np.transpose(w, (0, 2, 1))))
    assert np.array_equal(qc["codes"], qt["codes"]) and np.array_equal(qc["scales"], qt["scales"])
