"""Pins of the oracle's routed NF4 forward product (host only).

Y = X . DQ(W_e)^T per expert ("nf4moe -- QLoRA for a 743B Fused-MoE", "The
fix: dequant-on-forward for routed experts": each routed expert's weight is
dequantised and applied as F.linear(x, W[e])).  The oracle forms it with one
float64 matrix product per expert; these tests check it against a plain
triple loop over the same bf16 values (so a transposed operand or a wrong
expert offset fails), the layout rules (token rows grouped by expert, empty
experts), the bound |Y| <= |X| . |DQ|^T, and exact sums.
"""
import numpy as np
import pytest

from test_oracle_nvfp4 import bf16


def _bits_to_f64(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(oracle_mod, E, out, inn, counts, seed):
    rng = np.random.default_rng(seed)
    q = oracle_mod.nf4_quantize(bf16(rng.standard_normal((E, out, inn)) * 0.05))
    x = bf16(rng.standard_normal((sum(counts), inn)))
    return q, x


@pytest.mark.parametrize("E,out,inn,counts", [(1, 4, 64, [3]), (3, 6, 64, [2, 0, 3]), (2, 5, 128, [1, 4])])
def test_nf4_linear_against_triple_loop(oracle_mod, E, out, inn, counts):
    q, x = _case(oracle_mod, E, out, inn, counts, seed=E * 11 + out)
    y, bound = oracle_mod.nf4_routed_linear(x, counts, q["codes"], q["absmax"], out, inn)
    assert y.shape == (sum(counts), out)
    t0 = 0
    for e, c in enumerate(counts):
        wd = _bits_to_f64(oracle_mod.nf4_dequant(q["codes"][e:e + 1], q["absmax"][e:e + 1], 1, out, inn)[0])
        for t in range(t0, t0 + c):
            a = _bits_to_f64(x[t])
            for o in range(out):
                s = sum(a[i] * wd[o, i] for i in range(inn))
                b = sum(abs(a[i] * wd[o, i]) for i in range(inn))
                assert abs(y[t, o] - s) <= 1e-12 * max(b, 1e-300)
                assert abs(bound[t, o] - b) <= 1e-12 * max(b, 1e-300)
        t0 += c
    assert np.all(np.abs(y) <= bound * (1 + 1e-12))


def test_nf4_linear_uses_each_experts_own_weight(oracle_mod):
    """Expert 1's weight is expert 0's times 2: the same codes, twice the
    absmax, so its dequantised weight is exactly twice as large and the same
    token row routed to each gives outputs in the ratio 2 exactly."""
    rng = np.random.default_rng(5)
    w = rng.standard_normal((1, 8, 64)) * 0.1
    q = oracle_mod.nf4_quantize(bf16(np.concatenate([w, 2 * w])))
    assert np.array_equal(q["codes"][0], q["codes"][1])
    x = bf16(np.repeat(rng.standard_normal((1, 64)), 2, axis=0))
    y, _ = oracle_mod.nf4_routed_linear(x, [1, 1], q["codes"], q["absmax"], 8, 64)
    assert np.array_equal(2 * y[0], y[1]) and np.any(y[0] != 0)
    y0, _ = oracle_mod.nf4_routed_linear(x, [2, 0], q["codes"], q["absmax"], 8, 64)
    assert np.array_equal(y0[0], y0[1]) and np.array_equal(y0[0], y[0])


def test_nf4_linear_of_exact_values_is_exact(oracle_mod):
    """Blocks whose absmax is 1 dequantise to the bf16 levels themselves
    (multiples of 2^-11 in [-1, 1]); with X in {-1, 0, 1} every sum is a
    float64- and float32-exact multiple of 2^-11."""
    rng = np.random.default_rng(8)
    out, inn = 4, 128
    w = rng.uniform(-1, 1, (1, out, inn))
    w[0, :, ::64] = 1.0
    q = oracle_mod.nf4_quantize(bf16(w))
    assert np.all(q["absmax"] == 1.0)
    xf = rng.integers(-1, 2, (6, inn)).astype(np.float64)
    y, _ = oracle_mod.nf4_routed_linear(bf16(xf), [6], q["codes"], q["absmax"], out, inn)
    wd = _bits_to_f64(oracle_mod.nf4_dequant(q["codes"], q["absmax"], 1, out, inn)[0])
    assert np.array_equal(y, xf @ wd.T)
    assert np.all((y * 2048) == np.round(y * 2048))
    assert np.array_equal(y.astype(np.float32).astype(np.float64), y)
