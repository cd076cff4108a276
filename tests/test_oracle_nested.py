"""Pins of the oracle's nested (double-quantised) NF4 absmax (host only).

The NF4 state of "nf4moe -- QLoRA for a 743B Fused-MoE" ("The fix") holds the
absmax and a "nested code"; the reading is QLoRA's double quantisation: the
slice's FP32 absmax values centred on their mean (a pairwise-tree FP32 sum,
divided by n in binary64), quantised to E4M3 in blocks of 256 with the block's
largest centred magnitude mapped to 448, decoded by one fused multiply-add.
The pins:
  * the summation order, by closed forms that a sequential sum gets wrong;
  * the mean's error against an exactly rounded sum (math.fsum), within the
    pairwise-summation bound;
  * closed forms of whole slices (equal values, two-valued blocks, signs,
    saturation at 448);
  * the codes against an independent encoding (torch's float8_e4m3fn cast);
  * the decoded absmax within the E4M3 error bound of the input.
"""
import math

import numpy as np
import pytest
import torch

F32_EPS = 2.0 ** -24


def test_tree_order_closed_forms(oracle_mod):
    u = 2.0 ** -24
    # (1 + u) rounds to 1 (tie to even), (u + u) = 2u exactly, 1 + 2u is exact:
    # a sequential sum would give 1 instead
    a = np.array([1.0, u, u, u], np.float32)
    assert float(oracle_mod.tree_sum(a)) == 1.0 + 2 * u
    assert float(oracle_mod.absmax_mean(a)) == float(np.float32((1.0 + 2 * u) / 4))
    # n = 5 pads to 8: ((u+u)+(u+u)) + ((1+0)+(0+0)) = 1 + 4u exactly
    a = np.array([u, u, u, u, 1.0], np.float32)
    assert float(oracle_mod.tree_sum(a)) == 1.0 + 4 * u
    assert float(oracle_mod.absmax_mean(a)) == float(np.float32((1.0 + 4 * u) / 5))
    # n = 3 pads to 4: (1 + u) + (u + 0) = 1 + u -> 1
    a = np.array([1.0, u, u], np.float32)
    assert float(oracle_mod.tree_sum(a)) == 1.0
    assert float(oracle_mod.absmax_mean(a)) == float(np.float32(1.0 / 3))


@pytest.mark.parametrize("n", [1, 2, 3, 255, 256, 1000, 8192, 8193, 100000])
def test_mean_error_bound(oracle_mod, n):
    rng = np.random.default_rng(n)
    a = (np.abs(rng.standard_normal(n)) * np.exp(rng.uniform(-3, 3, n))).astype(np.float32)
    exact = math.fsum(a.astype(np.float64).tolist()) / n
    mu = float(oracle_mod.absmax_mean(a))
    levels = max(1, math.ceil(math.log2(n))) if n > 1 else 0
    assert abs(mu - exact) <= (levels + 2) * F32_EPS * exact


def test_equal_values_are_exact(oracle_mod):
    for n in (1, 7, 256, 300):
        a = np.full((2, n), 0.375, np.float32)
        r = oracle_mod.nf4_absmax_nest(a)
        assert np.all(r["mean"] == np.float32(0.375))
        assert np.all(r["codes"] == 0) and np.all(r["c1"] == 0)
        assert np.array_equal(oracle_mod.nf4_absmax_unnest(r["codes"], r["c1"], r["mean"]), a)


def test_two_valued_block(oracle_mod):
    a = np.tile(np.array([2.0, 4.0], np.float32), 128)[None]   # mean 3, centred +-1
    r = oracle_mod.nf4_absmax_nest(a)
    assert r["mean"][0] == 3.0 and r["c1"][0, 0] == 1.0
    assert np.all(r["codes"][0, 0::2] == 0xFE) and np.all(r["codes"][0, 1::2] == 0x7E)
    assert np.array_equal(oracle_mod.nf4_absmax_unnest(r["codes"], r["c1"], r["mean"]), a)


def _torch_e4m3(x):
    t = torch.from_numpy(np.asarray(x, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("n", [5, 256, 700, 9000])
def test_codes_against_independent_encoding(oracle_mod, n):
    rng = np.random.default_rng(10 + n)
    a = (0.02 * (2.5 + 0.6 * np.abs(rng.standard_normal((3, n))))).astype(np.float32)
    a[1, : min(n, 40)] = 0.0                      # zero absmax blocks (all-zero weights)
    r = oracle_mod.nf4_absmax_nest(a)
    nb = (n + 255) // 256
    for e in range(3):
        mu = np.float32(oracle_mod.absmax_mean(a[e]))
        assert r["mean"][e] == mu
        v = (a[e] - mu).astype(np.float32)
        for b in range(nb):
            vb = v[256 * b: 256 * (b + 1)]
            c1 = np.float32(np.max(np.abs(vb)))
            assert r["c1"][e, b] == c1
            with np.errstate(divide="ignore"):
                k = np.float32(np.minimum(np.float32(448.0) / c1, np.finfo(np.float32).max))
            x = (vb * k).astype(np.float32)
            assert np.array_equal(r["codes"][e, 256 * b: 256 * (b + 1)], _torch_e4m3(x)), (e, b)


def test_unnest_error_bound(oracle_mod):
    rng = np.random.default_rng(3)
    a = (0.01 * np.exp(rng.uniform(-1, 1, (2, 3000)))).astype(np.float32)
    r = oracle_mod.nf4_absmax_nest(a)
    d = oracle_mod.nf4_absmax_unnest(r["codes"], r["c1"], r["mean"]).astype(np.float64)
    nb = r["c1"].shape[1]
    for e in range(2):
        v = np.abs(a[e].astype(np.float64) - float(r["mean"][e]))
        rr = np.repeat(r["c1"][e].astype(np.float64) / 448.0, 256)[: a.shape[1]]
        bound = (2.0 ** -4 * v * (1 + 2.0 ** -20) + 2.0 ** -10 * rr * (1 + 2.0 ** -20)
                 + 4 * F32_EPS * v + F32_EPS * np.abs(d[e]))
        assert np.all(np.abs(d[e] - a[e]) <= bound)
    # the block maxima map to +-448 exactly
    for e in range(2):
        v = a[e] - r["mean"][e]
        for b in range(nb):
            j = 256 * b + int(np.argmax(np.abs(v[256 * b: 256 * (b + 1)])))
            assert r["codes"][e, j] & 0x7F == 0x7E
            assert (r["codes"][e, j] >> 7) == (1 if v[j] < 0 else 0)
