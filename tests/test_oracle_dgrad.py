"""Pins of the oracle's dgrad through the dequantised weight (host only).

dX = dY . DQ(Q(W_e)) per expert ("The 4-bitter Lesson", "Key claims":
dequantised backward).  The oracle forms it with one float64 matrix product
per expert; these tests check it against a plain triple loop over the same
bf16 values, against the layout rules (token rows grouped by expert, empty
experts), and the bound |dX| <= |dY| . |DQ|.
"""
import numpy as np
import pytest


def _bits_to_f64(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(oracle_mod, E, out, inn, counts, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((E, out, inn)) * 0.05).astype(np.float32)
    wb = (w.view(np.uint32) >> 16).astype(np.uint16)
    q = oracle_mod.nvfp4_quantize(wb, four_over_six=True)
    T = sum(counts)
    dy = ((rng.standard_normal((T, out)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    return q, dy


@pytest.mark.parametrize("E,out,inn,counts", [(1, 16, 16, [3]), (3, 32, 16, [2, 0, 3]), (2, 48, 32, [1, 4])])
def test_dgrad_against_triple_loop(oracle_mod, E, out, inn, counts):
    q, dy = _case(oracle_mod, E, out, inn, counts, seed=E * 7 + out)
    dx, bound = oracle_mod.nvfp4_dgrad(dy, counts, q["codes"], q["scales"], q["G"], out, inn)
    t0 = 0
    for e, c in enumerate(counts):
        wd = _bits_to_f64(oracle_mod.nvfp4_dequant(q["codes"][e:e + 1], q["scales"][e:e + 1],
                                                    q["G"][e:e + 1], out, inn)[0])
        for t in range(t0, t0 + c):
            a = _bits_to_f64(dy[t])
            for i in range(inn):
                s = sum(a[o] * wd[o, i] for o in range(out))
                b = sum(abs(a[o] * wd[o, i]) for o in range(out))
                assert abs(dx[t, i] - s) <= 1e-12 * max(b, 1e-300)
                assert abs(bound[t, i] - b) <= 1e-12 * max(b, 1e-300)
        t0 += c
    assert np.all(np.abs(dx) <= bound * (1 + 1e-12))


def test_dgrad_of_exact_values_is_exact(oracle_mod):
    """A weight whose dequantised values are small dyadic numbers and an
    integer dY give exact sums: the oracle must return them exactly."""
    out, inn = 32, 16
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    rng = np.random.default_rng(3)
    w = grid[rng.integers(0, 8, (1, out, inn))] * np.where(rng.random((1, out, inn)) < 0.5, -1, 1)
    w[0, :, 0] = 6.0                     # every 16-block has amax 6
    w[0, 0, 1] = 1536.0                  # tensor amax 1536: G = 1 under Four-Over-Six
    wb = (w.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q = oracle_mod.nvfp4_quantize(wb, four_over_six=True)
    assert q["G"][0] == 1.0
    dyf = rng.integers(-2, 3, (5, out)).astype(np.float32)
    dy = (dyf.view(np.uint32) >> 16).astype(np.uint16)
    dx, _ = oracle_mod.nvfp4_dgrad(dy, [5], q["codes"], q["scales"], q["G"], out, inn)
    wd = _bits_to_f64(oracle_mod.nvfp4_dequant(q["codes"], q["scales"], q["G"], out, inn)[0])
    assert np.array_equal(dx, dyf.astype(np.float64) @ wd)
    assert np.array_equal(wd[:, 2:16][wd[:, 2:16] != 0] % 0.5, np.zeros(np.count_nonzero(wd[:, 2:16])))
