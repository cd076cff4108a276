"""Randomised grouped GEMMs: nvfp4_dgrad and nf4_routed_linear on seeded
random expert counts, shapes and per-expert token counts (zeros, single
tokens, counts just past a 128-row half tile), each checked against the
oracle's float64 product within the FP32-accumulation bound of its own test
file.  The cases are drawn once from a fixed seed."""
import numpy as np
import pytest

import test_gpu_dgrad as dg
import test_gpu_nf4_linear as nl

pytestmark = pytest.mark.gpu

_RNG = np.random.default_rng(4242)


def _counts(E):
    c = []
    for _ in range(E):
        r = _RNG.random()
        if r < 0.2:
            c.append(0)
        elif r < 0.3:
            c.append(1)
        elif r < 0.5:
            c.append(int(_RNG.choice([127, 128, 129, 255, 256, 257])))
        else:
            c.append(int(_RNG.integers(2, 400)))
    if sum(c) == 0:
        c[0] = 3
    return c


def _cases(n, out_mult, in_mult, max_out, max_in):
    out = []
    for _ in range(n):
        E = int(_RNG.integers(1, 12))
        o = int(_RNG.integers(1, max_out // out_mult + 1)) * out_mult
        i = int(_RNG.integers(1, max_in // in_mult + 1)) * in_mult
        out.append((E, o, i, _counts(E)))
    return out


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


@pytest.mark.parametrize("E,out,inn,counts", _cases(6, 64, 256, 640, 1280))
def test_dgrad_random(nvq, oracle_mod, E, out, inn, counts):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(E, out, inn, seed=E * 31 + out + inn, device="cuda")
    dy = synth.activations(sum(counts), out, seed=out + 7, device="cuda")
    dg._check(nvq, oracle_mod, w, dy, counts)


@pytest.mark.parametrize("E,out,inn,counts", _cases(6, 256, 256, 1024, 1280))
def test_nf4_linear_random(nvq, oracle_mod, E, out, inn, counts):
    nl._check(nvq, oracle_mod, E, out, inn, counts, seed=E * 37 + out + inn)
