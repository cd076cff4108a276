"""Y = X . DQ(W_e)^T on the tensor cores, fused with the NF4 dequantisation of
each routed expert ("nf4moe -- QLoRA for a 743B Fused-MoE", "The fix:
dequant-on-forward for routed experts"), against the oracle's float64
evaluation.

Both sides read the same NF4 codes and absmax, made by the oracle.  The
tensor cores accumulate in FP32 in an order of their own and Y is the bf16
round to nearest even of that sum, so the check is
|Y - Y_exact| <= 2^-8 (|Y_exact| + d) + d with d = in * 2^-23 * (|X| . |DQ|^T):
every FP32 partial sum is a sum of at most `in` products, each addition
rounded once (2^-23 rather than 2^-24 to allow for truncation), and the bf16
rounding adds at most half a bf16 unit, 2^-8 relative.  A separate case uses
blocks with absmax 1 and X in {-1, 0, 1}, where every sum is exact in FP32 and
the result must be the bf16 round of the exact value, bit for bit.
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


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_rne_of_f32(v):
    """float32-exact values -> bf16 bits (round to nearest even)."""
    u = np.asarray(v, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _run(nvq, oq, xh, counts):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = nvq.nf4_routed_linear(bf16_from_u16(xh), counts, torch.from_numpy(oq["codes"]).cuda(),
                              torch.from_numpy(oq["absmax"]).cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return u16(y)


def _check(nvq, oracle_mod, E, out, inn, counts, seed):
    from rl_nvfp4_quantize_gb300 import synth
    oq = oracle_mod.nf4_quantize(u16(synth.expert_weights(E, out, inn, seed=seed)))
    xh = u16(synth.activations(sum(counts), inn, seed=seed + 1))
    got = _f64(_run(nvq, oq, xh, counts))
    ref, bound = oracle_mod.nf4_routed_linear(xh, counts, oq["codes"], oq["absmax"], out, inn)
    d = inn * 2.0 ** -23 * bound
    tol = 2.0 ** -8 * (np.abs(ref) + d) + d
    err = np.abs(got - ref)
    assert np.all(err <= tol), "max excess %g at %s" % (
        (err - tol).max(), np.unravel_index(np.argmax(err - tol), err.shape))


@pytest.mark.parametrize("E,out,inn,counts", [
    (1, 256, 256, [128]),     # one tile, four K steps (one absmax fetch)
    (1, 256, 256, [1]),       # one token
    (1, 512, 512, [300]),     # two token tiles (ragged), two column tiles, eight K steps
])
def test_nf4_linear_tiny(nvq, oracle_mod, E, out, inn, counts):
    _check(nvq, oracle_mod, E, out, inn, counts, seed=out + inn)


@pytest.mark.parametrize("E,out,inn,counts", [
    (3, 256, 256, [5, 0, 130]),
    (2, 512, 512, [200, 77]),
    (4, 512, 768, [129, 128, 0, 300]),
    (5, 768, 1280, [64, 1, 255, 256, 257]),
])
def test_nf4_linear_grouped_ragged(nvq, oracle_mod, E, out, inn, counts):
    _check(nvq, oracle_mod, E, out, inn, counts, seed=out * 3 + inn)


def test_nf4_linear_exact_values_bit_identical(nvq, oracle_mod):
    """Blocks with absmax 1 dequantise to the bf16 levels (multiples of 2^-11
    in [-1, 1]); with X in {-1, 0, 1} every partial sum is exact in FP32, so Y
    is the bf16 round of the exact sum."""
    from test_oracle_nvfp4 import bf16
    E, out, inn = 2, 256, 512
    rng = np.random.default_rng(12)
    w = rng.uniform(-1, 1, (E, out, inn))
    w[:, :, ::64] = 1.0
    oq = oracle_mod.nf4_quantize(bf16(w))
    assert np.all(oq["absmax"] == 1.0)
    counts = [100, 156]
    xh = bf16(rng.integers(-1, 2, (sum(counts), inn)).astype(np.float64))
    got = _run(nvq, oq, xh, counts)
    ref, _ = oracle_mod.nf4_routed_linear(xh, counts, oq["codes"], oq["absmax"], out, inn)
    assert np.array_equal(got, _bf16_rne_of_f32(ref))


def test_nf4_linear_empty_and_zero_k(nvq):
    codes = torch.zeros((2, 256, 128), dtype=torch.uint8, device="cuda")
    absmax = torch.ones((2, 256, 4), dtype=torch.float32, device="cuda")
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    y = nvq.nf4_routed_linear(x, [0, 0], codes, absmax)
    assert y.shape == (0, 256)
    # an empty contraction writes zeros over whatever the output held
    x0 = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    y0 = torch.full((5, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    nvq.nf4_routed_linear(x0, [2, 3], torch.empty((2, 256, 0), dtype=torch.uint8, device="cuda"),
                          torch.empty((2, 256, 0), dtype=torch.float32, device="cuda"), out=y0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y0).item() == 0
