"""dX = dY . DQ(Q(W_e)) on the tensor cores, fused with the dequantisation of
the rowwise NVFP4 copy, against the oracle's float64 evaluation.

The tensor cores accumulate in FP32 in an order of their own, so the check is
|dX - dX_exact| <= out * 2^-23 * (|dY| . |DQ|): every partial sum is a sum of
at most `out` products, each addition rounded once (with 2^-23 instead of
2^-24 for the rounding unit, to allow for truncation).  A separate case uses a
weight whose dequantised values and an integer dY make every sum exact, where
the result must match bit for bit.  Both sides read the rowwise NVFP4 copy
the oracle makes of the weight.
"""
import numpy as np
import pytest
import torch

from nvq_testutil import u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def _check(nvq, oracle_mod, w, dy, counts):
    """Both sides read the rowwise copy the oracle makes of w."""
    E, out, inn = w.shape
    q = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dx = nvq.nvfp4_dgrad(dy, counts, torch.from_numpy(q["codes"]).cuda(),
                         torch.from_numpy(q["scales"]).cuda(), torch.from_numpy(q["G"]).cuda(),
                         status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, bound = oracle_mod.nvfp4_dgrad(u16(dy), counts, q["codes"], q["scales"], q["G"], out, inn)
    got = dx.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    tol = out * 2.0 ** -23 * bound + 1e-30
    assert np.all(err <= tol), "max err %g at %s (tol %g)" % (
        err.max(), np.unravel_index(np.argmax(err - tol), err.shape), tol.flat[np.argmax(err - tol)])
    return got, ref


@pytest.mark.parametrize("E,out,inn,counts", [
    (1, 64, 256, [128]),      # one tile, one K step
    (1, 64, 256, [1]),        # one token
    (1, 128, 512, [130]),     # two token tiles (ragged), two column tiles, two K steps
])
def test_dgrad_tiny(nvq, oracle_mod, E, out, inn, counts):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(E, out, inn, seed=out + inn, device="cuda")
    dy = synth.activations(sum(counts), out, seed=5, device="cuda")
    _check(nvq, oracle_mod, w, dy, counts)


@pytest.mark.parametrize("E,out,inn,counts", [
    (3, 128, 256, [5, 0, 130]),
    (2, 256, 512, [200, 77]),
    (4, 512, 768, [129, 128, 0, 300]),
    (5, 1024, 1024, [64, 1, 255, 256, 257]),
])
def test_dgrad_grouped_ragged(nvq, oracle_mod, E, out, inn, counts):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(E, out, inn, seed=out * 3 + inn, device="cuda")
    dy = synth.activations(sum(counts), out, seed=inn, device="cuda")
    _check(nvq, oracle_mod, w, dy, counts)


def test_dgrad_exact_values_bit_identical(nvq, oracle_mod):
    """Dequantised weight values on the E2M1 grid (G = 1, S = 1 for the
    blocks) and dY in {-1, 0, 1}: every product and partial sum is exact in
    FP32, so the tensor-core result equals the exact one bit for bit."""
    E, out, inn = 2, 256, 512
    rng = np.random.default_rng(11)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    w = grid[rng.integers(0, 8, (E, out, inn))] * np.where(rng.random((E, out, inn)) < 0.5, -1, 1)
    w[:, :, ::16] = 6.0          # every 16-block has amax 6 ...
    w[:, 0, 1] = 1536.0          # ... and each slice amax 1536, so G = 1 under Four-Over-Six
    wt = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).cuda()
    counts = [100, 156]
    dyf = rng.integers(-1, 2, (sum(counts), out)).astype(np.float32)
    dy = torch.from_numpy(dyf).to(torch.bfloat16).cuda()
    got, ref = _check(nvq, oracle_mod, wt, dy, counts)
    assert np.array_equal(got, ref)


def test_dgrad_status_and_empty(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(2, 64, 256, seed=1, device="cuda")
    q = nvq.nvfp4_quantize(w, four_over_six=True)
    dy = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    dx = nvq.nvfp4_dgrad(dy, [0, 0], q["codes"], q["scales"], q["tensor_scale"])
    assert dx.shape == (0, 256)
    # an empty contraction (out = 0) writes zeros over whatever dX held
    u8 = torch.uint8
    dx0 = torch.full((5, 256), 7.0, dtype=torch.float32, device="cuda")
    nvq.nvfp4_dgrad(torch.empty((5, 0), dtype=torch.bfloat16, device="cuda"), [2, 3],
                    torch.empty((2, 0, 128), dtype=u8, device="cuda"),
                    torch.empty((2, 0, 16), dtype=u8, device="cuda"), q["tensor_scale"], out=dx0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dx0).item() == 0
