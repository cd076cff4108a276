"""GPU parity of the nested (double-quantised) NF4 absmax against the oracle:
nf4_absmax_nest bit for bit (codes, block maxima c1, slice means) and
nf4_absmax_unnest bit for bit, over ragged lengths that exercise every load
and store path, several 4096-value chunks of the tree sum, the full
[256, 4096 x 6144 / 64] absmax of a gate_up stack, and the chain
NF4 quantise -> nest -> unnest -> NF4 dequantise."""
import numpy as np
import pytest
import torch

from nvq_testutil import Guarded, assert_same, f32, u8, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def _check_nest(nvq, oracle_mod, a_cpu):
    E, n = a_cpu.shape
    nb = (n + 255) // 256
    gc, g1, gm = Guarded((E, n), torch.uint8), Guarded((E, nb), torch.float32), Guarded((E,), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = nvq.nf4_absmax_nest(a_cpu.cuda(), status=status, out=dict(codes=gc.t, c1=g1.t, mean=gm.t))
    torch.cuda.synchronize()
    assert gc.intact() and g1.intact() and gm.intact()
    o = oracle_mod.nf4_absmax_nest(a_cpu.numpy())
    assert_same(f32(r["mean"]).view(np.uint32), o["mean"].view(np.uint32), "mean")
    assert_same(f32(r["c1"]).view(np.uint32), o["c1"].view(np.uint32), "c1")
    assert_same(u8(r["codes"]), o["codes"], "codes")
    assert int(status.item()) == 0
    gu = Guarded((E, n), torch.float32)
    d = nvq.nf4_absmax_unnest(torch.from_numpy(o["codes"]).cuda(), torch.from_numpy(o["c1"]).cuda(),
                              torch.from_numpy(o["mean"]).cuda(), out=gu.t)
    torch.cuda.synchronize()
    assert gu.intact()
    ref = oracle_mod.nf4_absmax_unnest(o["codes"], o["c1"], o["mean"])
    assert_same(f32(d).view(np.uint32), ref.view(np.uint32), "unnest")


@pytest.mark.parametrize("E,n", [(1, 1), (1, 5), (2, 255), (3, 256), (2, 257), (2, 1000), (2, 4096),
                                 (2, 4097), (3, 8192 + 13), (2, 40000), (1, 3 * 4096 * 5 + 8),
                                 (5, 96 * 64)])
def test_nest_unnest_parity(nvq, oracle_mod, E, n):
    from rl_nvfp4_quantize_gb300 import synth
    _check_nest(nvq, oracle_mod, synth.nf4_absmax_values(E, n, seed=E * 7919 + n))


def test_nest_degenerate_slices(nvq, oracle_mod):
    """All-equal slices (mean exact, every code 0), all-zero slices, and a
    slice with one large value."""
    a = torch.full((3, 700), 0.046875)
    a[1] = 0.0
    a[2, 123] = 1.0
    _check_nest(nvq, oracle_mod, a)


def test_nest_misaligned_input(nvq, oracle_mod):
    """A 4- but not 16-byte aligned absmax array takes the scalar loads."""
    from rl_nvfp4_quantize_gb300 import synth
    a = synth.nf4_absmax_values(2, 1024, seed=5)
    buf = torch.empty(a.numel() + 1, dtype=torch.float32, device="cuda")
    av = buf[1:].view(2, 1024)
    av.copy_(a.cuda())
    assert av.data_ptr() % 16 != 0
    r = nvq.nf4_absmax_nest(av)
    o = oracle_mod.nf4_absmax_nest(a.numpy())
    assert_same(u8(r["codes"]), o["codes"], "codes")
    assert_same(f32(r["mean"]).view(np.uint32), o["mean"].view(np.uint32), "mean")


def test_nest_empty_and_nonfinite(nvq):
    r = nvq.nf4_absmax_nest(torch.empty((3, 0), dtype=torch.float32, device="cuda"))
    assert r["codes"].shape == (3, 0) and torch.equal(r["mean"], torch.zeros(3, device="cuda"))
    a = torch.full((2, 300), 0.5, device="cuda")
    a[1, 7] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nvq.nf4_absmax_nest(a, status=status)
    assert int(status.item()) & nvq.STATUS_NONFINITE


def test_nest_full_gate_up_every_element(nvq, oracle_mod):
    """The absmax of a [256, 4096, 6144] stack: 256 slices of 393216 values."""
    from rl_nvfp4_quantize_gb300 import synth
    _check_nest(nvq, oracle_mod, synth.nf4_absmax_values(256, 4096 * 6144 // 64, seed=11))


def test_nf4_chain_with_nested_absmax(nvq, oracle_mod):
    """NF4 quantise -> nest the absmax -> unnest -> dequantise, each step on the
    GPU, equals the same chain in the oracle."""
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 3, 96, 640
    w = synth.expert_weights(E, R, K, seed=21)
    q = nvq.nf4_quantize(w.cuda())
    nest = nvq.nf4_absmax_nest(q["absmax"])
    am = nvq.nf4_absmax_unnest(nest["codes"], nest["c1"], nest["mean"], shape=q["absmax"].shape)
    d = nvq.nf4_dequant(q["codes"], am)
    o = oracle_mod.nf4_quantize(u16(w))
    on = oracle_mod.nf4_absmax_nest(o["absmax"].reshape(E, -1))
    oam = oracle_mod.nf4_absmax_unnest(on["codes"], on["c1"], on["mean"]).reshape(o["absmax"].shape)
    assert_same(f32(am).view(np.uint32), oam.view(np.uint32), "unnested absmax")
    assert_same(u16(d), oracle_mod.nf4_dequant(o["codes"], oam, E, R, K), "dequant")
