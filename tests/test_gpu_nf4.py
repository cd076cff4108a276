"""GPU parity of the NF4 entry points and the routed union against the oracle."""
import numpy as np
import pytest
import torch

from nvq_testutil import Guarded, assert_same, f32, u8, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


@pytest.mark.parametrize("shape", [(1, 1, 64), (1, 4, 64), (3, 17, 192), (2, 64, 6144), (5, 33, 128),
                                   (1, 2, 64 * 1000)])
def test_nf4_quantize_dequant_parity(nvq, oracle_mod, shape):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(*shape, seed=sum(shape))
    E, R, K = shape
    gc, ga = Guarded((E, R, K // 2), torch.uint8), Guarded((E, R, K // 64), torch.float32)
    r = nvq.nf4_quantize(w.cuda(), out=dict(codes=gc.t, absmax=ga.t))
    gd = Guarded((E, R, K), torch.bfloat16)
    d = nvq.nf4_dequant(r["codes"], r["absmax"], out=gd.t)
    torch.cuda.synchronize()
    assert gc.intact() and ga.intact() and gd.intact()
    o = oracle_mod.nf4_quantize(u16(w))
    assert_same(f32(r["absmax"]).view(np.uint32), o["absmax"].view(np.uint32), "absmax")
    assert_same(u8(r["codes"]), o["codes"], "codes")
    assert_same(u16(d), oracle_mod.nf4_dequant(o["codes"], o["absmax"], E, R, K), "dequant")


def test_nf4_stack_16_byte_aligned(nvq, oracle_mod):
    """A stack that is 16- but not 32-byte aligned takes the 16-byte loads
    instead of the 32-byte ones: same bytes as the oracle."""
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 2, 48, 320
    w = synth.expert_weights(E, R, K, seed=91)
    buf = torch.empty(w.numel() + 8, dtype=torch.bfloat16, device="cuda")
    wv = buf[8:].view(E, R, K)
    wv.copy_(w.cuda())
    assert wv.data_ptr() % 32 == 16
    r = nvq.nf4_quantize(wv)
    o = oracle_mod.nf4_quantize(u16(w))
    assert_same(f32(r["absmax"]).view(np.uint32), o["absmax"].view(np.uint32), "absmax")
    assert_same(u8(r["codes"]), o["codes"], "codes")


def test_nf4_every_bf16_value(nvq, oracle_mod):
    """All finite bf16 patterns, in blocks whose maximum is 1.0 and 300.0."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    for A in (1.0, 300.0):
        keep = pats[np.isfinite(f) & (np.abs(f) <= A)]
        keep = keep[: (keep.size // 63) * 63].reshape(-1, 63)
        head = torch.tensor([A], dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]
        blocks = np.concatenate([np.full((keep.shape[0], 1), head, np.uint16), keep], 1).reshape(1, -1, 64)
        w = torch.from_numpy(blocks.view(np.int16).copy()).view(torch.bfloat16)
        r = nvq.nf4_quantize(w.cuda())
        o = oracle_mod.nf4_quantize(blocks)
        assert_same(u8(r["codes"]), o["codes"], "codes A=%g" % A)


def test_nf4_zero_and_status(nvq, oracle_mod):
    w = torch.zeros((1, 2, 128), dtype=torch.bfloat16)
    w[0, 1, 70] = -2.0
    w[0, 1, 71] = -0.0
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = nvq.nf4_quantize(w.cuda(), status=st)
    o = oracle_mod.nf4_quantize(u16(w))
    assert_same(u8(r["codes"]), o["codes"])
    assert int(st.item()) == 0
    w[0, 0, 5] = float("nan")
    nvq.nf4_quantize(w.cuda(), status=st)
    assert int(st.item()) & nvq.STATUS_NONFINITE


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (5, 2, 7), (8, 8, 256), (32, 8, 256), (8192, 8, 256),
                                   (3000, 4, 4096)])
def test_routed_dequant_parity(nvq, oracle_mod, T, k, E):
    from rl_nvfp4_quantize_gb300 import synth
    R, K = 4, 128
    w = synth.expert_weights(E, R, K, seed=T + E)
    q = nvq.nf4_quantize(w.cuda())
    topk = synth.zipf_router(T, E, k, seed=T * 7 + E)
    dst = torch.full((E, R, K), 12345, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    d, hl, nh = nvq.nf4_dequant_routed(q["codes"], q["absmax"], topk.cuda(), dst=dst)
    ref = np.full((E, R, K), 12345, np.uint16)
    hit, n, st = oracle_mod.nf4_dequant_routed(u8(q["codes"]), f32(q["absmax"]), E, R, K,
                                               topk.numpy(), ref)
    assert int(nh.item()) == n
    assert_same(hl.cpu().numpy(), hit, "hit_list")
    assert_same(u16(d), ref, "dst")


def test_routed_union_bad_indices_and_empty(nvq, oracle_mod):
    E, R, K = 6, 2, 64
    w = torch.randn(E, R, K).to(torch.bfloat16)
    q = nvq.nf4_quantize(w.cuda())
    topk = torch.tensor([[0, 5], [9, -1], [5, 2]], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d, hl, nh = nvq.nf4_dequant_routed(q["codes"], q["absmax"], topk.cuda(), status=st)
    assert int(nh.item()) == 3 and hl.cpu().tolist() == [0, 2, 5, -1, -1, -1]
    assert int(st.item()) == nvq.STATUS_BAD_INDEX
    empty = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    d, hl, nh = nvq.nf4_dequant_routed(q["codes"], q["absmax"], empty)
    assert int(nh.item()) == 0 and hl.cpu().tolist() == [-1] * E
