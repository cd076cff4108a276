"""Bit-exact parity over EVERY element of the full-size workloads.

The GPU runs each workload in the launch configuration the benchmark uses;
the oracle then recomputes every output on the host, one expert slice (or one
chunk of tokens) per task on a thread pool (the oracle's C calls release the
interpreter lock, so the tasks run on all host cores):

  * dual-layout NVFP4 + Four-Over-Six of a 32-expert gate_up stack
    [32, 4096, 6144] (four launches with the look-ahead amax), plus the
    transposed dequant of its rowwise copy;
  * the same for the whole 256-expert MoE layer: gate_up [256, 4096, 6144]
    and down [256, 6144, 2048];
  * per-token NVFP4 + Four-Over-Six of activations [16384, 6144] and
    [32768, 2048];
  * NF4 of the 256-expert gate_up stack [256, 4096, 6144] and the routed
    dequant of an 8192-token top-8 Zipf(1.1) router (all 256 experts hit);
  * MXFP8 rowwise + columnwise of the 32-expert stack [32, 4096, 6144] and
    the dequant of its rowwise copy.

Every code byte, scale byte, FP32 scale and absmax, every bf16 output and the
hit list must be identical.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from nvq_testutil import u16

pytestmark = pytest.mark.gpu

WORKERS = max(1, min(32, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def _run(tasks):
    with ThreadPoolExecutor(WORKERS) as ex:
        for f in [ex.submit(t) for t in tasks]:
            f.result()          # re-raises the first mismatch


def _same(a, b, what):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    if not np.array_equal(a.view(np.uint8), b.view(np.uint8)):
        bad = np.argwhere(a.view(np.uint8).reshape(a.shape[0], -1) != b.view(np.uint8).reshape(b.shape[0], -1))
        raise AssertionError("%s differs at %d places, first %s" % (what, len(bad), bad[:3].tolist()))


def test_dual_32_experts_every_element(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 32, 4096, 6144
    w = synth.expert_weights(E, R, K, seed=2, device="cuda")
    r = nvq.nvfp4_quantize_dual(w, four_over_six=True)
    dt = nvq.nvfp4_dequant_t(r["codes_row"], r["scales_row"], r["tensor_scale"])
    torch.cuda.synchronize()
    wh = u16(w)
    h = {k: v.cpu().numpy() for k, v in r.items()}
    dth = u16(dt)
    del w, r, dt
    torch.cuda.empty_cache()

    def one(e):
        x = wh[e:e + 1]
        o = oracle_mod.nvfp4_quantize(x, four_over_six=True)
        _same(h["codes_row"][e:e + 1], o["codes"], "codes_row[%d]" % e)
        _same(h["scales_row"][e:e + 1], o["scales"], "scales_row[%d]" % e)
        _same(h["amax"][e:e + 1], o["amax"], "amax[%d]" % e)
        _same(h["tensor_scale"][e:e + 1], o["G"], "tensor_scale[%d]" % e)
        oc = oracle_mod.nvfp4_quantize_colwise(x, four_over_six=True)
        _same(h["codes_col"][e:e + 1], oc["codes"], "codes_col[%d]" % e)
        _same(h["scales_col"][e:e + 1], oc["scales"], "scales_col[%d]" % e)
        odt = oracle_mod.nvfp4_dequant_t(o["codes"], o["scales"], o["G"], R, K)
        _same(dth[e:e + 1], odt, "dequant_t[%d]" % e)
    _run([lambda e=e: one(e) for e in range(E)])


@pytest.mark.parametrize("E,R,K,seed", [(256, 4096, 6144, 3), (256, 6144, 2048, 4)])
def test_moe_layer_dual_and_dequant_t_every_element(nvq, oracle_mod, E, R, K, seed):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(E, R, K, seed=seed, device="cuda")
    r = nvq.nvfp4_quantize_dual(w, four_over_six=True)
    dt = nvq.nvfp4_dequant_t(r["codes_row"], r["scales_row"], r["tensor_scale"])
    torch.cuda.synchronize()
    chunk = 16                       # experts copied to the host at a time
    for e0 in range(0, E, chunk):
        e1 = min(E, e0 + chunk)
        wh = u16(w[e0:e1])
        h = {k: v[e0:e1].cpu().numpy() for k, v in r.items()}
        dth = u16(dt[e0:e1])

        def one(i, e0=e0, wh=wh, h=h, dth=dth):
            x = wh[i:i + 1]
            o = oracle_mod.nvfp4_quantize(x, four_over_six=True)
            _same(h["codes_row"][i:i + 1], o["codes"], "codes_row[%d]" % (e0 + i))
            _same(h["scales_row"][i:i + 1], o["scales"], "scales_row[%d]" % (e0 + i))
            _same(h["amax"][i:i + 1], o["amax"], "amax[%d]" % (e0 + i))
            _same(h["tensor_scale"][i:i + 1], o["G"], "tensor_scale[%d]" % (e0 + i))
            oc = oracle_mod.nvfp4_quantize_colwise(x, four_over_six=True)
            _same(h["codes_col"][i:i + 1], oc["codes"], "codes_col[%d]" % (e0 + i))
            _same(h["scales_col"][i:i + 1], oc["scales"], "scales_col[%d]" % (e0 + i))
            odt = oracle_mod.nvfp4_dequant_t(o["codes"], o["scales"], o["G"], R, K)
            _same(dth[i:i + 1], odt, "dequant_t[%d]" % (e0 + i))
        _run([lambda i=i: one(i) for i in range(e1 - e0)])
    del w, r, dt
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,H,seed", [(16384, 6144, 5), (32768, 2048, 6)])
def test_activations_every_token(nvq, oracle_mod, T, H, seed):
    from rl_nvfp4_quantize_gb300 import synth
    x = synth.activations(T, H, seed=seed, device="cuda")
    r = nvq.act_quantize_per_token(x, four_over_six=True)
    torch.cuda.synchronize()
    xh = u16(x)
    h = {k: v.cpu().numpy() for k, v in r.items()}
    step = 1024

    def one(t0):
        o = oracle_mod.act_quantize_per_token(xh[t0:t0 + step], four_over_six=True)
        _same(h["codes"][t0:t0 + step], o["codes"], "codes[%d:]" % t0)
        _same(h["scales"][t0:t0 + step], o["scales"], "scales[%d:]" % t0)
        _same(h["token_scale"][t0:t0 + step], o["token_scale"], "token_scale[%d:]" % t0)
    _run([lambda t0=t0: one(t0) for t0 in range(0, T, step)])


def test_nf4_256_experts_and_routed_dequant_every_element(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 256, 4096, 6144
    w = synth.expert_weights(E, R, K, seed=7, device="cuda")
    q = nvq.nf4_quantize(w)
    topk = synth.zipf_router(8192, E, 8, seed=8, device="cuda")
    d, hl, nh = nvq.nf4_dequant_routed(q["codes"], q["absmax"], topk)
    torch.cuda.synchronize()
    hit, n, st = oracle_mod.routed_union(topk.cpu().numpy(), E)
    assert int(nh.item()) == n and st == 0
    _same(hl.cpu().numpy(), hit, "hit list")
    hitset = set(hit[:n].tolist())
    chunk = 16                       # experts copied to the host at a time

    for e0 in range(0, E, chunk):
        wh = u16(w[e0:e0 + chunk])
        ch = q["codes"][e0:e0 + chunk].cpu().numpy()
        ah = q["absmax"][e0:e0 + chunk].cpu().numpy()
        dh = u16(d[e0:e0 + chunk])

        def one(i, e0=e0, wh=wh, ch=ch, ah=ah, dh=dh):
            o = oracle_mod.nf4_quantize(wh[i:i + 1])
            _same(ch[i:i + 1], o["codes"], "nf4 codes[%d]" % (e0 + i))
            _same(ah[i:i + 1], o["absmax"], "nf4 absmax[%d]" % (e0 + i))
            if e0 + i in hitset:
                od = oracle_mod.nf4_dequant(o["codes"], o["absmax"], 1, R, K)
                _same(dh[i:i + 1], od, "routed dequant[%d]" % (e0 + i))
        _run([lambda i=i: one(i) for i in range(min(chunk, E - e0))])
    del w, q, d
    torch.cuda.empty_cache()


def test_mxfp8_32_experts_every_element(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 32, 4096, 6144
    w = synth.expert_weights(E, R, K, seed=23, device="cuda")
    q = nvq.mxfp8_quantize(w, columnwise=True)
    d = nvq.mxfp8_dequant(q["codes_row"], q["scales_row"])
    torch.cuda.synchronize()
    wh = u16(w)
    h = {k: v.cpu().numpy() for k, v in q.items()}
    dh = u16(d)
    del w, q, d
    torch.cuda.empty_cache()

    def one(e):
        x = wh[e:e + 1]
        o = oracle_mod.mxfp8_quantize(x)
        _same(h["codes_row"][e:e + 1], o["codes"], "mx codes_row[%d]" % e)
        _same(h["scales_row"][e:e + 1], o["scales"], "mx scales_row[%d]" % e)
        oc = oracle_mod.mxfp8_quantize_colwise(x)
        _same(h["codes_col"][e:e + 1], oc["codes"], "mx codes_col[%d]" % e)
        _same(h["scales_col"][e:e + 1], oc["scales"], "mx scales_col[%d]" % e)
        _same(dh[e:e + 1], oracle_mod.mxfp8_dequant(o["codes"], o["scales"]), "mx dequant[%d]" % e)
    _run([lambda e=e: one(e) for e in range(E)])
