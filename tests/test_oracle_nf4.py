"""Pins of the oracle's NF4 path and routed-expert union.

The NF4 levels are pinned to the published NF4 values of the QLoRA paper
(tests/golden/nf4_levels_qlora.json) and re-derived with scipy's normal
quantile function (independent of the oracle's bisection over erfc); the
quantiser is checked against a brute-force nearest-level search; dequant
against torch's bfloat16 cast of the FP32 products; the union against a
Python set.  Source: "nf4moe -- QLoRA for a 743B Fused-MoE", "The fix:
dequant-on-forward for routed experts" (NF4, blocksize 64, one-hot union of
top_k_index).
"""
import json
from pathlib import Path

import numpy as np
import pytest
import torch
from scipy.stats import norm

from test_oracle_nvfp4 import bf16, bf16_to_float


GOLDEN = Path(__file__).parent / "golden" / "nf4_levels_qlora.json"


def test_codebook_equals_published_nf4(oracle_mod):
    """The oracle's levels are the published NF4 values (QLoRA appendix),
    bit for bit as binary32 and to the printed precision."""
    pub = np.array(json.loads(GOLDEN.read_text())["values"], np.float64)
    cb = oracle_mod.nf4_codebook()
    assert np.array_equal(cb.view(np.uint32), pub.astype(np.float32).view(np.uint32))
    assert np.all(np.abs(cb.astype(np.float64) - pub) < 5e-8)


def test_codebook_is_the_normal_quantile_construction(oracle_mod):
    """Independent restatement with scipy's normal quantile, everything in
    double, at the outer probability 1 - (1/32 + 1/30)/2: every level agrees
    within a few binary32 units (the binary32 probabilities of the published
    values move them by less than 1e-6).  The same construction at the
    outer probability 31/32 is far off, so a wrong offset cannot pass."""
    def construct(delta):
        top = norm.ppf(delta)
        neg = [-norm.ppf(0.5 + j * (delta - 0.5) / 7) / top for j in range(7, 0, -1)]
        pos = [norm.ppf(0.5 + j * (delta - 0.5) / 8) / top for j in range(1, 9)]
        return np.array(neg + [0.0] + pos)

    cb = oracle_mod.nf4_codebook().astype(np.float64)
    assert np.max(np.abs(cb - construct(1 - (1 / 32 + 1 / 30) / 2))) < 1e-6
    assert np.max(np.abs(cb - construct(31 / 32))) > 1e-3


def test_codebook_structure(oracle_mod):
    cb = oracle_mod.nf4_codebook()
    assert cb.shape == (16,) and np.all(np.diff(cb) > 0)
    assert cb[0] == -1.0 and cb[7] == 0.0 and cb[15] == 1.0
    assert (cb < 0).sum() == 7 and (cb > 0).sum() == 8
    # normal quantiles: levels thin out towards the tails
    assert np.all(np.diff(cb[7:]) [1:] >= np.diff(cb[7:])[:-1] * 0.99)


def _nearest_level(v, cb):
    """Brute force: nearest level in float64, exact ties to the lower index."""
    d = np.abs(v[:, None].astype(np.float64) - cb[None, :].astype(np.float64))
    return np.argmin(d, axis=1).astype(np.uint8)  # argmin returns the first (lower) index


def _unpack(codes):
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


def test_nf4_quantize_brute_force(oracle_mod):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 8, 128)) * 0.02
    x[rng.random(x.shape) < 0.01] *= 30
    w = bf16(x)
    r = oracle_mod.nf4_quantize(w)
    cb = oracle_mod.nf4_codebook()
    xf = bf16_to_float(w).reshape(-1, 64)
    am = np.abs(xf).max(axis=1)
    assert np.array_equal(r["absmax"].ravel(), am.astype(np.float32))
    v = (xf * (np.float32(1) / am.astype(np.float32))[:, None]).astype(np.float32)
    ref = _nearest_level(v.ravel(), cb)
    got = _unpack(r["codes"]).ravel()
    mids = ((cb[:-1] + cb[1:]) * np.float32(0.5)).astype(np.float32)
    near_mid = np.min(np.abs(v.ravel()[:, None] - mids[None, :]), axis=1) < 1e-6
    assert np.array_equal(got[~near_mid], ref[~near_mid])


def test_nf4_all_bf16_inputs_match_brute_force(oracle_mod):
    """Every finite bf16 value in [-A, A] under several block maxima A.

    No bf16 input lands exactly on an FP32 midpoint of this level table (a
    search over all normal bf16 block maxima found none), so the stated tie
    rule never decides a code; the nearest level is unique everywhere."""
    cb = oracle_mod.nf4_codebook()
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = bf16_to_float(pats)
    for A in (1.0, 0.0234375, 3.5, 300.0):
        keep = np.isfinite(f) & (np.abs(f) <= A)
        vals = pats[keep]
        vals = vals[: (vals.size // 63) * 63].reshape(-1, 63)
        head = np.full((vals.shape[0], 1), bf16([A])[0], np.uint16)
        blocks = np.concatenate([head, vals], axis=1)
        r = oracle_mod.nf4_quantize(blocks.reshape(1, -1, 64))
        assert np.all(r["absmax"] == np.float32(A))
        v = (bf16_to_float(blocks) * (np.float32(1) / np.float32(A))).astype(np.float32).ravel()
        mids = ((cb[:-1] + cb[1:]) * np.float32(0.5)).astype(np.float32)
        assert not np.isin(v, mids).any()
        assert np.array_equal(_unpack(r["codes"]).ravel(), _nearest_level(v, cb))


def test_nf4_dequant_matches_torch(oracle_mod):
    rng = np.random.default_rng(3)
    w = bf16(rng.standard_normal((1, 4, 192)) * 0.05)
    r = oracle_mod.nf4_quantize(w)
    d = oracle_mod.nf4_dequant(r["codes"], r["absmax"], 1, 4, 192)
    cb = oracle_mod.nf4_codebook()
    c = _unpack(r["codes"])
    y = (cb[c] * np.repeat(r["absmax"], 64, axis=-1)).astype(np.float32)
    assert np.array_equal(d, bf16(y))


def test_nf4_bounded_and_idempotent(oracle_mod):
    rng = np.random.default_rng(4)
    w = bf16(rng.standard_normal((2, 16, 128)) * rng.uniform(0.01, 2))
    r1 = oracle_mod.nf4_quantize(w)
    d1 = oracle_mod.nf4_dequant(r1["codes"], r1["absmax"], 2, 16, 128)
    assert np.all(np.abs(bf16_to_float(d1)).reshape(-1, 64).max(axis=1)
                  <= r1["absmax"].ravel())
    r2 = oracle_mod.nf4_quantize(d1)
    assert np.array_equal(r1["codes"], r2["codes"])
    assert np.array_equal(r1["absmax"], r2["absmax"])


def test_nf4_zero_block_and_status(oracle_mod):
    w = np.zeros((1, 1, 128), np.uint16)
    w[0, 0, 64] = bf16([-2.0])[0]
    w[0, 0, 65] = 0x8000  # -0
    r = oracle_mod.nf4_quantize(w)
    assert r["absmax"][0, 0, 0] == 0 and r["absmax"][0, 0, 1] == 2.0
    c = _unpack(r["codes"]).ravel()
    assert np.all(c[:64] == 7) and c[64] == 0 and c[65] == 7
    w[0, 0, 3] = 0x7F80  # +inf
    assert oracle_mod.nf4_quantize(w)["status"] & oracle_mod.STATUS_NONFINITE


def test_routed_union_against_set(oracle_mod):
    rng = np.random.default_rng(5)
    for T, k, E in ((1, 1, 1), (7, 2, 5), (64, 8, 256), (300, 4, 40)):
        topk = rng.integers(0, E, (T, k)).astype(np.int32)
        hit, n, st = oracle_mod.routed_union(topk, E)
        ref = sorted(set(topk.ravel().tolist()))
        assert n == len(ref) and list(hit[:n]) == ref and np.all(hit[n:] == -1) and st == 0
    topk = np.array([[0, 3], [9, -1]], np.int32)
    hit, n, st = oracle_mod.routed_union(topk, 4)
    assert list(hit[:n]) == [0, 3] and st == oracle_mod.STATUS_BAD_INDEX


def test_routed_dequant_writes_only_hit_slices(oracle_mod):
    rng = np.random.default_rng(6)
    E, R, C = 6, 4, 128
    w = bf16(rng.standard_normal((E, R, C)) * 0.02)
    r = oracle_mod.nf4_quantize(w)
    full = oracle_mod.nf4_dequant(r["codes"], r["absmax"], E, R, C)
    topk = np.array([[4, 1], [1, 4], [0, 4]], np.int32)
    dst = np.full((E, R, C), 0xABCD, np.uint16)
    hit, n, st = oracle_mod.nf4_dequant_routed(r["codes"], r["absmax"], E, R, C, topk, dst)
    assert list(hit[:n]) == [0, 1, 4]
    for e in range(E):
        if e in (0, 1, 4):
            assert np.array_equal(dst[e], full[e])
        else:
            assert np.all(dst[e] == 0xABCD)
