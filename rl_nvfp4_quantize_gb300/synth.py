"""Seeded synthetic workloads (inputs only -- no quantisation arithmetic here).

The shapes and value distributions stand in for the workloads the sources
describe; no dataset or checkpoint is used:

* expert weights of a fused MoE layer, stored as 3-D stacks used as
  F.linear(x, W[e]) -- gate_up [256, 2*2048, 6144] and down [256, 6144, 2048]
  ("nf4moe", "Why every quantizer misses 95% of the model") -- drawn
  N(0, 0.02 * u_e) per expert with u_e ~ U(0.5, 2) and a small fraction of
  outliers multiplied by a constant;
* the 512 x 256 single weight, N(0, 0.02) with 0.1 % outliers x 20;
* activations: Student-t (nu = 3) values times 0.5 with 8 outlier channels
  x 50 ("The 4-bitter Lesson" quantises activations per token);
* NF4 block absmax values (the input of the nested absmax): for N(0, sigma)
  weights the largest magnitude of 64 values sits near 2.4 sigma with a
  spread of about 0.4 sigma, so sigma_e * max(0.5, 2.4 + 0.4 z), z ~ N(0, 1),
  with sigma_e = 0.02 * u_e as for the weights, rounded to bf16 (the absmax
  of bf16 weights is a bf16 value) and a small fraction of zero blocks;
* router choices: top-8 of 256 experts per token with Zipf(1.1) popularity
  over a seeded permutation of the experts; each token draws 8 distinct
  experts by the Gumbel-top-k trick.

Generators run on the given device with a seeded torch.Generator (CPU or
CUDA); the same seed on the same device gives the same tensor.
"""
from __future__ import annotations

import torch


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def expert_weights(nexp, rows, cols, seed, device="cpu", std=0.02, jitter=(0.5, 2.0),
                   outlier_frac=0.0005, outlier_mult=30.0, chunk_elems=1 << 27, out=None):
    """bf16 [nexp, rows, cols]: N(0, std * u_e), u_e ~ U(jitter), outliers x mult.

    Generated expert by expert (in chunks) so full-size stacks need no fp32
    copy of the whole tensor."""
    g = _gen(device, seed)
    w = out if out is not None else torch.empty((nexp, rows, cols), dtype=torch.bfloat16,
                                                device=device)
    u = torch.empty(nexp, device=device).uniform_(jitter[0], jitter[1], generator=g)
    per = rows * cols
    flat = w.view(nexp, per)
    step = max(1, chunk_elems // max(per, 1))
    for e0 in range(0, nexp, step):
        e1 = min(nexp, e0 + step)
        x = torch.randn((e1 - e0, per), device=device, generator=g)
        x.mul_((std * u[e0:e1]).unsqueeze(1))
        if outlier_frac > 0:
            m = torch.rand((e1 - e0, per), device=device, generator=g) < outlier_frac
            x[m] *= outlier_mult
        flat[e0:e1].copy_(x)
    return w


def nf4_absmax_values(nexp, n, seed, device="cpu", zero_frac=0.0002):
    """f32 [nexp, n]: bf16-representable block maxima, sigma_e * max(0.5, 2.4 + 0.4 z)."""
    g = _gen(device, seed)
    u = torch.empty(nexp, device=device).uniform_(0.5, 2.0, generator=g)
    z = torch.randn((nexp, n), device=device, generator=g)
    a = (0.02 * u.unsqueeze(1)) * torch.clamp(2.4 + 0.4 * z, min=0.5)
    if zero_frac > 0:
        a[torch.rand((nexp, n), device=device, generator=g) < zero_frac] = 0.0
    return a.to(torch.bfloat16).to(torch.float32)


def single_weight(rows=512, cols=256, seed=0, device="cpu"):
    """bf16 [rows, cols]: N(0, 0.02) with 0.1 % of elements x 20."""
    return expert_weights(1, rows, cols, seed, device=device, jitter=(1.0, 1.0),
                          outlier_frac=0.001, outlier_mult=20.0)[0]


def activations(T, H, seed, device="cpu", nu=3, scale=0.5, n_outlier_ch=8, outlier_mult=50.0):
    """bf16 [T, H]: Student-t(nu) * scale, n_outlier_ch channels x mult."""
    g = _gen(device, seed)
    z = torch.randn((T, H), device=device, generator=g)
    chi = torch.zeros((T, H), device=device)
    for _ in range(nu):
        chi.add_(torch.randn((T, H), device=device, generator=g).square_())
    x = z / torch.sqrt(chi / nu) * scale
    ch = torch.randperm(H, device=device, generator=g)[:n_outlier_ch]
    x[:, ch] *= outlier_mult
    return x.to(torch.bfloat16)


def zipf_router(T, nexp, k, seed, device="cpu", s=1.1):
    """int32 [T, k]: per token, k distinct experts; popularity of expert e is
    proportional to (rank(e) + 1)^-s for a seeded rank permutation."""
    g = _gen(device, seed)
    rank = torch.randperm(nexp, device=device, generator=g).to(torch.float32)
    logp = -s * torch.log(rank + 1.0)
    u = torch.rand((T, nexp), device=device, generator=g).clamp_(1e-12, 1.0 - 1e-7)
    gumbel = -torch.log(-torch.log(u))
    return torch.topk(logp.unsqueeze(0) + gumbel, k, dim=1).indices.to(torch.int32)


# Workloads named by what they are, with their sizes.
WORKLOADS = {
    "single_weight_512x256": dict(kind="single", rows=512, cols=256),
    "gate_up_32x4096x6144": dict(kind="experts", nexp=32, rows=4096, cols=6144),
    "moe_layer_256x(4096x6144,6144x2048)": dict(
        kind="layer", gate_up=(256, 4096, 6144), down=(256, 6144, 2048)),
    "act_16384x6144+32768x2048": dict(kind="act", shapes=((16384, 6144), (32768, 2048))),
    "nf4_gate_up_256x4096x6144_router_8192x8": dict(
        kind="nf4", nexp=256, rows=4096, cols=6144, tokens=8192, k=8),
}

