"""Parity at the full workload sizes, in the launch configuration the benchmark
times, checked on sampled outputs the oracle computes one by one.

Workloads (seeded, synthetic, generated on the GPU):
  * the dgrad GEMM through the rowwise NVFP4 copy and the NF4 forward GEMM of
    the 256-expert gate_up stack for the 8192-token top-8 Zipf(1.1) router
    (65536 grouped token rows), sampled rows of the largest, the smallest and
    six other routed experts;
  * expert stack [32, 4096, 6144] and the 256-expert layer gate_up
    [256, 4096, 6144] + down [256, 6144, 2048], N(0, 0.02 u_e) with 0.05 %
    outliers x 30: dual-layout NVFP4 + Four-Over-Six, then the transposed
    dequant of the rowwise copy;
  * activations [16384, 6144] and [32768, 2048] (Student-t, outlier
    channels): per-token NVFP4 + Four-Over-Six;
  * NF4 of gate_up [256, 4096, 6144] and the routed dequant for an
    8192-token top-8 Zipf(1.1) router.
For every sampled block the oracle recomputes the slice amax over the whole
expert (exact), the block's scale byte and codes, and the bf16 dequantised
values; per-token rows and NF4 blocks are independent and are recomputed
directly.
"""
import numpy as np
import pytest
import torch

from nvq_testutil import assert_same, u16

pytestmark = pytest.mark.gpu

N_BLOCKS = 48     # sampled blocks per layout per stack
N_EXPERTS = 6     # experts the samples are drawn from (each needs a full-slice amax)


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def _pack(codes16):
    return (codes16[0::2] | (codes16[1::2] << 4)).astype(np.uint8)


def _check_dual_sampled(oracle_mod, w, r, rng, four_over_six=True):
    E, R, K = w.shape
    experts = rng.choice(E, size=min(N_EXPERTS, E), replace=False)
    for e in experts:
        xe = u16(w[e])                                   # [R, K] host copy of one expert
        amax = oracle_mod.amax_bf16(xe)
        G, Ev = oracle_mod.tensor_scales(amax, four_over_six)
        assert float(r["amax"][e]) == amax
        assert np.float32(r["tensor_scale"][e].item()) == np.float32(G)
        # rowwise blocks
        rows = rng.integers(0, R, N_BLOCKS // len(experts) + 1)
        bcols = rng.integers(0, K // 16, rows.size)
        cr = r["codes_row"][e].cpu().numpy()
        sr = r["scales_row"][e].cpu().numpy()
        for i, b in zip(rows, bcols):
            s, c, _, _ = oracle_mod.nvfp4_block(np.ascontiguousarray(xe[i, 16 * b:16 * b + 16]), Ev,
                                                four_over_six)
            assert sr[i, b] == s, (e, i, b)
            assert np.array_equal(cr[i, 8 * b:8 * b + 8], _pack(c)), (e, i, b)
        # columnwise blocks: 16 rows at one column, stored transposed
        cols = rng.integers(0, K, N_BLOCKS // len(experts) + 1)
        brows = rng.integers(0, R // 16, cols.size)
        cc = r["codes_col"][e].cpu().numpy()
        sc = r["scales_col"][e].cpu().numpy()
        for j, b in zip(cols, brows):
            s, c, _, _ = oracle_mod.nvfp4_block(np.ascontiguousarray(xe[16 * b:16 * b + 16, j]), Ev,
                                                four_over_six)
            assert sc[j, b] == s, (e, j, b)
            assert np.array_equal(cc[j, 8 * b:8 * b + 8], _pack(c)), (e, j, b)
    return experts


def _check_dequant_t_sampled(oracle_mod, w, dt, experts, rng):
    """Columns of DQ(Q(w))^T against the oracle's own quantisation of the
    same weight rows (under the expert's amax, computed by the oracle)."""
    E, R, K = w.shape
    for e in experts:
        xe = u16(w[e])
        amax = np.array([oracle_mod.amax_bf16(xe)], np.float32)
        got = u16(dt[e])                                  # [K, R]
        for i in rng.integers(0, R, 4):
            o = oracle_mod.nvfp4_quantize(xe[i:i + 1].reshape(1, 1, K), four_over_six=True, amax=amax)
            ref = oracle_mod.nvfp4_dequant(o["codes"], o["scales"], o["G"], 1, K)[0, 0]
            assert_same(got[:, i], ref, "dequant_t column %d of expert %d" % (i, e))


@pytest.mark.parametrize("shape", [(32, 4096, 6144)])
def test_dual_32_experts_sampled(nvq, oracle_mod, shape):
    from rl_nvfp4_quantize_gb300 import synth
    w = synth.expert_weights(*shape, seed=2, device="cuda")
    r = nvq.nvfp4_quantize_dual(w, four_over_six=True)
    dt = nvq.nvfp4_dequant_t(r["codes_row"], r["scales_row"], r["tensor_scale"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(22)
    experts = _check_dual_sampled(oracle_mod, w, r, rng)
    _check_dequant_t_sampled(oracle_mod, w, dt, experts, rng)
    del w, r, dt
    torch.cuda.empty_cache()


def test_moe_layer_256_experts_sampled(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    rng = np.random.default_rng(33)
    for seed, shape in ((3, (256, 4096, 6144)), (4, (256, 6144, 2048))):
        w = synth.expert_weights(*shape, seed=seed, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        r = nvq.nvfp4_quantize_dual(w, four_over_six=True, status=st)
        dt = nvq.nvfp4_dequant_t(r["codes_row"], r["scales_row"], r["tensor_scale"])
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        experts = _check_dual_sampled(oracle_mod, w, r, rng)
        _check_dequant_t_sampled(oracle_mod, w, dt, experts, rng)
        # every slice scale is consistent with its amax (all 256, exactly)
        am = r["amax"].cpu().numpy()
        G = r["tensor_scale"].cpu().numpy()
        for e in range(shape[0]):
            assert np.float32(G[e]) == np.float32(oracle_mod.tensor_scales(float(am[e]), True)[0])
        del w, r, dt
        torch.cuda.empty_cache()


def test_activations_full_size_sampled(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    rng = np.random.default_rng(44)
    for seed, (T, H) in ((5, (16384, 6144)), (6, (32768, 2048))):
        x = synth.activations(T, H, seed=seed, device="cuda")
        r = nvq.act_quantize_per_token(x, four_over_six=True)
        torch.cuda.synchronize()
        rows = np.sort(rng.choice(T, 64, replace=False))
        sub = u16(x[torch.from_numpy(rows).cuda()])
        o = oracle_mod.act_quantize_per_token(sub, four_over_six=True)
        assert_same(r["codes"][torch.from_numpy(rows).cuda()].cpu().numpy(), o["codes"], "act codes")
        assert_same(r["scales"][torch.from_numpy(rows).cuda()].cpu().numpy(), o["scales"], "act scales")
        assert_same(r["token_scale"][torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint32),
                    o["token_scale"].view(np.uint32), "token scales")


def test_nf4_routed_full_size_sampled(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 256, 4096, 6144
    w = synth.expert_weights(E, R, K, seed=7, device="cuda")
    q = nvq.nf4_quantize(w)
    topk = synth.zipf_router(8192, E, 8, seed=8, device="cuda")
    dst = torch.empty((E, R, K), dtype=torch.bfloat16, device="cuda")
    d, hl, nh = nvq.nf4_dequant_routed(q["codes"], q["absmax"], topk, dst=dst)
    torch.cuda.synchronize()
    hit, n, st = oracle_mod.routed_union(topk.cpu().numpy(), E)
    assert int(nh.item()) == n and st == 0
    assert_same(hl.cpu().numpy(), hit, "hit list")
    rng = np.random.default_rng(55)
    for _ in range(64):
        e, i, b = int(rng.integers(E)), int(rng.integers(R)), int(rng.integers(K // 64))
        blk = u16(w[e, i, 64 * b:64 * b + 64]).reshape(1, 1, 64)
        o = oracle_mod.nf4_quantize(blk)
        assert np.array_equal(q["codes"][e, i, 32 * b:32 * b + 32].cpu().numpy(), o["codes"].ravel())
        assert np.float32(q["absmax"][e, i, b].item()) == o["absmax"].ravel()[0]
        ref = oracle_mod.nf4_dequant(o["codes"], o["absmax"], 1, 1, 64).ravel()
        assert_same(u16(d[e, i, 64 * b:64 * b + 64]), ref, "routed dequant")
    del w, q, dst, d
    torch.cuda.empty_cache()


def test_nf4_routed_few_tokens_leaves_unrouted_slices(nvq, oracle_mod):
    """8 tokens of the same router reach only a few of the 256 experts; every
    other slice of the output keeps its previous contents."""
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 256, 512, 6144
    w = synth.expert_weights(E, R, K, seed=9, device="cuda")
    q = nvq.nf4_quantize(w)
    topk = synth.zipf_router(8, E, 8, seed=10, device="cuda")
    dst = torch.full((E, R, K), 0x7A7A, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    d, hl, nh = nvq.nf4_dequant_routed(q["codes"], q["absmax"], topk, dst=dst)
    full = nvq.nf4_dequant(q["codes"], q["absmax"])
    torch.cuda.synchronize()
    hit, n, _ = oracle_mod.routed_union(topk.cpu().numpy(), E)
    assert int(nh.item()) == n and 8 <= n <= 64
    hitset = set(hit[:n].tolist())
    dv, fv = d.view(torch.int16), full.view(torch.int16)
    for e in range(E):
        if e in hitset:
            assert torch.equal(dv[e], fv[e]), e
        else:
            assert bool((dv[e] == 0x7A7A).all()), e


def _sample_rows(counts, rng):
    """Token rows to check: the first and last row of the largest expert, of
    the smallest routed one and of six others, plus two random rows of each;
    returns (expert, rows of that expert as offsets into the grouped rows)."""
    offs = np.concatenate([[0], np.cumsum(counts)])
    routed = [e for e in range(len(counts)) if counts[e] > 0]
    pick = {int(np.argmax(counts)), min(routed, key=lambda e: counts[e])}
    pick.update(int(e) for e in rng.choice(routed, 6, replace=False))
    out = []
    for e in sorted(pick):
        r = {offs[e], offs[e + 1] - 1} | set(int(x) for x in rng.integers(offs[e], offs[e + 1], 2))
        out.append((e, np.array(sorted(r))))
    return out


def test_dgrad_full_size_sampled(nvq, oracle_mod):
    """dX = dY . DQ(Q(W_e)) for the 256-expert gate_up stack and the
    8192-token top-8 Zipf(1.1) router (65536 grouped rows), as the benchmark
    times it; sampled rows against the oracle, which quantises the sampled
    experts itself.  Tolerance as in the small dgrad tests."""
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 256, 4096, 6144
    w = synth.expert_weights(E, R, K, seed=12, device="cuda")
    q = nvq.nvfp4_quantize(w, four_over_six=True)
    topk = synth.zipf_router(8192, E, 8, seed=13, device="cuda")
    counts = torch.bincount(topk.flatten().long(), minlength=E).cpu().numpy()
    T = int(counts.sum())
    dy = synth.activations(T, R, seed=14, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dx = nvq.nvfp4_dgrad(dy, counts.tolist(), q["codes"], q["scales"], q["tensor_scale"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(66)
    for e, rows in _sample_rows(counts, rng):
        o = oracle_mod.nvfp4_quantize(u16(w[e:e + 1]), four_over_six=True)
        idx = torch.from_numpy(rows).cuda()
        ref, bound = oracle_mod.nvfp4_dgrad(u16(dy[idx]), [len(rows)], o["codes"], o["scales"],
                                            o["G"], R, K)
        got = dx[idx].cpu().numpy().astype(np.float64)
        tol = R * 2.0 ** -23 * bound + 1e-30
        assert np.all(np.abs(got - ref) <= tol), (e, float((np.abs(got - ref) - tol).max()))
    del w, q, dy, dx
    torch.cuda.empty_cache()


def test_nf4_linear_full_size_sampled(nvq, oracle_mod):
    """Y = X . DQ(W_e)^T for the 256-expert NF4 gate_up stack and the same
    router, as the benchmark times it; sampled rows against the oracle, which
    quantises the sampled experts itself.  Tolerance as in the small NF4
    forward tests."""
    from rl_nvfp4_quantize_gb300 import synth
    E, R, K = 256, 4096, 6144
    w = synth.expert_weights(E, R, K, seed=15, device="cuda")
    q = nvq.nf4_quantize(w)
    topk = synth.zipf_router(8192, E, 8, seed=16, device="cuda")
    counts = torch.bincount(topk.flatten().long(), minlength=E).cpu().numpy()
    T = int(counts.sum())
    x = synth.activations(T, K, seed=17, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = nvq.nf4_routed_linear(x, counts.tolist(), q["codes"], q["absmax"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(77)
    for e, rows in _sample_rows(counts, rng):
        o = oracle_mod.nf4_quantize(u16(w[e:e + 1]))
        idx = torch.from_numpy(rows).cuda()
        ref, bound = oracle_mod.nf4_routed_linear(u16(x[idx]), [len(rows)], o["codes"], o["absmax"],
                                                  R, K)
        got = (u16(y[idx]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        d = K * 2.0 ** -23 * bound
        tol = 2.0 ** -8 * (np.abs(ref) + d) + d
        assert np.all(np.abs(got - ref) <= tol), (e, float((np.abs(got - ref) - tol).max()))
    del w, q, x, y
    torch.cuda.empty_cache()
