"""GPU parity of the NVFP4 entry points against the oracle, bit for bit.

Codes, E4M3 scale bytes, FP32 tensor/token scales and bf16 dequantised
values must equal the oracle's on the same seeded inputs.  Shapes span
several tiles with ragged tails (the kernels tile 64 x 256 for quantising
and 128 x 256 for the transposed dequant); outputs carry canary guard bands
that must survive every call."""
import numpy as np
import pytest
import torch

from nvq_testutil import Guarded, assert_same, bf16_from_u16, f32, u8, u16

pytestmark = pytest.mark.gpu

SHAPES = [(1, 16, 16), (2, 16, 32), (3, 48, 80), (1, 512, 256), (2, 144, 528), (5, 80, 48),
          (1, 64, 4096), (3, 272, 304)]


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def weights(shape, seed, **kw):
    from rl_nvfp4_quantize_gb300 import synth
    return synth.expert_weights(*shape, seed=seed, **kw)


def run_quant(nvq, w, f46, amax=None):
    E, R, K = w.shape
    g = dict(codes=Guarded((E, R, K // 2), torch.uint8), scales=Guarded((E, R, K // 16), torch.uint8),
             amax=Guarded((E,), torch.float32), tensor_scale=Guarded((E,), torch.float32))
    out = {k: v.t for k, v in g.items()}
    if amax is not None:
        out.pop("amax")
    r = nvq.nvfp4_quantize(w.cuda(), four_over_six=f46, amax=amax, out=out)
    torch.cuda.synchronize()
    for k, v in g.items():
        if amax is None or k != "amax":
            assert v.intact(), "guard band of %s overwritten" % k
    return r


@pytest.mark.parametrize("f46", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_rowwise_quantize_parity(nvq, oracle_mod, shape, f46):
    w = weights(shape, seed=sum(shape) + f46)
    r = run_quant(nvq, w, f46)
    o = oracle_mod.nvfp4_quantize(u16(w), four_over_six=f46)
    assert_same(f32(r["amax"]).view(np.uint32), o["amax"].view(np.uint32), "amax")
    assert_same(f32(r["tensor_scale"]).view(np.uint32), o["G"].view(np.uint32), "G")
    assert_same(u8(r["scales"]), o["scales"], "scales")
    assert_same(u8(r["codes"]), o["codes"], "codes")


@pytest.mark.parametrize("f46", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_dual_quantize_parity(nvq, oracle_mod, shape, f46):
    w = weights(shape, seed=1000 + sum(shape) + f46)
    E, R, K = shape
    g = dict(codes_row=Guarded((E, R, K // 2), torch.uint8),
             scales_row=Guarded((E, R, K // 16), torch.uint8),
             codes_col=Guarded((E, K, R // 2), torch.uint8),
             scales_col=Guarded((E, K, R // 16), torch.uint8),
             amax=Guarded((E,), torch.float32), tensor_scale=Guarded((E,), torch.float32))
    r = nvq.nvfp4_quantize_dual(w.cuda(), four_over_six=f46, out={k: v.t for k, v in g.items()})
    torch.cuda.synchronize()
    for k, v in g.items():
        assert v.intact(), k
    wn = u16(w)
    orow = oracle_mod.nvfp4_quantize(wn, four_over_six=f46)
    ocol = oracle_mod.nvfp4_quantize_colwise(wn, four_over_six=f46)
    assert_same(f32(r["tensor_scale"]).view(np.uint32), orow["G"].view(np.uint32), "G")
    assert_same(u8(r["scales_row"]), orow["scales"], "scales_row")
    assert_same(u8(r["codes_row"]), orow["codes"], "codes_row")
    assert_same(u8(r["scales_col"]), ocol["scales"], "scales_col")
    assert_same(u8(r["codes_col"]), ocol["codes"], "codes_col")


@pytest.mark.parametrize("shape", [(1, 512, 256), (3, 48, 80), (2, 144, 528), (2, 272, 304)])
def test_dequant_and_transposed_dequant_parity(nvq, oracle_mod, shape):
    w = weights(shape, seed=2000 + sum(shape))
    E, R, K = shape
    r = nvq.nvfp4_quantize(w.cuda(), four_over_six=True)
    gd = Guarded((E, R, K), torch.bfloat16)
    gt = Guarded((E, K, R), torch.bfloat16)
    d = nvq.nvfp4_dequant(r["codes"], r["scales"], r["tensor_scale"], out=gd.t)
    dt = nvq.nvfp4_dequant_t(r["codes"], r["scales"], r["tensor_scale"], out=gt.t)
    torch.cuda.synchronize()
    assert gd.intact() and gt.intact()
    codes, scales, G = u8(r["codes"]), u8(r["scales"]), f32(r["tensor_scale"])
    assert_same(u16(d), oracle_mod.nvfp4_dequant(codes, scales, G, R, K), "dequant")
    assert_same(u16(dt), oracle_mod.nvfp4_dequant_t(codes, scales, G, R, K), "dequant_t")
    # cross-check the bf16 rounding with torch's own cast of the FP32 products
    c = np.empty(codes.shape[:-1] + (K,), np.uint8)
    c[..., 0::2] = codes & 15
    c[..., 1::2] = codes >> 4
    mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)[c & 7]
    S = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).float().numpy()
    y = (mag * np.repeat(S, 16, axis=-1)).astype(np.float32) * G[:, None, None]
    y = np.where(c & 8, -y, y).astype(np.float32)
    assert_same(u16(d), u16(torch.from_numpy(y).to(torch.bfloat16)), "dequant vs torch")


@pytest.mark.parametrize("f46", [False, True])
@pytest.mark.parametrize("T,H", [(1, 16), (7, 48), (33, 6144), (5, 8192), (3, 16384), (64, 2048),
                                 (2, 22544)])
def test_act_per_token_parity(nvq, oracle_mod, T, H, f46):
    from rl_nvfp4_quantize_gb300 import synth
    x = synth.activations(T, H, seed=T * 31 + H + f46)
    g = dict(codes=Guarded((T, H // 2), torch.uint8), scales=Guarded((T, H // 16), torch.uint8),
             token_scale=Guarded((T,), torch.float32))
    r = nvq.act_quantize_per_token(x.cuda(), four_over_six=f46, out={k: v.t for k, v in g.items()})
    torch.cuda.synchronize()
    for k, v in g.items():
        assert v.intact(), k
    o = oracle_mod.act_quantize_per_token(u16(x), four_over_six=f46)
    assert_same(f32(r["token_scale"]).view(np.uint32), o["token_scale"].view(np.uint32), "token scale")
    assert_same(u8(r["scales"]), o["scales"], "scales")
    assert_same(u8(r["codes"]), o["codes"], "codes")


# ------------------------------------------------------------ edge cases

def _edge_tensor(kind, shape, seed=0):
    rng = np.random.default_rng(seed)
    E, R, K = shape
    if kind == "zeros":
        a = np.zeros(shape, np.float32)
    elif kind == "negzeros":
        a = -np.zeros(shape, np.float32)
    elif kind == "tiny":     # bf16 subnormals and tiny normals only
        a = rng.standard_normal(shape).astype(np.float32) * 1e-39
    elif kind == "huge":     # near the top of the bf16 range
        a = rng.standard_normal(shape).astype(np.float32) * 1e37
    elif kind == "wide":     # block maxima spread over 30 octaves -> E4M3 subnormal scales
        a = rng.standard_normal(shape) * np.exp2(rng.integers(-30, 1, (E, R, K // 16)).repeat(16, -1))
        a = a.astype(np.float32)
    elif kind == "equal":
        a = np.full(shape, 0.75, np.float32)
    elif kind == "ties":     # values on E2M1 midpoints after scaling (E = 1 when amax = 6M)
        a = rng.choice(np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 4.5, -0.25, -5.0]), shape)
        a[:, 0, 0] = 1536.0
    else:
        raise ValueError(kind)
    return torch.from_numpy(a).to(torch.bfloat16)


@pytest.mark.parametrize("f46", [False, True])
@pytest.mark.parametrize("kind", ["zeros", "negzeros", "tiny", "huge", "wide", "equal", "ties"])
def test_edge_inputs_dual_parity(nvq, oracle_mod, kind, f46):
    shape = (2, 48, 288)
    w = _edge_tensor(kind, shape, seed=5)
    r = nvq.nvfp4_quantize_dual(w.cuda(), four_over_six=f46)
    wn = u16(w)
    orow = oracle_mod.nvfp4_quantize(wn, four_over_six=f46)
    ocol = oracle_mod.nvfp4_quantize_colwise(wn, four_over_six=f46)
    assert_same(f32(r["tensor_scale"]).view(np.uint32), orow["G"].view(np.uint32), "G")
    assert_same(u8(r["scales_row"]), orow["scales"], "scales_row")
    assert_same(u8(r["codes_row"]), orow["codes"], "codes_row")
    assert_same(u8(r["scales_col"]), ocol["scales"], "scales_col")
    assert_same(u8(r["codes_col"]), ocol["codes"], "codes_col")
    dt = nvq.nvfp4_dequant_t(r["codes_row"], r["scales_row"], r["tensor_scale"])
    assert_same(u16(dt), oracle_mod.nvfp4_dequant_t(orow["codes"], orow["scales"], orow["G"],
                                                    shape[1], shape[2]), "dequant_t")


def test_amax_given_matches(nvq, oracle_mod):
    w = weights((3, 64, 96), seed=77)
    o = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    am = torch.from_numpy(o["amax"] * np.float32(1.5)).cuda()  # a larger given amax is allowed
    r = nvq.nvfp4_quantize_dual(w.cuda(), four_over_six=True, amax=am)
    o2 = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True, amax=o["amax"] * np.float32(1.5))
    assert_same(u8(r["codes_row"]), o2["codes"], "codes")
    assert_same(f32(r["tensor_scale"]).view(np.uint32), o2["G"].view(np.uint32), "G")


def test_status_reports_nonfinite(nvq):
    w = weights((2, 32, 64), seed=3)
    w[1, 5, 7] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nvq.nvfp4_quantize_dual(w.cuda(), status=st)
    assert int(st.item()) & nvq.STATUS_NONFINITE
    st.zero_()
    nvq.nvfp4_quantize_dual(weights((2, 32, 64), seed=3).cuda(), status=st)
    assert int(st.item()) == 0
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    x[2, 3] = float("inf")
    nvq.act_quantize_per_token(x.cuda(), status=st)
    assert int(st.item()) & nvq.STATUS_NONFINITE


def test_empty_inputs(nvq, oracle_mod):
    w = torch.zeros((3, 0, 32), dtype=torch.bfloat16, device="cuda")
    r = nvq.nvfp4_quantize(w)
    assert torch.all(r["amax"] == 0) and torch.all(r["tensor_scale"] == 0)
    w0 = torch.zeros((0, 16, 32), dtype=torch.bfloat16, device="cuda")
    r0 = nvq.nvfp4_quantize_dual(w0)
    assert r0["codes_row"].numel() == 0
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    assert nvq.act_quantize_per_token(x)["codes"].numel() == 0


def test_stream_ordering_on_side_stream(nvq, oracle_mod):
    w = weights((4, 128, 512), seed=9)
    s = torch.cuda.Stream()
    wc = w.cuda()
    torch.cuda.current_stream().synchronize()
    with torch.cuda.stream(s):
        r = nvq.nvfp4_quantize_dual(wc, four_over_six=True)
        dt = nvq.nvfp4_dequant_t(r["codes_row"], r["scales_row"], r["tensor_scale"])
    s.synchronize()
    o = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    assert_same(u16(dt), oracle_mod.nvfp4_dequant_t(o["codes"], o["scales"], o["G"], 128, 512))


@pytest.fixture
def quant_lead(nvq):
    """Sets the quantisers' look-ahead lead for one test, then restores 2."""
    yield nvq.debug_set_quant_lead
    nvq.debug_set_quant_lead(2)


@pytest.mark.parametrize("lead", [2, 3, 6])
@pytest.mark.parametrize("shape", [(7, 80, 336), (5, 64, 256), (4, 144, 528), (40, 64, 256),
                                   (3, 1040, 96)])
def test_single_pass_amax(nvq, oracle_mod, shape, lead, quant_lead):
    """The slice amax is reduced inside the quantising pass from tiles loaded
    one slice plus `lead` grid waves ahead (2: the least lead, the least
    slack before a slice's amax is needed).  Ragged
    row tiles (80, 144 and 1040 rows) load rows of the next slice, which the
    look-ahead must leave out.  Outputs are those of the oracle."""
    quant_lead(lead)
    w = weights(shape, seed=300 + lead + sum(shape))
    wn = u16(w)
    for f46 in (False, True):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        r = nvq.nvfp4_quantize_dual(w.cuda(), four_over_six=f46, status=st)
        orow = oracle_mod.nvfp4_quantize(wn, four_over_six=f46)
        ocol = oracle_mod.nvfp4_quantize_colwise(wn, four_over_six=f46)
        assert int(st.item()) == 0
        assert_same(f32(r["amax"]).view(np.uint32), orow["amax"].view(np.uint32), "amax")
        assert_same(f32(r["tensor_scale"]).view(np.uint32), orow["G"].view(np.uint32), "G")
        assert_same(u8(r["codes_row"]), orow["codes"], "codes_row")
        assert_same(u8(r["scales_row"]), orow["scales"], "scales_row")
        assert_same(u8(r["codes_col"]), ocol["codes"], "codes_col")
        assert_same(u8(r["scales_col"]), ocol["scales"], "scales_col")
        r1 = nvq.nvfp4_quantize(w.cuda(), four_over_six=f46, status=st)
        assert int(st.item()) == 0
        assert_same(u8(r1["codes"]), orow["codes"], "rowwise-only codes")
        assert_same(u8(r1["scales"]), orow["scales"], "rowwise-only scales")
        assert_same(f32(r1["tensor_scale"]).view(np.uint32), orow["G"].view(np.uint32), "G")


def test_slice_amax_outlier_in_last_ragged_rows(nvq, oracle_mod):
    """An outlier in the last rows of a slice whose row count is not a
    multiple of the 64-row tile: it must raise that slice's amax only."""
    w = weights((3, 80, 256), seed=91)
    w[1, 79, 200] = 50.0
    w[0, 70, 3] = -40.0
    wn = u16(w)
    r = nvq.nvfp4_quantize_dual(w.cuda(), four_over_six=True)
    o = oracle_mod.nvfp4_quantize(wn, four_over_six=True)
    assert_same(f32(r["amax"]).view(np.uint32), o["amax"].view(np.uint32), "amax")
    assert_same(u8(r["codes_row"]), o["codes"], "codes_row")


def test_stack_16_byte_aligned(nvq, oracle_mod):
    """A stack that is 16- but not 32-byte aligned (the copies need 16)."""
    w = weights((3, 64, 256), seed=77)
    buf = torch.empty(w.numel() + 8, dtype=torch.bfloat16, device="cuda")
    wv = buf[8:].view(3, 64, 256)
    wv.copy_(w.cuda())
    assert wv.data_ptr() % 32 == 16
    r = nvq.nvfp4_quantize_dual(wv, four_over_six=True)
    o = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    assert_same(u8(r["codes_row"]), o["codes"], "codes_row")
    assert_same(f32(r["amax"]).view(np.uint32), o["amax"].view(np.uint32), "amax")


def test_codes_col_16_byte_aligned(nvq, oracle_mod):
    """Columnwise codes into a buffer that is 16- but not 32-byte aligned take
    the two 16-byte stores instead of one 32-byte store; both give the same
    bytes."""
    w = weights((2, 128, 512), seed=78)
    buf = torch.empty(2 * 512 * 64 + 16, dtype=torch.uint8, device="cuda")
    cc = buf[16:].view(2, 512, 64)
    assert cc.data_ptr() % 32 == 16
    r = nvq.nvfp4_quantize_dual(w.cuda(), four_over_six=True, out={"codes_col": cc})
    ocol = oracle_mod.nvfp4_quantize_colwise(u16(w), four_over_six=True)
    assert_same(u8(cc), ocol["codes"], "codes_col")
    assert_same(u8(r["scales_col"]), ocol["scales"], "scales_col")


@pytest.mark.parametrize("shape", [(1, 16, 16), (2, 80, 96), (3, 528, 272), (2, 1040, 64),
                                   (1, 512, 1024), (2, 1536, 144)])
def test_transposed_dequant_ragged_tiles(nvq, oracle_mod, shape):
    """The transposed dequant over shapes ragged against its 128 x 256 tiles
    (out and in not multiples of the tile, slices smaller than a tile):
    same bytes as the oracle, guard bands intact."""
    w = weights(shape, seed=4000 + sum(shape))
    E, R, K = shape
    r = nvq.nvfp4_quantize(w.cuda(), four_over_six=True)
    gt = Guarded((E, K, R), torch.bfloat16)
    dt = nvq.nvfp4_dequant_t(r["codes"], r["scales"], r["tensor_scale"], out=gt.t)
    torch.cuda.synchronize()
    assert gt.intact()
    codes, scales, G = u8(r["codes"]), u8(r["scales"]), f32(r["tensor_scale"])
    assert_same(u16(dt), oracle_mod.nvfp4_dequant_t(codes, scales, G, R, K), "dequant_t")


@pytest.mark.parametrize("H", [2048, 208])
def test_act_rows_16_byte_aligned(nvq, oracle_mod, H):
    """Activations 16- but not 32-byte aligned (the loads are 16-byte ones):
    same bytes as the oracle."""
    from rl_nvfp4_quantize_gb300 import synth
    T = 37
    x = synth.activations(T, H, seed=H + 5)
    buf = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device="cuda")
    xv = buf[8:].view(T, H)
    xv.copy_(x.cuda())
    assert xv.data_ptr() % 32 == 16
    r = nvq.act_quantize_per_token(xv, four_over_six=True)
    o = oracle_mod.act_quantize_per_token(u16(x), four_over_six=True)
    assert_same(u8(r["codes"]), o["codes"], "codes")
    assert_same(u8(r["scales"]), o["scales"], "scales")
    assert_same(f32(r["token_scale"]).view(np.uint32), o["token_scale"].view(np.uint32), "token_scale")


@pytest.mark.parametrize("T,H", [(8000, 2064), (2500, 6400), (4097, 6144), (300, 2080),
                                 (257, 3216)])
def test_act_streamed_rows_wrap_the_ring(nvq, oracle_mod, T, H):
    """Rows of 2048 < H <= 6400 values stream through each warp's ring of
    row buffers; with more rows per warp than buffers the ring wraps (its
    barriers change phase); 6144, 6400 and 3216 leave one buffer per warp,
    2064 and 2080 several: same bytes as the oracle."""
    from rl_nvfp4_quantize_gb300 import synth
    x = synth.activations(T, H, seed=T + H)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = nvq.act_quantize_per_token(x.cuda(), four_over_six=True, status=st)
    o = oracle_mod.act_quantize_per_token(u16(x), four_over_six=True)
    assert int(st.item()) == 0
    assert_same(u8(r["codes"]), o["codes"], "codes")
    assert_same(u8(r["scales"]), o["scales"], "scales")
    assert_same(f32(r["token_scale"]).view(np.uint32), o["token_scale"].view(np.uint32), "token_scale")
