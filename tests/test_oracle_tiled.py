"""Host checks of the oracle's tiled block-scale layout and FP4 block values.

The tiled layout is the scale operand of the block-scaled FP4 GEMM ("Getting
GLM-5.2 NVFP4 Post-Training off the ground", "Why can't we just transpose
the one copy?": scales swizzled for the tensor-core tile).  Its bytes are
pinned on the GPU, where that GEMM consumes them; here the layout's shape
rules are checked: every (row, block column) of the padded matrix has its own
byte, the 512-byte tiles hold exactly the scales of their 128 x 4 window, and
padding is zero.  The block values c * S are checked against the E2M1 and
E4M3 definitions written out by hand.
"""
import numpy as np
import pytest


@pytest.mark.parametrize("R,C", [(128, 4), (256, 12), (100, 3), (300, 5), (1, 1)])
def test_tiled_layout_is_a_bijection_with_zero_padding(oracle_mod, R, C):
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    # label every entry of the padded matrix with a distinct 16-bit value
    idx = np.arange(Rp * Cp).reshape(Rp, Cp)
    lo = oracle_mod.scales_tiled((idx & 0xFF).astype(np.uint8)).astype(np.int64)
    hi = oracle_mod.scales_tiled((idx >> 8).astype(np.uint8)).astype(np.int64)
    assert np.array_equal(np.sort(lo | (hi << 8)), np.arange(Rp * Cp))
    # the real [R, C] window alone: ones inside, zeros in the padding
    t = oracle_mod.scales_tiled(np.ones((R, C), np.uint8))
    assert t.shape == (Rp * Cp,) and int(t.sum()) == R * C


def test_tiles_hold_their_128x4_windows(oracle_mod):
    R, C = 256, 8
    rng = np.random.default_rng(0)
    lin = rng.integers(1, 127, (R, C)).astype(np.uint8)
    t = oracle_mod.scales_tiled(lin)
    for ti in range(2):
        for tj in range(2):
            tile = t[(ti * 2 + tj) * 512:(ti * 2 + tj + 1) * 512]
            window = lin[128 * ti:128 * ti + 128, 4 * tj:4 * tj + 4]
            assert np.array_equal(np.sort(tile), np.sort(window.ravel()))
            # 32-row groups: bytes 16 r' .. 16 r' + 15 hold rows r', r'+32,
            # r'+64, r'+96 of the window, 4 block columns each
            for rr in (0, 7, 31):
                got = tile[16 * rr:16 * rr + 16].reshape(4, 4)
                assert np.array_equal(got, window[[rr, rr + 32, rr + 64, rr + 96]])


def test_block_values(oracle_mod):
    e2 = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}
    codes = np.array([[0x71, 0xF8, 0x2A] + [0] * 5], np.uint8)   # 16 elements
    scales = np.array([[0x38]], np.uint8)                          # E4M3 0x38 = 1.0
    v = oracle_mod.nvfp4_block_values(codes, scales)
    assert v.shape == (1, 16)
    assert list(v[0, :6]) == [e2[1], e2[7], -0.0, -e2[7], -e2[2], e2[2]]
    scales2 = np.array([[0x01]], np.uint8)                         # smallest subnormal 2^-9
    v2 = oracle_mod.nvfp4_block_values(codes, scales2)
    assert v2[0, 1] == 6.0 * 2.0 ** -9
    y, b = oracle_mod.nvfp4_scaled_product(codes, scales, codes, scales2)
    assert y[0, 0] == np.dot(v[0], v2[0]) and b[0, 0] == np.abs(v[0]) @ np.abs(v2[0])
