"""Pins of the oracle's 2-D weight-block NVFP4 quantizer: one E4M3 scale per 16 rows x 16
contraction elements (NVIDIA AI releases Nemotron 3 Ultra, architecture paragraph: weights
quantized in two-dimensional blocks; 16 x 16 is this project's reading).  The decode is the
tests' own (torch float8_e4m3fn and the E2M1 table), not the oracle's."""
import numpy as np

import oracle
from test_oracle_quant import E2M1, E4M3, dequant, e4m3_codes_positive


def test_round_trip_on_hand_built_16x16_blocks():
    # tensor amax 336 -> s_enc = 8, s_dec = 1/8 exactly.  Each 16 x 16 block: a scale value v,
    # elements g * v / 8 with g on the E2M1 grid and exactly one |g| = 6 in the whole block, so
    # the block amax * s_enc / 6 == v and every element sits on the block's grid.
    rng = np.random.default_rng(4)
    vals = E4M3[e4m3_codes_positive()]
    vals = vals[(vals >= 2.0 ** -6) & (vals <= 448)]
    R, K = 64, 96
    x = np.empty((R, K), np.float64)
    blocks = {}
    for gr in range(R // 16):
        for b in range(K // 16):
            v = 448.0 if (gr, b) == (0, 0) else rng.choice(vals)
            g = rng.choice(E2M1[np.abs(E2M1) < 6], (16, 16))
            i, j = rng.integers(16), rng.integers(16)
            g[i, j] = rng.choice([6.0, -6.0])
            x[16 * gr:16 * gr + 16, 16 * b:16 * b + 16] = g * v / 8.0
            blocks[(gr, b)] = v
    x32 = x.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x)
    codes, sf, sdec = oracle.quantize_nvfp4_2d(x32, amax=336.0)
    assert sdec == 0.125
    assert np.array_equal(dequant(codes, sf, sdec), x)
    for (gr, b), v in blocks.items():            # one scale per block, on all 16 of its rows
        assert np.all(E4M3[sf[16 * gr:16 * gr + 16, b]] == v)


def test_equals_1d_when_every_row_block_shares_the_block_amax():
    rng = np.random.default_rng(5)
    R, K = 32, 64
    x = rng.normal(0, 1, (R, K)).astype(np.float32)
    x = np.clip(x, -2.5, 2.5)
    for gr in range(R // 16):
        for b in range(K // 16):
            m = np.float32(rng.uniform(3, 4))
            for r in range(16):                     # every row of the block reaches the block max
                x[16 * gr + r, 16 * b + rng.integers(16)] = m if r % 2 else -m
    c1, s1, d1 = oracle.quantize_nvfp4(x)
    c2, s2, d2 = oracle.quantize_nvfp4_2d(x)
    assert d1 == d2
    assert np.array_equal(s1, s2) and np.array_equal(c1, c2)


def test_small_rows_share_the_large_rows_scale():
    # block rows 0..14 hold 1.0; row 15 holds +-0.05: under the shared scale (block max 6 ->
    # element step 0.5 at the bottom of the grid) 0.05 is below a quarter step and flushes to a
    # signed zero, while a 1-D quantizer would keep it
    x = np.ones((16, 16), np.float32)
    x[0, 0] = 6.0
    x[15] = np.where(np.arange(16) % 2 == 0, 0.05, -0.05)
    codes, sf, sdec = oracle.quantize_nvfp4_2d(x, amax=6.0)
    d = dequant(codes, sf, sdec)
    assert np.all(d[15] == 0.0)
    assert np.all((codes[15] & 0x77) == 0) and np.all((codes[15] & 0x88) == 0x80)  # -0 on odd elements
    c1, s1, d1 = oracle.quantize_nvfp4(x, amax=6.0)
    assert np.all(dequant(c1, s1, d1)[15] != 0.0)


def test_zero_tensor_2d():
    codes, sf, sdec = oracle.quantize_nvfp4_2d(np.zeros((16, 32), np.float32))
    assert sdec == 1.0 and not codes.any() and not sf.any()
