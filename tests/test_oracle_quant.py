"""Pins of the oracle's NVFP4 quantizer and block-scaled dot product.

The format (shengxinai.com Nemotron 3 blog, section 3.1.1 "NVFP4 格式解析"): E2M1 elements,
16-element micro-blocks, one E4M3 block scale; plus one FP32 tensor scale.  The decode used
here is written from the format (tables below and torch's float8_e4m3fn decode), not from
the oracle.
"""
import numpy as np
import pytest
import torch

import oracle

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0,
                 -4.0, -6.0])
E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant(codes, sf, s_dec):
    """Independent NVFP4 decode: [R][K/2] codes (low nibble = even element), [R][K/16] sf."""
    lo = E2M1[codes & 15]
    hi = E2M1[codes >> 4]
    R = codes.shape[0]
    v = np.stack([lo, hi], axis=-1).reshape(R, -1)
    return v * np.repeat(E4M3[sf], 16, axis=1) * float(s_dec)


def e4m3_codes_positive():
    return [c for c in range(1, 0x7F) if np.isfinite(E4M3[c])]


def test_round_trip_on_hand_built_blocks():
    # tensor amax 336 -> s_enc = 8, s_dec = 1/8 exactly.  Each block: a scale value v
    # (an E4M3 value), elements g * v / 8 with g on the E2M1 grid and one |g| = 6, so
    # amax_b * s_enc / 6 == v and every element sits on the block's grid.
    rng = np.random.default_rng(0)
    vals = E4M3[e4m3_codes_positive()]
    vals = vals[(vals >= 2.0 ** -6) & (vals <= 448)]
    R, K = 64, 256
    x = np.empty((R, K), np.float64)
    for r in range(R):
        for b in range(K // 16):
            v = rng.choice(vals)
            g = rng.choice(E2M1, 16)
            g[rng.integers(16)] = rng.choice([6.0, -6.0])
            x[r, 16 * b:16 * b + 16] = g * v / 8.0
    x32 = x.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x)
    codes, sf, sdec = oracle.quantize_nvfp4(x32, amax=336.0)
    assert sdec == 0.125
    assert np.array_equal(dequant(codes, sf, sdec), x)


def test_packing_low_nibble_is_even_element():
    x = np.zeros((1, 16), np.float32)
    x[0, 0], x[0, 1] = 6.0, -1.0           # amax 6 -> block scale decodes to 1 * s_dec
    codes, sf, sdec = oracle.quantize_nvfp4(x, amax=6.0 * 448 / 448)
    # the block amax equals the tensor amax -> block scale 448, bd = 448 * 6/2688 = 1
    assert E4M3[sf[0, 0]] == 448.0
    assert codes[0, 0] == (7 | (0b1010 << 4))


def test_zero_tensor():
    codes, sf, sdec = oracle.quantize_nvfp4(np.zeros((3, 32), np.float32))
    assert sdec == 1.0 and not codes.any() and not sf.any()


def test_flush_to_zero_block():
    x = np.zeros((1, 32), np.float32)
    x[0, :16] = 300.0
    x[0, 16:] = np.linspace(-1e-9, 1e-9, 16, dtype=np.float32)
    codes, sf, sdec = oracle.quantize_nvfp4(x)
    assert sf[0, 1] == 0
    assert set((codes[0, 8:] & 0x77).tolist()) == {0}      # every element is a signed zero


def test_saturating_block_with_static_amax():
    x = np.full((1, 16), 100.0, np.float32)
    x[0, ::2] = -3.0
    codes, sf, sdec = oracle.quantize_nvfp4(x, amax=1.0)
    assert sf[0, 0] == 0x7E
    d = dequant(codes, sf, sdec)
    assert np.allclose(d[0, 1::2], 1.0) and np.allclose(d[0, ::2], -1.0)


def test_error_bound_half_spacing():
    # Each element lands on the grid {0,.5,...,6} * bd with bd = value(sf) * s_dec; the
    # largest grid spacing is 2, so |x - dequant| <= bd for unsaturated, unflushed blocks.
    rng = np.random.default_rng(3)
    x = (rng.normal(0, 1, (128, 512)) * np.exp(rng.normal(0, 2, (128, 1)))).astype(np.float32)
    codes, sf, sdec = oracle.quantize_nvfp4(x)
    d = dequant(codes, sf, sdec)
    bd = np.repeat(E4M3[sf], 16, axis=1) * sdec
    ok = bd > 0
    assert np.all(np.abs(d - x)[ok] <= bd[ok] * (1 + 1e-6))
    assert np.all(np.abs(x)[~ok] < 2.0 ** -10 * 6 * sdec * 1.01)


def test_block_dot_is_exact():
    rng = np.random.default_rng(4)
    for K in (16, 64, 2048):
        a = rng.normal(0, 1, (1, K)).astype(np.float32)
        b = rng.normal(0, 3, (1, K)).astype(np.float32)
        qa, sa, da = oracle.quantize_nvfp4(a)
        qb, sb, db = oracle.quantize_nvfp4(b)
        want = float(np.dot(dequant(qa, sa, 1.0)[0], dequant(qb, sb, 1.0)[0]))
        got = oracle.nvfp4_dot(qa[0], sa[0], qb[0], sb[0])
        assert got == pytest.approx(want, rel=1e-14, abs=1e-300)


def test_tensor_scale_formula():
    x = np.random.default_rng(5).normal(0, 1, (4, 64)).astype(np.float32)
    amax = float(np.abs(x).max())
    _, _, sdec = oracle.quantize_nvfp4(x)
    assert sdec == np.float32(amax) / np.float32(2688.0)
