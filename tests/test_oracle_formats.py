"""Pins of the oracle's number formats against the format definitions and library routines.

E2M1 / E4M3 are the element and block-scale formats of NVFP4 (shengxinai.com Nemotron 3
blog, section 3.1.1 "NVFP4 格式解析").  bf16 is the precision of the latent projections
(same blog, section 3.1.3 mixed-precision table).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_e2m1_decode_matches_format_table():
    g = _golden("e2m1_format.json")
    for c, v in enumerate(g["codes_0_to_7"]):
        assert oracle.e2m1_value(c) == v
        neg = oracle.e2m1_value(c | g["sign_bit"])
        assert neg == -v and np.signbit(neg)


def test_e2m1_round_to_nearest_even_ties_and_saturation():
    g = _golden("e2m1_format.json")
    grid = g["codes_0_to_7"]
    for x, want in g["round_to_nearest_even_ties"] + g["saturation"]:
        for s in (1.0, -1.0):
            code = int(oracle.f32_to_e2m1(s * x)[0])
            assert oracle.e2m1_value(code) == s * want, (x, s, code)
    for x, code in g["signed_zero"]:
        assert int(oracle.f32_to_e2m1(x)[0]) == code
    assert len(grid) == 8


def _brute_e2m1(v):
    """Nearest E2M1 value by exhaustive search, ties to the even code, saturating."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    a = abs(float(v))
    dist = np.abs(grid - a)
    best = np.flatnonzero(dist == dist.min())
    c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (8 if np.signbit(v) else 0)


def test_e2m1_matches_brute_force_nearest():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-8, 8, 20000), rng.normal(0, 0.3, 5000),
                        np.arange(-28, 29) * 0.25]).astype(np.float32)
    got = oracle.f32_to_e2m1(v)
    want = np.array([_brute_e2m1(x) for x in v], np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_decode_matches_torch_for_all_codes():
    raw = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for c in range(256):
        v = oracle.e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert np.isnan(v)
        else:
            assert v == raw[c].item(), c
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_inside_range():
    rng = np.random.default_rng(1)
    codes = np.arange(0, 0x7E + 1)
    vals = np.array([oracle.e4m3_value(int(c)) for c in codes])
    mids = (vals[:-1] + vals[1:]) / 2          # exact ties: round to the even code
    v = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(447.0), 50000))])
    v = np.concatenate([v, -v]).astype(np.float32)
    got = oracle.f32_to_e4m3(v)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_e4m3_saturates():
    for x in (448.0, 449.0, 464.0, 1e6, 3e38):
        assert int(oracle.f32_to_e4m3(x)[0]) == 0x7E
        assert int(oracle.f32_to_e4m3(-x)[0]) == 0xFE


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-30, 1000),
                        rng.normal(0, 1e30, 1000)]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(x)) for x in v])
    assert np.array_equal(got, want)


def test_bf16_rounding_at_the_ends_of_its_range_matches_torch():
    # the largest bf16 value (255/128) 2^127, whose ulp is 2^120: a quarter ulp above it rounds
    # down to it, half an ulp above is a tie that goes to the even neighbour 2^128 (overflow to
    # inf); and the subnormal ties around the smallest bf16 subnormal 2^-133
    top = 255.0 / 128.0 * 2.0 ** 127
    vals = [top, top + 2.0 ** 118, top + 2.0 ** 119, top + 3 * 2.0 ** 118, 3.4028234663852886e38,
            2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134, 5 * 2.0 ** -134, 2.0 ** -127, 2.0 ** -126 - 2.0 ** -140]
    v = np.array(vals + [-x for x in vals], np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(x)) for x in v])
    assert np.array_equal(got, want)
    assert want[0] == top and want[1] == top and np.isinf(want[2]) and want[6] == 0.0
