"""Exhaustive checks of the hardware conversions the quantizers rely on, against the oracle's
conversions (which the format pins fix):

  * E4M3 (block scales; the FP8 shared expert): every finite fp32 bit pattern, through
    lmoe_quantize_fp8 with amax 448, which makes s_enc = 448/448 = 1 so each code is the
    conversion of the value itself;
  * E2M1 (NVFP4 elements): every fp32 bit pattern with 2^-10 <= |x| <= 6, and zero, through
    lmoe_quantize_nvfp4 with amax 10.5 (s_enc = 256, s_dec = 2^-8): a block led by 6 gets the
    scale 256, so bd = 1 and every other element is converted unscaled.
Chunks of 2^26 values; both sides see the same fp32 inputs.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


def test_e4m3_every_finite_fp32():
    import nvfp4_latentmoe_fwd_02_b300 as lm
    checked = 0
    for start in range(0, 1 << 32, CHUNK):
        bits = np.arange(start, start + CHUNK, dtype=np.uint64).astype(np.uint32)
        exp = (bits >> 23) & 0xFF
        v = bits[exp != 0xFF].view(np.float32)             # NaN and Inf are outside the contract
        if v.size == 0:
            continue
        codes, ts = lm.lmoe_quantize_fp8(torch.from_numpy(v).cuda(), 448.0)
        got = codes.cpu().numpy()
        want = oracle.f32_to_e4m3(v)
        assert float(ts.cpu()[0]) == 1.0
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (v[bad[:5]], got[bad[:5]], want[bad[:5]])
        checked += v.size
    assert checked == (1 << 32) - (1 << 24)


def test_e2m1_every_fp32_up_to_6():
    import nvfp4_latentmoe_fwd_02_b300 as lm
    lo = np.float32(2.0 ** -10).view(np.uint32)
    hi = np.float32(6.0).view(np.uint32)
    mags = np.arange(lo, hi + 1, dtype=np.uint64).astype(np.uint32)
    checked = 0
    for sign in (0, 0x80000000):
        for s in range(0, mags.size, CHUNK):
            v = (mags[s:s + CHUNK] | np.uint32(sign)).view(np.float32)
            n = (v.size + 14) // 15 * 15
            vv = np.concatenate([v, np.zeros(n - v.size, np.float32)]).reshape(-1, 15)
            x = np.concatenate([np.full((vv.shape[0], 1), 6.0, np.float32), vv], axis=1)
            codes, sf, ts = lm.lmoe_quantize_nvfp4(torch.from_numpy(x).cuda(), 10.5)
            c = codes.cpu().numpy()
            assert float(ts.cpu()[0]) == 2.0 ** -8 and np.all(sf.cpu().numpy() == 0x78)
            got = np.stack([c & 15, c >> 4], -1).reshape(-1, 16)[:, 1:].ravel()[:v.size]
            want = oracle.f32_to_e2m1(v)
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, (v[bad[:5]], got[bad[:5]], want[bad[:5]])
            checked += v.size
    assert checked == 2 * mags.size
