"""Pins of the oracle's layer composition.

LatentMoE (shengxinai.com Nemotron 3 blog, section 2.2, steps 1-3; Nemotron 3 Super page,
"潜在MoE"): project d -> l, route and run the experts in l, combine, project l -> d.
Pins:
  * l = d with identity projections reduces to a textbook top-k MoE (unquantized mode);
  * E = k = 1 reduces to a plain squared-ReLU FFN (unquantized mode);
  * the quantized expert stage equals dense products of the independently decoded NVFP4
    operands (numpy matmul as the library step), step by step through z, h, c and y.
"""
import numpy as np
import pytest
import torch

import lmoe_synth
import oracle
from test_oracle_quant import dequant


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _layer(dims, seed, zipf=0.0, identity=False):
    L = lmoe_synth.layer(dims, seed, "cpu", zipf)
    wd, wu = L.w_down.float().numpy(), L.w_up.float().numpy()
    if identity:
        assert dims.l == dims.d
        wd = np.eye(dims.d, dtype=np.float32)
        wu = np.eye(dims.d, dtype=np.float32)
    w1, w2 = L.w1.float().numpy(), L.w2.float().numpy()
    ol = oracle.OracleLayer(dims.d, dims.l, dims.E, dims.k, dims.ffn, wd, wu,
                            L.w_router.numpy(), L.b_router.numpy(),
                            lambda e: (w1[e], w2[e]))
    return ol, (wd, wu, L.w_router.numpy().astype(np.float64), L.b_router.numpy(), w1, w2)


def _textbook_moe(x, Wr, b, w1, w2, k):
    """y = sum_j softmax(topk(x Wr^T + b))_j * W2_e (relu(W1_e x))^2, all fp64."""
    logits = x @ Wr.T + b
    y = np.zeros((x.shape[0], w2.shape[1]))
    sets = []
    for t in range(x.shape[0]):
        order = sorted(range(len(logits[t])), key=lambda e: (-logits[t, e], e))
        sel = sorted(order[:k])
        sets.append(sel)
        s = logits[t, sel]
        p = np.exp(s - s.max())
        p /= p.sum()
        for pj, e in zip(p, sel):
            u = w1[e].astype(np.float64) @ x[t]
            y[t] += pj * (w2[e].astype(np.float64) @ np.maximum(u, 0) ** 2)
    return y, sets


def test_identity_projections_reduce_to_textbook_moe():
    dims = lmoe_synth.Dims(d=64, l=64, E=8, k=3, ffn=32)
    ol, (wd, wu, Wr, b, w1, w2) = _layer(dims, 11, identity=True)
    x = lmoe_synth.tokens(24, dims.d, 11).float().numpy()
    res = ol.forward(x, quant=False, want=("y64",))
    y_ref, sets = _textbook_moe(x.astype(np.float64), Wr, b, w1, w2, dims.k)
    assert [list(r) for r in res["idx"]] == sets
    assert np.allclose(res["y64"], y_ref, rtol=1e-5, atol=1e-6 * np.abs(y_ref).max())


def test_router_bias_decides_the_selection():
    # A bias of +1000 on two experts (k = 2) outweighs every logit of this layer (all below 100
    # in magnitude), so every token selects exactly those two; moving the bias moves the choice.
    dims = lmoe_synth.Dims(d=64, l=64, E=8, k=2, ffn=32)
    _, (wd, wu, Wr, b, w1, w2) = _layer(dims, 13)
    x = lmoe_synth.tokens(16, dims.d, 13).float().numpy()
    assert np.abs(x.astype(np.float64) @ Wr.T).max() < 100
    for hot in ((2, 5), (0, 7)):
        bias = np.zeros(dims.E, np.float32)
        bias[list(hot)] = 1000.0
        ol = oracle.OracleLayer(dims.d, dims.l, dims.E, dims.k, dims.ffn, wd, wu, Wr.astype(np.float32),
                                bias, lambda e: (w1[e], w2[e]))
        res = ol.forward(x, quant=False, want=("y64",))
        assert np.array_equal(res["idx"], np.tile(np.array(hot, np.int32), (16, 1)))


def test_single_expert_reduces_to_plain_relu2_ffn():
    dims = lmoe_synth.Dims(d=128, l=32, E=1, k=1, ffn=64)
    ol, (wd, wu, Wr, b, w1, w2) = _layer(dims, 12)
    x = lmoe_synth.tokens(16, dims.d, 12).float().numpy().astype(np.float64)
    res = ol.forward(x, quant=False, want=("y64",))
    z = x @ wd.T.astype(np.float64)
    h = np.maximum(z @ w1[0].T.astype(np.float64), 0) ** 2
    y = (h @ w2[0].T.astype(np.float64)) @ wu.T.astype(np.float64)
    assert np.all(res["w"] == 1.0)
    assert np.allclose(res["y64"], y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


@pytest.fixture(scope="module")
def tiny():
    dims = lmoe_synth.TINY
    ol, mats = _layer(dims, 0)
    xc = lmoe_synth.calibration_tokens(64, dims.d, 0).float().numpy()
    ol.calibrate(xc)
    x = lmoe_synth.tokens(64, dims.d, 0).float().numpy()
    want = ("z", "zq_codes", "zq_sf", "h", "hq_codes", "hq_sf", "c64", "c", "y64", "y")
    return dims, ol, mats, x, ol.forward(x, quant=True, want=want)


def test_quantized_down_projection(tiny):
    dims, ol, (wd, wu, Wr, b, w1, w2), x, res = tiny
    z = x.astype(np.float64) @ wd.T.astype(np.float64)
    assert np.array_equal(res["z"], _bf16(z))  # fp64 products of bf16 values then one rounding
    c, s, _ = oracle.quantize_nvfp4(res["z"], amax=ol.amax_z)
    assert np.array_equal(c, res["zq_codes"]) and np.array_equal(s, res["zq_sf"])


def test_quantized_expert_stage_equals_decoded_matmuls(tiny):
    dims, ol, (wd, wu, Wr, b, w1, w2), x, res = tiny
    F, l = dims.ffn, dims.l
    s_z = np.float32(ol.amax_z) / np.float32(2688.0)
    s_h = np.float32(ol.amax_h) / np.float32(2688.0)
    zq = dequant(res["zq_codes"], res["zq_sf"], 1.0) * float(s_z)
    idx = res["idx"]
    for t in range(x.shape[0]):
        c = np.zeros(l)
        for j, e in enumerate(idx[t]):
            c1, s1, d1, c2, s2, d2 = ol.quantized(int(e))
            u = dequant(c1, s1, d1) @ zq[t]
            h = np.maximum(u, 0.0) ** 2
            got_h = res["h"][t, j]
            # one bf16 rounding of the exact value (ties aside): within half an ulp
            assert np.all(np.abs(got_h - h) <= np.abs(h) * 2.0 ** -8 * 1.0001 + 1e-30)
            hq = dequant(res["hq_codes"][t, j][None], res["hq_sf"][t, j][None], 1.0)[0] * float(s_h)
            o = dequant(c2, s2, d2) @ hq
            # the weight used by the combine is the softmax in fp64; w is its float rounding
            c += float(res["w"][t, j]) * o
        assert np.allclose(res["c64"][t], c, rtol=1e-6, atol=1e-6 * np.abs(c).max())
    assert np.array_equal(res["c"], _bf16(res["c64"]))


def test_quantized_up_projection(tiny):
    dims, ol, (wd, wu, Wr, b, w1, w2), x, res = tiny
    y = res["c"].astype(np.float64) @ wu.T.astype(np.float64)
    assert np.allclose(res["y64"], y, rtol=1e-12, atol=1e-12)
    assert np.array_equal(res["y"], np.array([[oracle.round_bf16(v) for v in row] for row in y],
                                             np.float32))


def test_hq_is_the_quantizer_applied_to_h(tiny):
    dims, ol, mats, x, res = tiny
    h = res["h"].reshape(-1, dims.ffn)
    c, s, _ = oracle.quantize_nvfp4(h, amax=ol.amax_h)
    assert np.array_equal(c, res["hq_codes"].reshape(c.shape))
    assert np.array_equal(s, res["hq_sf"].reshape(s.shape))


def test_calibration_amax_is_attained(tiny):
    dims, ol, mats, x, res = tiny
    xc = lmoe_synth.calibration_tokens(64, dims.d, 0).float().numpy()
    r = ol.forward(xc, quant=True, want=("z", "h"))
    assert np.abs(r["z"]).max() == np.float32(ol.amax_z)
    assert r["h"].max() == np.float32(ol.amax_h)


def test_storage_arithmetic_ultra():
    # bytes per expert: two l x ffn matrices, 4-bit codes + one byte per 16 + one fp32 each
    d = lmoe_synth.ULTRA
    per = 2 * (d.l * d.ffn // 2 + d.l * d.ffn // 16 + 4)
    assert per == 4_718_600
    assert abs(per * d.E / 1e9 - 2.416) < 1e-3


def test_forward_from_a_given_zq(tiny):
    """The layer fed a given zq: with the oracle's own zq it reproduces the plain forward bit for
    bit; with a zq one neighbouring code away in some tokens (a z one bf16 ulp away can quantize
    so), its expert stage equals the dense products of that zq's independently decoded values,
    and the outputs of the untouched tokens do not change."""
    dims, ol, mats, x, res = tiny
    want = ("zq_codes", "zq_sf", "hq_codes", "hq_sf", "c64", "c", "y")
    same = ol.forward(x, quant=True, want=want, zq=(res["zq_codes"], res["zq_sf"]))
    for k in want + ("idx", "w", "counts"):
        assert np.array_equal(same[k], res[k]), k
    zc = res["zq_codes"].copy()
    moved = [3, 17, 40]
    for t in moved:                    # raise the magnitude code of one element by one step
        lo = int(zc[t, 5]) & 15
        zc[t, 5] = (zc[t, 5] & 0xF0) | ((lo & 8) | min((lo & 7) + 1, 7))
    alt = ol.forward(x, quant=True, want=("c64", "y"), zq=(zc, res["zq_sf"]))
    keep = np.setdiff1d(np.arange(x.shape[0]), moved)
    assert np.array_equal(alt["y"][keep], res["y"][keep])
    assert not np.array_equal(alt["c64"][moved], res["c64"][moved])
    s_z = np.float32(ol.amax_z) / np.float32(2688.0)
    s_h = np.float32(ol.amax_h) / np.float32(2688.0)
    zq = dequant(zc, res["zq_sf"], 1.0) * float(s_z)
    for t in moved:
        c = np.zeros(dims.l)
        for j, e in enumerate(res["idx"][t]):
            c1, s1, d1, c2, s2, d2 = ol.quantized(int(e))
            h = _bf16(np.maximum(dequant(c1, s1, d1) @ zq[t], 0.0) ** 2)
            hc, hs, _ = oracle.quantize_nvfp4(h[None], amax=ol.amax_h)
            c += float(res["w"][t, j]) * (dequant(c2, s2, d2) @ (dequant(hc, hs, 1.0)[0] * float(s_h)))
        assert np.allclose(alt["c64"][t], c, rtol=1e-6, atol=1e-6 * np.abs(c).max())
