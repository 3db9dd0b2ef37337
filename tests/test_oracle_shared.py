"""Pins of the oracle's shared expert: FP8 E4M3 with one per-tensor scale.

The shared expert stays at the hidden width d (shengxinai.com Nemotron 3 blog, section 2.2,
closing remark) and is FP8 (NVIDIA AI releases Nemotron 3 Ultra, quantization paragraph:
NVFP4 routed experts mixed with an FP8 shared expert).  Pins:
  * FP8 quantize / decode round trip on values of the E4M3 grid, ties to even, saturation,
    signed zero, the all-zero tensor;
  * the exact E4M3 dot product against rational arithmetic;
  * a closed form of the whole shared expert: selection matrices with unit entries (one
    extra entry fixes each tensor amax to 7, so every scale is a power of two) make
    u = x[pi1(f)], h = relu(u)^2 and s_j = sign_j h[pi2(j)] exact; a transposed operand,
    a dropped scale, a wrong sign or a missing ReLU breaks it;
  * the composition with the layer: w_up = 0 gives y == s; an all-zero Ws2 gives the layer
    without a shared expert, bit for bit;
  * calibration: amax_xs = max |x| and amax_hs = max h, in the closed form above.
The decode used here is torch's float8_e4m3fn, not the oracle's.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import lmoe_synth
import oracle

E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_fp8_round_trip_on_grid_values():
    # amax 56 -> s_enc = 448/56 = 8 and s_dec = 56/448 = 1/8, both exact: every E4M3 value
    # divided by 8 quantizes to its own code and decodes back exactly.
    codes = np.array([c for c in range(256) if np.isfinite(E4M3[c])], np.uint8)
    x = (E4M3[codes] / 8.0).astype(np.float32)
    q, sdec = oracle.quantize_fp8(x, 56.0)
    assert sdec == 0.125
    assert np.array_equal(E4M3[q], E4M3[codes])           # -0 and +0 decode equal
    assert np.array_equal(E4M3[q] * sdec, x.astype(np.float64))
    # computed amax: max |x| = 448/8 = 56
    q2, sdec2 = oracle.quantize_fp8(x, -1.0)
    assert sdec2 == 0.125 and np.array_equal(q2, q)


def test_fp8_ties_saturation_sign_and_zero():
    # s_enc = 1 (amax 448).  1.0625 lies halfway between 1.0 (mantissa 000) and 1.125
    # (001): ties go to the even mantissa, 1.0.  1.1875 lies between 1.125 (001) and 1.25
    # (010): -> 1.25.  Beyond 448 saturates to 448; -0.0 keeps its sign; 2^-10 is half of
    # the smallest subnormal 2^-9: a tie with 0 -> 0; 3 * 2^-10 -> 2^-9 * 2 (tie to even).
    x = np.array([1.0625, 1.1875, 500.0, -1000.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -10], np.float32)
    q, sdec = oracle.quantize_fp8(x, 448.0)
    assert sdec == 1.0
    assert list(E4M3[q]) == [1.0, 1.25, 448.0, -448.0, 0.0, 0.0, 2.0 ** -8]
    assert q[4] == 0x80 and q[5] == 0x00
    q, sdec = oracle.quantize_fp8(np.zeros(8, np.float32), -1.0)
    assert sdec == 1.0 and not q.any()


def test_fp8_dot_is_exact():
    rng = np.random.default_rng(3)
    finite = np.array([c for c in range(256) if np.isfinite(E4M3[c])], np.uint8)
    for K in (1, 31, 1000, 8192):
        a = rng.choice(finite, K)
        b = rng.choice(finite, K)
        exact = sum(Fraction(float(E4M3[i])) * Fraction(float(E4M3[j])) for i, j in zip(a, b))
        assert Fraction(oracle.fp8_dot(a, b)) == exact
    # the largest products do not overflow: 8192 * 448^2
    a = np.full(8192, 0x7E, np.uint8)
    assert oracle.fp8_dot(a, a) == 8192 * 448.0 ** 2


def _selection_case(d=64, F=40, T=12, seed=5, amax_xs=7.0, amax_hs=7.0):
    """Closed-form shared expert: returns (layer, x, expected h, expected s)."""
    rng = np.random.default_rng(seed)
    pi1 = rng.permutation(d - 1)[:F]                  # f -> column of x (never d - 1)
    pi2 = rng.integers(0, F - 1, d)                   # j -> row of h (never F - 1)
    sign = rng.choice([-1.0, 1.0], d)
    ws1 = np.zeros((F, d), np.float32)
    ws1[np.arange(F), pi1] = 1.0
    ws1[0, d - 1] = 7.0                               # amax 7: s_enc 64, s_dec 2^-6
    ws2 = np.zeros((d, F), np.float32)
    ws2[np.arange(d), pi2] = sign
    ws2[3, F - 1] = 7.0
    grid = np.array([0.25, 0.5, 1.0, 1.5, 2.0, -0.25, -0.5, -1.0, -1.5, -2.0], np.float32)
    x = rng.choice(grid, (T, d)).astype(np.float32)
    x[:, d - 1] = 0.0                                 # meets the amax entry of ws1
    x[:, pi1[F - 1]] = -np.abs(x[:, pi1[F - 1]])      # u[F-1] <= 0, so h[F-1] = 0
    u = x[:, pi1]
    h = np.maximum(u, 0.0) ** 2                       # {0, 1/16, 1/4, 1, 9/4, 4}: exact in bf16
    s = sign[None, :] * h[:, pi2]
    dims = lmoe_synth.Dims(d=d, l=16, E=4, k=2, ffn=32)
    L = lmoe_synth.layer(dims, seed, "cpu")
    ol = oracle.OracleLayer(d, 16, 4, 2, 32, L.w_down.float().numpy(), L.w_up.float().numpy(),
                            L.w_router.numpy(), None,
                            lambda e: (L.w1[e].float().numpy(), L.w2[e].float().numpy()),
                            amax_z=4.0, amax_h=16.0, shared=(ws1, ws2), amax_xs=amax_xs, amax_hs=amax_hs)
    return ol, x, h, s


def test_shared_expert_selection_closed_form():
    ol, x, h, s = _selection_case()
    c1, d1, c2, d2 = ol.quantized_shared()
    assert d1 == 2.0 ** -6 and d2 == 2.0 ** -6
    r = ol.shared_forward(x, quant=True)
    assert np.array_equal(E4M3[r["xs_q"]] * 2.0 ** -6, x.astype(np.float64))
    assert np.array_equal(r["hs"], h.astype(np.float32))
    # h * 64 lies on the E4M3 grid (16, 64, 144, 256 and 4): the codes decode back to h
    assert np.array_equal(E4M3[r["hs_q"]] * 2.0 ** -6, h)
    assert np.array_equal(r["s"], s.astype(np.float32))
    # the unquantized path gives the same exact values here
    r0 = ol.shared_forward(x, quant=False)
    assert np.array_equal(r0["s"], s.astype(np.float32))


def test_shared_expert_activation_scales_are_separate():
    # amax_xs = 3.5 (s_enc 128, s_dec 2^-7) and amax_hs = 7 (s_enc 64, s_dec 2^-6): x * 128 and
    # h * 64 still lie on the E4M3 grid, so xs_q, hs_q and s stay exact.  Quantizing h with the
    # x scale instead would saturate h = 4 at 448 / 128 = 3.5.
    ol, x, h, s = _selection_case(amax_xs=3.5, amax_hs=7.0)
    assert h.max() == 4.0
    r = ol.shared_forward(x, quant=True)
    assert np.array_equal(E4M3[r["xs_q"]] * 2.0 ** -7, x.astype(np.float64))
    assert np.array_equal(E4M3[r["hs_q"]] * 2.0 ** -6, h)
    assert np.array_equal(r["s"], s.astype(np.float32))


def test_calibrate_shared_closed_form():
    ol, x, h, _ = _selection_case(T=20, seed=8)
    ax, ah = ol.calibrate_shared(x)
    assert ax == float(np.abs(x).max())
    assert ah == float(h.max())


def test_calibrate_shared_uses_magnitudes():
    # amax_xs = max |x|: one entry of -3, beyond every other |x| <= 2, sets it
    ol, x, _, _ = _selection_case(T=20, seed=8)
    x = x.copy()
    x[4, 7] = -3.0
    ax, _ = ol.calibrate_shared(x)
    assert ax == 3.0


def test_layer_composition_with_shared_expert():
    ol, x, _, s = _selection_case(T=10, seed=9)
    # w_up = 0: c Wu^T = 0 and y = bf16(0 + s) = s (s already holds bf16 values)
    ol_up0 = oracle.OracleLayer(ol.d, ol.l, ol.E, ol.k, ol.ffn, ol.w_down,
                                np.zeros_like(ol.w_up), ol.w_router, None, ol.expert_fn,
                                amax_z=ol.amax_z, amax_h=ol.amax_h, shared=ol.shared,
                                amax_xs=7.0, amax_hs=7.0)
    r = ol_up0.forward(x, want=("y", "s"))
    assert np.array_equal(r["y"], s.astype(np.float32))
    assert np.array_equal(r["s"], s.astype(np.float32))
    # all-zero Ws2 (amax 0: codes 0, s_dec 1): s = 0 and y is the layer without it
    ws1, ws2 = ol.shared
    ol_s0 = oracle.OracleLayer(ol.d, ol.l, ol.E, ol.k, ol.ffn, ol.w_down, ol.w_up, ol.w_router,
                               None, ol.expert_fn, amax_z=ol.amax_z, amax_h=ol.amax_h,
                               shared=(ws1, np.zeros_like(ws2)), amax_xs=7.0, amax_hs=7.0)
    ol_none = oracle.OracleLayer(ol.d, ol.l, ol.E, ol.k, ol.ffn, ol.w_down, ol.w_up, ol.w_router,
                                 None, ol.expert_fn, amax_z=ol.amax_z, amax_h=ol.amax_h)
    y_s0 = ol_s0.forward(x, want=("y", "s"))
    y_none = ol_none.forward(x, want=("y",))
    assert not y_s0["s"].any()
    assert np.array_equal(y_s0["y"], y_none["y"])
    # with both parts live, y = bf16(y64_without + s) where both are exact sums here
    r2 = ol.forward(x, want=("y", "y64"))
    r_none = ol_none.forward(x, want=("y64",))
    assert np.allclose(r2["y64"], r_none["y64"] + s, rtol=0, atol=1e-9)
    assert np.array_equal(r2["y"], torch.from_numpy(r2["y64"]).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("quant", [True, False])
def test_shared_expert_outputs_agree_between_layer_and_alone(quant):
    rng = np.random.default_rng(12)
    d, F = 64, 48
    ws1 = torch.from_numpy(rng.normal(0, d ** -0.5, (F, d)).astype(np.float32)).bfloat16().float().numpy()
    ws2 = torch.from_numpy(rng.normal(0, F ** -0.5, (d, F)).astype(np.float32)).bfloat16().float().numpy()
    ol, x, _, _ = _selection_case(d=d, T=6, seed=12)
    ol = oracle.OracleLayer(ol.d, ol.l, ol.E, ol.k, ol.ffn, ol.w_down, ol.w_up, ol.w_router, None,
                            ol.expert_fn, amax_z=ol.amax_z, amax_h=ol.amax_h, shared=(ws1, ws2))
    ol.calibrate_shared(x)
    a = ol.shared_forward(x, quant=quant)
    b = ol.forward(x, quant=quant, want=("xs_q", "hs", "hs_q", "s"))
    for n in (("xs_q", "hs", "hs_q", "s") if quant else ("hs", "s")):
        assert np.array_equal(a[n], b[n]), n
