"""Pins of the oracle's W4A16 form: NVFP4 expert weights, bf16 activations with no activation
quantization (NVIDIA AI releases Nemotron 3 Ultra, quantization paragraph: the NVFP4
checkpoint runs as W4A16 on Hopper; here it is a B300 option of the same layer).

  u = s_w1 (z . dq(W1q)),  h = bf16(relu(u)^2),  o = s_w2 (h . dq(W2q)),  c = bf16(sum w o)

Pins: a closed form with permutation weights whose NVFP4 codes decode exactly (one entry
value 1.3125 = 2688 * 2^-11 makes the tensor scales powers of two), and agreement with numpy
products of independently decoded weights on a random layer."""
import numpy as np
import torch

import lmoe_synth
import oracle
from test_oracle_quant import dequant


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float64)).to(torch.bfloat16).double().numpy()


def test_permutation_closed_form():
    n = 64
    rng = np.random.default_rng(6)
    p1, p2 = rng.permutation(n), rng.permutation(n)
    w1 = np.zeros((n, n), np.float32)
    w1[np.arange(n), p1] = 1.3125                      # u_f = 1.3125 x[p1[f]]
    w2 = np.zeros((n, n), np.float32)
    w2[np.arange(n), p2] = 1.3125                      # o_j = 1.3125 h[p2[j]]
    eye = np.eye(n, dtype=np.float32)
    wr = np.zeros((1, n), np.float32)
    ol = oracle.OracleLayer(n, n, 1, 1, n, eye, eye, wr, None, lambda e: (w1, w2),
                            amax_z=1.0, amax_h=1.0)
    c1, s1, d1, c2, s2, d2 = ol.quantized(0)
    assert d1 == 2.0 ** -11 and d2 == 2.0 ** -11
    assert np.array_equal(dequant(c1, s1, d1), w1) and np.array_equal(dequant(c2, s2, d2), w2)
    x = rng.choice([0.0, 0.5, -0.5, 1.0, -1.0, 1.5, 2.0, -3.0], (9, n)).astype(np.float32)
    r = ol.forward(x, quant="w4a16", want=("z", "h", "c", "y"))
    h = _bf16(np.maximum(1.3125 * x[:, p1], 0.0) ** 2)
    assert np.array_equal(r["z"], x)
    assert np.array_equal(r["h"][:, 0, :], h.astype(np.float32))
    y = _bf16(_bf16(1.3125 * h[:, p2]))
    assert np.array_equal(r["c"], y.astype(np.float32))
    assert np.array_equal(r["y"], y.astype(np.float32))


def test_matches_independently_decoded_weights():
    dims = lmoe_synth.TINY
    L = lmoe_synth.layer(dims, 4, "cpu", 0.0)
    w1, w2 = L.w1.float().numpy(), L.w2.float().numpy()
    ol = oracle.OracleLayer(dims.d, dims.l, dims.E, dims.k, dims.ffn, L.w_down.float().numpy(),
                            L.w_up.float().numpy(), L.w_router.numpy(), None,
                            lambda e: (w1[e], w2[e]), amax_z=4.0, amax_h=16.0)
    x = lmoe_synth.tokens(12, dims.d, 8).float().numpy()
    r = ol.forward(x, quant="w4a16", want=("z", "h", "c"))
    for t in range(x.shape[0]):
        acc = np.zeros(dims.l)
        for j, e in enumerate(r["idx"][t]):
            c1, s1, d1, c2, s2, d2 = ol.quantized(int(e))
            u = dequant(c1, s1, d1) @ r["z"][t].astype(np.float64)
            h = _bf16(np.maximum(u, 0.0) ** 2)
            assert np.allclose(r["h"][t, j], h, rtol=1e-2, atol=0) and \
                np.mean(r["h"][t, j] == h) > 0.99            # equal but for bf16 ties
            acc += float(r["w"][t, j]) * (dequant(c2, s2, d2) @ r["h"][t, j].astype(np.float64))
        assert np.allclose(r["c"][t], _bf16(acc), rtol=1e-2, atol=1e-30)
        assert np.mean(r["c"][t] == _bf16(acc)) > 0.99
