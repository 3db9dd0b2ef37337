"""Layer-level drift of the NVFP4 method against its BF16-expert form, on the CPU oracle alone
(the pages' analogue is the BF16-vs-NVFP4 greedy-token agreement of the whole model, "Heidi 在
Fireworks 上训练并部署 NVIDIA Nemotron 3 Ultra", NVFP4 paragraph; here measured for one layer).

Reference: the oracle's unquantized mode (fp64, the bf16 master weights, no quantization of
weights or activations, no intermediate rounding).  Reported: relative L2 per token of y and c,
the routing agreement (the router reads x before any quantization, so it is 1 by construction),
and the flush-to-zero rate of z and h (non-zero values whose NVFP4 code is +-0).
"""
import numpy as np

import lmoe_synth
import oracle
from lmoe_cases import rel_l2_rows


def drift(case_dims, seed, T, zipf=0.0):
    L = lmoe_synth.layer(case_dims, seed, "cpu", zipf)
    w1, w2 = L.w1.float().numpy(), L.w2.float().numpy()
    ol = oracle.OracleLayer(case_dims.d, case_dims.l, case_dims.E, case_dims.k, case_dims.ffn,
                            L.w_down.float().numpy(), L.w_up.float().numpy(), L.w_router.numpy(),
                            L.b_router.numpy(), lambda e: (w1[e], w2[e]))
    ol.calibrate(lmoe_synth.calibration_tokens(64, case_dims.d, seed).float().numpy())
    x = lmoe_synth.tokens(T, case_dims.d, seed + 77).float().numpy()
    q = ol.forward(x, quant=True, want=("z", "zq_codes", "h", "hq_codes", "c", "y"))
    u = ol.forward(x, quant=False, want=("c64", "y64"))
    zero = lambda codes: ((codes & 7) == 0) & True
    zc = np.stack([q["zq_codes"] & 15, q["zq_codes"] >> 4], -1).reshape(T, -1)
    hc = np.stack([q["hq_codes"] & 15, q["hq_codes"] >> 4], -1).reshape(T, case_dims.k, -1)
    ftz_z = (zero(zc) & (q["z"] != 0)).sum() / max(1, (q["z"] != 0).sum())
    ftz_h = (zero(hc) & (q["h"] != 0)).sum() / max(1, (q["h"] != 0).sum())
    return {
        "y_rel_l2_mean": float(rel_l2_rows(q["y"], u["y64"]).mean()),
        "y_rel_l2_max": float(rel_l2_rows(q["y"], u["y64"]).max()),
        "c_rel_l2_mean": float(rel_l2_rows(q["c"], u["c64"]).mean()),
        "routing_agreement": float((q["idx"] == u["idx"]).all(axis=1).mean()),
        "ftz_rate_z": float(ftz_z), "ftz_rate_h": float(ftz_h),
    }


def test_tiny_layer_drift_against_bf16_experts():
    r = drift(lmoe_synth.TINY, 0, 128)
    print("drift tiny:", r)
    assert r["routing_agreement"] == 1.0
    # A measurement, not a pin: four 4-bit quantizations (z, W1, h, W2) of random, untrained
    # weights each add ~10 % relative error (E2M1 steps are 1/8 to 1/4 of a binade), and h =
    # relu(u)^2 is heavy-tailed inside its 16-blocks, so values below 1/24 of their block's
    # largest flush to zero.  Measured here: y 0.21 mean / 0.35 max, FTZ z 6.7 %, h 27 %.
    # The bounds only catch a broken quantized path (e.g. a dropped scale gives ~1).
    assert 0.05 < r["y_rel_l2_mean"] < 0.35 and r["y_rel_l2_max"] < 0.6
    assert r["ftz_rate_z"] < 0.15 and r["ftz_rate_h"] < 0.5
