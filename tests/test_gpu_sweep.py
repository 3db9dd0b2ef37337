"""GPU parity over the full-block sweep: the Ultra layer with its FP8 shared expert (d = shared
ffn = 8192) at every T in {1, 8, 64, 512, 4096, 16384, 65536} and every routing skew in
{uniform, Zipf 1.1, Zipf 2.0} (NVIDIA AI releases Nemotron 3 Ultra, architecture and
quantization paragraphs; shengxinai.com Nemotron 3 blog, section 2.2).

Per point: the routing invariants on every token, and on the first and the last token (the
ragged M tile) the oracle's expert indices exactly and its output y within the layer's
tolerance (for tokens whose zq equals the oracle's; a z on a rounding boundary can take the
neighbouring code, as in the stage-by-stage tests).  The static activation scales are the
stored ones of the long-prompt layer (same weights), so no calibration pass runs here.
"""
import json
import os

import numpy as np
import pytest
import torch

import lmoe_synth
from lmoe_cases import Case, rel_l2_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_OUT = 2e-2
HERE = os.path.dirname(os.path.abspath(__file__))


def _calib():
    with open(os.path.join(HERE, "golden", "calibration.json")) as f:
        c = json.load(f)[lmoe_synth.SWEEP_BASE]
    return (c["amax_z"], c["amax_h"], c["amax_xs"], c["amax_hs"])


@pytest.mark.parametrize("skew", lmoe_synth.SWEEP_SKEW)
def test_sweep_block(skew):
    base = lmoe_synth.CONFIGS[lmoe_synth.SWEEP_BASE]
    case = Case(base["dims"], seed=base["seed"], zipf=skew, gen_device="cuda", calib=_calib())
    try:
        moe = case.gpu(debug=False)
        d = case.dims
        for p in (q for q in lmoe_synth.sweep_points() if q["zipf"] == skew):
            T = p["T"]
            x = lmoe_synth.tokens(T, d.d, p["seed"], "cuda")
            y = moe.forward(x)
            moe.check()
            idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
            counts = moe.stage("counts", T, torch.int32).cpu().numpy()
            assert counts.sum() == T * d.k
            assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=d.E))
            assert np.all(np.diff(idx, axis=1) > 0)              # ascending expert id per token
            zc = moe.stage("zq_codes", T).view(T, d.l // 2).cpu().numpy()
            zs = moe.stage("zq_sf", T).view(T, d.l // 16).cpu().numpy()
            sample = np.array([0]) if T == 1 else np.array([0, T - 1])
            ref = case.ol.forward(x[sample].float().cpu().numpy(), quant=True,
                                  want=("zq_codes", "zq_sf", "y"))
            assert np.array_equal(idx[sample], ref["idx"]), (T, skew)
            same = np.all(zc[sample] == ref["zq_codes"], axis=1) & np.all(zs[sample] == ref["zq_sf"], axis=1)
            assert same.sum() >= len(sample) - 1, (T, skew)
            err = rel_l2_rows(y[sample].float().cpu().numpy()[same], ref["y"][same])
            assert err.max() <= TOL_OUT, (T, skew, err)
            case.ol._m.clear()                                   # fp32 masters: 32 MB per expert
            del x, y
    finally:
        case.close()
