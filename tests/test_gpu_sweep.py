"""GPU parity over the full-block sweep: the Ultra layer with its FP8 shared expert (d = shared
ffn = 8192) at every T in {1, 8, 64, 512, 4096, 16384, 65536} and every routing skew in
{uniform, Zipf 1.1, Zipf 2.0} (NVIDIA AI releases Nemotron 3 Ultra, architecture and
quantization paragraphs; shengxinai.com Nemotron 3 blog, section 2.2).

Per point: the expert indices and per-expert counts of every token against the oracle's router
(exact), ascending expert ids per token, and the output y of 64 sampled tokens (all tokens when
T <= 64; the first and the last, i.e. the ragged M tile, always among them) within the layer's
tolerance, every sampled token included (a token whose zq took a neighbouring code against the
oracle fed that zq; see lmoe_cases.check_outputs_all_tokens).  The static activation scales are
the stored ones of the long-prompt layer (same weights), so no calibration pass runs here.
"""
import numpy as np
import pytest
import torch

import lmoe_synth
from lmoe_cases import Case, check_outputs_all_tokens, check_routing_all_tokens, sample_tokens, stored_calib

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_OUT = 2e-2


@pytest.mark.parametrize("skew", lmoe_synth.SWEEP_SKEW)
def test_sweep_block(skew):
    base = lmoe_synth.CONFIGS[lmoe_synth.SWEEP_BASE]
    case = Case(base["dims"], seed=base["seed"], zipf=skew, gen_device="cuda",
                calib=stored_calib(lmoe_synth.SWEEP_BASE))
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
            assert np.all(np.diff(idx, axis=1) > 0)              # ascending expert id per token
            check_routing_all_tokens(case, T, x, idx, counts)
            zc = moe.stage("zq_codes", T).view(T, d.l // 2).cpu().numpy()
            zs = moe.stage("zq_sf", T).view(T, d.l // 16).cpu().numpy()
            sample = sample_tokens(T, 64, seed=p["seed"])
            xs = x[sample].float().cpu().numpy()
            ref = case.ol.forward(xs, quant=True, want=("zq_codes", "zq_sf", "y"))
            assert np.array_equal(idx[sample], ref["idx"]), (T, skew)
            moved, worst = check_outputs_all_tokens(case, xs, zc[sample], zs[sample],
                                                    {"y": y[sample].float().cpu().numpy()}, ref, TOL_OUT)
            print(f"T={T} skew={skew}: {moved} of {len(sample)} sampled tokens took a neighbouring "
                  f"zq code (their worst rel L2 against the oracle's own zq: {worst:.3e})")
            case.ol._m.clear()                                   # fp32 masters: 32 MB per expert
            del x, y
    finally:
        case.close()
