"""Write tests/golden/calibration.json: the static activation amax (z, h; with a shared
expert also its x and h) of each named workload, computed by the CPU oracle's calibration pass (post-training calibration on
synthetic prompts, "Heidi 在 Fireworks 上训练并部署 NVIDIA Nemotron 3 Ultra", NVFP4 paragraph).

Calls only the oracle and the seeded input generators.  Ultra-size inputs are drawn by
torch's generator on the GPU, so this script runs on a B300 host for those entries.
Usage: python tests/golden/make_calibration.py [config ...]
"""
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import lmoe_synth  # noqa: E402
import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "calibration.json")


def calibrate(name):
    cfg = lmoe_synth.CONFIGS[name]
    dims, gen = cfg["dims"], cfg["gen"]
    L = lmoe_synth.layer(dims, cfg["seed"], gen, cfg["zipf"])
    host = {n: getattr(L, n).float().cpu().numpy() for n in ("w_down", "w_up", "w_router", "b_router")}
    shared = None
    if dims.shared_ffn:
        shared = (L.ws1.float().cpu().numpy(), L.ws2.float().cpu().numpy())
    ol = oracle.OracleLayer(dims.d, dims.l, dims.E, dims.k, dims.ffn, host["w_down"], host["w_up"],
                            host["w_router"], host["b_router"],
                            lambda e: (L.w1[e].float().cpu().numpy(), L.w2[e].float().cpu().numpy()),
                            shared=shared)
    xc = lmoe_synth.calibration_tokens(cfg["calib_T"], dims.d, cfg["seed"], gen).float().cpu().numpy()
    az, ah = ol.calibrate(xc)
    rec = {"amax_z": az, "amax_h": ah, "calib_T": cfg["calib_T"], "torch": torch.__version__,
           "gen": gen}
    if shared is not None:
        rec["amax_xs"], rec["amax_hs"] = ol.calibrate_shared(xc)
    if gen == "cuda":
        p = torch.cuda.get_device_properties(0)
        rec["gpu"] = p.name
        rec["sm_count"] = p.multi_processor_count
    return rec


def main(names):
    data = json.load(open(OUT)) if os.path.exists(OUT) else {}
    for n in names or list(lmoe_synth.CONFIGS):
        data[n] = calibrate(n)
        print(n, data[n], flush=True)
    with open(OUT, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:])
