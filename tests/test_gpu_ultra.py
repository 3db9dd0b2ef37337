"""GPU parity at the Ultra layer size (d = 8192, l = 2048, E = 512, top-22, ffn = 2048;
NVIDIA AI releases Nemotron 3 Ultra, architecture paragraph; l = d/4 from the shengxinai.com
Nemotron 3 blog, section 2.2), in the launch configuration the benchmark times.

Both workloads use the benchmark's layer (weights of seed 1) and its stored static activation
scales (calibrated by the oracle on 1024 tokens).  Decode (T = 8, uniform routing): every token
against the oracle.  Prefill (T = 4096, Zipf(1.1) router bias): expert indices and per-expert
counts against the oracle's router on every token, the other stages on 256 sampled tokens
(tokens are independent under static scales), every sampled token at the layer's tolerance.
"""
import numpy as np
import pytest
import torch

import lmoe_synth
import oracle
from lmoe_cases import (Case, check_outputs_all_tokens, check_routing_all_tokens, real_rows,
                        rel_l2_rows, sample_tokens, stored_calib, w_tol)

pytestmark = pytest.mark.gpu

TOL_INTER = 5e-3
TOL_OUT = 2e-2


DECODE = "ultra_decode_T8"
PREFILL = "ultra_prefill_T4096_zipf1.1"


def _case(name):
    cfg = lmoe_synth.CONFIGS[name]
    return Case(cfg["dims"], seed=cfg["seed"], zipf=cfg["zipf"], gen_device="cuda",
                calib=stored_calib(name))


@pytest.fixture(scope="module")
def ultra_uniform():
    case = _case(DECODE)
    yield case
    case.close()


@pytest.fixture(scope="module")
def ultra_zipf():
    case = _case(PREFILL)
    yield case
    case.close()


def _check_tokens(case, T, x, y, sample):
    d = case.dims
    moe = case.moe
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
    counts = moe.stage("counts", T, torch.int32).cpu().numpy()
    w = moe.stage("w", T, torch.float32).view(T, d.k).cpu().numpy()
    check_routing_all_tokens(case, T, x, idx, counts, w)
    xs = x[sample].float().cpu().numpy()
    ref = case.ol.forward(xs, quant=True, want=("z", "zq_codes", "zq_sf", "c", "y"))
    assert np.array_equal(idx[sample], ref["idx"])
    w = moe.stage("w", T, torch.float32).view(T, d.k).cpu().numpy()
    assert np.allclose(w[sample], ref["w"], **w_tol(T))
    z = moe.stage("z", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()[sample]
    assert rel_l2_rows(z, ref["z"]).max() <= TOL_INTER
    zc = moe.stage("zq_codes", T).view(T, d.l // 2).cpu().numpy()[sample]
    zs = moe.stage("zq_sf", T).view(T, d.l // 16).cpu().numpy()[sample]
    oc, os_, _ = oracle.quantize_nvfp4(z, case.amax_z)
    assert np.array_equal(zs, os_) and np.array_equal(zc, oc)
    c = moe.stage("c", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()[sample]
    moved, worst = check_outputs_all_tokens(case, xs, zc, zs, {"c": c, "y": y[sample].float().cpu().numpy()},
                                            ref, TOL_OUT)
    print(f"T={T}: {moved} of {len(sample)} sampled tokens took a neighbouring zq code "
          f"(their worst rel L2 against the oracle's own zq: {worst:.3e})")


def test_ultra_expert_weights_sampled(ultra_uniform):
    case = ultra_uniform
    moe = case.gpu(debug=True)
    d = case.dims
    codes = torch.empty((d.ffn, d.l // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((d.ffn, d.l // 16), dtype=torch.uint8, device="cuda")
    for e in (0, 137, 511):
        for which in (1, 2):
            sdec = case.lm.lmoe_get_expert_nvfp4(moe.ctx, which, e, codes, sf)
            q = case.ol.quantized(e)
            oc, os_, od = (q[0], q[1], q[2]) if which == 1 else (q[3], q[4], q[5])
            assert sdec == od
            assert np.array_equal(sf.cpu().numpy(), os_)
            assert np.array_equal(codes.cpu().numpy(), oc)


def test_ultra_decode_T8(ultra_uniform):
    case = ultra_uniform
    moe = case.gpu(debug=True)
    T = 8
    x = case.tokens(T).cuda()
    y = moe.forward(x)
    moe.check()
    _check_tokens(case, T, x, y, np.arange(T))


def test_ultra_prefill_T4096_zipf(ultra_zipf):
    case = ultra_zipf
    moe = case.gpu(debug=True)
    T = 4096
    x = case.tokens(T).cuda()
    y = moe.forward(x)
    moe.check()
    counts = moe.stage("counts", T, torch.int32).cpu().numpy()
    assert (counts == 0).sum() > 0 and counts.max() > 1000      # the skew the workload asks for
    # saturation under the static scales (calibrated on 1024 other tokens): |z| > amax_z, h > amax_h
    d = case.dims
    z = moe.stage("z", T, torch.bfloat16).view(T, d.l).float()
    nrows = int(moe.stage("nrows", T, torch.int32).cpu()[0])
    R = moe.stage("rows", T, torch.int32).numel()
    live = torch.from_numpy(real_rows(counts, nrows)).cuda()
    h = moe.stage("h", T, torch.bfloat16).view(R, d.ffn)[:nrows][live].float()
    print(f"saturation at T={T}: z {float((z.abs() > case.amax_z).float().mean()):.3e}, "
          f"h {float((h > case.amax_h).float().mean()):.3e} (amax_z {case.amax_z}, amax_h {case.amax_h})")
    _check_tokens(case, T, x, y, sample_tokens(T))


def test_ultra_router_margin_and_routing_on_many_tokens(ultra_zipf):
    """T = 4096: routing of every token against the oracle, and the tensor-core logits of 256
    sampled tokens against the canonical ones: the observed error must sit far inside the
    certified margin (whose floor is 2^-16 |x| max|w_e|)."""
    case = ultra_zipf
    moe = case.gpu(debug=True)
    d = case.dims
    T = 4096
    x = case.tokens(T, seed_offset=31).cuda()
    moe.forward(x)
    moe.check()
    check_routing_all_tokens(case, T, x, moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy(),
                             moe.stage("counts", T, torch.int32).cpu().numpy())
    sample = np.sort(np.random.default_rng(1).choice(T, 256, replace=False))
    xs = x[sample].float().cpu().numpy()
    logits, oidx, ow, _ = oracle.router(xs, case.ol.w_router, case.ol.b_router, d.k)
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()[sample]
    assert np.array_equal(idx, oidx)
    approx = moe.stage("router", T, torch.float32).view(T, d.E).cpu().numpy()[sample]
    approx = (approx + case.ol.b_router[None, :]).astype(np.float64)
    nx = np.linalg.norm(xs.astype(np.float64), axis=1)
    wn = np.linalg.norm(case.ol.w_router.astype(np.float64), axis=1).max()
    ratio = (np.abs(approx - logits) / (nx * wn)[:, None]).max()
    print(f"max |tensor-core - canonical| / (|x| max|w|) = {ratio:.3e} (margin floor 2^-16 = {2**-16:.3e})")
    assert ratio < 2.0 ** -16 / 4


def test_ultra_drift_against_bf16_experts(ultra_uniform):
    """Layer-level drift at Ultra dims, T = 8: the GPU's NVFP4 layer against the oracle's
    BF16-expert layer (unquantized mode: fp64, bf16 master weights, no quantization), with the
    flush-to-zero rates of the GPU's z and h.  The inputs, weights and static scales are
    seeded, so these are reproducible measurements (on a B300: y rel L2 mean 0.1965, max
    0.2038, c 0.1955, FTZ z 0.0649, FTZ h 0.2750); the bounds sit about 15% around them, so a
    quantizer that rounds, scales or flushes differently fails here."""
    case = ultra_uniform
    moe = case.gpu(debug=True)
    d = case.dims
    T = 8
    x = case.tokens(T, seed_offset=55).cuda()
    y = moe.forward(x)
    moe.check()
    u = case.ol.forward(x.float().cpu().numpy(), quant=False, want=("c64", "y64"))
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
    ry = rel_l2_rows(y.float().cpu().numpy(), u["y64"])
    c = moe.stage("c", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()
    z = moe.stage("z", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()
    zc = moe.stage("zq_codes", T).view(T, d.l // 2).cpu().numpy()
    zn = np.stack([zc & 15, zc >> 4], -1).reshape(T, -1)
    nrows = int(moe.stage("nrows", T, torch.int32).cpu()[0])
    R = moe.stage("rows", T, torch.int32).numel()
    live = real_rows(moe.stage("counts", T, torch.int32).cpu().numpy(), nrows)
    h = moe.stage("h", T, torch.bfloat16).view(R, d.ffn)[:nrows].float().cpu().numpy()[live]
    hc = moe.stage("hq_codes", T).view(R, d.ffn // 2)[:nrows].cpu().numpy()[live]
    hn = np.stack([hc & 15, hc >> 4], -1).reshape(hc.shape[0], -1)
    r = {"y_rel_l2_mean": float(ry.mean()), "y_rel_l2_max": float(ry.max()),
         "c_rel_l2_mean": float(rel_l2_rows(c, u["c64"]).mean()),
         "routing_agreement": float((idx == u["idx"]).all(axis=1).mean()),
         "ftz_rate_z": float((((zn & 7) == 0) & (z != 0)).sum() / max(1, (z != 0).sum())),
         "ftz_rate_h": float((((hn & 7) == 0) & (h != 0)).sum() / max(1, (h != 0).sum()))}
    print("drift ultra T=8:", r)
    assert r["routing_agreement"] == 1.0
    assert 0.17 < r["y_rel_l2_mean"] < 0.23 and r["y_rel_l2_max"] < 0.24
    assert 0.17 < r["c_rel_l2_mean"] < 0.23
    assert 0.055 < r["ftz_rate_z"] < 0.075 and 0.235 < r["ftz_rate_h"] < 0.315


@pytest.mark.parametrize("which,T", [("uniform", 8), ("zipf", 4096)])
def test_ultra_timed_configuration(ultra_uniform, ultra_zipf, which, T):
    """The benchmark times the layer with debug copies off; that forward (same kernels, no
    intermediate copies) gives the oracle's routing on every token and its output y on every
    sampled token (256 at T = 4096) within the layer's tolerance.  A z on a rounding boundary
    can take the neighbouring zq code (counted and printed; such tokens must be rare)."""
    case = ultra_uniform if which == "uniform" else ultra_zipf
    moe = case.gpu(debug=True)
    d = case.dims
    x = case.tokens(T, seed_offset=5).cuda()
    case.lm.lmoe_set_debug(moe.ctx, False)
    try:
        y = moe.forward(x)
        moe.check()
        idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
        counts = moe.stage("counts", T, torch.int32).cpu().numpy()
        zc = moe.stage("zq_codes", T).view(T, d.l // 2).cpu().numpy()
        zs = moe.stage("zq_sf", T).view(T, d.l // 16).cpu().numpy()
    finally:
        case.lm.lmoe_set_debug(moe.ctx, True)
    check_routing_all_tokens(case, T, x, idx, counts)
    sample = sample_tokens(T, seed=5)
    xs = x[sample].float().cpu().numpy()
    ref = case.ol.forward(xs, quant=True, want=("zq_codes", "zq_sf", "y"))
    assert np.array_equal(idx[sample], ref["idx"])
    moved, worst = check_outputs_all_tokens(case, xs, zc[sample], zs[sample],
                                            {"y": y[sample].float().cpu().numpy()}, ref, TOL_OUT)
    print(f"T={T}: {moved} of {len(sample)} sampled tokens took a neighbouring zq code "
          f"(their worst rel L2 against the oracle's own zq: {worst:.3e})")
