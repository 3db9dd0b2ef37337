"""GPU parity of the FP8 shared expert against the CPU oracle, through the C ABI.

The shared expert stays at the width d (shengxinai.com Nemotron 3 blog, section 2.2, closing
remark) and is FP8 E4M3 with per-tensor scales (NVIDIA AI releases Nemotron 3 Ultra,
quantization paragraph); its output joins the up-projection before the final rounding.
Bit-exact: the FP8 quantizer, the shared weight codes and tensor scales, the codes of x, and
the GPU's own h re-quantized by the oracle vs. the GPU's codes of h.  Float outputs: relative
L2 per row <= 5e-3 for h, <= 2e-2 for s and y.
"""
import numpy as np
import pytest
import torch

import lmoe_synth
import oracle
from lmoe_cases import Case, rel_l2_rows, stored_calib, check_routing_all_tokens, sample_tokens

pytestmark = pytest.mark.gpu

TOL_INTER = 5e-3
TOL_OUT = 2e-2


@pytest.fixture(scope="module")
def tiny_shared():
    case = Case(lmoe_synth.TINY_SHARED, seed=0)
    yield case
    case.close()


def _special_values(n, rng):
    v = rng.normal(0, 3, n).astype(np.float32)
    # ties of the E4M3 grid at s_enc = 1, signed zeros, saturation and subnormals
    extra = np.array([1.0625, 1.1875, -1.0625, 0.0, -0.0, 447.9, 448.0, 464.0, 500.0, -1e6,
                      2.0 ** -10, 3 * 2.0 ** -10, -(2.0 ** -9), 2.0 ** -7 * 1.5, 0.01171875], np.float32)
    v[: len(extra)] = extra
    return v


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("amax", [448.0, 3.5, -1.0, 0.0])
def test_fp8_quantizer_matches_oracle(dtype, amax):
    import nvfp4_latentmoe_fwd_02_b300 as lm
    rng = np.random.default_rng(7)
    n = 4096 + 16 * 37
    v = torch.from_numpy(_special_values(n, rng)).to(dtype)
    if amax == 0.0:
        v = torch.zeros(n, dtype=dtype)
    codes, ts = lm.lmoe_quantize_fp8(v.cuda(), amax)
    torch.cuda.synchronize()
    oc, osd = oracle.quantize_fp8(v.float().numpy(), amax)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert float(ts.cpu()[0]) == osd


def test_fp8_quantizer_empty_and_invalid():
    import nvfp4_latentmoe_fwd_02_b300 as lm
    v = torch.zeros(0, dtype=torch.float32, device="cuda")
    lm.lmoe_quantize_fp8(v, 1.0)                          # n = 0 is a no-op
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_quantize_fp8(torch.zeros(24, dtype=torch.float32, device="cuda"), 1.0)
    assert ei.value.status == lm.LMOE_EINVAL              # n % 16 != 0


def test_shared_weights_match_oracle(tiny_shared):
    moe = tiny_shared.gpu()
    d = tiny_shared.dims
    c1, d1, c2, d2 = tiny_shared.ol.quantized_shared()
    for which, (oc, od, shape) in ((1, (c1, d1, (d.shared_ffn, d.d))), (2, (c2, d2, (d.d, d.shared_ffn)))):
        codes = torch.empty(shape, dtype=torch.uint8, device="cuda")
        sdec = tiny_shared.lm.lmoe_get_shared_fp8(moe.ctx, which, codes)
        assert sdec == od
        assert np.array_equal(codes.cpu().numpy(), oc)


def _check_shared(case, T, x, y, sample=None):
    d = case.dims
    moe = case.moe
    FS = d.shared_ffn
    sel = np.arange(T) if sample is None else sample
    xs = x[sel].float().cpu().numpy()
    ref = case.ol.forward(xs, quant=True, want=("xs_q", "hs", "s", "y"))
    xq = moe.stage("xs_q", T).view(T, d.d).cpu().numpy()[sel]
    oq, _ = oracle.quantize_fp8(xs, case.amax_xs)
    assert np.array_equal(xq, oq)
    assert np.array_equal(xq, ref["xs_q"])
    hs = moe.stage("hs", T, torch.bfloat16).view(T, FS).float().cpu().numpy()[sel]
    assert rel_l2_rows(hs, ref["hs"]).max() <= TOL_INTER
    hq = moe.stage("hs_q", T).view(T, FS).cpu().numpy()[sel]
    oh, _ = oracle.quantize_fp8(hs, case.amax_hs)
    assert np.array_equal(hq, oh)
    s = moe.stage("s", T, torch.bfloat16).view(T, d.d).float().cpu().numpy()[sel]
    assert rel_l2_rows(s, ref["s"]).max() <= TOL_OUT
    assert rel_l2_rows(y[sel].float().cpu().numpy(), ref["y"]).max() <= TOL_OUT


@pytest.mark.parametrize("T", [1, 5, 64, 129, 300, 5000])
def test_forward_with_shared_expert_matches_oracle(tiny_shared, T):
    # T = 5000 takes the up-projection without split-K (the addend joins in the GEMM epilogue);
    # the smaller T split it (the addend joins in the finalize)
    moe = tiny_shared.gpu(debug=True)
    x = tiny_shared.tokens(T, seed_offset=2000 + T)
    y = moe.forward(x.cuda())
    moe.check()
    d = tiny_shared.dims
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
    sample = None if T <= 300 else np.random.default_rng(T).choice(T, 256, replace=False)
    _check_shared(tiny_shared, T, x, y, sample)
    _, oidx, _, _ = tiny_shared.ol.route(x.float().numpy())
    assert np.array_equal(idx, oidx)


def test_shared_kernel_count(tiny_shared):
    moe = tiny_shared.gpu()
    plain = Case(lmoe_synth.TINY, seed=0)
    try:
        base = plain.gpu()
        for T in (1, 300, 5000):
            assert (tiny_shared.lm.lmoe_forward_kernel_count(moe.ctx, T) ==
                    tiny_shared.lm.lmoe_forward_kernel_count(base.ctx, T) + 3)
    finally:
        plain.close()


def test_create_rejects_bad_shared_arguments(tiny_shared):
    lm = tiny_shared.lm
    D = tiny_shared.dev
    d = tiny_shared.dims
    args = [D[n] for n in ("w_down", "w_up", "w_router", "b_router", "w1", "w2")]
    bad = D["ws1"][: 100].contiguous()                  # shared_ffn = 100: not a multiple of 64
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_create(d.d, d.l, d.E, d.k, d.ffn, *args, 1.0, 1.0, None, bad, D["ws2"], 1.0, 1.0)
    assert ei.value.status == lm.LMOE_EINVAL
    with pytest.raises(lm.LmoeError) as ei:                # amax_xs must be > 0
        lm.lmoe_create(d.d, d.l, d.E, d.k, d.ffn, *args, 1.0, 1.0, None, D["ws1"], D["ws2"], 0.0, 1.0)
    assert ei.value.status == lm.LMOE_EINVAL


@pytest.fixture(scope="module")
def ultra_shared():
    cfg = lmoe_synth.CONFIGS["ultra_long_T32768_shared"]
    case = Case(cfg["dims"], seed=cfg["seed"], zipf=cfg["zipf"], gen_device="cuda",
                calib=stored_calib("ultra_long_T32768_shared"))
    yield case
    case.close()


@pytest.mark.slow
def test_ultra_long_prompt_with_shared_expert(ultra_shared):
    """T = 32768 (one long prompt), Ultra dims, shared expert d = ffn = 8192: expert indices and
    per-expert counts against the oracle's router on every token; the shared expert's stages
    and y on 64 sampled tokens (the first and the last among them)."""
    T = lmoe_synth.CONFIGS["ultra_long_T32768_shared"]["T"]
    moe = ultra_shared.gpu(debug=True)
    d = ultra_shared.dims
    x = lmoe_synth.tokens(T, d.d, 4242, "cuda")
    y = moe.forward(x)
    moe.check()
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
    counts = moe.stage("counts", T, torch.int32).cpu().numpy()
    check_routing_all_tokens(ultra_shared, T, x, idx, counts)
    sample = sample_tokens(T, 64, seed=3)
    _check_shared(ultra_shared, T, x, y, sample)
