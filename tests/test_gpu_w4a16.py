"""GPU parity of the W4A16 form of the layer (NVFP4 expert weights decoded to bf16: into tensor
memory at decode size, T <= 32, with 16- or 32-row token tiles; into shared memory above that;
bf16 z and h; NVIDIA AI releases Nemotron 3 Ultra, quantization paragraph: the
checkpoint's W4A16 form) against the oracle's W4A16 mode: routing exact, z and h within
5e-3, c and y within 2e-2 relative L2 per row."""
import numpy as np
import pytest
import torch

import lmoe_synth
from lmoe_cases import Case, real_rows, rel_l2_rows, w_tol, stored_calib

pytestmark = pytest.mark.gpu

TOL_INTER = 5e-3
TOL_OUT = 2e-2


@pytest.fixture(scope="module", params=["tiny", "mid"])
def w4(request):
    if request.param == "tiny":
        case = Case(lmoe_synth.TINY, seed=0, w4a16=True)
    else:
        case = Case(lmoe_synth.Dims(d=1024, l=512, E=32, k=4, ffn=512), seed=9, zipf=1.1, w4a16=True)
    yield case
    case.close()


def gpu_h_rows(case, T, sample):
    """The GPU's h rows of the sampled tokens in (token, slot) order, from the expert segments."""
    d = case.dims
    moe = case.moe
    nrows = int(moe.stage("nrows", T, torch.int32).cpu()[0])
    R = moe.stage("rows", T, torch.int32).numel()
    rows = moe.stage("rows", T, torch.int32).cpu().numpy()[:nrows]
    h = moe.stage("h", T, torch.bfloat16).view(R, d.ffn)[:nrows].float().cpu().numpy()
    counts = moe.stage("counts", T, torch.int32).cpu().numpy()
    live = real_rows(counts, nrows)
    pos = {int(sl): i for i, sl in enumerate(rows) if live[i]}
    return np.stack([h[pos[int(t) * d.k + j]] for t in sample for j in range(d.k)])


def check_w4a16(case, T, x, y, sample):
    d = case.dims
    moe = case.moe
    ref = case.ol.forward(x[sample].float().cpu().numpy(), quant="w4a16", want=("z", "h", "c", "y"))
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()[sample]
    assert np.array_equal(idx, ref["idx"])
    w = moe.stage("w", T, torch.float32).view(T, d.k).cpu().numpy()[sample]
    assert np.allclose(w, ref["w"], **w_tol(T))
    z = moe.stage("z", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()[sample]
    assert rel_l2_rows(z, ref["z"]).max() <= TOL_INTER
    hr = gpu_h_rows(case, T, sample)
    assert rel_l2_rows(hr, ref["h"].reshape(-1, d.ffn)).max() <= TOL_INTER
    c = moe.stage("c", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()[sample]
    assert rel_l2_rows(c, ref["c"]).max() <= TOL_OUT
    assert rel_l2_rows(y[sample].float().cpu().numpy(), ref["y"]).max() <= TOL_OUT


@pytest.mark.parametrize("T", [1, 5, 16, 17, 32, 40, 129, 600])
def test_forward_w4a16_matches_oracle(w4, T):
    moe = w4.gpu(debug=True)
    x = w4.tokens(T, seed_offset=700 + T)
    y = moe.forward(x.cuda())
    moe.check()
    sample = np.arange(T) if T <= 200 else np.sort(np.random.default_rng(T).choice(T, 150, replace=False))
    check_w4a16(w4, T, x, y, sample)


@pytest.fixture(scope="module")
def ultra_w4():
    case = Case(lmoe_synth.ULTRA, seed=1, zipf=0.0, gen_device="cuda", w4a16=True,
                calib=stored_calib("ultra_decode_T8"))
    yield case
    case.close()


@pytest.mark.parametrize("T", [8, 24])
def test_ultra_decode_w4a16(ultra_w4, T):
    moe = ultra_w4.gpu(debug=True)
    x = ultra_w4.tokens(T).cuda()
    y = moe.forward(x)
    moe.check()
    check_w4a16(ultra_w4, T, x, y, np.arange(T))


@pytest.mark.parametrize("T", [8, 16])
def test_ultra_decode_w4a16_repeated(ultra_w4, T):
    """The 16-token-tile decode kernel (three converter groups sharing the rings) run 24 times on
    the same tokens: every run completes with no bounded wait running out, and every run's h rows
    and y match the oracle.  An MMA that read a ring stage before its fill had landed would show
    up here as a wrong h row, or as a timeout, in some run."""
    moe = ultra_w4.gpu(debug=True)
    d = ultra_w4.dims
    x = ultra_w4.tokens(T, seed_offset=900 + T).cuda()
    sample = np.arange(T)
    ref = ultra_w4.ol.forward(x.float().cpu().numpy(), quant="w4a16", want=("h", "y"))
    href = ref["h"].reshape(-1, d.ffn)
    for run in range(24):
        y = moe.forward(x)
        moe.check()
        assert rel_l2_rows(gpu_h_rows(ultra_w4, T, sample), href).max() <= TOL_INTER, f"run {run}"
        assert rel_l2_rows(y.float().cpu().numpy(), ref["y"]).max() <= TOL_OUT, f"run {run}"
