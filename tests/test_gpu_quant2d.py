"""GPU parity of the 2-D weight-block variant (one E4M3 scale per 16 rows x 16 contraction
elements; NVIDIA AI releases Nemotron 3 Ultra, architecture paragraph: two-dimensional weight
blocks) against the CPU oracle: the quantizer and the expert weights bit-exact, the layer's
outputs within the float tolerances.  The GEMMs are the 1-D ones (each row carries its block's
scale)."""
import numpy as np
import pytest
import torch

import lmoe_synth
import oracle
from lmoe_cases import Case, rel_l2_rows, w_tol, check_outputs_all_tokens

pytestmark = pytest.mark.gpu

TOL_INTER = 5e-3
TOL_OUT = 2e-2


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,K,amax", [(16, 64, -1.0), (48, 256, 3.0), (400, 512, -1.0), (128, 2048, 0.5)])
def test_quantizer_2d_matches_oracle(dtype, rows, K, amax):
    import nvfp4_latentmoe_fwd_02_b300 as lm
    rng = np.random.default_rng(rows + K)
    x = rng.normal(0, 1, (rows, K)) * rng.choice([1e-3, 1.0, 30.0], (rows, 1))
    x[rows // 2, :16] = 0.0                               # an all-zero 1 x 16 piece
    xt = torch.from_numpy(x.astype(np.float32)).to(dtype)
    codes, sf, ts = lm.lmoe_quantize_nvfp4_2d(xt.cuda(), amax)
    torch.cuda.synchronize()
    oc, os_, od = oracle.quantize_nvfp4_2d(xt.float().numpy(), amax)
    assert float(ts.cpu()[0]) == od
    assert np.array_equal(sf.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


def test_quantizer_2d_rejects_ragged_rows():
    import nvfp4_latentmoe_fwd_02_b300 as lm
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_quantize_nvfp4_2d(torch.zeros((24, 64), device="cuda"), 1.0)
    assert ei.value.status == lm.LMOE_EINVAL


@pytest.fixture(scope="module")
def tiny2d():
    case = Case(lmoe_synth.TINY, seed=3, zipf=1.1, weight_blocks_2d=True)
    yield case
    case.close()


def test_expert_weights_2d_match_oracle(tiny2d):
    moe = tiny2d.gpu()
    d = tiny2d.dims
    for which, (N, K) in ((1, (d.ffn, d.l)), (2, (d.l, d.ffn))):
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
        sf = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
        for e in range(d.E):
            sdec = tiny2d.lm.lmoe_get_expert_nvfp4(moe.ctx, which, e, codes, sf)
            q = tiny2d.ol.quantized(e)
            oc, os_, od = (q[0], q[1], q[2]) if which == 1 else (q[3], q[4], q[5])
            assert sdec == od
            assert np.array_equal(sf.cpu().numpy(), os_)
            assert np.array_equal(codes.cpu().numpy(), oc)
            # one scale per 16 x 16 block
            s = sf.cpu().numpy().reshape(N // 16, 16, K // 16)
            assert np.all(s == s[:, :1, :])


@pytest.mark.parametrize("T", [5, 64, 300])
def test_forward_2d_matches_oracle(tiny2d, T):
    moe = tiny2d.gpu(debug=True)
    d = tiny2d.dims
    x = tiny2d.tokens(T, seed_offset=500 + T)
    y = moe.forward(x.cuda())
    moe.check()
    ref = tiny2d.ol.forward(x.float().numpy(), quant=True, want=("z", "zq_codes", "zq_sf", "c", "y"))
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
    assert np.array_equal(idx, ref["idx"])
    w = moe.stage("w", T, torch.float32).view(T, d.k).cpu().numpy()
    assert np.allclose(w, ref["w"], **w_tol(T))
    z = moe.stage("z", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()
    assert rel_l2_rows(z, ref["z"]).max() <= TOL_INTER
    zc = moe.stage("zq_codes", T).view(T, d.l // 2).cpu().numpy()
    zs = moe.stage("zq_sf", T).view(T, d.l // 16).cpu().numpy()
    c = moe.stage("c", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()
    moved, worst = check_outputs_all_tokens(tiny2d, x.float().numpy(), zc, zs,
                                            {"c": c, "y": y.float().cpu().numpy()}, ref, TOL_OUT)
    print(f"T={T}: {moved} of {T} tokens took a neighbouring zq code (worst rel L2 against the "
          f"oracle's own zq: {worst:.3e})")
