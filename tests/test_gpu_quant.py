"""GPU parity of the NVFP4 quantizer (lmoe_quantize_nvfp4) against the CPU oracle.

Format: shengxinai.com Nemotron 3 blog, section 3.1.1 (E2M1 elements, 16-element blocks,
E4M3 block scale) plus one FP32 tensor scale.  Codes, scales and tensor scale must be
bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _lm():
    import nvfp4_latentmoe_fwd_02_b300 as lm
    return lm


def _run(x: torch.Tensor, amax: float):
    lm = _lm()
    codes, sf, ts = lm.lmoe_quantize_nvfp4(x.cuda().contiguous(), amax)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), sf.cpu().numpy(), float(ts.cpu()[0])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,K", [(1, 16), (3, 48), (129, 64), (1000, 2048), (7, 8192)])
@pytest.mark.parametrize("static", [False, True])
def test_quantize_matches_oracle(dtype, rows, K, static):
    g = torch.Generator().manual_seed(rows * 7 + K)
    x = (torch.randn(rows, K, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 2)).to(dtype)
    xf = x.float().numpy()
    amax = float(np.abs(xf).max()) * 0.7 if static else -1.0   # static: some blocks saturate
    c, s, ts = _run(x, amax)
    oc, os_, ots = oracle.quantize_nvfp4(xf, amax)
    assert ts == ots
    assert np.array_equal(s, os_)
    assert np.array_equal(c, oc)


def test_zero_tensor_and_zero_rows():
    c, s, ts = _run(torch.zeros(4, 32), -1.0)
    assert ts == 1.0 and not c.any() and not s.any()
    lm = _lm()
    lm.lmoe_quantize_nvfp4(torch.zeros(0, 32, device="cuda"))   # no-op, no error


def test_invalid_arguments():
    lm = _lm()
    x = torch.zeros(2, 24, device="cuda")
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_quantize_nvfp4(x)
    assert ei.value.status == lm.LMOE_EINVAL


def _boundary_values(grid: np.ndarray, span: int) -> np.ndarray:
    """Every fp32 within `span` ulps of each grid value and each midpoint between neighbours."""
    pts = np.concatenate([grid, (grid[:-1] + grid[1:]) / 2]).astype(np.float32)
    bits = pts.view(np.int32)[:, None] + np.arange(-span, span + 1, dtype=np.int32)[None, :]
    v = bits.ravel().view(np.float32)
    v = v[np.isfinite(v)]
    return np.unique(np.concatenate([v, -v]))


def test_e2m1_conversion_at_every_rounding_boundary():
    # Static tensor amax 10.5 gives s_enc = 256 and s_dec = 2^-8 exactly; a block whose first
    # element is 6 gets scale e4m3(6 * 256/6) = 256, so bd = 1 and rcp = 1: each other element
    # is converted by the hardware E2M1 conversion unscaled.  Compared with the oracle's own
    # conversion of the same fp32 values (which the format pins fix).
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    v = _boundary_values(grid, 2048)
    v = v[np.abs(v) <= 6.0]
    rng = np.random.default_rng(0)
    extra = rng.uniform(-6, 6, 200000).astype(np.float32)
    tiny = (np.arange(1, 4096, dtype=np.int32)).view(np.float32)   # denormals
    v = np.concatenate([v, extra, tiny, -tiny, np.array([0.0, -0.0], np.float32)])
    n = (len(v) + 14) // 15 * 15
    v = np.concatenate([v, np.zeros(n - len(v), np.float32)])
    blocks = v.reshape(-1, 15)
    x = np.concatenate([np.full((len(blocks), 1), 6.0, np.float32), blocks], axis=1)
    c, s, ts = _run(torch.from_numpy(x), 10.5)
    assert ts == 2.0 ** -8
    assert np.all(s == 0x78)             # e4m3 code of 256
    lo, hi = c & 15, c >> 4
    codes = np.stack([lo, hi], -1).reshape(-1, 16)[:, 1:].ravel()
    want = oracle.f32_to_e2m1(blocks.ravel())
    assert np.array_equal(codes, want)


def test_e4m3_conversion_at_every_rounding_boundary():
    # Static tensor amax 448 gives s_enc = 6 and s_enc6 = 1 exactly, so a block's scale is the
    # hardware E4M3 conversion of the block amax itself.
    vals = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    v = _boundary_values(vals, 256)
    v = v[(v >= 0) & (v < 600.0)]
    rng = np.random.default_rng(1)
    v = np.concatenate([v, np.exp(rng.uniform(np.log(1e-5), np.log(500), 100000)).astype(np.float32),
                        (np.arange(0, 4096, dtype=np.int32)).view(np.float32)])
    x = np.zeros((len(v), 16), np.float32)
    x[:, 3] = v
    x[:, 7] = -v * 0.5
    c, s, ts = _run(torch.from_numpy(x), 448.0)
    assert np.array_equal(s[:, 0], oracle.f32_to_e4m3(v))
