"""Reads of unwritten memory and writes out of bounds (a substitute for a memory sanitizer).

The forward runs twice on the same tokens: once on a workspace filled with zeros, once on a
workspace filled with 0xFF (a NaN in every float view, -1 in every int32 view, E2M1 code -6 and
a NaN E4M3 scale in the NVFP4 views), with the timed configuration's kernels (debug copies off).
If any kernel read a byte of the workspace before writing it in the same forward (a padding row,
a stale accumulator, an unset table entry) the two runs would differ.  Both runs also place
1 MiB guard regions filled with 0xFF before and after the workspace and y; the guards must be
unchanged afterwards.  Compared: expert indices and counts exactly; routing weights, the
quantized z, y and c nearly: the fp32 router logits, combine and split-K reductions use atomics,
whose order differs between runs, so z may land one bf16 ulp apart and a rare token take a
neighbouring zq code (a few bytes of its row).  y and c must be finite everywhere and within
5e-3 relative L2 on the tokens whose zq is the same in both runs.
"""
import numpy as np
import pytest
import torch

import lmoe_synth
from lmoe_cases import Case, rel_l2_rows, stored_calib

pytestmark = pytest.mark.gpu

GUARD = 1 << 20
TOL_RUNS = 5e-3


def _run(case, x, T, fill):
    lm = case.lm
    moe = case.moe
    d = case.dims
    need = lm.lmoe_workspace_size(moe.ctx, T)
    buf = torch.full((need + 2 * GUARD,), fill, dtype=torch.uint8, device="cuda")
    buf[:GUARD] = 0xFF
    buf[GUARD + need:] = 0xFF
    ws = buf[GUARD:GUARD + need]
    ybuf = torch.full((T * d.d * 2 + 2 * GUARD,), 0xFF, dtype=torch.uint8, device="cuda")
    y = ybuf[GUARD:GUARD + T * d.d * 2].view(torch.bfloat16).view(T, d.d)
    lm.lmoe_forward(moe.ctx, x, T, y, ws, need)
    moe.check()
    for b in (buf, ybuf):
        n = b.numel()
        assert bool((b[:GUARD] == 0xFF).all()) and bool((b[n - GUARD:] == 0xFF).all()), "guard overwritten"

    def stage(name, dtype=torch.uint8):
        off, nb = lm.lmoe_workspace_range(moe.ctx, T, name)
        t = ws[off:off + nb].view(dtype)
        return (t.float() if dtype == torch.bfloat16 else t).cpu().numpy()

    return {"y": y.float().cpu().numpy(), "idx": stage("idx", torch.int32),
            "counts": stage("counts", torch.int32), "w": stage("w", torch.float32),
            "zq_codes": stage("zq_codes"), "zq_sf": stage("zq_sf"), "c": stage("c", torch.bfloat16)}


def _compare(case, T, seed):
    moe = case.gpu(debug=False)
    x = lmoe_synth.tokens(T, case.dims.d, seed, "cuda")
    clean = _run(case, x, T, 0x00)
    poisoned = _run(case, x, T, 0xFF)
    for k in ("idx", "counts"):
        assert np.array_equal(clean[k], poisoned[k]), k
    # the routing weights above 64 tokens and z at small T come from fp32 reductions with
    # atomics: between two runs they may differ in the last bits (and z then in a rare code)
    assert np.allclose(clean["w"], poisoned["w"], rtol=1e-4, atol=1e-6)
    if case.w4a16:
        same = np.ones(T, dtype=bool)       # no activation quantizer in the W4A16 form
    else:
        zc_a, zc_b = clean["zq_codes"].reshape(T, -1), poisoned["zq_codes"].reshape(T, -1)
        zs_a, zs_b = clean["zq_sf"].reshape(T, -1), poisoned["zq_sf"].reshape(T, -1)
        same = np.all(zc_a == zc_b, axis=1) & np.all(zs_a == zs_b, axis=1)
        assert same.mean() >= 0.95
        assert np.all((zc_a != zc_b).sum(axis=1) <= 16) and np.all((zs_a != zs_b).sum(axis=1) <= 2)
    for k in ("y", "c"):
        a, b = clean[k].reshape(T, -1), poisoned[k].reshape(T, -1)
        assert np.isfinite(a).all() and np.isfinite(b).all(), k
        assert rel_l2_rows(b[same], a[same]).max() <= TOL_RUNS, k


@pytest.fixture(scope="module")
def tiny():
    case = Case(lmoe_synth.TINY, seed=5, zipf=1.1)
    yield case
    case.close()


@pytest.fixture(scope="module")
def mid():
    case = Case(lmoe_synth.Dims(d=1024, l=512, E=32, k=4, ffn=512), seed=9, zipf=1.1)
    yield case
    case.close()


@pytest.fixture(scope="module")
def ultra():
    cfg = lmoe_synth.CONFIGS["ultra_prefill_T4096_zipf1.1"]
    case = Case(cfg["dims"], seed=cfg["seed"], zipf=cfg["zipf"], gen_device="cuda",
                calib=stored_calib("ultra_prefill_T4096_zipf1.1"))
    yield case
    case.close()


@pytest.mark.parametrize("T", [1, 5, 64, 65, 300])
def test_poisoned_workspace_tiny(tiny, T):
    _compare(tiny, T, 700 + T)


@pytest.mark.parametrize("T", [8, 40, 1000])
def test_poisoned_workspace_mid(mid, T):
    _compare(mid, T, 800 + T)


@pytest.mark.parametrize("T", [8, 4096])
def test_poisoned_workspace_ultra(ultra, T):
    _compare(ultra, T, 900 + T)


@pytest.fixture(scope="module")
def mid_w4():
    case = Case(lmoe_synth.Dims(d=1024, l=512, E=32, k=4, ffn=512), seed=9, zipf=1.1, w4a16=True)
    yield case
    case.close()


# W4A16: the decode kernel (T <= 32) reads 16 or 32 token rows of each expert segment, past the
# segment's count, into accumulator columns it never stores; T = 40 takes the shared-memory path
@pytest.mark.parametrize("T", [1, 8, 20, 40])
def test_poisoned_workspace_w4a16(mid_w4, T):
    _compare(mid_w4, T, 850 + T)
