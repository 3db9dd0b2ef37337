"""GPU routing above 64 tokens: tensor-core logits with a certified margin, canonical logits
for the candidates the margin leaves open (NVIDIA AI releases Nemotron 3 Ultra, architecture
paragraph: top-k of E experts; the canonical fp32 logit order is this project's reading).

Exact ties (integer-valued tokens and weights), all-zero tokens (every logit equal: the margin
cannot separate more than 32 candidates, so the block falls back to every canonical logit),
ordinary tokens, and at the Ultra router width tokens whose ranks k and k + 1 lie a few fp32
ulps apart, against the oracle: idx and counts bit-exact, weights within the float tolerance.
"""
import numpy as np
import pytest
import torch

import lmoe_synth
import oracle
from lmoe_cases import w_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wide():
    """d = 256, E = 64 (> 32: wider than one sorted list), k = 6."""
    import nvfp4_latentmoe_fwd_02_b300 as lm
    dims = lmoe_synth.Dims(d=256, l=64, E=64, k=6, ffn=128)
    L = lmoe_synth.layer(dims, 21, "cpu", 0.0)
    rng = np.random.default_rng(21)
    W_int = rng.integers(-1, 2, (dims.E, dims.d)).astype(np.float32)
    ctxs = {}
    for name, W, b in (("normal", L.w_router.numpy(), None),
                       ("integer", W_int, rng.integers(-2, 3, dims.E).astype(np.float32))):
        ctx = lm.lmoe_create(dims.d, dims.l, dims.E, dims.k, dims.ffn, L.w_down.cuda(), L.w_up.cuda(),
                             torch.from_numpy(W).cuda(), None if b is None else torch.from_numpy(b).cuda(),
                             L.w1.cuda(), L.w2.cuda(), 4.0, 16.0)
        ctxs[name] = (ctx, W, b)
    yield lm, dims, ctxs
    for ctx, _, _ in ctxs.values():
        lm.lmoe_destroy(ctx)


def _route(lm, ctx, x, k, E):
    T = x.shape[0]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    lm.lmoe_route(ctx, x.cuda(), T, idx, w, counts)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("T", [65, 200, 1000])
def test_integer_ties_zero_and_normal_tokens(wide, T):
    lm, dims, ctxs = wide
    rng = np.random.default_rng(T)
    x = np.zeros((T, dims.d), np.float32)
    n_int = T // 3
    x[:n_int] = rng.integers(-2, 3, (n_int, dims.d))            # exact integer logits: ties
    x[n_int + 10:] = rng.normal(0, 1, (T - n_int - 10, dims.d))  # ten all-zero tokens between
    xb = torch.from_numpy(x).to(torch.bfloat16)
    for name, (ctx, W, b) in ctxs.items():
        idx, w, counts = _route(lm, ctx, xb, dims.k, dims.E)
        _, oidx, ow, ocounts = oracle.router(xb.float().numpy(), W, b, dims.k)
        assert np.array_equal(idx, oidx), name
        assert np.array_equal(counts, ocounts), name
        assert np.allclose(w, ow, **w_tol(T)), name


def test_zero_tokens_pick_the_lowest_indices(wide):
    lm, dims, ctxs = wide
    ctx, W, _ = ctxs["normal"]
    T = 100
    idx, w, _ = _route(lm, ctx, torch.zeros((T, dims.d), dtype=torch.bfloat16), dims.k, dims.E)
    assert np.array_equal(idx, np.tile(np.arange(dims.k), (T, 1)))
    assert np.allclose(w, 1.0 / dims.k, rtol=1e-6)


@pytest.fixture(scope="module")
def ultra_near_ties():
    """The Ultra router width (d = 8192, E = 512, top-22; NVIDIA AI releases Nemotron 3 Ultra,
    architecture paragraph) with weights built in groups of four experts: e = 4 g + r has the row
    B_g (r = 0, 1: an exact duplicate, so an exact tie broken by the lower index), B_g with one
    element raised by 2^-21 (r = 2) or one other element lowered by 2^-21 (r = 3).  A token's
    logits inside a group then differ by a few fp32 ulps, far below the certified margin of the
    tensor-core logits (about 2^-16 |x| max|w|), while groups sit ~0.1 apart; top-22 takes five
    whole groups and two of the sixth, so ranks 22 and 23 always fall inside one near-tied group
    and only the canonical fp32 order decides them.  The experts are tiny (l = ffn = 64): only
    routing is checked."""
    import nvfp4_latentmoe_fwd_02_b300 as lm
    dims = lmoe_synth.Dims(d=8192, l=64, E=512, k=22, ffn=64)
    L = lmoe_synth.layer(dims, 31, "cpu", 0.0)
    rng = np.random.default_rng(31)
    G = dims.E // 4
    base = (rng.standard_normal((G, dims.d)) / np.sqrt(dims.d)).astype(np.float32)
    W = np.repeat(base, 4, axis=0)
    j2 = rng.integers(0, dims.d, G)
    j3 = (j2 + 1 + rng.integers(0, dims.d - 1, G)) % dims.d
    W[4 * np.arange(G) + 2, j2] += np.float32(2.0 ** -21)
    W[4 * np.arange(G) + 3, j3] -= np.float32(2.0 ** -21)
    ctx = lm.lmoe_create(dims.d, dims.l, dims.E, dims.k, dims.ffn, L.w_down.cuda(), L.w_up.cuda(),
                         torch.from_numpy(W).cuda(), None, L.w1.cuda(), L.w2.cuda(), 4.0, 16.0)
    yield lm, dims, ctx, W
    lm.lmoe_destroy(ctx)


@pytest.mark.parametrize("T", [8, 64, 65, 256, 1000])
def test_ultra_width_near_ties(ultra_near_ties, T):
    lm, dims, ctx, W = ultra_near_ties
    x = lmoe_synth.tokens(T, dims.d, 900 + T)
    idx, w, counts = _route(lm, ctx, x, dims.k, dims.E)
    logits, oidx, ow, ocounts = oracle.router(x.float().numpy(), W, None, dims.k)
    # the construction: ranks k and k + 1 (canonical order) lie a few ulps apart, or tie exactly
    srt = -np.sort(-logits, axis=1)
    gap = srt[:, dims.k - 1] - srt[:, dims.k]
    ulp = np.spacing(np.abs(srt[:, dims.k - 1]).astype(np.float32))
    assert np.all(gap <= 64 * ulp), "ranks k and k+1 are not near-tied"
    print(f"T={T}: exact ties at the boundary {int((gap == 0).sum())}, median gap "
          f"{np.median(gap / ulp):.1f} ulp")
    bad = np.flatnonzero(np.any(idx != oidx, axis=1))
    assert bad.size == 0, f"{bad.size} tokens routed differently, first {bad[:8]}"
    assert np.array_equal(counts, ocounts)
    assert np.allclose(w, ow, **w_tol(T))
