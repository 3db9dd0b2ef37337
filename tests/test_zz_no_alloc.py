"""The allocation-free routing entry point, lmoe_route_static.

It exists for callers that cannot allocate device memory when they route (allocator or
memory-pool callbacks, serving loops with memory fixed at start-up, embedders that give the
library no allocator).  It must give the same results as lmoe_route, the regular entry point,
on consecutive calls that reuse its one fixed scratch array.  This file is collected last so a
run that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import lmoe_synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    import nvfp4_latentmoe_fwd_02_b300 as lm
    dims = lmoe_synth.TINY
    L = lmoe_synth.layer(dims, 3, "cpu", 1.1)
    dev = {n: getattr(L, n).cuda() for n in ("w_down", "w_up", "w_router", "b_router", "w1", "w2")}
    ctx = lm.lmoe_create(dims.d, dims.l, dims.E, dims.k, dims.ffn, dev["w_down"], dev["w_up"],
                         dev["w_router"], dev["b_router"], dev["w1"], dev["w2"], 4.0, 20.0)
    yield lm, dims, ctx
    lm.lmoe_destroy(ctx)


def _route(lm, fn, ctx, x, k, E):
    T = x.shape[0]
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    counts = torch.full((E,), 12345, dtype=torch.int32, device="cuda")
    fn(ctx, x, T, idx, w, counts)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("T", [37, 300])
def test_route_static_matches_route_on_two_calls(layer, T):
    lm, dims, ctx = layer
    for call in range(2):
        x = lmoe_synth.tokens(T, dims.d, 900 + 10 * T + call).cuda()
        ref = _route(lm, lm.lmoe_route, ctx, x, dims.k, dims.E)
        got = _route(lm, lm.lmoe_route_static, ctx, x, dims.k, dims.E)
        assert np.array_equal(got[0], ref[0])
        # T > 64: the weights come from tensor-core logits summed by fp32 reductions in no
        # fixed order, so two calls agree to about 1e-6 relative, not bit for bit
        assert np.allclose(got[1], ref[1], rtol=2e-6 if T <= 64 else 1e-4, atol=1e-7)
        assert np.array_equal(got[2], ref[2])
        assert got[2].sum() == T * dims.k


def test_route_static_rejects_more_tokens_than_its_scratch(layer):
    lm, dims, ctx = layer
    T = (16 << 20) // (dims.E * 4) + 1
    x = torch.zeros((T, dims.d), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, dims.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, dims.k), dtype=torch.float32, device="cuda")
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_route_static(ctx, x, T, idx, w, None)
    assert ei.value.status == lm.LMOE_EINVAL
