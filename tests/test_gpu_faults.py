"""Failure paths of the library, exercised without faulting, trapping or hanging the GPU.

  * A device-side wait forced to run out: LMOE_FAULT=wait makes the latent-up GEMM wait on a
    barrier nothing arrives at, under a short wait limit (lmoe_set_wait_limit); the kernel
    records LMOE_ETIMEOUT, drains its copies and tensor-core work, frees its tensor memory and
    returns.  lmoe_check (and lmoe_forward_host) then report LMOE_ETIMEOUT, and the next forward
    with the default limit matches the oracle.
  * Host-side injected failures: LMOE_FAULT=alloc:N fails the N-th device allocation of a call
    (LMOE_ENOMEM, nothing leaked), LMOE_FAULT=launch:N fails the N-th kernel launch of a forward
    before it launches (LMOE_ECUDA); the context stays usable.
  * Argument errors caught on the host before anything is launched: misaligned x, a stream that
    is being captured for lmoe_forward_host.
"""
import numpy as np
import pytest
import torch

import lmoe_synth
from lmoe_cases import Case, rel_l2_rows, w_tol

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-2


@pytest.fixture(scope="module")
def tiny():
    case = Case(lmoe_synth.TINY, seed=0)
    yield case
    case.close()


def _matches_oracle(case, T, seed_offset):
    moe = case.gpu()
    d = case.dims
    x = case.tokens(T, seed_offset=seed_offset)
    y = moe.forward(x.cuda())
    moe.check()
    ref = case.ol.forward(x.float().numpy(), quant=True, want=("y",))
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
    assert np.array_equal(idx, ref["idx"])
    assert np.array_equal(moe.stage("counts", T, torch.int32).cpu().numpy(), ref["counts"])
    assert np.allclose(moe.stage("w", T, torch.float32).view(T, d.k).cpu().numpy(), ref["w"], **w_tol(T))
    assert rel_l2_rows(y.float().cpu().numpy(), ref["y"]).max() <= TOL_OUT


@pytest.mark.parametrize("T", [8, 64, 300])
def test_injected_wait_times_out_then_recovers(tiny, monkeypatch, T):
    lm = tiny.lm
    moe = tiny.gpu()
    x = tiny.tokens(T, seed_offset=7).cuda()
    lm.lmoe_set_wait_limit(moe.ctx, 200_000)              # about 0.1 ms of SM clock
    monkeypatch.setenv("LMOE_FAULT", "wait")
    try:
        moe.forward(x)                                    # asynchronous: returns LMOE_OK
        with pytest.raises(lm.LmoeError) as ei:
            moe.check()
        assert ei.value.status == lm.LMOE_ETIMEOUT
        moe.check()                                       # reported once, then cleared
    finally:
        monkeypatch.delenv("LMOE_FAULT")
        lm.lmoe_set_wait_limit(moe.ctx, 0)
    _matches_oracle(tiny, T, seed_offset=8)


def test_forward_host_reports_the_timeout(tiny, monkeypatch):
    lm = tiny.lm
    moe = tiny.gpu()
    d = tiny.dims
    T = 32
    x = tiny.tokens(T, seed_offset=9).pin_memory()
    y = torch.empty((T, d.d), dtype=torch.bfloat16).pin_memory()
    nb = lm.lmoe_host_workspace_size(moe.ctx, T)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    lm.lmoe_set_wait_limit(moe.ctx, 200_000)
    monkeypatch.setenv("LMOE_FAULT", "wait")
    try:
        with pytest.raises(lm.LmoeError) as ei:
            lm.lmoe_forward_host(moe.ctx, x, T, y, ws, nb, s)
        assert ei.value.status == lm.LMOE_ETIMEOUT
    finally:
        monkeypatch.delenv("LMOE_FAULT")
        lm.lmoe_set_wait_limit(moe.ctx, 0)
    lm.lmoe_forward_host(moe.ctx, x, T, y, ws, nb, s)     # recaptured without the fault
    ref = tiny.ol.forward(x.float().numpy(), quant=True, want=("y",))
    assert rel_l2_rows(y.float().numpy(), ref["y"]).max() <= TOL_OUT


def _create(case):
    d, D = case.dims, case.dev
    return case.lm.lmoe_create(d.d, d.l, d.E, d.k, d.ffn, D["w_down"], D["w_up"], D["w_router"],
                               D["b_router"], D["w1"], D["w2"], case.amax_z, case.amax_h)


def test_create_allocation_failures_leak_nothing(monkeypatch):
    """Each of lmoe_create's device allocations failed in turn: LMOE_ENOMEM every time, and after
    three rounds the free device memory is where it started."""
    case = Case(lmoe_synth.Dims(d=1024, l=512, E=32, k=4, ffn=512), seed=9, calib_T=64)
    lm = case.lm
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    n_fail = 0
    for _ in range(3):
        n = 1
        while True:
            monkeypatch.setenv("LMOE_FAULT", f"alloc:{n}")
            try:
                ctx = _create(case)
            except lm.LmoeError as e:
                assert e.status == lm.LMOE_ENOMEM, n
                n_fail += 1
                n += 1
                continue
            finally:
                monkeypatch.delenv("LMOE_FAULT")
            lm.lmoe_destroy(ctx)                          # no allocation left to fail
            break
        assert n > 10                                     # every buffer of the context was tried
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    print(f"{n_fail} failed creations; free device memory {free0} -> {free1}")
    assert abs(free0 - free1) <= 8 << 20
    case.close()


def test_route_allocation_failure(tiny, monkeypatch):
    lm = tiny.lm
    ctx = _create(tiny)                                   # fresh context: no routing scratch yet
    try:
        T = 200
        x = tiny.tokens(T, seed_offset=11).cuda()
        idx = torch.empty((T, tiny.dims.k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, tiny.dims.k), dtype=torch.float32, device="cuda")
        monkeypatch.setenv("LMOE_FAULT", "alloc:1")
        try:
            with pytest.raises(lm.LmoeError) as ei:
                lm.lmoe_route(ctx, x, T, idx, w)
            assert ei.value.status == lm.LMOE_ENOMEM
        finally:
            monkeypatch.delenv("LMOE_FAULT")
        lm.lmoe_route(ctx, x, T, idx, w)
        torch.cuda.synchronize()
        _, oidx, _, _ = tiny.ol.route(x.float().cpu().numpy())
        assert np.array_equal(idx.cpu().numpy(), oidx)
    finally:
        lm.lmoe_destroy(ctx)


@pytest.mark.parametrize("T", [8, 300])
def test_forward_launch_failures(tiny, monkeypatch, T):
    """The n-th launch of a forward failed, for every n: LMOE_ECUDA, no device error latched,
    and the next forward is correct."""
    lm = tiny.lm
    moe = tiny.gpu()
    x = tiny.tokens(T, seed_offset=13).cuda()
    n = lm.lmoe_forward_kernel_count(moe.ctx, T)
    for i in range(1, n + 1):
        monkeypatch.setenv("LMOE_FAULT", f"launch:{i}")
        try:
            with pytest.raises(lm.LmoeError) as ei:
                moe.forward(x)
            assert ei.value.status == lm.LMOE_ECUDA, i
        finally:
            monkeypatch.delenv("LMOE_FAULT")
        moe.check()
    monkeypatch.setenv("LMOE_FAULT", f"launch:{n + 1}")   # past the last launch: nothing fails
    try:
        moe.forward(x)
    finally:
        monkeypatch.delenv("LMOE_FAULT")
    moe.check()
    _matches_oracle(tiny, T, seed_offset=14)


def test_misaligned_inputs_are_refused(tiny):
    lm = tiny.lm
    moe = tiny.gpu()
    d = tiny.dims
    T = 16
    buf = torch.zeros(T * d.d + 8, dtype=torch.bfloat16, device="cuda")
    x_bad = buf[1:1 + T * d.d]                            # 2 bytes past a 16-byte boundary
    idx = torch.empty((T, d.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, d.k), dtype=torch.float32, device="cuda")
    for f in (lm.lmoe_route, lm.lmoe_route_static):
        with pytest.raises(lm.LmoeError) as ei:
            f(moe.ctx, x_bad, T, idx, w)
        assert ei.value.status == lm.LMOE_EINVAL
    y = torch.empty((T, d.d), dtype=torch.bfloat16, device="cuda")
    ws = moe.workspace(T)
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_forward(moe.ctx, x_bad, T, y, ws, ws.numel())
    assert ei.value.status == lm.LMOE_EINVAL
    moe.check()


def test_forward_host_refuses_a_capturing_stream(tiny):
    lm = tiny.lm
    moe = tiny.gpu()
    d = tiny.dims
    T = 8
    x = tiny.tokens(T, seed_offset=15).pin_memory()
    y = torch.empty((T, d.d), dtype=torch.bfloat16).pin_memory()
    nb = lm.lmoe_host_workspace_size(moe.ctx, T)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    scratch = torch.zeros(16, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        scratch.add_(1.0)                                 # the captured graph is not empty
        st = lm.lib().lmoe_forward_host(moe.ctx, x.data_ptr(), T, y.data_ptr(), ws.data_ptr(), nb,
                                        s.cuda_stream)
    assert st == lm.LMOE_EINVAL
    torch.cuda.synchronize()
    lm.lmoe_forward_host(moe.ctx, x, T, y, ws, nb, s)     # outside a capture the call works
    ref = tiny.ol.forward(x.float().numpy(), quant=True, want=("y",))
    assert rel_l2_rows(y.float().numpy(), ref["y"]).max() <= TOL_OUT
