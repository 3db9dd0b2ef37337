"""GPU parity of the LatentMoE layer (tiny dims) against the CPU oracle, through the C ABI.

Layer: shengxinai.com Nemotron 3 blog, section 2.2 (project d -> l, route, latent experts,
combine, project back); routing top-k of E (NVIDIA AI releases Nemotron 3 Ultra).
Bit-exact: expert weight codes / scales / tensor scales, expert indices, per-expert counts,
and the GPU's own z and h re-quantized by the oracle vs. the GPU's codes.  Float outputs:
relative L2 per row <= 5e-3 for z and h, <= 2e-2 for c and y.
"""
import numpy as np
import pytest
import torch

import lmoe_synth
import oracle
from lmoe_cases import Case, atoms_to_rows, check_outputs_all_tokens, real_rows, rel_l2_rows, w_tol
from test_oracle_quant import dequant

pytestmark = pytest.mark.gpu

TOL_INTER = 5e-3
TOL_OUT = 2e-2


@pytest.fixture(scope="module", params=[0.0, 1.1], ids=["uniform", "zipf1.1"])
def tiny(request):
    case = Case(lmoe_synth.TINY, seed=0 if request.param == 0.0 else 5, zipf=request.param)
    yield case
    case.close()


def test_expert_weights_match_oracle(tiny):
    moe = tiny.gpu()
    d = tiny.dims
    for which, (N, K) in ((1, (d.ffn, d.l)), (2, (d.l, d.ffn))):
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
        sf = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
        for e in range(d.E):
            sdec = tiny.lm.lmoe_get_expert_nvfp4(moe.ctx, which, e, codes, sf)
            q = tiny.ol.quantized(e)
            oc, os_, od = (q[0], q[1], q[2]) if which == 1 else (q[3], q[4], q[5])
            assert sdec == od
            assert np.array_equal(sf.cpu().numpy(), os_)
            assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("T", [1, 7, 64, 65, 300])
def test_route_matches_oracle(tiny, T):
    moe = tiny.gpu()
    x = tiny.tokens(T, seed_offset=T)
    k, E = tiny.dims.k, tiny.dims.E
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    tiny.lm.lmoe_route(moe.ctx, x.cuda(), T, idx, w, counts)
    torch.cuda.synchronize()
    _, oidx, ow, ocounts = tiny.ol.route(x.float().numpy())
    assert np.array_equal(idx.cpu().numpy(), oidx)
    assert np.array_equal(counts.cpu().numpy(), ocounts)
    assert np.allclose(w.cpu().numpy(), ow, **w_tol(T))


@pytest.mark.parametrize("T", [1, 5, 64, 129, 300])
def test_forward_matches_oracle(tiny, T):
    moe = tiny.gpu(debug=True)
    d = tiny.dims
    x = tiny.tokens(T, seed_offset=1000 + T)
    y = moe.forward(x.cuda())
    moe.check()
    want = ("z", "zq_codes", "zq_sf", "h", "hq_codes", "hq_sf", "c", "y")
    ref = tiny.ol.forward(x.float().numpy(), quant=True, want=want)

    # routing: exact
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()
    counts = moe.stage("counts", T, torch.int32).cpu().numpy()
    assert np.array_equal(idx, ref["idx"])
    assert np.array_equal(counts, ref["counts"])
    w = moe.stage("w", T, torch.float32).view(T, d.k).cpu().numpy()
    assert np.allclose(w, ref["w"], **w_tol(T))

    # z: float within tolerance; the GPU's codes are the oracle's quantizer on the GPU's z
    z = moe.stage("z", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()
    assert rel_l2_rows(z, ref["z"]).max() <= TOL_INTER
    zc = moe.stage("zq_codes", T).view(T, d.l // 2).cpu().numpy()
    zs = moe.stage("zq_sf", T).view(T, d.l // 16).cpu().numpy()
    oc, os_, _ = oracle.quantize_nvfp4(z, tiny.amax_z)
    assert np.array_equal(zs, os_) and np.array_equal(zc, oc)

    # permuted rows: a valid grouping of all T*k slots by expert (padding rows carry no slot)
    nrows = int(moe.stage("nrows", T, torch.int32).cpu()[0])
    rows = moe.stage("rows", T, torch.int32).cpu().numpy()[:nrows]
    live = real_rows(counts, nrows)
    slots = rows[live]
    assert np.array_equal(np.sort(slots), np.arange(T * d.k))
    flat_idx = idx.ravel()
    start = 0
    for e in range(d.E):
        n = int(counts[e])
        assert np.all(flat_idx[rows[start:start + n]] == e)
        start += ((n + 127) // 128) * 128
    assert start == nrows

    # h per slot: float within tolerance; hq codes = oracle quantizer on the GPU's h
    R = moe.stage("rows", T, torch.int32).numel()
    h = moe.stage("h", T, torch.bfloat16).view(R, d.ffn)[:nrows].float().cpu().numpy()
    hc = moe.stage("hq_codes", T).view(R, d.ffn // 2)[:nrows].cpu().numpy()
    hs = atoms_to_rows(moe.stage("hq_sf", T).cpu().numpy()[: R * d.ffn // 16], R, d.ffn)[:nrows]
    s = rows[live]
    ref_h = ref["h"].reshape(T * d.k, d.ffn)[s]
    assert rel_l2_rows(h[live], ref_h).max() <= TOL_INTER
    oc, os_, _ = oracle.quantize_nvfp4(h[live], tiny.amax_h)
    assert np.array_equal(hs[live], os_)
    assert np.array_equal(hc[live], oc)

    # combine and output
    c = moe.stage("c", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()
    assert rel_l2_rows(c, ref["c"]).max() <= TOL_OUT
    assert rel_l2_rows(y.float().cpu().numpy(), ref["y"]).max() <= TOL_OUT


def test_forward_host_matches_device(tiny):
    moe = tiny.gpu()
    T = 37
    x = tiny.tokens(T, seed_offset=77)
    y_dev = moe.forward(x.cuda()).cpu()
    lm = tiny.lm
    nb = lm.lmoe_host_workspace_size(moe.ctx, T)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    xh = x.pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    lm.lmoe_forward_host(moe.ctx, xh, T, yh, ws, nb)
    # combine uses fp32 atomics; results agree to the last bf16 place almost everywhere
    assert rel_l2_rows(yh.float().numpy(), y_dev.float().numpy()).max() <= 1e-2
    # on a created stream: the first call captures a graph, the next ones replay it; a replay
    # reads the current contents of x_host
    st = torch.cuda.Stream()
    x2 = tiny.tokens(T, seed_offset=78)
    y2_dev = moe.forward(x2.cuda()).cpu()
    for _ in range(3):
        yh.zero_()
        lm.lmoe_forward_host(moe.ctx, xh, T, yh, ws, nb, st)
        assert rel_l2_rows(yh.float().numpy(), y_dev.float().numpy()).max() <= 1e-2
    xh.copy_(x2)
    lm.lmoe_forward_host(moe.ctx, xh, T, yh, ws, nb, st)
    assert rel_l2_rows(yh.float().numpy(), y2_dev.float().numpy()).max() <= 1e-2
    # another T captures anew
    T3 = 5
    xh3 = x2[:T3].contiguous().pin_memory()
    yh3 = torch.empty_like(xh3).pin_memory()
    lm.lmoe_forward_host(moe.ctx, xh3, T3, yh3, ws, nb, st)
    assert rel_l2_rows(yh3.float().numpy(), y2_dev[:T3].float().numpy()).max() <= 1e-2


def test_routing_is_deterministic_across_calls(tiny):
    moe = tiny.gpu()
    T = 100
    x = tiny.tokens(T, seed_offset=5).cuda()
    moe.forward(x)
    a = moe.stage("idx", T, torch.int32).clone()
    moe.forward(x)
    b = moe.stage("idx", T, torch.int32)
    assert torch.equal(a, b)


def test_invalid_arguments(tiny):
    lm = tiny.lm
    moe = tiny.gpu()
    x = tiny.tokens(4).cuda()
    y = torch.empty_like(x)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_forward(moe.ctx, x, 4, y, ws, 16)
    assert ei.value.status == lm.LMOE_ENOMEM
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_create(100, 64, 16, 4, 128, *[tiny.dev[n] for n in ("w_down", "w_up", "w_router", "b_router", "w1", "w2")], 1.0, 1.0)
    assert ei.value.status == lm.LMOE_EINVAL
    lm.lmoe_forward(moe.ctx, x, 0, y, ws, 16)   # T = 0 is a no-op


@pytest.fixture(scope="module")
def mid():
    """ℓ = ffn = 512 (four n-tiles per expert GEMM), Zipf(1.1) routing over 32 experts: several
    M tiles per hot expert, empty experts, ragged segments."""
    case = Case(lmoe_synth.Dims(d=1024, l=512, E=32, k=4, ffn=512), seed=9, zipf=1.1)
    yield case
    case.close()


@pytest.mark.parametrize("T", [8, 40, 300, 1000])
def test_forward_mid_size_stage_by_stage(mid, T):
    """Each stage against the oracle's arithmetic applied to the GPU's own inputs of that stage
    (decoded independently), then c and y against the oracle end to end on every sampled token.
    A token whose z sits on a rounding boundary can get a zq code other than the oracle's (both
    are correct quantizations of their own z); such tokens must be rare, and their c and y are
    checked against the oracle fed the GPU's zq (lmoe_cases.check_outputs_all_tokens)."""
    moe = mid.gpu(debug=True)
    d = mid.dims
    x = mid.tokens(T, seed_offset=3000 + T)
    y = moe.forward(x.cuda())
    moe.check()
    sample = np.arange(T) if T <= 300 else np.sort(np.random.default_rng(T).choice(T, 200, replace=False))
    ref = mid.ol.forward(x[sample].float().numpy(), quant=True, want=("z", "zq_codes", "zq_sf", "c", "y"))
    idx = moe.stage("idx", T, torch.int32).view(T, d.k).cpu().numpy()[sample]
    assert np.array_equal(idx, ref["idx"])
    w = moe.stage("w", T, torch.float32).view(T, d.k).cpu().numpy()[sample]
    # z within tolerance; the GPU's zq is the oracle's quantizer on the GPU's z
    z = moe.stage("z", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()[sample]
    assert rel_l2_rows(z, ref["z"]).max() <= TOL_INTER
    zc = moe.stage("zq_codes", T).view(T, d.l // 2).cpu().numpy()[sample]
    zs = moe.stage("zq_sf", T).view(T, d.l // 16).cpu().numpy()[sample]
    oc, os_, sdz = oracle.quantize_nvfp4(z, mid.amax_z)
    assert np.array_equal(zc, oc) and np.array_equal(zs, os_)
    same_zq = np.all(zc == ref["zq_codes"], axis=1)
    assert same_zq.mean() >= 0.98
    # h of every slot from the GPU's zq; hq = the oracle's quantizer on the GPU's h; c from the
    # GPU's hq and routing weights
    nrows = int(moe.stage("nrows", T, torch.int32).cpu()[0])
    R = moe.stage("rows", T, torch.int32).numel()
    rows = moe.stage("rows", T, torch.int32).cpu().numpy()[:nrows]
    h = moe.stage("h", T, torch.bfloat16).view(R, d.ffn)[:nrows].float().cpu().numpy()
    hc = moe.stage("hq_codes", T).view(R, d.ffn // 2)[:nrows].cpu().numpy()
    hsf = atoms_to_rows(moe.stage("hq_sf", T).cpu().numpy()[: R * d.ffn // 16], R, d.ffn)[:nrows]
    counts = moe.stage("counts", T, torch.int32).cpu().numpy()
    live = real_rows(counts, nrows)
    pos = {int(sl): i for i, sl in enumerate(rows) if live[i]}
    zdec = dequant(zc, zs, sdz)
    _, _, sdh = oracle.quantize_nvfp4(np.ones((1, 16), np.float32), mid.amax_h)
    c = moe.stage("c", T, torch.bfloat16).view(T, d.l).float().cpu().numpy()[sample]
    for n, t in enumerate(sample):
        acc = np.zeros(d.l)
        for j in range(d.k):
            e = int(idx[n, j])
            c1, s1, d1, c2, s2, d2 = mid.ol.quantized(e)
            r = pos[int(t) * d.k + j]
            u = dequant(c1, s1, d1) @ zdec[n]
            href = torch.from_numpy(np.maximum(u, 0.0) ** 2).to(torch.bfloat16).double().numpy()
            assert rel_l2_rows(h[r:r + 1], href[None]).max() <= TOL_INTER
            qc, qs, _ = oracle.quantize_nvfp4(h[r:r + 1], mid.amax_h)
            assert np.array_equal(hc[r:r + 1], qc) and np.array_equal(hsf[r:r + 1], qs)
            acc += float(w[n, j]) * (dequant(c2, s2, d2) @ dequant(hc[r:r + 1], hsf[r:r + 1], sdh)[0])
        cref = torch.from_numpy(acc).to(torch.bfloat16).double().numpy()
        assert rel_l2_rows(c[n:n + 1], cref[None]).max() <= TOL_INTER
    # end to end, every sampled token
    moved, worst = check_outputs_all_tokens(mid, x[sample].float().numpy(), zc, zs,
                                            {"c": c, "y": y[sample].float().cpu().numpy()}, ref, TOL_OUT)
    print(f"T={T}: {moved} of {len(sample)} tokens took a neighbouring zq code "
          f"(their worst rel L2 against the oracle's own zq: {worst:.3e})")
