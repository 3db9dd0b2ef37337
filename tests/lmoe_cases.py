"""Shared set-up for the GPU parity tests: one layer instance fed identically to the CUDA
library (through its C ABI binding) and to the CPU oracle."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import lmoe_synth
import oracle

E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def stored_calib(name):
    """The stored static activation scales of a named workload (written by
    tests/golden/make_calibration.py, which calls only the oracle): (amax_z, amax_h, amax_xs,
    amax_hs), the last two 0 without a shared expert."""
    with open(os.path.join(GOLDEN, "calibration.json")) as f:
        c = json.load(f)[name]
    assert c["calib_T"] == lmoe_synth.CONFIGS[name]["calib_T"], "stale calibration record"
    return (c["amax_z"], c["amax_h"], c.get("amax_xs", 0.0), c.get("amax_hs", 0.0))


def w_tol(T):
    """Tolerance of the routing weights: T <= 64 computes every canonical logit (rtol 2e-6);
    above, the weights come from tensor-core logits within about 1e-5 of the canonical ones
    (float outputs; the layer's float tolerance is 2e-2 relative L2 per token)."""
    return dict(rtol=2e-6, atol=1e-7) if T <= 64 else dict(rtol=1e-4, atol=1e-6)


def real_rows(counts, nrows):
    """Mask of the permuted rows that hold a routing slot: the first counts[e] rows of each
    expert's 128-row-padded segment (padding rows are never written or read)."""
    mask = np.zeros(nrows, bool)
    start = 0
    for c in np.asarray(counts):
        mask[start:start + int(c)] = True
        start += (int(c) + 127) // 128 * 128
    assert start == nrows
    return mask


def check_routing_all_tokens(case, T, x, idx, counts, w=None):
    """Expert indices and per-expert counts of every token against the oracle's router (exact),
    routing weights within their tolerance."""
    d = case.dims
    _, oidx, ow, ocounts = case.ol.route(x.float().cpu().numpy())
    bad = np.flatnonzero(np.any(idx != oidx, axis=1))
    assert bad.size == 0, f"T={T}: {bad.size} tokens routed differently, first {bad[:8]}"
    assert np.array_equal(counts, ocounts)
    assert counts.sum() == T * d.k
    if w is not None:
        assert np.allclose(w, ow, **w_tol(T))


def sample_tokens(T, n=256, seed=0):
    """n sorted token indices including the first and the last (the ragged M tile)."""
    if T <= n:
        return np.arange(T)
    s = np.sort(np.random.default_rng(seed).choice(np.arange(1, T - 1), n - 2, replace=False))
    return np.concatenate([[0], s, [T - 1]])


def check_outputs_all_tokens(case, x, zq_codes, zq_sf, outs, ref, tol=2e-2, max_moved=0.1):
    """Every sampled token's float outputs at the layer's tolerance.  x: the sampled tokens
    [n][d]; zq_codes / zq_sf: the GPU's quantized z of those tokens; outs: {name: GPU values
    [n][...]} for names among c, y; ref: the oracle's forward of x with want >= outs, zq_codes,
    zq_sf.  z is the bf16 rounding of a sum whose fp32 accumulation order the method leaves
    open, so the GPU's z may sit one bf16 ulp from the oracle's at a quantization boundary and
    its zq take a neighbouring code (or block scale); one E2M1 step of one element is up to a
    third of its value, which moves c and y by a few percent.  Those tokens are checked against
    the oracle's layer fed the GPU's zq (oracle_layer_forward_zq); they must be rare, and their
    zq must differ from the oracle's in a few bytes only.  Returns (moved, worst error of a
    moved token against the plain oracle) as a measurement."""
    n = x.shape[0]
    same = np.all(zq_codes == ref["zq_codes"], axis=1) & np.all(zq_sf == ref["zq_sf"], axis=1)
    moved = np.flatnonzero(~same)
    assert moved.size <= max(1, max_moved * n), f"{moved.size} of {n} tokens with another zq"
    for name, got in outs.items():
        err = rel_l2_rows(got[same], ref[name][same]) if same.any() else np.zeros(1)
        assert err.max() <= tol, (name, float(err.max()))
    worst = 0.0
    if moved.size:
        assert np.all((zq_codes[moved] != ref["zq_codes"][moved]).sum(axis=1) <= 16)
        assert np.all((zq_sf[moved] != ref["zq_sf"][moved]).sum(axis=1) <= 2)
        alt = case.ol.forward(np.asarray(x)[moved], quant=True, want=tuple(outs),
                              zq=(zq_codes[moved], zq_sf[moved]))
        for name, got in outs.items():
            err = rel_l2_rows(got[moved], alt[name])
            assert err.max() <= tol, (name, "zq-fed", float(err.max()))
            worst = max(worst, float(rel_l2_rows(got[moved], ref[name][moved]).max()))
    return moved.size, worst


def rel_l2_rows(a, b):
    a = np.asarray(a, np.float64).reshape(a.shape[0], -1)
    b = np.asarray(b, np.float64).reshape(b.shape[0], -1)
    num = np.linalg.norm(a - b, axis=1)
    den = np.maximum(np.linalg.norm(b, axis=1), 1e-30)
    return num / den


def atoms_to_rows(atoms: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Tensor-core scale-atom layout [rows/128][K/64][512] -> row-major [rows][K/16]."""
    a = atoms.reshape(rows // 128, K // 64, 32, 4, 4)          # [rb][kb][r0][r1][j]
    a = a.transpose(0, 3, 2, 1, 4)                             # [rb][r1][r0][kb][j]
    return a.reshape(rows, K // 16)


class Case:
    """A layer (dims, seed, routing skew) with its calibration, on the GPU and in the oracle."""

    def __init__(self, dims: lmoe_synth.Dims, seed: int, zipf: float = 0.0, calib_T: int = 1024,
                 gen_device: str = "cpu", weight_blocks_2d: bool = False, w4a16: bool = False,
                 calib=None):
        """calib: stored static scales (amax_z, amax_h, amax_xs, amax_hs) instead of the
        oracle's calibration pass."""
        import nvfp4_latentmoe_fwd_02_b300 as lm
        self.lm = lm
        self.dims, self.seed, self.zipf = dims, seed, zipf
        self.weight_blocks_2d = weight_blocks_2d
        self.w4a16 = w4a16
        L = lmoe_synth.layer(dims, seed, gen_device, zipf)
        self.L = L
        self.dev = {n: getattr(L, n).cuda() for n in
                    ("w_down", "w_up", "w_router", "b_router", "w1", "w2")}
        host = {n: getattr(L, n).float().cpu().numpy() for n in
                ("w_down", "w_up", "w_router", "b_router")}
        self._w1, self._w2 = L.w1, L.w2
        shared = None
        if dims.shared_ffn:
            self.dev["ws1"], self.dev["ws2"] = L.ws1.cuda(), L.ws2.cuda()
            shared = (L.ws1.float().cpu().numpy(), L.ws2.float().cpu().numpy())
        self.ol = oracle.OracleLayer(dims.d, dims.l, dims.E, dims.k, dims.ffn, host["w_down"],
                                     host["w_up"], host["w_router"], host["b_router"],
                                     self._expert_master, shared=shared,
                                     weight_blocks_2d=weight_blocks_2d)
        if calib is not None:
            self.amax_z, self.amax_h, self.amax_xs, self.amax_hs = (float(v) for v in calib)
            self.ol.amax_z, self.ol.amax_h = self.amax_z, self.amax_h
            self.ol.amax_xs, self.ol.amax_hs = self.amax_xs, self.amax_hs
        else:
            xc = lmoe_synth.calibration_tokens(calib_T, dims.d, seed, gen_device).float().cpu().numpy()
            self.amax_z, self.amax_h = self.ol.calibrate(xc)
            self.amax_xs, self.amax_hs = self.ol.calibrate_shared(xc) if shared else (0.0, 0.0)
        self.moe = None

    def _expert_master(self, e):
        return (self._w1[e].float().cpu().numpy(), self._w2[e].float().cpu().numpy())

    def gpu(self, debug=True):
        if self.moe is None:
            d = self.dims
            D = self.dev
            self.moe = self.lm.LatentMoE(d.d, d.l, d.E, d.k, d.ffn, D["w_down"], D["w_up"],
                                         D["w_router"], D["b_router"], D["w1"], D["w2"],
                                         self.amax_z, self.amax_h, debug=debug,
                                         ws1=D.get("ws1"), ws2=D.get("ws2"),
                                         amax_xs=self.amax_xs, amax_hs=self.amax_hs,
                                         weight_blocks_2d=self.weight_blocks_2d, w4a16=self.w4a16)
        return self.moe

    def tokens(self, T, seed_offset=0):
        return lmoe_synth.tokens(T, self.dims.d, self.seed * 7919 + 13 + seed_offset, "cpu")

    def close(self):
        if self.moe is not None:
            self.moe.close()
            self.moe = None
