"""Seeded synthetic inputs for the LatentMoE expert layer.

This module only draws random numbers; it holds none of the layer's arithmetic.  Both the
CPU oracle (through the tests) and the CUDA library receive the very same tensors from it.

Recipe (every tensor from its own torch Philox / CPU generator stream, seeded from the
config seed and a fixed tag, so any one expert can be regenerated alone):
  x         [T][d]          ~ N(0, 1)            rounded to bf16
  w_down    [l][d]          ~ N(0, 1/d)          rounded to bf16    (z = x w_down^T)
  w_up      [d][l]          ~ N(0, 1/l)          rounded to bf16    (y = c w_up^T)
  w_router  [E][d]          ~ N(0, 1/d)          fp32
  b_router  [E]             0 ("uniform") or Zipf: b[pi(r)] = -s ln r, r = 1..E, pi a seeded
                            permutation (so expert popularity follows a Zipf(s) law)
  w1[e]     [ffn][l]        ~ N(0, 1/l)          rounded to bf16    (u = zq w1_e^T)
  w2[e]     [l][ffn]        ~ N(0, 1/ffn)        rounded to bf16    (o = hq w2_e^T)
  ws1       [shared_ffn][d] ~ N(0, 1/d)          rounded to bf16    (shared expert, optional)
  ws2       [d][shared_ffn] ~ N(0, 1/shared_ffn) rounded to bf16
  x_cal     [T_cal][d]      ~ N(0, 1) bf16, seed + 1: the calibration batch
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Dims:
    d: int
    l: int
    E: int
    k: int
    ffn: int
    shared_ffn: int = 0      # 0: no shared expert


TINY = Dims(d=256, l=64, E=16, k=4, ffn=128)
ULTRA = Dims(d=8192, l=2048, E=512, k=22, ffn=2048)
TINY_SHARED = Dims(d=256, l=64, E=16, k=4, ffn=128, shared_ffn=320)
ULTRA_SHARED = Dims(d=8192, l=2048, E=512, k=22, ffn=2048, shared_ffn=8192)

_TAG = {"x": 1, "w_down": 2, "w_up": 3, "w_router": 4, "perm": 5, "w1": 1000, "w2": 2000000,
        "x_cal": 7, "ws1": 8, "ws2": 9}


def _gen(device, seed: int, tag: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tag) % (2 ** 63))
    return g


def _normal(shape, std, device, seed, tag, dtype):
    g = _gen(device, seed, tag)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def tokens(T: int, d: int, seed: int, device="cpu", tag: str = "x") -> torch.Tensor:
    """x ~ N(0,1) as bf16 [T][d]."""
    return _normal((T, d), 1.0, device, seed, _TAG[tag], torch.bfloat16)


def projections(dims: Dims, seed: int, device="cpu"):
    wd = _normal((dims.l, dims.d), 1.0 / math.sqrt(dims.d), device, seed, _TAG["w_down"],
                 torch.bfloat16)
    wu = _normal((dims.d, dims.l), 1.0 / math.sqrt(dims.l), device, seed, _TAG["w_up"],
                 torch.bfloat16)
    return wd, wu


def router(dims: Dims, seed: int, device="cpu", zipf_s: float = 0.0):
    wr = _normal((dims.E, dims.d), 1.0 / math.sqrt(dims.d), device, seed, _TAG["w_router"],
                 torch.float32)
    if zipf_s <= 0.0:
        b = torch.zeros(dims.E, dtype=torch.float32, device=device)
    else:
        g = _gen("cpu", seed, _TAG["perm"])
        perm = torch.randperm(dims.E, generator=g)
        r = torch.arange(1, dims.E + 1, dtype=torch.float64)
        b = torch.empty(dims.E, dtype=torch.float64)
        b[perm] = -zipf_s * torch.log(r)
        b = b.to(torch.float32).to(device)
    return wr, b


def expert(dims: Dims, seed: int, e: int, device="cpu"):
    """(w1_e [ffn][l], w2_e [l][ffn]) bf16 for expert e."""
    w1 = _normal((dims.ffn, dims.l), 1.0 / math.sqrt(dims.l), device, seed, _TAG["w1"] + e,
                 torch.bfloat16)
    w2 = _normal((dims.l, dims.ffn), 1.0 / math.sqrt(dims.ffn), device, seed, _TAG["w2"] + e,
                 torch.bfloat16)
    return w1, w2


def experts(dims: Dims, seed: int, device="cpu"):
    """All experts stacked: (w1 [E][ffn][l], w2 [E][l][ffn]) bf16."""
    w1 = torch.empty((dims.E, dims.ffn, dims.l), dtype=torch.bfloat16, device=device)
    w2 = torch.empty((dims.E, dims.l, dims.ffn), dtype=torch.bfloat16, device=device)
    for e in range(dims.E):
        a, b = expert(dims, seed, e, device)
        w1[e].copy_(a)
        w2[e].copy_(b)
    return w1, w2


def shared_expert(dims: Dims, seed: int, device="cpu"):
    """(ws1 [shared_ffn][d], ws2 [d][shared_ffn]) bf16, or (None, None) without one."""
    if not dims.shared_ffn:
        return None, None
    ws1 = _normal((dims.shared_ffn, dims.d), 1.0 / math.sqrt(dims.d), device, seed, _TAG["ws1"],
                  torch.bfloat16)
    ws2 = _normal((dims.d, dims.shared_ffn), 1.0 / math.sqrt(dims.shared_ffn), device, seed,
                  _TAG["ws2"], torch.bfloat16)
    return ws1, ws2


@dataclasses.dataclass
class Layer:
    """All inputs of one layer instance (tensors on `device`)."""
    dims: Dims
    seed: int
    zipf_s: float
    w_down: torch.Tensor
    w_up: torch.Tensor
    w_router: torch.Tensor
    b_router: torch.Tensor
    w1: torch.Tensor
    w2: torch.Tensor
    ws1: torch.Tensor = None
    ws2: torch.Tensor = None


def layer(dims: Dims, seed: int, device="cpu", zipf_s: float = 0.0) -> Layer:
    wd, wu = projections(dims, seed, device)
    wr, b = router(dims, seed, device, zipf_s)
    w1, w2 = experts(dims, seed, device)
    ws1, ws2 = shared_expert(dims, seed, device)
    return Layer(dims, seed, zipf_s, wd, wu, wr, b, w1, w2, ws1, ws2)


def calibration_tokens(T: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """The calibration batch: N(0,1) bf16 tokens drawn with seed + 1."""
    return tokens(T, d, seed + 1, device, tag="x_cal")


# Named workloads.  calib_T: size of the calibration batch (1024 tokens drawn with seed + 1)
# whose activation amax fixes the static scales.  "gen" is the device whose torch generator draws the inputs (Ultra-size
# weights are drawn on the GPU, so their values are reproducible on the same GPU model).
CONFIGS = {
    "tiny": dict(dims=TINY, seed=0, zipf=0.0, T=64, calib_T=1024, gen="cpu"),
    "ultra_decode_T8": dict(dims=ULTRA, seed=1, zipf=0.0, T=8, calib_T=1024, gen="cuda"),
    "ultra_prefill_T4096_zipf1.1": dict(dims=ULTRA, seed=1, zipf=1.1, T=4096, calib_T=1024,
                                        gen="cuda"),
    # with the FP8 shared expert at width d
    "tiny_shared": dict(dims=TINY_SHARED, seed=0, zipf=0.0, T=64, calib_T=1024, gen="cpu"),
    "ultra_long_T32768_shared": dict(dims=ULTRA_SHARED, seed=1, zipf=0.0, T=32768, calib_T=1024,
                                     gen="cuda"),
}

# The full-block sweep (Ultra dims with the FP8 shared expert): every T against every routing
# skew.  Point i (T-major order) draws its tokens with seed 100 + i; all points share the
# weights of "ultra_long_T32768_shared" (seed 1, drawn on the GPU) and its static activation
# scales; the router bias of a point is that seed's Zipf(s) bias (s = 0: none).
SWEEP_T = (1, 8, 64, 512, 4096, 16384, 65536)
SWEEP_SKEW = (0.0, 1.1, 2.0)
SWEEP_BASE = "ultra_long_T32768_shared"


def sweep_points():
    """[{"i", "T", "zipf", "seed"}] in T-major order."""
    pts = []
    for T in SWEEP_T:
        for s in SWEEP_SKEW:
            pts.append(dict(i=len(pts), T=T, zipf=s, seed=100 + len(pts)))
    return pts
