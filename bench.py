#!/usr/bin/env python
"""bench.py -- LatentMoE layer forward throughput on B300 (tokens/s and roofline fraction).

Workload (one "step" = one whole forward of the layer over one batch):
  headline: decode-size batch, T = 8 tokens at Ultra dims (d = 8192, l = 2048, E = 512,
            top-22, ffn = 2048), uniform routing, NVFP4 experts, BF16 projections;
  also:     prefill, T = 4096 at Ultra dims with a Zipf(1.1) router bias (reported under
            "prefill"), and one long prompt, T = 32768 at Ultra dims plus the FP8 shared expert
            (d = shared ffn = 8192), uniform routing (reported under "long_shared").
Inputs are seeded synthetic tensors (lmoe_synth); the static activation scales come from
tests/golden/calibration.json (the oracle's calibration pass, written by
tests/golden/make_calibration.py).

Timing: each step is one CUDA-graph replay of lmoe_forward; L2 is flushed (256 MB write)
before every step, outside the step's own event pair; K steps are bracketed by a barrier and
a device synchronize; the reported time is the sum of the per-step event times, max over
ranks.  N > 1 (torchrun): independent replicas, one per GPU ("weak" scaling, no data-path
collective).  --impl reference times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import lmoe_synth  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
HEADLINE = "ultra_decode_T8"
PREFILL = "ultra_prefill_T4096_zipf1.1"
LONG = "ultra_long_T32768_shared"


def args_():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="lmoe", choices=["lmoe", "reference"])
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-long", action="store_true")
    p.add_argument("--no-w4a16", action="store_true")
    p.add_argument("--long-steps", type=int, default=5)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--prefill-steps", type=int, default=20)
    p.add_argument("--only-prefill", action="store_true",
                   help="profiling aid: build and run only the prefill workload, print its line")
    p.add_argument("--sweep", action="store_true",
                   help="the full-block sweep instead (Ultra + FP8 shared expert, T x routing "
                        "skew): one JSON line per point")
    p.add_argument("--only-long", action="store_true",
                   help="profiling aid: build and run only the long-prompt workload, print its line")
    return p.parse_args()


# ----------------------------------------------------------------------------------------
# distributed plumbing (timing only; no data-path collective)
# ----------------------------------------------------------------------------------------
class Dist:
    """One process per GPU (torchrun env).  Only timing is exchanged: a barrier around the
    timed region and the max of the per-rank elapsed times.  backend "gloo" runs on CPU."""

    def __init__(self, backend: str = "nccl"):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cuda" if backend == "nccl" else "cpu"
        if self.world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                torch.cuda.set_device(self.local)
                dist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
            else:
                dist.init_process_group("gloo")
            self.pg = dist
        elif backend == "nccl":
            torch.cuda.set_device(0)

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------
# workload set-up
# ----------------------------------------------------------------------------------------
def calibration(name):
    with open(os.path.join(ROOT, "tests", "golden", "calibration.json")) as f:
        return json.load(f)[name]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "src": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "src": "fallback"}


def csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "nvfp4_latentmoe_fwd_02_b300", "csrc")
    for n in sorted(os.listdir(d)):
        with open(os.path.join(d, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def build_layers(names):
    """One set of weights (seed of the first config) and one context per routing config."""
    import nvfp4_latentmoe_fwd_02_b300 as lm
    cfgs = [lmoe_synth.CONFIGS[n] for n in names]
    dims, seed = cfgs[0]["dims"], cfgs[0]["seed"]
    assert all(c["dims"] == dims and c["seed"] == seed for c in cfgs)
    L = lmoe_synth.layer(dims, seed, "cuda", 0.0)
    out = {}
    for n, c in zip(names, cfgs):
        _, b = lmoe_synth.router(dims, seed, "cuda", c["zipf"])
        cal = calibration(n)
        moe = lm.LatentMoE(dims.d, dims.l, dims.E, dims.k, dims.ffn, L.w_down, L.w_up,
                           L.w_router, b, L.w1, L.w2, cal["amax_z"], cal["amax_h"])
        out[n] = moe
    torch.cuda.synchronize()
    L.w1 = L.w2 = None            # the contexts hold the quantized experts; masters not kept
    torch.cuda.empty_cache()
    return L, out


def build_long():
    """The long-prompt layer with its FP8 shared expert (own weights draw of the same seed)."""
    import nvfp4_latentmoe_fwd_02_b300 as lm
    c = lmoe_synth.CONFIGS[LONG]
    dims = c["dims"]
    L = lmoe_synth.layer(dims, c["seed"], "cuda", c["zipf"])
    cal = calibration(LONG)
    moe = lm.LatentMoE(dims.d, dims.l, dims.E, dims.k, dims.ffn, L.w_down, L.w_up, L.w_router,
                       L.b_router, L.w1, L.w2, cal["amax_z"], cal["amax_h"], ws1=L.ws1, ws2=L.ws2,
                       amax_xs=cal["amax_xs"], amax_hs=cal["amax_hs"])
    torch.cuda.synchronize()
    del L
    torch.cuda.empty_cache()
    return moe


class Runner:
    """CUDA graphs of lmoe_forward over a small pool of distinct token batches."""

    def __init__(self, moe, T, seed, pool=4):
        import nvfp4_latentmoe_fwd_02_b300 as lm
        self.lm, self.moe, self.T = lm, moe, T
        d = moe.d
        self.xs = [lmoe_synth.tokens(T, d, seed * 7919 + 101 + i, "cuda") for i in range(pool)]
        self.y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
        self.ws = moe.workspace(T)
        self.nbytes = self.ws.numel()
        self.stream = torch.cuda.Stream()
        self.graphs = []
        with torch.cuda.stream(self.stream):
            for x in self.xs:             # warm (lazy module loading) before capture
                lm.lmoe_forward(moe.ctx, x, T, self.y, self.ws, self.nbytes, self.stream)
            self.stream.synchronize()
            for x in self.xs:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    lm.lmoe_forward(moe.ctx, x, T, self.y, self.ws, self.nbytes, self.stream)
                self.graphs.append(g)
        torch.cuda.synchronize()
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.flush_src = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
        self.flush_sink = torch.empty(1, dtype=torch.int64, device="cuda")

    def flush(self):
        """Write 256 MB (evicts L2), then read another 256 MB (writes the dirty lines back)."""
        with torch.cuda.stream(self.stream):
            self.flush_buf.fill_(1)
            self.flush_sink.copy_(self.flush_src.sum(dtype=torch.int64).view(1))

    def timed_steps(self, K, warmup):
        for i in range(warmup):
            self.flush()
            with torch.cuda.stream(self.stream):
                self.graphs[i % len(self.graphs)].replay()
        self.stream.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for i in range(K):
            self.flush()
            with torch.cuda.stream(self.stream):
                evs[i][0].record(self.stream)
                self.graphs[i % len(self.graphs)].replay()
                evs[i][1].record(self.stream)
        self.stream.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def profile(self, reps=5):
        """Per-kernel times (ms) of non-graph forwards with cold L2, averaged over reps."""
        lm = self.lm
        lm.lmoe_set_profile(self.moe.ctx, True)
        acc = {}
        order = []
        try:
            for r in range(reps):
                self.flush()
                with torch.cuda.stream(self.stream):
                    lm.lmoe_forward(self.moe.ctx, self.xs[r % len(self.xs)], self.T, self.y,
                                    self.ws, self.nbytes, self.stream)
                for n, ms in lm.lmoe_profile_read(self.moe.ctx):
                    if n not in acc:
                        acc[n] = []
                        order.append(n)
                    acc[n].append(ms)
        finally:
            lm.lmoe_set_profile(self.moe.ctx, False)
        return [(n, sum(acc[n]) / len(acc[n])) for n in order]


def expert_bytes(moe, T):
    """Algorithmic bytes of the two expert GEMM launches of the last forward (device counts):
    the touched experts' weights only (codes, block scales, FP32 tensor scale of one matrix per
    expert).  The activations these launches read and write (zq, hq, the fp32 combine
    accumulator) are intermediates of the layer, which the algorithmic bytes exclude; they are
    reported beside it as `with_activations`."""
    d = moe
    counts = moe.stage("counts", T, torch.int32).cpu()
    touched = int((counts > 0).sum())
    slots = int(counts.sum())
    l, F = d.l, d.ffn
    w_bytes = l * F // 2 + l * F // 16 + 4          # one matrix of one expert (codes, scales, fp32)
    act_in_up = slots * (l // 2 + l // 16)
    act_out_up = slots * (F // 2 + F // 16)
    act_in_dn = slots * (F // 2 + F // 16)
    out_dn = T * l * 4                               # fp32 combine accumulator (read-modify-write once)
    return {"expert_up": touched * w_bytes, "expert_down": touched * w_bytes,
            "with_activations": {"expert_up": touched * w_bytes + act_in_up + act_out_up,
                                 "expert_down": touched * w_bytes + act_in_dn + out_dn},
            "touched": touched, "slots": slots}


def layer_bytes(moe, T, eb):
    d, l = moe.d, moe.l
    return (2 * eb["touched"] * (l * moe.ffn // 2 + l * moe.ffn // 16 + 4) + 2 * d * l * 2 +
            moe.E * d * 4 + 2 * T * d * 2)


def flops_expert(moe, slots):
    return 4 * moe.l * moe.ffn * slots


def ncu_traffic(kernel_key):
    """dram bytes per launch from a committed ncu summary, if taken on the current kernels."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(kernel_key)
    if not rec or rec.get("csrc_hash") != csrc_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def cpu_baseline(T, L, cfg_name, budget_s=20.0):
    """The oracle, as it stands, on the same workload (token batch of the headline step)."""
    import numpy as np

    import oracle
    cfg = lmoe_synth.CONFIGS[cfg_name]
    dims = cfg["dims"]
    host = {n: getattr(L, n).float().cpu().numpy() for n in ("w_down", "w_up", "w_router")}
    _, b = lmoe_synth.router(dims, cfg["seed"], "cpu", cfg["zipf"])
    cal = calibration(cfg_name)
    ol = oracle.OracleLayer(dims.d, dims.l, dims.E, dims.k, dims.ffn, host["w_down"], host["w_up"],
                            host["w_router"], b.numpy(),
                            lambda e: tuple(t.float().cpu().numpy()
                                            for t in lmoe_synth.expert(dims, cfg["seed"], e, "cuda")),
                            cal["amax_z"], cal["amax_h"])
    x = lmoe_synth.tokens(T, dims.d, cfg["seed"] * 7919 + 101, "cuda").float().cpu().numpy()
    _, idx, _, _ = ol.route(x)
    for e in sorted(set(int(v) for v in np.unique(idx))):
        ol.quantized(e)                      # weight quantization is set-up, not the step
    t0 = time.perf_counter()
    ol.forward(x, quant=True, want=("y",))
    t1 = time.perf_counter() - t0
    reps = max(1, min(50, int(budget_s / max(t1, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(reps):
        ol.forward(x, quant=True, want=("y",))
    el = time.perf_counter() - t0
    cores = min(os.cpu_count() or 1, T)
    return {"value": T * reps / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} full forwards of the T={T} batch (all {T} tokens), "
                      f"{dims.E} experts top-{dims.k}; expert weight quantization excluded"}, ol, x


# ----------------------------------------------------------------------------------------
def run_reference(a, dist):
    if dist.rank != 0:
        return
    cfg = lmoe_synth.CONFIGS[HEADLINE]
    dims, T = cfg["dims"], cfg["T"]
    wd, wu = lmoe_synth.projections(dims, cfg["seed"], "cuda")
    wr, b = lmoe_synth.router(dims, cfg["seed"], "cuda", 0.0)
    L = lmoe_synth.Layer(dims, cfg["seed"], 0.0, wd, wu, wr, b, None, None)
    cb, ol, x = cpu_baseline(T, L, HEADLINE, budget_s=1.0)
    for _ in range(a.warmup):
        ol.forward(x, quant=True, want=("y",))
    t0 = time.perf_counter()
    for _ in range(a.steps):
        ol.forward(x, quant=True, want=("y",))
    el = time.perf_counter() - t0
    v = T * a.steps / el
    cb["value"] = v
    cb["sample"] = f"{a.steps} timed forwards of the full T={T} batch"
    line = {"impl": "reference", "metric": "LatentMoE layer tokens/s (T=8, Ultra dims)",
            "value": v, "unit": "tokens/s", "n_gpus": a.gpus, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": el / a.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (exact nvfp4 block dots)",
            "data": "synthetic", "config": workload_config(HEADLINE),
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(name):
    c = lmoe_synth.CONFIGS[name]
    d = c["dims"]
    sh = f", + FP8 shared expert ffn={d.shared_ffn}" if d.shared_ffn else ""
    return {"workload": f"LatentMoE forward, T={c['T']}, d={d.d}, l={d.l}, E={d.E}, top-{d.k}, "
                        f"ffn={d.ffn}, routing {'uniform' if c['zipf'] == 0 else 'Zipf(%g)' % c['zipf']}{sh}",
            "T": c["T"], "d": d.d, "l": d.l, "E": d.E, "k": d.k, "ffn": d.ffn,
            **({"shared_ffn": d.shared_ffn} if d.shared_ffn else {}),
            "routing": "uniform" if c["zipf"] == 0 else f"zipf{c['zipf']}",
            "l2": "flushed before every step (256 MB write + 256 MB read, outside the step's events)",
            "graph": "one CUDA graph replay per step"}


def roofline_entry(prof, moe, T, pk):
    eb = expert_bytes(moe, T)
    times = dict(prof)
    dom = max(("expert_up", "expert_down"), key=lambda n: times.get(n, 0.0))
    ms = times[dom]
    achieved = eb[dom] / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": ncu_traffic(f"{dom}_T{T}"),
            "algorithmic_bytes": eb[dom], "bytes_counted": "touched expert weights (intermediates excluded)",
            "frac_with_activations": eb["with_activations"][dom] / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "launch_ms": ms, "peak_src": f"{pk['src']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"}, eb


def long_entry(a, dist, pk):
    """The long-prompt point: T = 32768 plus the FP8 shared expert."""
    c = lmoe_synth.CONFIGS[LONG]
    moe = build_long()
    T = c["T"]
    r = Runner(moe, T, c["seed"], pool=2)
    K = max(3, a.long_steps)
    with Clocks(torch.cuda.current_device()) as clk:
        ms = r.timed_steps(K, 3)
    tot = dist.max(sum(ms))
    prof = r.profile(reps=2)
    times = dict(prof)
    d, FS = moe.d, moe.shared_ffn
    # per-kernel FLOPs of the contractions (dense math of the definitions)
    eb = expert_bytes(moe, T)
    flops = {"shared_up": 2 * T * d * FS, "shared_down": 2 * T * d * FS,
             "down_proj": 2 * T * d * moe.l, "up_proj": 2 * T * d * moe.l,
             "expert_up": 2 * eb["slots"] * moe.l * moe.ffn,
             "expert_down": 2 * eb["slots"] * moe.l * moe.ffn,
             "router_approx": 2 * T * 2 * d * moe.E}
    ratio = {"shared_up": 2.0, "shared_down": 2.0, "expert_up": 6.0, "expert_down": 6.0,
             "down_proj": 1.0, "up_proj": 1.0, "router_approx": 1.0}
    dom = max(flops, key=lambda n: times.get(n, 0.0))
    ach = flops[dom] / (times[dom] * 1e-3) / 1e12
    peak = pk["bf16_tflops"] * ratio[dom]
    dtype = {2.0: "fp8", 6.0: "nvfp4", 1.0: "bf16"}[ratio[dom]]
    moe.close()
    del r
    torch.cuda.empty_cache()
    return {
        "config": workload_config(LONG), "steps": K,
        "tokens_per_s": T * K * dist.world / (tot * 1e-3), "ms_per_step": tot / K,
        "per_kernel_ms": {n: round(v, 4) for n, v in prof},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak,
                     "unit": "TFLOP/s", "frac": ach / peak, "traffic": None,
                     "dtype": dtype, "flops_per_launch": flops[dom], "launch_ms": times[dom],
                     "peak_src": f"{pk['src']} bf16 cuBLAS (MEASURED_PEAKS.json bf16_tflops) x "
                                 f"{ratio[dom]:g}, the nominal {dtype}/bf16 dense ratio"},
        "clocks": clk.summary(),
    }


def sweep(a, dist, pk):
    """The full Ultra block with its FP8 shared expert over every T x routing skew of the sweep
    (lmoe_synth.sweep_points): one weight draw, one context per skew, the long-prompt layer's
    static scales.  Per point: tokens/s and two roofline fractions,
      experts: max(touched expert bytes / HBM, expert FLOPs / NVFP4 peak) / expert-stage time,
      layer:   max(algorithmic bytes / HBM, sum over precisions of FLOPs / peak) / step time,
    peaks: measured HBM copy, measured bf16 x the nominal dense ratios (nvfp4 6, fp8 2)."""
    import nvfp4_latentmoe_fwd_02_b300 as lm
    base = lmoe_synth.CONFIGS[lmoe_synth.SWEEP_BASE]
    dims, seed = base["dims"], base["seed"]
    cal = calibration(lmoe_synth.SWEEP_BASE)
    L = lmoe_synth.layer(dims, seed, "cuda", 0.0)
    moes = {}
    for s in lmoe_synth.SWEEP_SKEW:
        _, b = lmoe_synth.router(dims, seed, "cuda", s)
        moes[s] = lm.LatentMoE(dims.d, dims.l, dims.E, dims.k, dims.ffn, L.w_down, L.w_up,
                               L.w_router, b, L.w1, L.w2, cal["amax_z"], cal["amax_h"],
                               ws1=L.ws1, ws2=L.ws2, amax_xs=cal["amax_xs"], amax_hs=cal["amax_hs"])
    torch.cuda.synchronize()
    del L
    torch.cuda.empty_cache()
    bw = pk["hbm_gbs"] * 1e9
    p_bf16 = pk["bf16_tflops"] * 1e12
    d, l, E, F, FS = dims.d, dims.l, dims.E, dims.ffn, dims.shared_ffn
    w_e = l * F // 2 + l * F // 16 + 4                  # one expert matrix: codes, scales, fp32
    for p in lmoe_synth.sweep_points():
        T, moe = p["T"], moes[p["zipf"]]
        r = Runner(moe, T, p["seed"], pool=1)
        K = 5 if T <= 4096 else 3
        with Clocks(torch.cuda.current_device()) as clk:
            ms = r.timed_steps(K, 3)
        tot = dist.max(sum(ms))
        prof = dict(r.profile(reps=1))
        eb = expert_bytes(moe, T)
        t_exp = (prof.get("expert_up", 0.0) + prof.get("expert_down", 0.0)) * 1e-3
        fl_e = 4 * l * F * eb["slots"]
        roof_e = max(2 * eb["touched"] * w_e / bw, fl_e / (6 * p_bf16))
        bytes_layer = layer_bytes(moe, T, eb) + 2 * d * FS       # + the shared expert's FP8 weights
        t_comp = fl_e / (6 * p_bf16) + (4 * T * d * l + 2 * T * d * E) / p_bf16 + 4 * T * d * FS / (2 * p_bf16)
        roof_l = max(bytes_layer / bw, t_comp)
        step = tot / K * 1e-3
        if dist.rank == 0:
            print(json.dumps({
                "sweep_point": p["i"], "T": T, "routing": "uniform" if p["zipf"] == 0 else f"zipf{p['zipf']}",
                "seed": p["seed"], "steps": K, "ms_per_step": tot / K,
                "tokens_per_s": T * K * dist.world / (tot * 1e-3),
                "touched_experts": eb["touched"], "slots": eb["slots"],
                "expert_stage_ms": t_exp * 1e3,
                "roofline_experts": {"time_ms": roof_e * 1e3, "frac": roof_e / t_exp if t_exp else None,
                                     "bound": "hbm" if 2 * eb["touched"] * w_e / bw >= fl_e / (6 * p_bf16) else "nvfp4"},
                "roofline_layer": {"time_ms": roof_l * 1e3, "frac": roof_l / step,
                                   "bound": "hbm" if bytes_layer / bw >= t_comp else "compute"},
                "per_kernel_ms": {n: round(v, 4) for n, v in prof.items()},
                "clocks": clk.summary(),
                "config": {"workload": f"LatentMoE forward + FP8 shared expert, T={T}, d={d}, l={l}, "
                                       f"E={E}, top-{dims.k}, ffn={F}, shared ffn={FS}",
                           "l2": "flushed before every step", "graph": "one CUDA graph replay per step"},
            }), flush=True)
        del r
        torch.cuda.empty_cache()
    for m in moes.values():
        m.close()


def main():
    a = args_()
    dist = Dist("nccl")
    if a.impl == "reference":
        run_reference(a, dist)
        dist.close()
        return
    import nvfp4_latentmoe_fwd_02_b300 as lm
    pk = peaks()
    if a.sweep:
        sweep(a, dist, pk)
        dist.close()
        return
    if a.only_prefill:
        L, moes = build_layers([PREFILL])
        pc = lmoe_synth.CONFIGS[PREFILL]
        pr = Runner(moes[PREFILL], pc["T"], pc["seed"], pool=2)
        pms = pr.timed_steps(a.steps, max(3, a.warmup))
        if dist.rank == 0:
            print(json.dumps({"workload": PREFILL, "ms_per_step": sum(pms) / len(pms),
                              "per_kernel_ms": dict(pr.profile(reps=2))}), flush=True)
        dist.close()
        return
    if a.only_long:
        e = long_entry(a, dist, pk)
        if dist.rank == 0:
            print(json.dumps({"workload": LONG, **e}), flush=True)
        dist.close()
        return
    names = [HEADLINE] + ([] if a.no_prefill else [PREFILL])
    L, moes = build_layers(names)
    cfg = lmoe_synth.CONFIGS[HEADLINE]
    T = cfg["T"]
    moe = moes[HEADLINE]
    run = Runner(moe, T, cfg["seed"])

    # ---- headline: K timed steps
    dist.barrier()
    torch.cuda.synchronize()
    with Clocks(torch.cuda.current_device()) as clk:
        step_ms = run.timed_steps(a.steps, max(3, a.warmup))
    torch.cuda.synchronize()
    dist.barrier()
    total_ms = dist.max(sum(step_ms))
    ms_per_step = total_ms / a.steps
    value = T * a.steps * dist.world / (total_ms * 1e-3)

    # ---- per-kernel profile (cold L2), roofline of the dominant kernel
    prof = run.profile()
    roof, eb = roofline_entry(prof, moe, T, pk)
    lb = layer_bytes(moe, T, eb)

    # ---- end to end through the C ABI with host buffers
    nb = lm.lmoe_host_workspace_size(moe.ctx, T)
    ws_h = torch.empty(nb, dtype=torch.uint8, device="cuda")
    xh = run.xs[0].cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(3):
        lm.lmoe_forward_host(moe.ctx, xh, T, yh, ws_h, nb, run.stream)
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(a.steps):
        lm.lmoe_forward_host(moe.ctx, xh, T, yh, ws_h, nb, run.stream)
    e2e_s = dist.max(time.perf_counter() - t0)
    e2e = {"value": T * a.steps * dist.world / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": T * moe.d * 2, "d2h_bytes_per_step": T * moe.d * 2,
           "path": "lmoe_forward_host (pinned host x/y, copies + forward + sync per step)"}

    line = {
        "metric": "LatentMoE layer tokens/s (T=8, Ultra dims)",
        "value": value, "unit": "tokens/s", "n_gpus": dist.world, "steps": a.steps,
        "warmup": max(3, a.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3 scales, fp32 acc) + bf16",
        "data": "synthetic (seeded; random-init weights of the Ultra layer)",
        "config": workload_config(HEADLINE),
        "roofline": roof,
        "layer": {"bytes_per_step": lb, "achieved_gbs": lb / (ms_per_step * 1e-3) / 1e9,
                  "frac_hbm": lb / (ms_per_step * 1e-3) / 1e9 / pk["hbm_gbs"],
                  "touched_experts": eb["touched"], "slots": eb["slots"]},
        "per_kernel_ms": {n: round(ms, 5) for n, ms in prof},
        "gpu_launches": lm.lmoe_forward_kernel_count(moe.ctx, T) * a.steps,
        "e2e": e2e,
        "clocks": clk.summary(),
        "csrc_hash": csrc_hash(),
    }

    # ---- the W4A16 form of the same decode step (NVFP4 weights decoded on chip, bf16 z and h)
    if not a.no_w4a16:
        import nvfp4_latentmoe_fwd_02_b300 as lm2
        Lw = lmoe_synth.layer(cfg["dims"], cfg["seed"], "cuda", cfg["zipf"])
        cal = calibration(HEADLINE)
        d_ = cfg["dims"]
        mw = lm2.LatentMoE(d_.d, d_.l, d_.E, d_.k, d_.ffn, Lw.w_down, Lw.w_up, Lw.w_router, Lw.b_router,
                           Lw.w1, Lw.w2, cal["amax_z"], cal["amax_h"], w4a16=True)
        del Lw
        torch.cuda.empty_cache()
        rw = Runner(mw, T, cfg["seed"])
        with Clocks(torch.cuda.current_device()) as clkw:
            wms = rw.timed_steps(a.steps, max(3, a.warmup))
        wtot = dist.max(sum(wms))
        wprof = rw.profile()
        web = expert_bytes(mw, T)
        wt = dict(wprof)
        line["w4a16_decode"] = {
            "config": {**workload_config(HEADLINE), "experts": "W4A16 (NVFP4 weights, bf16 activations)"},
            "tokens_per_s": T * a.steps * dist.world / (wtot * 1e-3), "ms_per_step": wtot / a.steps,
            "per_kernel_ms": {n: round(v, 5) for n, v in wprof},
            "expert_up_hbm_frac": web["expert_up"] / (wt["expert_up"] * 1e-3) / 1e9 / pk["hbm_gbs"],
            "clocks": clkw.summary(),
        }
        mw.close()
        del rw
        torch.cuda.empty_cache()

    # ---- prefill point
    if not a.no_prefill:
        pc = lmoe_synth.CONFIGS[PREFILL]
        pm = moes[PREFILL]
        Tp = pc["T"]
        pr = Runner(pm, Tp, pc["seed"], pool=2)
        K2 = max(3, min(a.prefill_steps, a.steps))
        with Clocks(torch.cuda.current_device()) as clk2:
            pms = pr.timed_steps(K2, 3)
        pms_tot = dist.max(sum(pms))
        pprof = pr.profile(reps=3)
        proof, peb = roofline_entry(pprof, pm, Tp, pk)
        fl = flops_expert(pm, peb["slots"])
        exp_ms = dict(pprof)["expert_up"] + dict(pprof)["expert_down"]
        line["prefill"] = {
            "config": workload_config(PREFILL), "steps": K2,
            "tokens_per_s": Tp * K2 * dist.world / (pms_tot * 1e-3), "ms_per_step": pms_tot / K2,
            "per_kernel_ms": {n: round(ms, 4) for n, ms in pprof},
            "roofline": proof,
            "expert_stage": {"flops": fl, "ms": exp_ms, "tflops": fl / (exp_ms * 1e-3) / 1e12,
                             "touched_experts": peb["touched"], "slots": peb["slots"]},
            "clocks": clk2.summary(),
        }

    # ---- long prompt with the shared expert (its own layer and context)
    if not a.no_long:
        line["long_shared"] = long_entry(a, dist, pk)

    # ---- CPU baseline (rank 0, N = 1)
    if dist.world == 1 and not a.no_cpu_baseline:
        cb, _, _ = cpu_baseline(T, L, HEADLINE)
        line["cpu_baseline"] = cb
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
