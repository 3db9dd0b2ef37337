"""CPU oracle for the LatentMoE expert layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or runs anything here, and this package imports
nothing from the product.

The arithmetic lives in ``lmoe_oracle.c`` (plain C, built with ``-ffp-contract=off`` and no
fast-math); this module only builds it, loads it with ctypes and marshals numpy arrays.
Page names and the reading of each step are documented in ``lmoe_oracle.h``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lmoe_oracle.c")
_HDR = os.path.join(_HERE, "lmoe_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
# A library built from a modified copy of lmoe_oracle.c, loaded in place of liboracle.so: the
# mutation tests plant one mistake in such a copy and check that a pin fails.
LIB_ENV = "LMOE_ORACLE_LIB"
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle source `src` (liboracle.so from lmoe_oracle.c by default) with gcc (no
    fast-math, no FMA contraction); lmoe_oracle.h is taken from beside `src`."""
    hdr = os.path.join(os.path.dirname(os.path.abspath(src)), "lmoe_oracle.h")
    stale = (not os.path.exists(out)) or any(
        os.path.getmtime(p) > os.path.getmtime(out) for p in (src, hdr))
    if force or stale:
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-Wall", "-o", out, src, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
    return out


class _Layer(C.Structure):
    _fields_ = [
        ("d", C.c_int), ("l", C.c_int), ("E", C.c_int), ("k", C.c_int), ("ffn", C.c_int),
        ("w_down", C.c_void_p), ("w_up", C.c_void_p), ("w_router", C.c_void_p),
        ("b_router", C.c_void_p),
        ("w1_codes", C.c_void_p), ("w1_sf", C.c_void_p), ("w1_sdec", C.c_void_p),
        ("w2_codes", C.c_void_p), ("w2_sf", C.c_void_p), ("w2_sdec", C.c_void_p),
        ("w1", C.c_void_p), ("w2", C.c_void_p),
        ("amax_z", C.c_float), ("amax_h", C.c_float),
        ("shared_ffn", C.c_int),
        ("ws1_codes", C.c_void_p), ("ws1_sdec", C.c_float),
        ("ws2_codes", C.c_void_p), ("ws2_sdec", C.c_float),
        ("ws1", C.c_void_p), ("ws2", C.c_void_p),
        ("amax_xs", C.c_float), ("amax_hs", C.c_float),
    ]


class _Out(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "z", "zq_codes", "zq_sf", "logits", "idx", "w", "counts", "h", "hq_codes", "hq_sf",
        "c64", "c", "y64", "y", "xs_q", "hs", "hs_q", "s")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(os.environ.get(LIB_ENV) or build())
            L.oracle_e2m1_value.restype = C.c_double
            L.oracle_e2m1_value.argtypes = [C.c_uint8]
            L.oracle_e4m3_value.restype = C.c_double
            L.oracle_e4m3_value.argtypes = [C.c_uint8]
            L.oracle_f32_to_e2m1.restype = C.c_uint8
            L.oracle_f32_to_e2m1.argtypes = [C.c_float]
            L.oracle_f32_to_e4m3.restype = C.c_uint8
            L.oracle_f32_to_e4m3.argtypes = [C.c_float]
            L.oracle_round_bf16.restype = C.c_double
            L.oracle_round_bf16.argtypes = [C.c_double]
            for n in ("oracle_f32_to_e2m1_array", "oracle_f32_to_e4m3_array"):
                getattr(L, n).restype = None
                getattr(L, n).argtypes = [C.c_void_p, C.c_int64, C.c_void_p, C.c_int]
            L.oracle_quantize_nvfp4.restype = None
            L.oracle_quantize_nvfp4.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_float,
                                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_int]
            L.oracle_quantize_nvfp4_2d.restype = None
            L.oracle_quantize_nvfp4_2d.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_float,
                                                   C.c_void_p, C.c_void_p, C.c_void_p, C.c_int]
            L.oracle_nvfp4_dense_dot.restype = C.c_double
            L.oracle_nvfp4_dense_dot.argtypes = [C.c_void_p] * 3 + [C.c_int64]
            L.oracle_nvfp4_dot.restype = C.c_double
            L.oracle_nvfp4_dot.argtypes = [C.c_void_p] * 4 + [C.c_int64]
            L.oracle_quantize_fp8.restype = None
            L.oracle_quantize_fp8.argtypes = [C.c_void_p, C.c_int64, C.c_float, C.c_void_p,
                                              C.c_void_p, C.c_int]
            L.oracle_fp8_dot.restype = C.c_double
            L.oracle_fp8_dot.argtypes = [C.c_void_p, C.c_void_p, C.c_int64]
            L.oracle_shared_forward.restype = C.c_int
            L.oracle_shared_forward.argtypes = [C.POINTER(_Layer), C.c_void_p, C.c_int64, C.c_int,
                                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                                C.c_int]
            L.oracle_calibrate_shared.restype = C.c_int
            L.oracle_calibrate_shared.argtypes = [C.POINTER(_Layer), C.c_void_p, C.c_int64,
                                                  C.POINTER(C.c_float), C.POINTER(C.c_float),
                                                  C.c_int]
            L.oracle_router.restype = None
            L.oracle_router.argtypes = [C.c_void_p, C.c_int64, C.c_int, C.c_void_p, C.c_void_p,
                                        C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.c_int]
            L.oracle_layer_forward.restype = C.c_int
            L.oracle_layer_forward.argtypes = [C.POINTER(_Layer), C.c_void_p, C.c_int64, C.c_int,
                                               C.POINTER(_Out), C.c_int]
            L.oracle_layer_forward_zq.restype = C.c_int
            L.oracle_layer_forward_zq.argtypes = [C.POINTER(_Layer), C.c_void_p, C.c_void_p,
                                                  C.c_void_p, C.c_int64, C.POINTER(_Out), C.c_int]
            L.oracle_calibrate.restype = C.c_int
            L.oracle_calibrate.argtypes = [C.POINTER(_Layer), C.c_void_p, C.c_int64,
                                           C.POINTER(C.c_float), C.POINTER(C.c_float), C.c_int]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# --------------------------------------------------------------------------------------
# element conversions
# --------------------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(code)


def f32_to_e2m1(v) -> np.ndarray:
    v = _f32(np.atleast_1d(v))
    out = np.empty(v.shape, np.uint8)
    lib().oracle_f32_to_e2m1_array(_p(v), v.size, _p(out), 0)
    return out


def f32_to_e4m3(v) -> np.ndarray:
    v = _f32(np.atleast_1d(v))
    out = np.empty(v.shape, np.uint8)
    lib().oracle_f32_to_e4m3_array(_p(v), v.size, _p(out), 0)
    return out


def round_bf16(v: float) -> float:
    return lib().oracle_round_bf16(float(v))


# --------------------------------------------------------------------------------------
# NVFP4
# --------------------------------------------------------------------------------------
def quantize_nvfp4(x, amax: float = -1.0, nthreads: int = 0):
    """x: [R][K] -> (codes uint8 [R][K/2], sf uint8 [R][K/16], s_dec float)."""
    x = _f32(x)
    R, K = x.shape
    assert K % 16 == 0
    codes = np.empty((R, K // 2), np.uint8)
    sf = np.empty((R, K // 16), np.uint8)
    sdec = np.zeros(1, np.float32)
    lib().oracle_quantize_nvfp4(_p(x), R, K, float(amax), _p(codes), _p(sf), _p(sdec), nthreads)
    return codes, sf, float(sdec[0])


def quantize_nvfp4_2d(x, amax: float = -1.0, nthreads: int = 0):
    """x: [R][K] (R % 16 == 0) -> (codes [R][K/2], sf [R][K/16], s_dec): 16 x 16 weight blocks."""
    x = _f32(x)
    R, K = x.shape
    assert K % 16 == 0 and R % 16 == 0
    codes = np.empty((R, K // 2), np.uint8)
    sf = np.empty((R, K // 16), np.uint8)
    sdec = np.zeros(1, np.float32)
    lib().oracle_quantize_nvfp4_2d(_p(x), R, K, float(amax), _p(codes), _p(sf), _p(sdec), nthreads)
    return codes, sf, float(sdec[0])


def nvfp4_dot(qa, sfa, qb, sfb) -> float:
    qa, sfa, qb, sfb = (np.ascontiguousarray(a, np.uint8) for a in (qa, sfa, qb, sfb))
    return lib().oracle_nvfp4_dot(_p(qa), _p(sfa), _p(qb), _p(sfb), qa.size * 2)


# --------------------------------------------------------------------------------------
# FP8 E4M3, one per-tensor scale
# --------------------------------------------------------------------------------------
def quantize_fp8(x, amax: float = -1.0, nthreads: int = 0):
    """x: any shape -> (codes uint8 of that shape, s_dec float)."""
    x = _f32(x)
    codes = np.empty(x.shape, np.uint8)
    sdec = np.zeros(1, np.float32)
    lib().oracle_quantize_fp8(_p(x), x.size, float(amax), _p(codes), _p(sdec), nthreads)
    return codes, float(sdec[0])


def fp8_dot(a, b) -> float:
    a, b = (np.ascontiguousarray(v, np.uint8) for v in (a, b))
    assert a.size == b.size
    return lib().oracle_fp8_dot(_p(a), _p(b), a.size)


# --------------------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------------------
def router(x, w_router, b_router, k: int, nthreads: int = 0):
    """Returns (logits [T][E] f32, idx [T][k] i32, w [T][k] f32, counts [E] i32)."""
    x = _f32(x)
    Wr = _f32(w_router)
    T, d = x.shape
    E = Wr.shape[0]
    b = None if b_router is None else _f32(b_router)
    logits = np.empty((T, E), np.float32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    counts = np.empty(E, np.int32)
    lib().oracle_router(_p(x), T, d, _p(Wr), _p(b), E, k, _p(logits), _p(idx), _p(w),
                        _p(counts), nthreads)
    return logits, idx, w, counts


# --------------------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------------------
class OracleLayer:
    """The oracle's view of one layer.

    Masters are float32 arrays holding bf16 values (w_down [l][d], w_up [d][l],
    w_router [E][d] fp32, b_router [E] or None).  Expert masters are obtained from
    ``expert_fn(e) -> (w1 [ffn][l], w2 [l][ffn])`` on demand, so that at full size only
    the experts a token batch touches are ever quantized.
    """

    def __init__(self, d, l, E, k, ffn, w_down, w_up, w_router, b_router, expert_fn,
                 amax_z=0.0, amax_h=0.0, nthreads=0, shared=None, amax_xs=0.0, amax_hs=0.0,
                 weight_blocks_2d=False):
        self.d, self.l, self.E, self.k, self.ffn = d, l, E, k, ffn
        self.w_down = _f32(w_down)
        self.w_up = _f32(w_up)
        self.w_router = _f32(w_router)
        self.b_router = None if b_router is None else _f32(b_router)
        self.expert_fn = expert_fn
        self.amax_z, self.amax_h = float(amax_z), float(amax_h)
        self.nthreads = nthreads
        # optional shared expert: (ws1 [shared_ffn][d], ws2 [d][shared_ffn]) bf16 values
        self.shared = None if shared is None else (_f32(shared[0]), _f32(shared[1]))
        self.shared_ffn = 0 if shared is None else self.shared[0].shape[0]
        self.amax_xs, self.amax_hs = float(amax_xs), float(amax_hs)
        self.weight_blocks_2d = bool(weight_blocks_2d)   # 16 x 16 expert weight blocks
        self._sq = None    # (ws1 codes, ws1 s_dec, ws2 codes, ws2 s_dec)
        self._q = {}       # e -> (c1, s1, d1, c2, s2, d2)
        self._m = {}       # e -> (w1, w2) float32 masters
        self._arrays = {}

    # -- experts ---------------------------------------------------------------------
    def master(self, e):
        if e not in self._m:
            w1, w2 = self.expert_fn(e)
            self._m[e] = (_f32(w1), _f32(w2))
        return self._m[e]

    def quantized(self, e):
        """Oracle-quantized expert e: (w1 codes, w1 sf, w1 s_dec, w2 codes, w2 sf, w2 s_dec)."""
        if e not in self._q:
            w1, w2 = self.master(e)
            qf = quantize_nvfp4_2d if self.weight_blocks_2d else quantize_nvfp4
            c1, s1, d1 = qf(w1, -1.0, self.nthreads)
            c2, s2, d2 = qf(w2, -1.0, self.nthreads)
            self._q[e] = (c1, s1, d1, c2, s2, d2)
        return self._q[e]

    def quantized_shared(self):
        """Oracle-quantized shared expert: (ws1 codes, ws1 s_dec, ws2 codes, ws2 s_dec)."""
        if self._sq is None and self.shared is not None:
            c1, d1 = quantize_fp8(self.shared[0], -1.0, self.nthreads)
            c2, d2 = quantize_fp8(self.shared[1], -1.0, self.nthreads)
            self._sq = (c1, d1, c2, d2)
        return self._sq

    def route(self, x):
        return router(x, self.w_router, self.b_router, self.k, self.nthreads)

    def _struct(self, experts, quant):
        E = self.E
        P = C.c_void_p * E
        c1, s1, c2, s2, m1, m2 = P(), P(), P(), P(), P(), P()
        d1 = np.ones(E, np.float32)
        d2 = np.ones(E, np.float32)
        keep = []
        for e in experts:
            if quant:
                q = self.quantized(e)
                c1[e], s1[e], c2[e], s2[e] = (_p(q[0]), _p(q[1]), _p(q[3]), _p(q[4]))
                d1[e], d2[e] = q[2], q[5]
                keep.append(q)
            else:
                w1, w2 = self.master(e)
                m1[e], m2[e] = _p(w1), _p(w2)
                keep.append((w1, w2))
        sq = self.quantized_shared() if (quant and self.shared is not None) else None
        sm = self.shared if (not quant and self.shared is not None) else None
        st = _Layer(self.d, self.l, self.E, self.k, self.ffn,
                    _p(self.w_down), _p(self.w_up), _p(self.w_router), _p(self.b_router),
                    C.cast(c1, C.c_void_p), C.cast(s1, C.c_void_p), _p(d1),
                    C.cast(c2, C.c_void_p), C.cast(s2, C.c_void_p), _p(d2),
                    C.cast(m1, C.c_void_p), C.cast(m2, C.c_void_p),
                    self.amax_z, self.amax_h, self.shared_ffn,
                    _p(sq[0]) if sq else None, sq[1] if sq else 1.0,
                    _p(sq[2]) if sq else None, sq[3] if sq else 1.0,
                    _p(sm[0]) if sm else None, _p(sm[1]) if sm else None,
                    self.amax_xs, self.amax_hs)
        keep += [sq, sm]
        keep += [c1, s1, c2, s2, m1, m2, d1, d2]
        return st, keep

    def forward(self, x, quant=True, want=("y",), zq=None):
        """Run the layer on the token rows x [T][d]; returns a dict of requested outputs.
        quant: True (NVFP4 weights and activations), "w4a16" (NVFP4 weights, bf16 activations)
        or False (fp64 masters, no quantization).
        zq: optional (codes [T][l/2], scales [T][l/16]) uint8: the NVFP4 layer's steps after the
        quantization of z applied to this zq instead of the quantization of the oracle's own z
        (a z from another fp32 accumulation order may sit one bf16 ulp away and quantize to
        a neighbouring code; oracle_layer_forward_zq).

        Available: z, zq_codes, zq_sf, logits, idx, w, counts, h, hq_codes, hq_sf, c64, c,
        y64, y, and with a shared expert xs_q, hs, hs_q, s.  idx / w / counts are always
        returned."""
        x = _f32(x)
        T = x.shape[0]
        d, l, E, k, F = self.d, self.l, self.E, self.k, self.ffn
        _, idx, _, _ = self.route(x)
        experts = sorted(set(int(e) for e in np.unique(idx)))
        shapes = {
            "z": ((T, l), np.float32), "zq_codes": ((T, l // 2), np.uint8),
            "zq_sf": ((T, l // 16), np.uint8), "logits": ((T, E), np.float32),
            "idx": ((T, k), np.int32), "w": ((T, k), np.float32), "counts": ((E,), np.int32),
            "h": ((T, k, F), np.float32), "hq_codes": ((T, k, F // 2), np.uint8),
            "hq_sf": ((T, k, F // 16), np.uint8), "c64": ((T, l), np.float64),
            "c": ((T, l), np.float32), "y64": ((T, d), np.float64), "y": ((T, d), np.float32),
            "xs_q": ((T, d), np.uint8), "hs": ((T, max(self.shared_ffn, 1)), np.float32),
            "hs_q": ((T, max(self.shared_ffn, 1)), np.uint8), "s": ((T, d), np.float32),
        }
        names = set(want) | {"idx", "w", "counts"}
        res = {n: np.zeros(*shapes[n]) for n in names}
        out = _Out(**{n: _p(res[n]) for n in names})
        mode = 2 if quant == "w4a16" else (1 if quant else 0)
        st, keep = self._struct(experts, mode != 0)
        if zq is not None:
            assert mode == 1
            zc = np.ascontiguousarray(zq[0], dtype=np.uint8).reshape(T, l // 2)
            zs = np.ascontiguousarray(zq[1], dtype=np.uint8).reshape(T, l // 16)
            rc = lib().oracle_layer_forward_zq(C.byref(st), _p(x), _p(zc), _p(zs), T, C.byref(out),
                                               self.nthreads)
        else:
            rc = lib().oracle_layer_forward(C.byref(st), _p(x), T, mode, C.byref(out), self.nthreads)
        if rc != 0:
            raise RuntimeError("oracle_layer_forward: missing expert weights")
        del keep
        return res

    def shared_forward(self, x, quant=True):
        """The shared expert alone on x [T][d]: dict xs_q, hs, hs_q, s (codes only if quant)."""
        assert self.shared is not None
        x = _f32(x)
        T, F = x.shape[0], self.shared_ffn
        res = {"xs_q": np.zeros((T, self.d), np.uint8), "hs": np.zeros((T, F), np.float32),
               "hs_q": np.zeros((T, F), np.uint8), "s": np.zeros((T, self.d), np.float32)}
        st, keep = self._struct([], quant)
        rc = lib().oracle_shared_forward(C.byref(st), _p(x), T, 1 if quant else 0,
                                         _p(res["xs_q"]), _p(res["hs"]), _p(res["hs_q"]),
                                         _p(res["s"]), self.nthreads)
        if rc != 0:
            raise RuntimeError("oracle_shared_forward: no shared expert weights")
        del keep
        return res

    def calibrate_shared(self, x_cal):
        """Static amax of the shared expert's x and h; stores and returns them."""
        x = _f32(x_cal)
        st, keep = self._struct([], True)
        ax, ah = C.c_float(0), C.c_float(0)
        rc = lib().oracle_calibrate_shared(C.byref(st), _p(x), x.shape[0], C.byref(ax),
                                           C.byref(ah), self.nthreads)
        if rc != 0:
            raise RuntimeError("oracle_calibrate_shared: no shared expert weights")
        del keep
        self.amax_xs, self.amax_hs = float(ax.value), float(ah.value)
        return self.amax_xs, self.amax_hs

    def calibrate(self, x_cal):
        """Static activation amax (z, h) from a calibration batch; stores and returns them."""
        x = _f32(x_cal)
        _, idx, _, _ = self.route(x)
        experts = sorted(set(int(e) for e in np.unique(idx)))
        st, keep = self._struct(experts, True)
        az, ah = C.c_float(0), C.c_float(0)
        rc = lib().oracle_calibrate(C.byref(st), _p(x), x.shape[0], C.byref(az), C.byref(ah),
                                    self.nthreads)
        if rc != 0:
            raise RuntimeError("oracle_calibrate: missing expert weights")
        del keep
        self.amax_z, self.amax_h = float(az.value), float(ah.value)
        return self.amax_z, self.amax_h
