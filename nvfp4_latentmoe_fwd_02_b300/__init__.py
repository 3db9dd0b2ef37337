"""Python binding of liblmoe.so -- the LatentMoE expert layer forward on one B300.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``csrc/``.  Function names mirror the C ABI in ``include/lmoe.h``.  Tensors are torch
tensors (device memory and streams only); pointers and the current CUDA stream are passed
through unchanged.  There is no CPU fallback: if the library cannot be loaded, importing
the binding's functions raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblmoe.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "lmoe.h")

LMOE_OK, LMOE_EINVAL, LMOE_ENOMEM, LMOE_ECUDA, LMOE_EUNSUPPORTED, LMOE_ETIMEOUT, LMOE_EDEVICE = range(7)
LMOE_BF16, LMOE_FP32 = 0, 1
STAGES = {
    "idx": 0, "w": 1, "counts": 2, "zq_codes": 3, "zq_sf": 4, "c": 5, "z": 6, "rows": 7, "h": 8,
    "hq_codes": 9, "hq_sf": 10, "nrows": 11, "xs_q": 12, "hs": 13, "hs_q": 14, "s": 15,
    "router": 16,
}


class LmoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lmoe_status_string(status)} (status {status})")


class _Weights(C.Structure):
    _fields_ = [("w_down", C.c_void_p), ("w_up", C.c_void_p), ("w_router", C.c_void_p),
                ("b_router", C.c_void_p), ("w1", C.c_void_p), ("w2", C.c_void_p),
                ("amax_z", C.c_float), ("amax_h", C.c_float),
                ("ws1", C.c_void_p), ("ws2", C.c_void_p), ("shared_ffn", C.c_int),
                ("amax_xs", C.c_float), ("amax_hs", C.c_float), ("weight_blocks_2d", C.c_int),
                ("expert_w4a16", C.c_int)]


_lib = None


def lib() -> C.CDLL:
    """Load liblmoe.so (building it first if it is missing or stale and nvcc exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        from . import build as _build
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"liblmoe.so not found at {LIB_PATH}; run the build first")
    L = C.CDLL(LIB_PATH)
    vp, i64, sz = C.c_void_p, C.c_int64, C.c_size_t
    sig = {
        "lmoe_status_string": (C.c_char_p, [C.c_int]),
        "lmoe_create": (C.c_int, [C.c_int] * 5 + [C.POINTER(_Weights), vp, C.POINTER(vp)]),
        "lmoe_quantize_nvfp4": (C.c_int, [vp, C.c_int, i64, i64, C.c_float, vp, vp, vp, vp]),
        "lmoe_quantize_nvfp4_2d": (C.c_int, [vp, C.c_int, i64, i64, C.c_float, vp, vp, vp, vp]),
        "lmoe_quantize_fp8": (C.c_int, [vp, C.c_int, i64, C.c_float, vp, vp, vp]),
        "lmoe_get_shared_fp8": (C.c_int, [vp, C.c_int, vp, C.POINTER(C.c_float), vp]),
        "lmoe_route": (C.c_int, [vp, vp, i64, vp, vp, vp, vp]),
        "lmoe_route_static": (C.c_int, [vp, vp, i64, vp, vp, vp, vp]),
        "lmoe_workspace_size": (sz, [vp, i64]),
        "lmoe_forward": (C.c_int, [vp, vp, i64, vp, vp, sz, vp]),
        "lmoe_host_workspace_size": (sz, [vp, i64]),
        "lmoe_forward_host": (C.c_int, [vp, vp, i64, vp, vp, sz, vp]),
        "lmoe_workspace_range": (C.c_int, [vp, i64, C.c_int, C.POINTER(sz), C.POINTER(sz)]),
        "lmoe_set_debug": (C.c_int, [vp, C.c_int]),
        "lmoe_set_wait_limit": (C.c_int, [vp, C.c_longlong]),
        "lmoe_get_expert_nvfp4": (C.c_int, [vp, C.c_int, C.c_int, vp, vp, C.POINTER(C.c_float), vp]),
        "lmoe_check": (C.c_int, [vp, vp]),
        "lmoe_forward_kernel_count": (C.c_int, [vp, i64]),
        "lmoe_set_profile": (C.c_int, [vp, C.c_int]),
        "lmoe_profile_read": (C.c_int, [vp, C.POINTER(C.c_char_p), C.POINTER(C.c_float), C.c_int]),
        "lmoe_destroy": (None, [vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def header_functions() -> list[str]:
    """Names of every function include/lmoe.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lmoe_[a-z0-9_]+)\s*\(", src)))


def _check(st: int, where: str):
    if st != LMOE_OK:
        raise LmoeError(st, where)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def lmoe_status_string(status: int) -> str:
    return lib().lmoe_status_string(status).decode()


def lmoe_quantize_nvfp4(src: torch.Tensor, amax: float = -1.0, codes=None, sf=None,
                        tensor_scale=None, stream=None):
    """NVFP4-quantize a [rows][K] bf16/fp32 device tensor -> (codes, sf, tensor_scale)."""
    assert src.is_cuda and src.dim() == 2 and src.is_contiguous()
    rows, K = src.shape
    dt = {torch.bfloat16: LMOE_BF16, torch.float32: LMOE_FP32}[src.dtype]
    dev = src.device
    codes = codes if codes is not None else torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    sf = sf if sf is not None else torch.empty((rows, K // 16), dtype=torch.uint8, device=dev)
    tensor_scale = tensor_scale if tensor_scale is not None else torch.empty(1, dtype=torch.float32, device=dev)
    _check(lib().lmoe_quantize_nvfp4(_ptr(src), dt, rows, K, float(amax), _ptr(codes), _ptr(sf),
                                     _ptr(tensor_scale), _stream(stream)), "lmoe_quantize_nvfp4")
    return codes, sf, tensor_scale


def lmoe_quantize_nvfp4_2d(src: torch.Tensor, amax: float = -1.0, codes=None, sf=None,
                           tensor_scale=None, stream=None):
    """NVFP4 with 16 x 16 blocks of a [rows][K] bf16/fp32 device tensor (rows % 16 == 0)."""
    assert src.is_cuda and src.dim() == 2 and src.is_contiguous()
    rows, K = src.shape
    dt = {torch.bfloat16: LMOE_BF16, torch.float32: LMOE_FP32}[src.dtype]
    dev = src.device
    codes = codes if codes is not None else torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    sf = sf if sf is not None else torch.empty((rows, K // 16), dtype=torch.uint8, device=dev)
    tensor_scale = tensor_scale if tensor_scale is not None else torch.empty(1, dtype=torch.float32, device=dev)
    _check(lib().lmoe_quantize_nvfp4_2d(_ptr(src), dt, rows, K, float(amax), _ptr(codes), _ptr(sf),
                                        _ptr(tensor_scale), _stream(stream)), "lmoe_quantize_nvfp4_2d")
    return codes, sf, tensor_scale


def lmoe_quantize_fp8(src: torch.Tensor, amax: float = -1.0, codes=None, tensor_scale=None,
                      stream=None):
    """FP8 E4M3 per-tensor quantization of a bf16/fp32 device tensor -> (codes, tensor_scale)."""
    assert src.is_cuda and src.is_contiguous()
    dt = {torch.bfloat16: LMOE_BF16, torch.float32: LMOE_FP32}[src.dtype]
    codes = codes if codes is not None else torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    tensor_scale = tensor_scale if tensor_scale is not None else torch.empty(1, dtype=torch.float32, device=src.device)
    _check(lib().lmoe_quantize_fp8(_ptr(src), dt, src.numel(), float(amax), _ptr(codes),
                                   _ptr(tensor_scale), _stream(stream)), "lmoe_quantize_fp8")
    return codes, tensor_scale


def lmoe_create(d, l, E, k, ffn, w_down, w_up, w_router, b_router, w1, w2, amax_z, amax_h,
                stream=None, ws1=None, ws2=None, amax_xs=0.0, amax_hs=0.0,
                weight_blocks_2d=False, w4a16=False) -> int:
    """Create a context from device tensors: w_down bf16 [l][d], w_up bf16 [d][l], w_router fp32
    [E][d], b_router fp32 [E] or None, w1 bf16 [E][ffn][l], w2 bf16 [E][l][ffn]; optional
    shared expert ws1 bf16 [shared_ffn][d], ws2 bf16 [d][shared_ffn]."""
    for t in (w_down, w_up, w_router, w1, w2) + ((ws1, ws2) if ws1 is not None else ()):
        assert t.is_cuda and t.is_contiguous()
    ws = _Weights(_ptr(w_down), _ptr(w_up), _ptr(w_router), _ptr(b_router), _ptr(w1), _ptr(w2),
                  float(amax_z), float(amax_h), _ptr(ws1), _ptr(ws2),
                  0 if ws1 is None else ws1.shape[0], float(amax_xs), float(amax_hs),
                  1 if weight_blocks_2d else 0, 1 if w4a16 else 0)
    out = C.c_void_p()
    _check(lib().lmoe_create(d, l, E, k, ffn, C.byref(ws), _stream(stream), C.byref(out)), "lmoe_create")
    return out.value


def lmoe_destroy(ctx: int):
    lib().lmoe_destroy(ctx)


def lmoe_route(ctx, x, T, idx, w, counts=None, stream=None):
    _check(lib().lmoe_route(ctx, _ptr(x), T, _ptr(idx), _ptr(w), _ptr(counts), _stream(stream)),
           "lmoe_route")


def lmoe_route_static(ctx, x, T, idx, w, counts=None, stream=None):
    """lmoe_route without any device allocation (fixed scratch inside the library; see the
    header for the size limit and the first-call and concurrency rules)."""
    _check(lib().lmoe_route_static(ctx, _ptr(x), T, _ptr(idx), _ptr(w), _ptr(counts),
                                   _stream(stream)), "lmoe_route_static")


def lmoe_workspace_size(ctx, T) -> int:
    return lib().lmoe_workspace_size(ctx, T)


def lmoe_host_workspace_size(ctx, T) -> int:
    return lib().lmoe_host_workspace_size(ctx, T)


def lmoe_forward(ctx, x, T, y, ws, ws_bytes, stream=None):
    _check(lib().lmoe_forward(ctx, _ptr(x), T, _ptr(y), _ptr(ws), ws_bytes, _stream(stream)),
           "lmoe_forward")


def lmoe_forward_host(ctx, x_host, T, y_host, ws, ws_bytes, stream=None):
    """x_host / y_host: CPU tensors (pinned for overlap)."""
    _check(lib().lmoe_forward_host(ctx, _ptr(x_host), T, _ptr(y_host), _ptr(ws), ws_bytes,
                                   _stream(stream)), "lmoe_forward_host")


def lmoe_workspace_range(ctx, T, stage) -> tuple[int, int]:
    off, nb = C.c_size_t(), C.c_size_t()
    st = STAGES[stage] if isinstance(stage, str) else int(stage)
    _check(lib().lmoe_workspace_range(ctx, T, st, C.byref(off), C.byref(nb)), "lmoe_workspace_range")
    return off.value, nb.value


def lmoe_set_debug(ctx, on: bool):
    _check(lib().lmoe_set_debug(ctx, 1 if on else 0), "lmoe_set_debug")


def lmoe_set_wait_limit(ctx, cycles: int):
    _check(lib().lmoe_set_wait_limit(ctx, int(cycles)), "lmoe_set_wait_limit")


def lmoe_get_expert_nvfp4(ctx, which, e, codes, sf, stream=None) -> float:
    sd = C.c_float()
    _check(lib().lmoe_get_expert_nvfp4(ctx, which, e, _ptr(codes), _ptr(sf), C.byref(sd),
                                       _stream(stream)), "lmoe_get_expert_nvfp4")
    return sd.value


def lmoe_get_shared_fp8(ctx, which, codes, stream=None) -> float:
    sd = C.c_float()
    _check(lib().lmoe_get_shared_fp8(ctx, which, _ptr(codes), C.byref(sd), _stream(stream)),
           "lmoe_get_shared_fp8")
    return sd.value


def lmoe_forward_kernel_count(ctx, T) -> int:
    return lib().lmoe_forward_kernel_count(ctx, T)


def lmoe_set_profile(ctx, on: bool):
    _check(lib().lmoe_set_profile(ctx, 1 if on else 0), "lmoe_set_profile")


def lmoe_profile_read(ctx, max_kernels: int = 32) -> list[tuple[str, float]]:
    """[(kernel name, ms)] of the last forward run with profiling on."""
    names = (C.c_char_p * max_kernels)()
    ms = (C.c_float * max_kernels)()
    n = lib().lmoe_profile_read(ctx, names, ms, max_kernels)
    if n < 0:
        raise LmoeError(LMOE_EINVAL, "lmoe_profile_read")
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


def lmoe_check(ctx, stream=None):
    _check(lib().lmoe_check(ctx, _stream(stream)), "lmoe_check")


class LatentMoE:
    """Owns one context and a workspace; forward(x) -> y.  Marshalling only."""

    def __init__(self, d, l, E, k, ffn, w_down, w_up, w_router, b_router, w1, w2, amax_z, amax_h,
                 debug=False, stream=None, ws1=None, ws2=None, amax_xs=0.0, amax_hs=0.0,
                 weight_blocks_2d=False, w4a16=False):
        self.d, self.l, self.E, self.k, self.ffn = d, l, E, k, ffn
        self.shared_ffn = 0 if ws1 is None else ws1.shape[0]
        self.ctx = lmoe_create(d, l, E, k, ffn, w_down, w_up, w_router, b_router, w1, w2,
                               amax_z, amax_h, stream, ws1, ws2, amax_xs, amax_hs, weight_blocks_2d,
                               w4a16)
        if debug:
            lmoe_set_debug(self.ctx, True)
        self.ws = None
        self.ws_T = -1

    def workspace(self, T):
        need = lmoe_workspace_size(self.ctx, T)
        if self.ws is None or self.ws.numel() < need:
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        self.ws_T = T
        return self.ws

    def forward(self, x, y=None, stream=None):
        T = x.shape[0]
        assert x.dtype == torch.bfloat16 and x.shape[1] == self.d and x.is_contiguous()
        y = y if y is not None else torch.empty_like(x)
        ws = self.workspace(T)
        lmoe_forward(self.ctx, x, T, y, ws, ws.numel(), stream)
        return y

    def stage(self, name, T, dtype=torch.uint8):
        """View of an intermediate of the last forward (see lmoe_workspace_range)."""
        off, nb = lmoe_workspace_range(self.ctx, T, name)
        return self.ws[off:off + nb].view(dtype)

    def check(self, stream=None):
        lmoe_check(self.ctx, stream)

    def close(self):
        if self.ctx:
            lmoe_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
