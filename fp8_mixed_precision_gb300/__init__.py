"""Python binding of the GB300 FP8 linear-layer library (libfp8lin.so).

Argument marshalling only: every function below allocates its outputs with
torch on the current CUDA device, passes raw device pointers and the current
stream to the C ABI declared in include/fp8lin.h, and raises FP8Error on a
non-OK status.  Names follow the C ABI.  There is no fallback: if the
compiled library is missing, importing works but the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import torch

__all__ = [
    "FP8Error", "lib", "RECIPE", "ROLE", "FORMAT", "SCALING",
    "fp8_quantize", "fp8_scale_shape", "fp8_gemm", "fp8_linear_fwd", "fp8_linear_bwd",
    "fp8_gelu_fwd", "fp8_gelu_bwd", "fp8_grad_accumulate", "fp8_get_device_status",
    "fp8_launch_count", "fp8_profile_begin", "fp8_profile_end", "WeightCache", "LinearContext",
    "fp8_quantize_delayed", "fp8_debug_wait_timeout", "HostPipeline", "amax_partials_buffer",
    "fp8_amax_partials", "fp8_linear_fwd_after_amax", "fp8_linear_bwd_after_amax",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8lin.so")

RECIPE = {"tensorwise": 0, "block": 1, "delayed": 2}
ROLE = {"act": 0, "weight": 1, "grad": 2}
FORMAT = {"e4m3": 0, "e5m2": 1}
SCALING = {"tensor": 0, "1x128_128x128": 1, "1x128_1x128": 2}

_c_i64 = ctypes.c_int64
_c_p = ctypes.c_void_p
_c_sz = ctypes.c_size_t
_c_int = ctypes.c_int

_SIGS = {
    "fp8_status_string": (ctypes.c_char_p, [_c_int]),
    "fp8_launch_count": (ctypes.c_uint64, []),
    "fp8_quantize": (_c_int, [_c_p, _c_i64, _c_i64, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p,
                              _c_p, _c_p, _c_sz, _c_p]),
    "fp8_quantize_workspace_size": (_c_int, [_c_int, _c_i64, _c_i64, ctypes.POINTER(_c_sz)]),
    "fp8_scale_shape": (_c_int, [_c_int, _c_int, _c_i64, _c_i64, _c_int,
                                 ctypes.POINTER(_c_i64), ctypes.POINTER(_c_i64)]),
    "fp8_gemm": (_c_int, [_c_p, _c_int, _c_p, _c_p, _c_int, _c_p, _c_i64, _c_i64, _c_i64, _c_int,
                          _c_p, _c_p, _c_sz, _c_p]),
    "fp8_gemm_workspace_size": (_c_int, [_c_i64, _c_i64, _c_i64, _c_int, ctypes.POINTER(_c_sz)]),
    "fp8_weight_cache_create": (_c_int, [ctypes.POINTER(_c_p)]),
    "fp8_weight_cache_destroy": (None, [_c_p]),
    "fp8_weight_cache_register": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_int, _c_p, _c_p, _c_p,
                                           _c_p, _c_p, _c_p, _c_p, _c_sz,
                                           ctypes.POINTER(ctypes.c_int32)]),
    "fp8_weight_cache_begin_cycle": (_c_int, [_c_p]),
    "fp8_weight_cache_get": (_c_int, [_c_p, ctypes.c_int32, ctypes.c_uint64, _c_int, _c_p,
                                      ctypes.POINTER(_c_int)]),
    "fp8_linear_ctx_size": (_c_int, [_c_int, _c_i64, _c_i64, ctypes.POINTER(_c_sz)]),
    "fp8_linear_workspace_size": (_c_int, [_c_int, _c_i64, _c_i64, _c_i64, ctypes.POINTER(_c_sz)]),
    "fp8_linear_fwd": (_c_int, [_c_p, _c_i64, _c_i64, _c_p, ctypes.c_int32, _c_int, _c_p, _c_p,
                                _c_p, _c_sz, _c_p]),
    "fp8_linear_bwd": (_c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p, ctypes.c_int32, _c_int, _c_p,
                                _c_p, _c_p, _c_sz, _c_p]),
    "fp8_gelu_fwd": (_c_int, [_c_p, _c_p, _c_i64, _c_p]),
    "fp8_gelu_bwd": (_c_int, [_c_p, _c_p, _c_p, _c_i64, _c_p]),
    "fp8_grad_accumulate": (_c_int, [_c_p, _c_p, _c_i64, _c_p]),
    "fp8_get_device_status": (_c_int, [_c_p]),
    "fp8_profile_begin": (_c_int, []),
    "fp8_debug_wait_timeout": (_c_int, [ctypes.c_uint64, _c_p]),
    "fp8_quantize_delayed": (_c_int, [_c_p, _c_i64, _c_i64, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p,
                                      ctypes.c_int32, _c_i64, _c_p, _c_sz, _c_p]),
    "fp8_weight_cache_register_delayed": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p,
                                                   _c_p, _c_p, ctypes.c_int32, _c_p, _c_sz,
                                                   ctypes.POINTER(ctypes.c_int32)]),
    "fp8_gelu_quantize": (_c_int, [_c_p, _c_i64, _c_i64, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p,
                                   _c_p, _c_p]),
    "fp8_gelu_bwd_quantize": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_int, _c_p, _c_p, _c_p, _c_p,
                                       _c_p, _c_p, _c_p]),
    "fp8_linear_ctx_layout": (_c_int, [_c_int, _c_i64, _c_i64, _c_p, ctypes.POINTER(_c_p),
                                       ctypes.POINTER(_c_p), ctypes.POINTER(_c_p)]),
    "fp8_linear_fwd_quantized": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p, ctypes.c_int32, _c_int,
                                          _c_p, _c_p, _c_sz, _c_p]),
    "fp8_linear_bwd_quantized": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p,
                                          ctypes.c_int32, _c_int, _c_p, _c_p, _c_p, _c_sz, _c_p]),
}


class _HostIO(ctypes.Structure):
    _fields_ = [("X", _c_p), ("W", _c_p), ("dY", _c_p), ("Y", _c_p), ("dX", _c_p), ("dW", _c_p)]


class _DeviceIO(ctypes.Structure):
    _fields_ = [("X", _c_p), ("dY", _c_p), ("Y", _c_p), ("dX", _c_p), ("dW", _c_p),
                ("ctx", _c_p), ("ws", _c_p), ("ws_bytes", _c_sz)]


_SIGS.update({
    "fp8_amax_partials": (_c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_sz, _c_p]),
    "fp8_linear_fwd_after_amax": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p, ctypes.c_int32, _c_int,
                                           _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "fp8_linear_bwd_after_amax": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p, ctypes.c_int32,
                                           _c_int, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "fp8_host_pipeline_create": (_c_int, [_c_int, ctypes.POINTER(_c_p)]),
    "fp8_host_pipeline_destroy": (None, [_c_p]),
    "fp8_linear_step_host": (_c_int, [_c_p, _c_int, _c_i64, ctypes.POINTER(_HostIO),
                                      ctypes.POINTER(_DeviceIO), _c_p, ctypes.c_int32, _c_int,
                                      ctypes.c_uint64]),
    "fp8_host_pipeline_fork": (_c_int, [_c_p, _c_p]),
    "fp8_host_pipeline_join": (_c_int, [_c_p, _c_p]),
    "fp8_host_pipeline_sync": (_c_int, [_c_p]),
})


class _KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 64), ("launches", ctypes.c_uint64),
                ("total_ms", ctypes.c_double), ("bytes", ctypes.c_double),
                ("flops", ctypes.c_double), ("m", ctypes.c_int64), ("n", ctypes.c_int64),
                ("k", ctypes.c_int64)]

_lib = None


class FP8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().fp8_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: status {status} ({msg})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded C library (built in-tree by build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m fp8_mixed_precision_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        L.fp8_profile_end.restype = _c_int
        L.fp8_profile_end.argtypes = [ctypes.POINTER(_KernelStat), _c_int, ctypes.POINTER(_c_int)]
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise FP8Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_bf16_cuda(t, name):
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")


def fp8_launch_count() -> int:
    return int(lib().fp8_launch_count())


def fp8_scale_shape(recipe: str, role: str, rows: int, cols: int, colwise: bool):
    sr, sc = _c_i64(), _c_i64()
    _check(lib().fp8_scale_shape(RECIPE[recipe], ROLE[role], rows, cols, int(colwise),
                                 ctypes.byref(sr), ctypes.byref(sc)), "fp8_scale_shape")
    return (sr.value, sc.value)


def _quant_ws_bytes(recipe, rows, cols):
    b = _c_sz()
    _check(lib().fp8_quantize_workspace_size(RECIPE[recipe], rows, cols, ctypes.byref(b)),
           "fp8_quantize_workspace_size")
    return b.value


def _empty_bytes(n, device):
    return torch.empty(max(int(n), 16), dtype=torch.uint8, device=device)


def fp8_quantize(x: torch.Tensor, recipe: str, role: str, rowwise: bool = True,
                 colwise: bool = True, stream=None) -> dict:
    """Quantize a bf16 [R, C] tensor; returns dict(row, col, row_scale,
    row_scale_inv, col_scale, col_scale_inv) (absent layouts are None)."""
    _need_bf16_cuda(x, "x")
    R, C = x.shape
    dev = x.device
    out = dict(row=None, col=None, row_scale=None, row_scale_inv=None, col_scale=None,
               col_scale_inv=None)
    rs = fp8_scale_shape(recipe, role, R, C, False)
    cs = fp8_scale_shape(recipe, role, R, C, True)
    if rowwise or recipe == "tensorwise":
        out["row_scale"] = torch.empty(rs, dtype=torch.float32, device=dev)
        out["row_scale_inv"] = torch.empty(rs, dtype=torch.float32, device=dev)
    if colwise:
        out["col_scale"] = torch.empty(cs, dtype=torch.float32, device=dev)
        out["col_scale_inv"] = torch.empty(cs, dtype=torch.float32, device=dev)
    if rowwise:
        out["row"] = torch.empty((R, C), dtype=torch.uint8, device=dev)
    if colwise:
        out["col"] = torch.empty((C, R), dtype=torch.uint8, device=dev)
    wsb = _quant_ws_bytes(recipe, R, C)
    ws = _empty_bytes(wsb, dev)
    _check(lib().fp8_quantize(_ptr(x), R, C, RECIPE[recipe], ROLE[role], _ptr(out["row"]),
                              _ptr(out["col"]), _ptr(out["row_scale"]), _ptr(out["row_scale_inv"]),
                              _ptr(out["col_scale"]), _ptr(out["col_scale_inv"]), _ptr(ws),
                              ws.numel(), _stream(stream)), "fp8_quantize")
    return out


def fp8_quantize_delayed(x: torch.Tensor, role: str, history: torch.Tensor, step: int,
                         rowwise: bool = True, colwise: bool = True, stream=None) -> dict:
    """DelayedScaling quantize: scale from max(history), then history[step %
    len] = amax(x).  history: float32 CUDA tensor (updated in place)."""
    _need_bf16_cuda(x, "x")
    if history.dtype != torch.float32 or not history.is_cuda:
        raise ValueError("history must be a float32 CUDA tensor")
    R, C = x.shape
    dev = x.device
    out = dict(row=torch.empty((R, C), dtype=torch.uint8, device=dev) if rowwise else None,
               col=torch.empty((C, R), dtype=torch.uint8, device=dev) if colwise else None,
               scale=torch.empty(1, dtype=torch.float32, device=dev),
               scale_inv=torch.empty(1, dtype=torch.float32, device=dev))
    ws = _empty_bytes(_quant_ws_bytes("tensorwise", R, C), dev)
    _check(lib().fp8_quantize_delayed(_ptr(x), R, C, ROLE[role], _ptr(out["row"]), _ptr(out["col"]),
                                      _ptr(out["scale"]), _ptr(out["scale_inv"]), _ptr(history),
                                      history.numel(), int(step), _ptr(ws), ws.numel(),
                                      _stream(stream)), "fp8_quantize_delayed")
    return out


def fp8_gemm(a: torch.Tensor, a_fmt: str, a_scale_inv: torch.Tensor, b: torch.Tensor, b_fmt: str,
             b_scale_inv: torch.Tensor, scaling: str, out: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """C[M, N] bf16 = sum_k (a[m,k] sa)(b[n,k] sb); a [M, K], b [N, K] uint8."""
    M, K = a.shape
    N, K2 = b.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    dev = a.device
    C = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    wsb = _c_sz()
    _check(lib().fp8_gemm_workspace_size(M, N, K, SCALING[scaling], ctypes.byref(wsb)),
           "fp8_gemm_workspace_size")
    ws = _empty_bytes(wsb.value, dev)
    _check(lib().fp8_gemm(_ptr(a), FORMAT[a_fmt], _ptr(a_scale_inv), _ptr(b), FORMAT[b_fmt],
                          _ptr(b_scale_inv), M, N, K, SCALING[scaling], _ptr(C), _ptr(ws),
                          wsb.value, _stream(stream)), "fp8_gemm")
    return C


@dataclass
class _Entry:
    w: torch.Tensor
    recipe: str
    row: torch.Tensor
    col: torch.Tensor
    row_scale: torch.Tensor
    row_scale_inv: torch.Tensor
    col_scale: torch.Tensor
    col_scale_inv: torch.Tensor
    ws: torch.Tensor
    history: torch.Tensor | None = None


class WeightCache:
    """Owns an fp8_weight_cache and the device buffers of its FP8 weights."""

    def __init__(self):
        h = ctypes.c_void_p()
        _check(lib().fp8_weight_cache_create(ctypes.byref(h)), "fp8_weight_cache_create")
        self._h = h
        self.entries: list[_Entry] = []

    @property
    def handle(self):
        return self._h

    def register(self, w: torch.Tensor, recipe: str, history_len: int = 16) -> int:
        _need_bf16_cuda(w, "w")
        O, K = w.shape
        dev = w.device
        if recipe == "delayed":
            s = torch.empty(1, dtype=torch.float32, device=dev)
            si = torch.empty(1, dtype=torch.float32, device=dev)
            e = _Entry(w=w, recipe=recipe,
                       row=torch.empty((O, K), dtype=torch.uint8, device=dev),
                       col=torch.empty((K, O), dtype=torch.uint8, device=dev),
                       row_scale=s, row_scale_inv=si, col_scale=s, col_scale_inv=si,
                       ws=_empty_bytes(_quant_ws_bytes("tensorwise", O, K), dev),
                       history=torch.zeros(history_len, dtype=torch.float32, device=dev))
            out = ctypes.c_int32()
            _check(lib().fp8_weight_cache_register_delayed(
                self._h, _ptr(w), O, K, _ptr(e.row), _ptr(e.col), _ptr(s), _ptr(si),
                _ptr(e.history), history_len, _ptr(e.ws), e.ws.numel(), ctypes.byref(out)),
                "fp8_weight_cache_register_delayed")
            self.entries.append(e)
            return out.value
        rs = fp8_scale_shape(recipe, "weight", O, K, False)
        cs = fp8_scale_shape(recipe, "weight", O, K, True)
        e = _Entry(w=w, recipe=recipe,
                   row=torch.empty((O, K), dtype=torch.uint8, device=dev),
                   col=torch.empty((K, O), dtype=torch.uint8, device=dev),
                   row_scale=torch.empty(rs, dtype=torch.float32, device=dev),
                   row_scale_inv=torch.empty(rs, dtype=torch.float32, device=dev),
                   col_scale=torch.empty(cs, dtype=torch.float32, device=dev),
                   col_scale_inv=torch.empty(cs, dtype=torch.float32, device=dev),
                   ws=_empty_bytes(_quant_ws_bytes(recipe, O, K), dev))
        out = ctypes.c_int32()
        _check(lib().fp8_weight_cache_register(
            self._h, _ptr(w), O, K, RECIPE[recipe], _ptr(e.row), _ptr(e.col), _ptr(e.row_scale),
            _ptr(e.row_scale_inv), _ptr(e.col_scale), _ptr(e.col_scale_inv), _ptr(e.ws),
            e.ws.numel(), ctypes.byref(out)), "fp8_weight_cache_register")
        self.entries.append(e)
        return out.value

    def begin_cycle(self):
        _check(lib().fp8_weight_cache_begin_cycle(self._h), "fp8_weight_cache_begin_cycle")

    def get(self, h: int, version: int = 0, use_cache: bool = True, stream=None) -> bool:
        """Make weight h's FP8 copy current; True if it was re-quantized."""
        rq = ctypes.c_int()
        _check(lib().fp8_weight_cache_get(self._h, h, version, int(use_cache), _stream(stream),
                                          ctypes.byref(rq)), "fp8_weight_cache_get")
        return bool(rq.value)

    def __del__(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.fp8_weight_cache_destroy(self._h)
            self._h = None


@dataclass
class LinearContext:
    ctx: torch.Tensor
    N: int
    K: int
    extra: dict = field(default_factory=dict)


def _ctx_bytes(recipe, N, K):
    b = _c_sz()
    _check(lib().fp8_linear_ctx_size(RECIPE[recipe], N, K, ctypes.byref(b)), "fp8_linear_ctx_size")
    return b.value


def linear_workspace(recipe: str, N: int, K: int, O: int, device) -> torch.Tensor:
    b = _c_sz()
    _check(lib().fp8_linear_workspace_size(RECIPE[recipe], N, K, O, ctypes.byref(b)),
           "fp8_linear_workspace_size")
    return _empty_bytes(b.value, device)


def fp8_linear_fwd(x: torch.Tensor, cache: WeightCache, h: int, recipe: str,
                   ws: torch.Tensor | None = None, y: torch.Tensor | None = None,
                   ctx: LinearContext | None = None, stream=None):
    """Y = X W^T with FP8 operands; returns (Y, LinearContext)."""
    _need_bf16_cuda(x, "x")
    N, K = x.shape
    O = cache.entries[h].w.shape[0]
    dev = x.device
    if y is None:
        y = torch.empty((N, O), dtype=torch.bfloat16, device=dev)
    if ctx is None:
        ctx = LinearContext(_empty_bytes(_ctx_bytes(recipe, N, K), dev), N, K)
    if ws is None:
        ws = linear_workspace(recipe, N, K, O, dev)
    _check(lib().fp8_linear_fwd(_ptr(x), N, K, cache.handle, h, RECIPE[recipe], _ptr(y),
                                _ptr(ctx.ctx), _ptr(ws), ws.numel(), _stream(stream)),
           "fp8_linear_fwd")
    return y, ctx


def fp8_linear_bwd(dy: torch.Tensor, ctx: LinearContext, cache: WeightCache, h: int, recipe: str,
                   need_dx: bool = True, ws: torch.Tensor | None = None,
                   dx: torch.Tensor | None = None, dw: torch.Tensor | None = None, stream=None):
    """Returns (dX or None, dW) for Y = X W^T."""
    _need_bf16_cuda(dy, "dy")
    N, O = dy.shape
    K = ctx.K
    dev = dy.device
    if need_dx and dx is None:
        dx = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    if dw is None:
        dw = torch.empty((O, K), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = linear_workspace(recipe, N, K, O, dev)
    _check(lib().fp8_linear_bwd(_ptr(dy), N, O, _ptr(ctx.ctx), cache.handle, h, RECIPE[recipe],
                                _ptr(dx) if need_dx else None, _ptr(dw), _ptr(ws), ws.numel(),
                                _stream(stream)), "fp8_linear_bwd")
    return (dx if need_dx else None), dw


def fp8_gelu_fwd(h: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need_bf16_cuda(h, "h")
    a = out if out is not None else torch.empty_like(h)
    _check(lib().fp8_gelu_fwd(_ptr(h), _ptr(a), h.numel(), _stream(stream)), "fp8_gelu_fwd")
    return a


def fp8_gelu_bwd(da: torch.Tensor, h: torch.Tensor, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    _need_bf16_cuda(da, "da")
    _need_bf16_cuda(h, "h")
    dh = out if out is not None else torch.empty_like(h)
    _check(lib().fp8_gelu_bwd(_ptr(da), _ptr(h), _ptr(dh), h.numel(), _stream(stream)),
           "fp8_gelu_bwd")
    return dh


def fp8_grad_accumulate(acc: torch.Tensor, dw: torch.Tensor, stream=None) -> torch.Tensor:
    if acc.dtype != torch.float32 or not acc.is_cuda:
        raise ValueError("acc must be a float32 CUDA tensor")
    _need_bf16_cuda(dw, "dw")
    _check(lib().fp8_grad_accumulate(_ptr(acc), _ptr(dw), acc.numel(), _stream(stream)),
           "fp8_grad_accumulate")
    return acc


def fp8_get_device_status(stream=None) -> int:
    return int(lib().fp8_get_device_status(_stream(stream)))


def fp8_profile_begin():
    """Start per-kernel event timing of this library's launches."""
    _check(lib().fp8_profile_begin(), "fp8_profile_begin")


def fp8_profile_end(by_shape: bool = False) -> list:
    """Stop timing; one dict per kernel name (by_shape: per kernel name and
    launch shape) with launches, total_ms, bytes, flops (and m, n, k)."""
    cap = 512
    arr = (_KernelStat * cap)()
    n = _c_int()
    _check(lib().fp8_profile_end(arr, cap, ctypes.byref(n)), "fp8_profile_end")
    recs = [dict(name=arr[i].name.decode(), launches=int(arr[i].launches),
                 total_ms=float(arr[i].total_ms), bytes=float(arr[i].bytes),
                 flops=float(arr[i].flops), m=int(arr[i].m), n=int(arr[i].n), k=int(arr[i].k))
            for i in range(min(n.value, cap))]
    if by_shape:
        return recs
    agg = {}
    for r in recs:
        a = agg.setdefault(r["name"], dict(name=r["name"], launches=0, total_ms=0.0, bytes=0.0,
                                           flops=0.0))
        for key in ("launches", "total_ms", "bytes", "flops"):
            a[key] += r[key]
    return list(agg.values())


def fp8_debug_wait_timeout(limit_ns: int, stream=None):
    """Enqueue the bounded-wait probe (a wait that nothing satisfies)."""
    _check(lib().fp8_debug_wait_timeout(int(limit_ns), _stream(stream)), "fp8_debug_wait_timeout")


class QuantizedTensor:
    """Caller-owned FP8 buffers of one [R, C] tensor under the block recipe:
    row [R, C] + row scales, and the transposed layout, either owned here or
    placed inside a linear context (col_ptrs from fp8_linear_ctx_layout)."""

    def __init__(self, R: int, C: int, role: str, device, col_ptrs=None):
        self.R, self.C = R, C
        rs = fp8_scale_shape("block", role, R, C, False)
        cs = fp8_scale_shape("block", role, R, C, True)
        self.row = torch.empty((R, C), dtype=torch.uint8, device=device)
        self.row_scale = torch.empty(rs, dtype=torch.float32, device=device)
        self.row_scale_inv = torch.empty(rs, dtype=torch.float32, device=device)
        if col_ptrs is None:
            self.col = torch.empty((C, R), dtype=torch.uint8, device=device)
            self.col_scale = torch.empty(cs, dtype=torch.float32, device=device)
            self.col_scale_inv = torch.empty(cs, dtype=torch.float32, device=device)
            self.col_ptrs = (_ptr(self.col), _ptr(self.col_scale), _ptr(self.col_scale_inv))
        else:
            self.col = self.col_scale = self.col_scale_inv = None
            self.col_ptrs = col_ptrs


def fp8_linear_ctx_layout(recipe: str, ctx: LinearContext):
    """Device pointers of the transposed FP8 input and its scales inside ctx."""
    a, b_, c = _c_p(), _c_p(), _c_p()
    _check(lib().fp8_linear_ctx_layout(RECIPE[recipe], ctx.N, ctx.K, _ptr(ctx.ctx), ctypes.byref(a),
                                       ctypes.byref(b_), ctypes.byref(c)), "fp8_linear_ctx_layout")
    return (a, b_, c)


def fp8_gelu_quantize(h: torch.Tensor, q: QuantizedTensor, recipe: str = "block", stream=None):
    """q <- 1x128 E4M3 quantization of bf16(GELU(h)); the bf16 GELU output is not written."""
    _need_bf16_cuda(h, "h")
    R, C = h.shape
    _check(lib().fp8_gelu_quantize(_ptr(h), R, C, RECIPE[recipe], _ptr(q.row), q.col_ptrs[0],
                                   _ptr(q.row_scale), _ptr(q.row_scale_inv), q.col_ptrs[1],
                                   q.col_ptrs[2], _stream(stream)), "fp8_gelu_quantize")
    return q


def fp8_gelu_bwd_quantize(da: torch.Tensor, h: torch.Tensor, q: QuantizedTensor,
                          recipe: str = "block", stream=None):
    """q <- 1x128 E5M2 quantization of bf16(dA * GELU'(H)); dH is not written."""
    _need_bf16_cuda(da, "da")
    _need_bf16_cuda(h, "h")
    R, C = h.shape
    _check(lib().fp8_gelu_bwd_quantize(_ptr(da), _ptr(h), R, C, RECIPE[recipe], _ptr(q.row),
                                       q.col_ptrs[0], _ptr(q.row_scale), _ptr(q.row_scale_inv),
                                       q.col_ptrs[1], q.col_ptrs[2], _stream(stream)),
           "fp8_gelu_bwd_quantize")
    return q


def fp8_linear_fwd_quantized(xq: QuantizedTensor, cache: WeightCache, h: int, recipe: str,
                             ws: torch.Tensor, y: torch.Tensor, stream=None):
    _check(lib().fp8_linear_fwd_quantized(_ptr(xq.row), _ptr(xq.row_scale_inv), xq.R, xq.C,
                                          cache.handle, h, RECIPE[recipe], _ptr(y), _ptr(ws),
                                          ws.numel(), _stream(stream)), "fp8_linear_fwd_quantized")
    return y


def fp8_linear_bwd_quantized(gq: QuantizedTensor, ctx: LinearContext, cache: WeightCache, h: int,
                             recipe: str, ws: torch.Tensor, dx, dw: torch.Tensor, stream=None):
    _check(lib().fp8_linear_bwd_quantized(_ptr(gq.row), _ptr(gq.row_scale_inv), gq.col_ptrs[0],
                                          gq.col_ptrs[2], gq.R, gq.C, _ptr(ctx.ctx), cache.handle,
                                          h, RECIPE[recipe], _ptr(dx), _ptr(dw), _ptr(ws),
                                          ws.numel(), _stream(stream)), "fp8_linear_bwd_quantized")
    return dx, dw


class HostPipeline:
    """Owns an fp8_host_pipeline: one fwd+bwd of an isolated FP8 linear per
    step() call, with inputs and results in (pinned) host tensors and the
    host<->device copies done by the library on its own streams."""

    def __init__(self, slots: int):
        h = ctypes.c_void_p()
        _check(lib().fp8_host_pipeline_create(slots, ctypes.byref(h)), "fp8_host_pipeline_create")
        self._h = h

    def step(self, slot: int, host: dict, dev: dict, ctx: LinearContext, ws: torch.Tensor,
             cache: WeightCache, h: int, recipe: str, version: int):
        """host: X, W, dY, Y, dX (or None), dW as CPU bf16 tensors; dev: X, dY, Y,
        dX (or None), dW as CUDA bf16 tensors (W goes to the buffer registered
        for handle h)."""
        N = host["X"].shape[0]
        hio = _HostIO(*[_ptr(host[k]) for k in ("X", "W", "dY", "Y", "dX", "dW")])
        dio = _DeviceIO(*[_ptr(dev[k]) for k in ("X", "dY", "Y", "dX", "dW")], _ptr(ctx.ctx),
                        _ptr(ws), ws.numel())
        _check(lib().fp8_linear_step_host(self._h, slot, N, ctypes.byref(hio), ctypes.byref(dio),
                                          cache.handle, h, RECIPE[recipe], version),
               "fp8_linear_step_host")

    def fork(self, stream=None):
        _check(lib().fp8_host_pipeline_fork(self._h, _stream(stream)), "fp8_host_pipeline_fork")

    def join(self, stream=None):
        _check(lib().fp8_host_pipeline_join(self._h, _stream(stream)), "fp8_host_pipeline_join")

    def sync(self):
        _check(lib().fp8_host_pipeline_sync(self._h), "fp8_host_pipeline_sync")

    def __del__(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.fp8_host_pipeline_destroy(self._h)
            self._h = None


def amax_partials_buffer(rows: int, cols: int, device) -> torch.Tensor:
    """Device buffer for fp8_amax_partials of a [rows, cols] tensor."""
    return _empty_bytes(_quant_ws_bytes("tensorwise", rows, cols), device)


def fp8_amax_partials(x: torch.Tensor, partials: torch.Tensor, stream=None) -> torch.Tensor:
    """First tensorwise pass alone (per-CTA maxima of |x|) into `partials`."""
    _need_bf16_cuda(x, "x")
    R, C = x.shape
    _check(lib().fp8_amax_partials(_ptr(x), R, C, _ptr(partials), partials.numel(),
                                   _stream(stream)), "fp8_amax_partials")
    return partials


def fp8_linear_fwd_after_amax(x: torch.Tensor, x_partials: torch.Tensor, cache: WeightCache,
                              h: int, recipe: str, ws: torch.Tensor, y: torch.Tensor,
                              ctx: LinearContext, stream=None):
    """fp8_linear_fwd with X's amax pass already run by fp8_amax_partials."""
    _need_bf16_cuda(x, "x")
    N, K = x.shape
    _check(lib().fp8_linear_fwd_after_amax(_ptr(x), _ptr(x_partials), N, K, cache.handle, h,
                                           RECIPE[recipe], _ptr(y), _ptr(ctx.ctx), _ptr(ws),
                                           ws.numel(), _stream(stream)),
           "fp8_linear_fwd_after_amax")
    return y, ctx


def fp8_linear_bwd_after_amax(dy: torch.Tensor, dy_partials: torch.Tensor, ctx: LinearContext,
                              cache: WeightCache, h: int, recipe: str, ws: torch.Tensor,
                              dx: torch.Tensor | None, dw: torch.Tensor, stream=None):
    """fp8_linear_bwd with dY's amax pass already run by fp8_amax_partials."""
    _need_bf16_cuda(dy, "dy")
    N, O = dy.shape
    _check(lib().fp8_linear_bwd_after_amax(_ptr(dy), _ptr(dy_partials), N, O, _ptr(ctx.ctx),
                                           cache.handle, h, RECIPE[recipe], _ptr(dx), _ptr(dw),
                                           _ptr(ws), ws.numel(), _stream(stream)),
           "fp8_linear_bwd_after_amax")
    return dx, dw
