"""Reduced-width packed FP8 QKV projection for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libqkvp.so`` (declared in
``include/qkvp.h``).  This module only marshals arguments: it allocates the
output tensors with torch, passes raw device pointers and the current CUDA
stream, and turns status codes into exceptions.  Every step of the forward and
backward runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback, and every call raises if the library is missing.

The method: "96 is enough: shrinking attention's routing vectors", section
"The change" (packed projection, split, QK RMSNorm, RoPE) and "Track 1
(1.167 min on 8xH100, -5.15% same-node): Reduced-width QK and packed FP8
attention", section "Changes" (one FP8 GEMM, dual-layout FP8 bank cached per
optimizer update, fused norm/RoPE/layout, FP8 backward).
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqkvp.so")

STATUS = {
    0: "QKVP_OK", 1: "QKVP_ERR_INVALID_ARGUMENT", 2: "QKVP_ERR_UNSUPPORTED", 3: "QKVP_ERR_MISALIGNED",
    4: "QKVP_ERR_WORKSPACE_TOO_SMALL", 5: "QKVP_ERR_CUDA", 6: "QKVP_ERR_TIMEOUT", 7: "QKVP_ERR_DEVICE_INPUT",
}
OK, ERR_INVALID_ARGUMENT, ERR_UNSUPPORTED, ERR_MISALIGNED = 0, 1, 2, 3
ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_INPUT = 4, 5, 6, 7


class QKVPError(RuntimeError):
    """A non-OK qkvp_status from a library call; ``code`` holds the status."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class Dims(ctypes.Structure):
    """The C ``qkvp_dims`` struct."""

    _fields_ = [("T", ctypes.c_int), ("D", ctypes.c_int), ("H", ctypes.c_int),
                ("d_qk", ctypes.c_int), ("d_v", ctypes.c_int)]


_lib_handle = None
_P = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """The loaded libqkvp.so; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with fp8_packed_reduced_gb300.build.build()"
                               " (or __graft_entry__.build()); there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "qkvp_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "qkvp_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Dims)]),
            "qkvp_bank_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 5),
            "qkvp_workspace_init": (ctypes.c_int, [_P, ctypes.c_size_t, _P]),
            "qkvp_poll_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int), _P]),
            "qkvp_build_rope_table": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.c_double, _P]),
            "qkvp_quantize_bank": (ctypes.c_int, [ctypes.c_int] * 5 + [ctypes.POINTER(_P)] * 3 + [_P] * 4
                                   + [ctypes.c_size_t, _P]),
            "qkvp_forward": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.c_float, _P, ctypes.c_int] + [_P] * 11
                             + [ctypes.c_size_t, _P]),
            "qkvp_backward": (ctypes.c_int, [ctypes.POINTER(Dims), _P, ctypes.c_int] + [_P] * 16
                              + [ctypes.c_size_t, _P]),
            "qkvp_selftest_wait_timeout": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint, _P]),
            "qkvp_set_wait_timeout_ns": (ctypes.c_int, [ctypes.c_uint64]),
            "qkvp_set_timing_events": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int]),
            "qkvp_timing_events_recorded": (ctypes.c_int, []),
            "qkvp_set_cta_pairs": (ctypes.c_int, [ctypes.c_int]),
            "qkvp_weight_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 3),
            "qkvp_quantize_weight": (ctypes.c_int, [ctypes.c_int] * 3 + [ctypes.POINTER(_P)] + [_P] * 4
                                     + [ctypes.c_size_t, _P]),
            "qkvp_oproj_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 3),
            "qkvp_oproj_forward": (ctypes.c_int, [ctypes.c_int] * 3 + [_P] * 7 + [ctypes.c_size_t, _P]),
            "qkvp_oproj_backward": (ctypes.c_int, [ctypes.c_int] * 3 + [_P] * 10 + [ctypes.c_size_t, _P]),
            "qkvp_mlp_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 3),
            "qkvp_activation_workspace_bytes": (ctypes.c_size_t, []),
            "qkvp_quantize_activation": (ctypes.c_int, [_P, ctypes.c_int64, _P, _P, _P, ctypes.c_size_t, _P]),
            "qkvp_forward_quantized": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.c_float, _P, ctypes.c_int]
                                       + [_P] * 10 + [ctypes.c_size_t, _P]),
            "qkvp_mlp_forward": (ctypes.c_int, [ctypes.c_int] * 3 + [_P] * 12 + [ctypes.c_size_t, _P]),
            "qkvp_mlp_backward": (ctypes.c_int, [ctypes.c_int] * 3 + [_P] * 18 + [ctypes.c_size_t, _P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib_handle = L
    return _lib_handle


def _check(code: int, where: str):
    if code != OK:
        raise QKVPError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# ----------------------------------------------------------------------------
# Shapes and scratch
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Shape:
    """Problem shape of one layer: T tokens, model width D, H heads of
    d_qk (q, k) and d_v (v) columns."""

    T: int
    D: int
    H: int
    d_qk: int = 96
    d_v: int = 128

    @property
    def N(self) -> int:
        return self.H * (2 * self.d_qk + self.d_v)

    def dims(self) -> Dims:
        return Dims(self.T, self.D, self.H, self.d_qk, self.d_v)


def workspace_bytes(shape: Shape) -> int:
    """Bytes of workspace forward/backward need for ``shape`` (0: unsupported)."""
    d = shape.dims()
    return int(lib().qkvp_workspace_bytes(ctypes.byref(d)))


def new_workspace(shape: Shape, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace for forward/backward of ``shape``."""
    n = workspace_bytes(shape)
    if n == 0:
        raise QKVPError(ERR_UNSUPPORTED, "workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(lib().qkvp_workspace_init(_ptr(ws), n, _stream(ws.device)), "qkvp_workspace_init")
    return ws


def poll_device_status(ws: torch.Tensor):
    """(status, kernel id) recorded on the device since the last poll; clears it."""
    where = ctypes.c_int(0)
    code = lib().qkvp_poll_device_status(_ptr(ws), ctypes.byref(where), _stream(ws.device))
    return int(code), int(where.value)


def set_timing_events(events):
    """Arm the kernel-boundary timing hook with torch.cuda.Event objects
    (created with enable_timing=True); an empty list disarms it."""
    n = len(events)
    arr = (ctypes.c_void_p * max(n, 1))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().qkvp_set_timing_events(arr, n), "qkvp_set_timing_events")


def timing_events_recorded() -> int:
    """Events the armed timing hook has recorded so far."""
    return int(lib().qkvp_timing_events_recorded())


def set_cta_pairs(mask: int) -> int:
    """Choose which GEMMs run on 2-CTA clusters (bit 0 forward, bit 1 dX,
    bit 2 dW); returns the previous mask."""
    prev = int(lib().qkvp_set_cta_pairs(mask))
    if prev < 0:
        raise ValueError(f"cta pair mask {mask} outside 0..7")
    return prev


def set_wait_timeout_ns(ns: int):
    """Limit of every device-side wait in the library's kernels (ns); a wait
    that runs out records QKVP_ERR_TIMEOUT in the workspace's status word."""
    _check(lib().qkvp_set_wait_timeout_ns(ns), "qkvp_set_wait_timeout_ns")


def selftest_wait_timeout(ws: torch.Tensor, timeout_us: int):
    """Launch the self-test kernel whose bounded wait on a barrier that
    nothing arrives on runs out after ``timeout_us`` and records
    QKVP_ERR_TIMEOUT (the context stays usable)."""
    _check(lib().qkvp_selftest_wait_timeout(_ptr(ws), ws.numel(), timeout_us, _stream(ws.device)),
           "qkvp_selftest_wait_timeout")


def build_rope_table(max_pos: int, d_qk: int, base: float = 10000.0, device="cuda") -> torch.Tensor:
    """RoPE table [d_qk/4, max_pos, 4] float32: entry (j, p) holds
    cos(p w_2j), cos(p w_2j+1), sin(p w_2j), sin(p w_2j+1)."""
    t = torch.empty((d_qk // 4, max_pos, 4), dtype=torch.float32, device=device)
    _check(lib().qkvp_build_rope_table(_ptr(t), max_pos, d_qk, base, _stream(t.device)), "qkvp_build_rope_table")
    return t


# ----------------------------------------------------------------------------
# Bank refresh (once per optimizer update)
# ----------------------------------------------------------------------------

# Scratch of the weight refreshes, one per (device, stream): zeroed once when
# it is made, and left zeroed by every refresh (the counters its kernel's
# blocks share), so that refreshes on one stream reuse it and refreshes on
# different streams never share one.
_refresh_scratch = {}


def _refresh_ws(dev, nbytes: int) -> torch.Tensor:
    stream = torch.cuda.current_stream(dev)
    key = (torch.device(dev).index, stream.cuda_stream)
    ws = _refresh_scratch.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        _check(lib().qkvp_workspace_init(_ptr(ws), nbytes, _stream(ws.device)), "qkvp_workspace_init")
        _refresh_scratch[key] = ws
    return ws


def quantize_bank(layers: Sequence[Sequence[torch.Tensor]], H: int, d_qk: int = 96, d_v: int = 128,
                  out=None):
    """Quantise L layers of (W_q, W_k, W_v) bf16 into the dual-layout FP8 bank.

    Returns (W8 [L, N, D] uint8, W8T [L, D, N] uint8, w_scale [L] float32).
    """
    L = len(layers)
    D = layers[0][0].shape[1]
    dev = layers[0][0].device
    N = H * (2 * d_qk + d_v)
    for l, (wq, wk, wv) in enumerate(layers):
        for name, w, rows in (("Wq", wq, H * d_qk), ("Wk", wk, H * d_qk), ("Wv", wv, H * d_v)):
            _need_cuda(w, f"layer {l} {name}", torch.bfloat16)
            if tuple(w.shape) != (rows, D):
                raise ValueError(f"layer {l} {name}: expected {(rows, D)}, got {tuple(w.shape)}")
    if out is None:
        W8 = torch.empty((L, N, D), dtype=torch.uint8, device=dev)
        W8T = torch.empty((L, D, N), dtype=torch.uint8, device=dev)
        w_scale = torch.empty((L,), dtype=torch.float32, device=dev)
    else:
        W8, W8T, w_scale = out
    nws = int(lib().qkvp_bank_workspace_bytes(L, D, H, d_qk, d_v))
    if nws == 0:
        raise QKVPError(ERR_UNSUPPORTED, "qkvp_bank_workspace_bytes")
    ws = _refresh_ws(dev, nws)
    arr = lambda i: (ctypes.c_void_p * L)(*[ctypes.c_void_p(layers[l][i].data_ptr()) for l in range(L)])
    _check(lib().qkvp_quantize_bank(L, D, H, d_qk, d_v, arr(0), arr(1), arr(2), _ptr(W8), _ptr(W8T),
                                    _ptr(w_scale), _ptr(ws), ws.numel(), _stream(dev)), "qkvp_quantize_bank")
    return W8, W8T, w_scale


class QKVPBank:
    """The FP8 weight bank of L layers, refreshed once per optimizer update.

    ``refresh`` re-quantises when any weight tensor changed since the last
    refresh (tracked by the tensors' version counters and storage pointers),
    so the cached row-major and transposed views are never stale.
    """

    def __init__(self, layers, H: int, d_qk: int = 96, d_v: int = 128):
        self.layers = [tuple(l) for l in layers]
        self.H, self.d_qk, self.d_v = H, d_qk, d_v
        self._key = None
        self.W8 = self.W8T = self.w_scale = None
        self.refreshes = 0
        self.refresh()

    def _state(self):
        return tuple((w._version, w.data_ptr()) for l in self.layers for w in l)

    def refresh(self, force: bool = False) -> bool:
        key = self._state()
        if not force and key == self._key:
            return False
        out = None if self.W8 is None else (self.W8, self.W8T, self.w_scale)
        self.W8, self.W8T, self.w_scale = quantize_bank(self.layers, self.H, self.d_qk, self.d_v, out=out)
        self._key = key
        self.refreshes += 1
        return True

    def layer(self, l: int):
        return self.W8[l], self.W8T[l], self.w_scale[l:l + 1]


# ----------------------------------------------------------------------------
# Forward / backward
# ----------------------------------------------------------------------------

@dataclass
class Saved:
    """State the backward needs: saved outputs and the FP8 activations."""
    q: torch.Tensor
    k: torch.Tensor
    rstd: torch.Tensor
    x8: torch.Tensor
    x_scale: torch.Tensor
    pos: torch.Tensor


def forward(x, pos, W8, w_scale, H, rope_table, d_qk=96, d_v=128, eps=1e-6, ws=None, out=None):
    """Packed QKV forward for one layer.

    x [T, D] bf16, pos [T] int32, W8 [N, D] uint8, w_scale [1] float32,
    rope_table from build_rope_table.  Returns (q, k, v, Saved) with
    q, k [H, T, d_qk] and v [H, T, d_v] bf16; Saved holds what the backward
    needs (saved outputs, rstd, the FP8 activations x8 and their scale).
    """
    T, D = x.shape
    shape = Shape(T, D, H, d_qk, d_v)
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(pos, "pos", torch.int32, (T,))
    _need_cuda(W8, "W8", torch.uint8, (shape.N, D))
    _need_cuda(w_scale, "w_scale", torch.float32, (1,))
    _need_cuda(rope_table, "rope_table", torch.float32)
    if rope_table.dim() != 3 or rope_table.shape[0] != d_qk // 4 or rope_table.shape[2] != 4:
        raise ValueError("rope_table must be build_rope_table(max_pos, d_qk)")
    dev = x.device
    if ws is None:
        ws = new_workspace(shape, dev)
    if out is None:
        bf = dict(dtype=torch.bfloat16, device=dev)
        out = dict(q=torch.empty((H, T, d_qk), **bf), k=torch.empty((H, T, d_qk), **bf),
                   v=torch.empty((H, T, d_v), **bf),
                   rstd=torch.empty((2, H, T), dtype=torch.float32, device=dev),
                   x8=torch.empty((T, D), dtype=torch.uint8, device=dev),
                   x_scale=torch.empty((1,), dtype=torch.float32, device=dev))
    o = out
    for name, dt, shp in (("q", torch.bfloat16, (H, T, d_qk)), ("k", torch.bfloat16, (H, T, d_qk)),
                          ("v", torch.bfloat16, (H, T, d_v)), ("rstd", torch.float32, (2, H, T)),
                          ("x8", torch.uint8, (T, D)), ("x_scale", torch.float32, (1,))):
        _need_cuda(o[name], name, dt, shp)
    d = shape.dims()
    rc = lib().qkvp_forward(ctypes.byref(d), eps, _ptr(rope_table), rope_table.shape[1], _ptr(x), _ptr(pos),
                            _ptr(W8), _ptr(w_scale), _ptr(o["q"]), _ptr(o["k"]), _ptr(o["v"]), _ptr(o["rstd"]),
                            _ptr(o["x8"]), _ptr(o["x_scale"]), _ptr(ws), ws.numel(),
                            _stream(dev))
    _check(rc, "qkvp_forward")
    saved = Saved(q=o["q"], k=o["k"], rstd=o["rstd"], x8=o["x8"], x_scale=o["x_scale"], pos=pos)
    return o["q"], o["k"], o["v"], saved


def quantize_activation(x, ws, out=None):
    """Per-tensor E4M3 codes of a bf16 tensor (numel a multiple of 16).
    ``ws``: a zero-initialised workspace (new_workspace, or any workspace of
    this library).  Returns (codes uint8 shaped like x, scale [1] float32)."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(ws, "ws", torch.uint8)
    if out is None:
        out = (torch.empty(x.shape, dtype=torch.uint8, device=x.device),
               torch.empty((1,), dtype=torch.float32, device=x.device))
    x8, scale = out
    _need_cuda(x8, "x8", torch.uint8, tuple(x.shape))
    _need_cuda(scale, "scale", torch.float32, (1,))
    _check(lib().qkvp_quantize_activation(_ptr(x), x.numel(), _ptr(x8), _ptr(scale), _ptr(ws), ws.numel(),
                                          _stream(x.device)), "qkvp_quantize_activation")
    return x8, scale


def forward_quantized(x8, x_scale, pos, W8, w_scale, H, rope_table, d_qk=96, d_v=128, eps=1e-6, ws=None, out=None):
    """The forward's GEMM and fused epilogue from x8 [T, D] and x_scale
    (quantize_activation of x).  Returns (q, k, v, Saved) like forward()."""
    T, D = x8.shape
    shape = Shape(T, D, H, d_qk, d_v)
    _need_cuda(x8, "x8", torch.uint8)
    _need_cuda(x_scale, "x_scale", torch.float32, (1,))
    _need_cuda(pos, "pos", torch.int32, (T,))
    _need_cuda(W8, "W8", torch.uint8, (shape.N, D))
    _need_cuda(w_scale, "w_scale", torch.float32, (1,))
    _need_cuda(rope_table, "rope_table", torch.float32)
    if rope_table.dim() != 3 or rope_table.shape[0] != d_qk // 4 or rope_table.shape[2] != 4:
        raise ValueError("rope_table must be build_rope_table(max_pos, d_qk)")
    dev = x8.device
    if ws is None:
        ws = new_workspace(shape, dev)
    if out is None:
        bf = dict(dtype=torch.bfloat16, device=dev)
        out = dict(q=torch.empty((H, T, d_qk), **bf), k=torch.empty((H, T, d_qk), **bf),
                   v=torch.empty((H, T, d_v), **bf), rstd=torch.empty((2, H, T), dtype=torch.float32, device=dev))
    o = out
    for name, dt, shp in (("q", torch.bfloat16, (H, T, d_qk)), ("k", torch.bfloat16, (H, T, d_qk)),
                          ("v", torch.bfloat16, (H, T, d_v)), ("rstd", torch.float32, (2, H, T))):
        _need_cuda(o[name], name, dt, shp)
    d = shape.dims()
    _check(lib().qkvp_forward_quantized(ctypes.byref(d), eps, _ptr(rope_table), rope_table.shape[1], _ptr(x8),
                                        _ptr(x_scale), _ptr(pos), _ptr(W8), _ptr(w_scale), _ptr(o["q"]),
                                        _ptr(o["k"]), _ptr(o["v"]), _ptr(o["rstd"]), _ptr(ws), ws.numel(),
                                        _stream(dev)), "qkvp_forward_quantized")
    saved = Saved(q=o["q"], k=o["k"], rstd=o["rstd"], x8=x8, x_scale=x_scale, pos=pos)
    return o["q"], o["k"], o["v"], saved


def backward(dq, dk, dv, saved: Saved, W8T, w_scale, rope_table, ws=None, out=None):
    """Packed QKV backward for one layer.  Returns a dict with dx [T, D],
    dW [N, D] (bf16), dY8 [T, N] (uint8) and dy_scale [1]."""
    H, T, d_qk = dq.shape
    d_v = dv.shape[2]
    D = W8T.shape[0]
    shape = Shape(T, D, H, d_qk, d_v)
    _need_cuda(dq, "dq", torch.bfloat16)
    _need_cuda(dk, "dk", torch.bfloat16, (H, T, d_qk))
    _need_cuda(dv, "dv", torch.bfloat16, (H, T, d_v))
    _need_cuda(saved.q, "saved q", torch.bfloat16, (H, T, d_qk))
    _need_cuda(saved.k, "saved k", torch.bfloat16, (H, T, d_qk))
    _need_cuda(saved.rstd, "saved rstd", torch.float32, (2, H, T))
    _need_cuda(saved.pos, "pos", torch.int32, (T,))
    _need_cuda(saved.x8, "saved x8", torch.uint8, (T, D))
    _need_cuda(saved.x_scale, "saved x_scale", torch.float32, (1,))
    _need_cuda(W8T, "W8T", torch.uint8, (D, shape.N))
    _need_cuda(w_scale, "w_scale", torch.float32, (1,))
    _need_cuda(rope_table, "rope_table", torch.float32)
    if rope_table.dim() != 3 or rope_table.shape[0] != d_qk // 4 or rope_table.shape[2] != 4:
        raise ValueError("rope_table must be build_rope_table(max_pos, d_qk)")
    dev = dq.device
    if ws is None:
        ws = new_workspace(shape, dev)
    if out is None:
        out = dict(dx=torch.empty((T, D), dtype=torch.bfloat16, device=dev),
                   dW=torch.empty((shape.N, D), dtype=torch.bfloat16, device=dev),
                   dY8=torch.empty((T, shape.N), dtype=torch.uint8, device=dev),
                   dy_scale=torch.empty((1,), dtype=torch.float32, device=dev))
    o = out
    for name, dt, shp in (("dx", torch.bfloat16, (T, D)), ("dW", torch.bfloat16, (shape.N, D)),
                          ("dY8", torch.uint8, (T, shape.N)), ("dy_scale", torch.float32, (1,))):
        _need_cuda(o[name], name, dt, shp)
    d = shape.dims()
    rc = lib().qkvp_backward(ctypes.byref(d), _ptr(rope_table), rope_table.shape[1], _ptr(dq), _ptr(dk), _ptr(dv),
                             _ptr(saved.q), _ptr(saved.k), _ptr(saved.rstd), _ptr(saved.pos), _ptr(W8T),
                             _ptr(w_scale), _ptr(saved.x8), _ptr(saved.x_scale), _ptr(o["dx"]), _ptr(o["dW"]),
                             _ptr(o["dY8"]), _ptr(o["dy_scale"]), _ptr(ws), ws.numel(),
                             _stream(dev))
    _check(rc, "qkvp_backward")
    return o


# ----------------------------------------------------------------------------
# Output projection over the V/O bank
# ----------------------------------------------------------------------------

def quantize_weight(weights: Sequence[torch.Tensor], out=None):
    """Quantise L bf16 matrices [R, C] (one scale each) into both FP8 layouts.

    Returns (W8 [L, R, C] uint8, W8T [L, C, R] uint8, w_scale [L] float32)."""
    L = len(weights)
    R, C = weights[0].shape
    dev = weights[0].device
    for l, w in enumerate(weights):
        _need_cuda(w, f"weight {l}", torch.bfloat16, (R, C))
    if out is None:
        W8 = torch.empty((L, R, C), dtype=torch.uint8, device=dev)
        W8T = torch.empty((L, C, R), dtype=torch.uint8, device=dev)
        w_scale = torch.empty((L,), dtype=torch.float32, device=dev)
    else:
        W8, W8T, w_scale = out
        _need_cuda(W8, "W8", torch.uint8, (L, R, C))
        _need_cuda(W8T, "W8T", torch.uint8, (L, C, R))
        _need_cuda(w_scale, "w_scale", torch.float32, (L,))
    nws = int(lib().qkvp_weight_workspace_bytes(L, R, C))
    if nws == 0:
        raise QKVPError(ERR_UNSUPPORTED, "qkvp_weight_workspace_bytes")
    ws = _refresh_ws(dev, nws)
    arr = (ctypes.c_void_p * L)(*[ctypes.c_void_p(w.data_ptr()) for w in weights])
    _check(lib().qkvp_quantize_weight(L, R, C, arr, _ptr(W8), _ptr(W8T), _ptr(w_scale), _ptr(ws), ws.numel(),
                                      _stream(dev)), "qkvp_quantize_weight")
    return W8, W8T, w_scale


def new_oproj_workspace(T: int, D: int, K: int, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace for the O projection's forward/backward."""
    n = int(lib().qkvp_oproj_workspace_bytes(T, D, K))
    if n == 0:
        raise QKVPError(ERR_UNSUPPORTED, "qkvp_oproj_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(lib().qkvp_workspace_init(_ptr(ws), n, _stream(ws.device)), "qkvp_workspace_init")
    return ws


def oproj_forward(a, Wo8, wo_scale, ws=None, out=None):
    """out [T, D] = FP8 a [T, K] . W_o^T.  Returns (out, a8 [T, K] uint8, a_scale [1])."""
    T, K = a.shape
    D = Wo8.shape[0]
    _need_cuda(a, "a", torch.bfloat16)
    _need_cuda(Wo8, "Wo8", torch.uint8, (D, K))
    _need_cuda(wo_scale, "wo_scale", torch.float32, (1,))
    dev = a.device
    if ws is None:
        ws = new_oproj_workspace(T, D, K, dev)
    if out is None:
        out = dict(out=torch.empty((T, D), dtype=torch.bfloat16, device=dev),
                   a8=torch.empty((T, K), dtype=torch.uint8, device=dev),
                   a_scale=torch.empty((1,), dtype=torch.float32, device=dev))
    o = out
    for name, dt, shp in (("out", torch.bfloat16, (T, D)), ("a8", torch.uint8, (T, K)),
                          ("a_scale", torch.float32, (1,))):
        _need_cuda(o[name], name, dt, shp)
    _check(lib().qkvp_oproj_forward(T, D, K, _ptr(a), _ptr(Wo8), _ptr(wo_scale), _ptr(o["out"]), _ptr(o["a8"]),
                                    _ptr(o["a_scale"]), _ptr(ws), ws.numel(), _stream(dev)), "qkvp_oproj_forward")
    return o["out"], o["a8"], o["a_scale"]


def oproj_backward(dout, Wo8T, wo_scale, a8, a_scale, ws=None, out=None):
    """Backward of the O projection.  Returns a dict with da [T, K], dWo [D, K]
    (bf16), dout8 [T, D] (uint8) and dout_scale [1]."""
    T, D = dout.shape
    K = Wo8T.shape[0]
    _need_cuda(dout, "dout", torch.bfloat16)
    _need_cuda(Wo8T, "Wo8T", torch.uint8, (K, D))
    _need_cuda(wo_scale, "wo_scale", torch.float32, (1,))
    _need_cuda(a8, "a8", torch.uint8, (T, K))
    _need_cuda(a_scale, "a_scale", torch.float32, (1,))
    dev = dout.device
    if ws is None:
        ws = new_oproj_workspace(T, D, K, dev)
    if out is None:
        out = dict(da=torch.empty((T, K), dtype=torch.bfloat16, device=dev),
                   dWo=torch.empty((D, K), dtype=torch.bfloat16, device=dev),
                   dout8=torch.empty((T, D), dtype=torch.uint8, device=dev),
                   dout_scale=torch.empty((1,), dtype=torch.float32, device=dev))
    o = out
    for name, dt, shp in (("da", torch.bfloat16, (T, K)), ("dWo", torch.bfloat16, (D, K)),
                          ("dout8", torch.uint8, (T, D)), ("dout_scale", torch.float32, (1,))):
        _need_cuda(o[name], name, dt, shp)
    _check(lib().qkvp_oproj_backward(T, D, K, _ptr(dout), _ptr(Wo8T), _ptr(wo_scale), _ptr(a8), _ptr(a_scale),
                                     _ptr(o["da"]), _ptr(o["dWo"]), _ptr(o["dout8"]), _ptr(o["dout_scale"]),
                                     _ptr(ws), ws.numel(), _stream(dev)), "qkvp_oproj_backward")
    return o


# ----------------------------------------------------------------------------
# FP8 ReLU-squared MLP
# ----------------------------------------------------------------------------

def new_mlp_workspace(T: int, D: int, F: int, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace for the MLP's forward/backward."""
    n = int(lib().qkvp_mlp_workspace_bytes(T, D, F))
    if n == 0:
        raise QKVPError(ERR_UNSUPPORTED, "qkvp_mlp_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(lib().qkvp_workspace_init(_ptr(ws), n, _stream(ws.device)), "qkvp_workspace_init")
    return ws


def mlp_forward(x, W1_8, w1_scale, W2_8, w2_scale, ws=None, out=None):
    """out = relu(x . W_fc^T)^2 . W_proj^T in FP8.  Returns a dict with out
    [T, D] bf16, x8 [T, D], x_scale, h [T, F] bf16, h8 [T, F], h_scale."""
    T, D = x.shape
    F_ = W1_8.shape[0]
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(W1_8, "W1_8", torch.uint8, (F_, D))
    _need_cuda(W2_8, "W2_8", torch.uint8, (D, F_))
    _need_cuda(w1_scale, "w1_scale", torch.float32, (1,))
    _need_cuda(w2_scale, "w2_scale", torch.float32, (1,))
    dev = x.device
    if ws is None:
        ws = new_mlp_workspace(T, D, F_, dev)
    if out is None:
        u8, bf, f = (dict(dtype=torch.uint8, device=dev), dict(dtype=torch.bfloat16, device=dev),
                     dict(dtype=torch.float32, device=dev))
        out = dict(out=torch.empty((T, D), **bf), x8=torch.empty((T, D), **u8), x_scale=torch.empty((1,), **f),
                   h=torch.empty((T, F_), **bf), h8=torch.empty((T, F_), **u8), h_scale=torch.empty((1,), **f))
    o = out
    for name, dt, shp in (("out", torch.bfloat16, (T, D)), ("x8", torch.uint8, (T, D)),
                          ("x_scale", torch.float32, (1,)), ("h", torch.bfloat16, (T, F_)),
                          ("h8", torch.uint8, (T, F_)), ("h_scale", torch.float32, (1,))):
        _need_cuda(o[name], name, dt, shp)
    _check(lib().qkvp_mlp_forward(T, D, F_, _ptr(x), _ptr(W1_8), _ptr(w1_scale), _ptr(W2_8), _ptr(w2_scale),
                                  _ptr(o["out"]), _ptr(o["x8"]), _ptr(o["x_scale"]), _ptr(o["h"]), _ptr(o["h8"]),
                                  _ptr(o["h_scale"]), _ptr(ws), ws.numel(), _stream(dev)), "qkvp_mlp_forward")
    return o


def mlp_backward(dout, W1_8T, w1_scale, W2_8T, w2_scale, saved, ws=None, out=None):
    """Backward of mlp_forward from its saved codes (``saved``: the forward's
    dict, whose x8, x_scale, h8 and h_scale are read).  Returns a dict with dx
    [T, D], dW1 [F, D], dW2 [D, F] (bf16), dout8, dout_scale, dpre [T, F] bf16,
    dpre8 and dpre_scale."""
    T, D = dout.shape
    F_ = W2_8T.shape[0]
    _need_cuda(dout, "dout", torch.bfloat16)
    _need_cuda(W1_8T, "W1_8T", torch.uint8, (D, F_))
    _need_cuda(W2_8T, "W2_8T", torch.uint8, (F_, D))
    _need_cuda(w1_scale, "w1_scale", torch.float32, (1,))
    _need_cuda(w2_scale, "w2_scale", torch.float32, (1,))
    _need_cuda(saved["x8"], "saved x8", torch.uint8, (T, D))
    _need_cuda(saved["x_scale"], "saved x_scale", torch.float32, (1,))
    _need_cuda(saved["h8"], "saved h8", torch.uint8, (T, F_))
    _need_cuda(saved["h_scale"], "saved h_scale", torch.float32, (1,))
    dev = dout.device
    if ws is None:
        ws = new_mlp_workspace(T, D, F_, dev)
    if out is None:
        u8, bf, f = (dict(dtype=torch.uint8, device=dev), dict(dtype=torch.bfloat16, device=dev),
                     dict(dtype=torch.float32, device=dev))
        out = dict(dx=torch.empty((T, D), **bf), dW1=torch.empty((F_, D), **bf), dW2=torch.empty((D, F_), **bf),
                   dout8=torch.empty((T, D), **u8), dout_scale=torch.empty((1,), **f),
                   dpre=torch.empty((T, F_), **bf), dpre8=torch.empty((T, F_), **u8),
                   dpre_scale=torch.empty((1,), **f))
    o = out
    for name, dt, shp in (("dx", torch.bfloat16, (T, D)), ("dW1", torch.bfloat16, (F_, D)),
                          ("dW2", torch.bfloat16, (D, F_)), ("dout8", torch.uint8, (T, D)),
                          ("dout_scale", torch.float32, (1,)), ("dpre", torch.bfloat16, (T, F_)),
                          ("dpre8", torch.uint8, (T, F_)), ("dpre_scale", torch.float32, (1,))):
        _need_cuda(o[name], name, dt, shp)
    _check(lib().qkvp_mlp_backward(T, D, F_, _ptr(dout), _ptr(W1_8T), _ptr(w1_scale), _ptr(W2_8T), _ptr(w2_scale),
                                   _ptr(saved["x8"]), _ptr(saved["x_scale"]), _ptr(saved["h8"]),
                                   _ptr(saved["h_scale"]), _ptr(o["dx"]), _ptr(o["dW1"]), _ptr(o["dW2"]),
                                   _ptr(o["dout8"]), _ptr(o["dout_scale"]), _ptr(o["dpre"]), _ptr(o["dpre8"]),
                                   _ptr(o["dpre_scale"]), _ptr(ws), ws.numel(), _stream(dev)), "qkvp_mlp_backward")
    return o
