"""ctypes binding of libmoe.so (include/moe.h).  Argument marshalling only.

Every function takes torch tensors that already live on the GPU and passes their device
pointers to the C entry point of the same name; all computation happens in the library's
CUDA kernels.  Loading fails loudly if the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_WORKSPACE_TOO_SMALL",
                3: "MOE_ERR_UNSUPPORTED_SHAPE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_NOT_IMPLEMENTED"}

# Every symbol include/moe.h declares.
EXPORTS = ["moe_status_string", "moe_workspace_size", "moe_route", "moe_route_from_logits",
           "moe_permute", "moe_permute_noalloc", "moe_expert_ffn", "moe_combine", "moe_forward", "moe_check_status",
           "moe_plan_pieces", "moe_launch_count", "moe_timing_enable", "moe_timing_read",
           "moe_timing_name", "moe_timing_classes", "moe_selftest_wait", "moe_decode_chain",
           "moe_decode_chain_q8", "moe_quantize_e4m3", "moe_graph_create", "moe_graph_launch",
           "moe_graph_kernel_count", "moe_graph_destroy", "moe_forward_q8", "moe_debug_build",
           "moe_decode_chain_q4", "moe_quantize_q4"]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, STATUS_NAMES.get(status, "?"), status))


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("inter", ctypes.c_int), ("shared_inter", ctypes.c_int)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "b_router", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")]


class WeightsQ8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "b_router", "q_gate", "q_up", "q_down", "s_gate", "s_up", "s_down",
                 "qs_gate", "qs_up", "qs_down", "ss_gate", "ss_up", "ss_down")]


class WeightsQ4(ctypes.Structure):
    # the same fields as WeightsQ8: packed 4-bit codes and per-block scales (include/moe.h)
    _fields_ = WeightsQ8._fields_


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_lib = None


def load(path: str = LIB_PATH):
    """Load libmoe.so (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libmoe.so not built (%s); run __graft_entry__.build() or "
                          "python -m sparse_moe_router_gb300.build" % path)
    L = ctypes.CDLL(path)
    C, W = ctypes.POINTER(Config), ctypes.POINTER(Weights)
    L.moe_status_string.argtypes = [_I]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_workspace_size.argtypes = [C, _I]
    L.moe_workspace_size.restype = _SZ
    L.moe_route.argtypes = [C, W, _P, _I, _P, _P, _P, _P, _SZ, _P]
    L.moe_route_from_logits.argtypes = [C, _P, _I, _P, _P, _P]
    L.moe_permute.argtypes = [C, _P, _I, _P, _P, _P, _P, _SZ, _P]
    L.moe_permute_noalloc.argtypes = [C, _P, _I, _P, _P, _P, _P]
    L.moe_expert_ffn.argtypes = [C, W, _P, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_combine.argtypes = [C, _P, _P, _P, _P, _I, _P, _P]
    L.moe_forward.argtypes = [C, W, _P, _I, _P, _P, _P, _P, _SZ, _P]
    L.moe_decode_chain.argtypes = [C, W, _I, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_decode_chain_q8.argtypes = [C, ctypes.POINTER(WeightsQ8), _I, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_forward_q8.argtypes = [C, ctypes.POINTER(WeightsQ8), _P, _I, _P, _P, _P, _P, _SZ, _P]
    L.moe_quantize_e4m3.argtypes = [_P, _I, _I, _P, _P, _P]
    L.moe_decode_chain_q4.argtypes = [C, ctypes.POINTER(WeightsQ4), _I, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_quantize_q4.argtypes = [_P, _I, _I, _P, _P, _P]
    L.moe_check_status.argtypes = [_P, _SZ, ctypes.POINTER(_I), _P]
    L.moe_selftest_wait.argtypes = [_P, _SZ, ctypes.c_ulonglong, _I, _P]
    L.moe_graph_create.argtypes = [C, W, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, ctypes.POINTER(_P)]
    L.moe_graph_launch.argtypes = [_P, _P]
    L.moe_graph_kernel_count.argtypes = [_P]
    L.moe_graph_kernel_count.restype = _I
    L.moe_graph_destroy.argtypes = [_P]
    L.moe_plan_pieces.argtypes = [_I, ctypes.POINTER(_I), _I]
    L.moe_plan_pieces.restype = _I
    L.moe_launch_count.argtypes = []
    L.moe_launch_count.restype = ctypes.c_uint64
    L.moe_timing_enable.argtypes = [_I]
    L.moe_timing_read.argtypes = [ctypes.c_char_p, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_double)]
    L.moe_timing_name.argtypes = [_I]
    L.moe_timing_name.restype = ctypes.c_char_p
    L.moe_timing_classes.argtypes = []
    L.moe_debug_build.argtypes = []
    L.moe_debug_build.restype = _I
    for fn in ("moe_route", "moe_route_from_logits", "moe_permute", "moe_permute_noalloc", "moe_expert_ffn",
               "moe_combine", "moe_forward", "moe_check_status", "moe_timing_enable",
               "moe_timing_read", "moe_timing_classes", "moe_selftest_wait", "moe_decode_chain",
               "moe_decode_chain_q8", "moe_quantize_e4m3", "moe_graph_create", "moe_graph_launch",
               "moe_graph_destroy", "moe_forward_q8", "moe_decode_chain_q4", "moe_quantize_q4"):
        getattr(L, fn).restype = _I
    _lib = L
    return L


def lib():
    return load()


# ---------------------------------------------------------------------- helpers --

def config(hidden, n_experts, top_k, inter, shared_inter) -> Config:
    return Config(hidden, n_experts, top_k, inter, shared_inter)


def config_of(shape) -> Config:
    """Config from an object with hidden/n_experts/top_k/inter/shared_inter attributes."""
    return Config(shape.hidden, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def weights(layer: dict) -> Weights:
    """Weights struct from a dict of device tensors (keys as in include/moe.h)."""
    w = Weights()
    for name, _ in Weights._fields_:
        t = layer.get(name)
        setattr(w, name, None if t is None else t.data_ptr())
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("weight %s must be a contiguous CUDA tensor" % name)
    return w


def weights_q8(layer: dict) -> WeightsQ8:
    """WeightsQ8 struct from a dict of device tensors (keys as in include/moe.h)."""
    w = WeightsQ8()
    for name, _ in WeightsQ8._fields_:
        t = layer.get(name)
        setattr(w, name, None if t is None else t.data_ptr())
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("weight %s must be a contiguous CUDA tensor" % name)
    return w


def weights_q4(layer: dict) -> WeightsQ4:
    """WeightsQ4 struct from a dict of device tensors (keys as in include/moe.h)."""
    w = WeightsQ4()
    for name, _ in WeightsQ4._fields_:
        t = layer.get(name)
        setattr(w, name, None if t is None else t.data_ptr())
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("weight %s must be a contiguous CUDA tensor" % name)
    return w


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, st):
    if st != MOE_OK:
        raise MoeError(fn, st)


def workspace_size(cfg: Config, max_T: int) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(cfg), int(max_T)))


def alloc_workspace(cfg: Config, max_T: int, device="cuda") -> torch.Tensor:
    n = workspace_size(cfg, max_T)
    if n == 0:
        raise MoeError("moe_workspace_size", 3)
    # zeroed once: the first 256 bytes are the device status word
    return torch.zeros(n, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ entry points --

def moe_route(cfg, w: Weights, x, T, logits_out, topk_ids, topk_w, ws, stream=None):
    st = lib().moe_route(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), int(T), _ptr(logits_out),
                         _ptr(topk_ids), _ptr(topk_w), _ptr(ws), ws.numel(), _stream(stream))
    _check("moe_route", st)


def moe_route_from_logits(cfg, logits, T, topk_ids, topk_w, stream=None):
    st = lib().moe_route_from_logits(ctypes.byref(cfg), _ptr(logits), int(T), _ptr(topk_ids),
                                     _ptr(topk_w), _stream(stream))
    _check("moe_route_from_logits", st)


def moe_permute(cfg, topk_ids, T, offsets, perm, inv, ws, stream=None):
    st = lib().moe_permute(ctypes.byref(cfg), _ptr(topk_ids), int(T), _ptr(offsets), _ptr(perm),
                           _ptr(inv), _ptr(ws), ws.numel(), _stream(stream))
    _check("moe_permute", st)


def moe_permute_noalloc(cfg, topk_ids, T, offsets, perm, inv, stream=None):
    """moe_permute for callers that cannot allocate: no workspace argument."""
    st = lib().moe_permute_noalloc(ctypes.byref(cfg), _ptr(topk_ids), int(T), _ptr(offsets),
                                   _ptr(perm), _ptr(inv), _stream(stream))
    _check("moe_permute_noalloc", st)


def moe_expert_ffn(cfg, w: Weights, x, T, offsets, perm, h_rows, y_rows, shared_y, ws, stream=None):
    st = lib().moe_expert_ffn(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), int(T), _ptr(offsets),
                              _ptr(perm), _ptr(h_rows), _ptr(y_rows), _ptr(shared_y), _ptr(ws),
                              ws.numel(), _stream(stream))
    _check("moe_expert_ffn", st)


def moe_combine(cfg, y_rows, inv, topk_w, shared_y, T, out, stream=None):
    st = lib().moe_combine(ctypes.byref(cfg), _ptr(y_rows), _ptr(inv), _ptr(topk_w),
                           _ptr(shared_y), int(T), _ptr(out), _stream(stream))
    _check("moe_combine", st)


def moe_forward(cfg, w: Weights, x, T, out, x_next, ws, stream=None, resid=None):
    st = lib().moe_forward(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), int(T), _ptr(out),
                           _ptr(resid), _ptr(x_next), _ptr(ws), ws.numel(), _stream(stream))
    _check("moe_forward", st)


class Graph:
    """A layer stack captured by moe_graph_create; launch() replays it.  Holds references to
    every tensor the graph reads or writes, so none is freed while the graph lives."""

    def __init__(self, cfg, layers, T, x0, out, x_last, scratch, ws, stream=None, resid=None, keep=()):
        arr = (Weights * len(layers))(*layers)
        h = ctypes.c_void_p()
        st = lib().moe_graph_create(ctypes.byref(cfg), arr, len(layers), int(T), _ptr(x0), _ptr(resid), _ptr(out),
                                    _ptr(x_last), _ptr(scratch), _ptr(ws), ws.numel(), _stream(stream),
                                    ctypes.byref(h))
        _check("moe_graph_create", st)
        self._h = h
        self._keep = (x0, out, x_last, scratch, ws, resid, tuple(keep))

    @property
    def kernels(self) -> int:
        return int(lib().moe_graph_kernel_count(self._h))

    def launch(self, stream=None):
        _check("moe_graph_launch", lib().moe_graph_launch(self._h, _stream(stream)))

    def destroy(self):
        if self._h is not None and self._h.value:
            lib().moe_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def moe_forward_q8(cfg, w, x, T, out, x_next, ws, stream=None, resid=None):
    """The layer with E4M3 expert weights (a WeightsQ8): x [T,H] -> out (and x_next)."""
    st = lib().moe_forward_q8(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), int(T), _ptr(out), _ptr(resid),
                              _ptr(x_next), _ptr(ws), ws.numel(), _stream(stream))
    _check("moe_forward_q8", st)


def moe_decode_chain(cfg, layers, x0, out, x_last, ws, stream=None, resid=None):
    """One token through len(layers) layers (a list of Weights) in one launch."""
    arr = (Weights * len(layers))(*layers)
    st = lib().moe_decode_chain(ctypes.byref(cfg), arr, len(layers), _ptr(x0), _ptr(resid), _ptr(out),
                                _ptr(x_last), _ptr(ws), ws.numel(), _stream(stream))
    _check("moe_decode_chain", st)


def moe_decode_chain_q8(cfg, layers_q8, x0, out, x_last, ws, stream=None, resid=None):
    """One token through len(layers_q8) layers with E4M3 expert weights (WeightsQ8 list)."""
    arr = (WeightsQ8 * len(layers_q8))(*layers_q8)
    st = lib().moe_decode_chain_q8(ctypes.byref(cfg), arr, len(layers_q8), _ptr(x0), _ptr(resid), _ptr(out),
                                   _ptr(x_last), _ptr(ws), ws.numel(), _stream(stream))
    _check("moe_decode_chain_q8", st)


def moe_decode_chain_q4(cfg, layers_q4, x0, out, x_last, ws, stream=None, resid=None):
    """One token through len(layers_q4) layers with 4-bit expert weights (WeightsQ4 list)."""
    arr = (WeightsQ4 * len(layers_q4))(*layers_q4)
    st = lib().moe_decode_chain_q4(ctypes.byref(cfg), arr, len(layers_q4), _ptr(x0), _ptr(resid), _ptr(out),
                                   _ptr(x_last), _ptr(ws), ws.numel(), _stream(stream))
    _check("moe_decode_chain_q4", st)


def moe_quantize_q4(w, q, scale, stream=None):
    """Block-wise 4-bit codes q (uint8, w's shape with the last dimension halved) and fp32 scales
    (w's shape with the last dimension / 32) of a bf16 w whose last dimension is the row."""
    rows, cols = (w.numel() // w.shape[-1]) if w.dim() > 1 else 1, w.shape[-1]
    st = lib().moe_quantize_q4(_ptr(w), int(rows), int(cols), _ptr(q), _ptr(scale), _stream(stream))
    _check("moe_quantize_q4", st)


def quantize_layer_q4(layer: dict, stream=None) -> dict:
    """A layer's expert matrices as 4-bit codes and block scales (the router kept as it is), on
    the device, through moe_quantize_q4."""
    out = {"w_router": layer["w_router"], "b_router": layer.get("b_router")}
    for src, q, sc in (("w_gate", "q_gate", "s_gate"), ("w_up", "q_up", "s_up"), ("w_down", "q_down", "s_down"),
                       ("ws_gate", "qs_gate", "ss_gate"), ("ws_up", "qs_up", "ss_up"),
                       ("ws_down", "qs_down", "ss_down")):
        w = layer.get(src)
        if w is None:
            continue
        out[q] = torch.empty(w.shape[:-1] + (w.shape[-1] // 2,), dtype=torch.uint8, device=w.device)
        out[sc] = torch.empty(w.shape[:-1] + (w.shape[-1] // 32,), dtype=torch.float32, device=w.device)
        moe_quantize_q4(w, out[q], out[sc], stream)
    return out


def moe_quantize_e4m3(w, q, scale, stream=None):
    """Row-wise E4M3 codes q (uint8, w's shape) and fp32 scales (one per row) of a bf16 w whose
    last dimension is the row."""
    rows, cols = (w.numel() // w.shape[-1]) if w.dim() > 1 else 1, w.shape[-1]
    st = lib().moe_quantize_e4m3(_ptr(w), int(rows), int(cols), _ptr(q), _ptr(scale), _stream(stream))
    _check("moe_quantize_e4m3", st)


def quantize_layer(layer: dict, stream=None) -> dict:
    """A layer's expert matrices as E4M3 codes and row scales (the router kept as it is), on the
    device, through moe_quantize_e4m3."""
    out = {"w_router": layer["w_router"], "b_router": layer.get("b_router")}
    for src, q, sc in (("w_gate", "q_gate", "s_gate"), ("w_up", "q_up", "s_up"), ("w_down", "q_down", "s_down"),
                       ("ws_gate", "qs_gate", "ss_gate"), ("ws_up", "qs_up", "ss_up"),
                       ("ws_down", "qs_down", "ss_down")):
        w = layer.get(src)
        if w is None:
            continue
        out[q] = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
        out[sc] = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
        moe_quantize_e4m3(w, out[q], out[sc], stream)
    return out


def moe_forward_status(cfg, w: Weights, x, T, out, x_next, ws, stream=None, resid=None) -> int:
    """Like moe_forward but returns the status code instead of raising."""
    return int(lib().moe_forward(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), int(T), _ptr(out),
                                 _ptr(resid), _ptr(x_next), _ptr(ws), ws.numel(), _stream(stream)))


def moe_check_status(ws, stream=None) -> int:
    v = ctypes.c_int(0)
    st = lib().moe_check_status(_ptr(ws), ws.numel(), ctypes.byref(v), _stream(stream))
    _check("moe_check_status", st)
    return v.value


def moe_selftest_wait(ws, limit_ns: int, arrive: bool, stream=None):
    """Run the library's bounded device wait on a barrier that completes (arrive) or never does."""
    st = lib().moe_selftest_wait(_ptr(ws), ws.numel(), int(limit_ns), 1 if arrive else 0, _stream(stream))
    _check("moe_selftest_wait", st)


def moe_plan_pieces(T: int):
    n = lib().moe_plan_pieces(int(T), None, 0)
    if n < 0:
        raise ValueError("T < 0")
    buf = (ctypes.c_int * max(n, 1))()
    lib().moe_plan_pieces(int(T), buf, n)
    return [buf[i] for i in range(n)]


def moe_launch_count() -> int:
    return int(lib().moe_launch_count())


def timing_enable(on: bool):
    lib().moe_timing_enable(1 if on else 0)


def timing_classes():
    L = lib()
    return [L.moe_timing_name(i).decode() for i in range(L.moe_timing_classes())]


def timing_read(name: str):
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    st = lib().moe_timing_read(name.encode(), ctypes.byref(n), ctypes.byref(ms))
    _check("moe_timing_read", st)
    return n.value, ms.value


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()
