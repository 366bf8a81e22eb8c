"""ctypes wrapper around the plain C oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's CPU
baseline leg, never by the product path.  Arrays are numpy; bf16 tensors travel as their
uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build_oracle

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        _lib = ctypes.CDLL(path)
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int


def _declare(L):
    L.moe_ref_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.moe_ref_bf16_to_double.restype = ctypes.c_double
    L.moe_ref_double_to_bf16.argtypes = [ctypes.c_double]
    L.moe_ref_double_to_bf16.restype = ctypes.c_uint16
    L.moe_ref_silu.argtypes = [ctypes.c_double]
    L.moe_ref_silu.restype = ctypes.c_double
    L.moe_ref_router_logits.argtypes = [_I, _I, _I, _P, _P, _P, _P]
    L.moe_ref_router_logits.restype = None
    L.moe_ref_route_from_logits.argtypes = [_I, _I, _I, _P, _P, _P]
    L.moe_ref_route_from_logits.restype = None
    L.moe_ref_permute.argtypes = [_I, _I, _I, _P, _P, _P, _P]
    L.moe_ref_permute.restype = _I
    L.moe_ref_expert_ffn.argtypes = [_I] * 6 + [_P] * 13
    L.moe_ref_expert_ffn.restype = None
    L.moe_ref_combine.argtypes = [_I, _I, _I, _P, _P, _P, _P, _P]
    L.moe_ref_combine.restype = None
    L.moe_ref_forward.argtypes = ([_I] * 6 + [_P] * 11 + [_I, _I] + [_P] * 5)
    L.moe_ref_forward.restype = None
    L.moe_ref_dense_masked.argtypes = [_I] * 6 + [_P] * 9 + [_I, _P]
    L.moe_ref_dense_masked.restype = None
    L.moe_ref_threads.argtypes = [_I]
    L.moe_ref_threads.restype = _I
    L.moe_ref_e4m3_to_double.argtypes = [ctypes.c_uint8]
    L.moe_ref_e4m3_to_double.restype = ctypes.c_double
    L.moe_ref_float_to_e4m3.argtypes = [ctypes.c_float]
    L.moe_ref_float_to_e4m3.restype = ctypes.c_uint8
    L.moe_ref_quantize_e4m3_rows.argtypes = [_I, _I, _P, _P, _P]
    L.moe_ref_quantize_e4m3_rows.restype = None
    L.moe_ref_forward_q8.argtypes = [_I] * 6 + [_P] * 16
    L.moe_ref_forward_q8.restype = None
    L.moe_ref_quantize_q4_rows.argtypes = [_I, _I, _P, _P, _P]
    L.moe_ref_quantize_q4_rows.restype = None
    L.moe_ref_q4_code.argtypes = [_P, _I]
    L.moe_ref_q4_code.restype = _I
    L.moe_ref_forward_q4.argtypes = [_I] * 6 + [_P] * 16
    L.moe_ref_forward_q4.restype = None


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def bf16_to_f64(bits):
    """bf16 bit patterns -> float64 (exact), vectorised."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def double_to_bf16(v):
    return lib().moe_ref_double_to_bf16(float(v))


def silu(g):
    return lib().moe_ref_silu(float(g))


def router_logits(x, w_router, b_router=None):
    x, w_router = _u16(x), _u16(w_router)
    T, H = x.shape
    E = w_router.shape[0]
    b = _f32(b_router)
    out = np.empty((T, E), dtype=np.float32)
    lib().moe_ref_router_logits(H, E, T, _ptr(x), _ptr(w_router), _ptr(b), _ptr(out))
    return out


def route_from_logits(logits, k):
    logits = _f32(logits)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    lib().moe_ref_route_from_logits(E, k, T, _ptr(logits), _ptr(ids), _ptr(w))
    return ids, w


def permute(ids, E):
    ids = _i32(ids)
    T, k = ids.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    rc = lib().moe_ref_permute(E, k, T, _ptr(ids), _ptr(offsets), _ptr(perm), _ptr(inv))
    if rc != 0:
        raise ValueError("expert id out of range")
    return offsets, perm, inv


def expert_ffn(x, offsets, perm, k, w, h_in=None, want_shared=True):
    """Routed rows (permuted order) and the shared expert, unfused.

    ``w`` is a dict of uint16 arrays: w_gate [E,I,H], w_up, w_down [E,H,I], and optionally
    ws_gate [Is,H], ws_up, ws_down [H,Is].  Returns (h_rows [P,I] u16, y_rows [P,H] f32,
    shared_y [T,H] f32 or None).
    """
    x = _u16(x)
    T, H = x.shape
    wg, wu, wd = _u16(w["w_gate"]), _u16(w["w_up"]), _u16(w["w_down"])
    E, I, _ = wg.shape
    sg, su, sd = _u16(w.get("ws_gate")), _u16(w.get("ws_up")), _u16(w.get("ws_down"))
    Is = 0 if sg is None else sg.shape[0]
    offsets, perm = _i32(offsets), _i32(perm)
    P = T * k
    h_rows = np.empty((P, I), dtype=np.uint16)
    y_rows = np.empty((P, H), dtype=np.float32)
    shared_y = np.empty((T, H), dtype=np.float32) if (want_shared and Is > 0) else None
    h_in = _u16(h_in)
    lib().moe_ref_expert_ffn(H, E, k, I, Is, T, _ptr(x), _ptr(offsets), _ptr(perm), _ptr(wg),
                             _ptr(wu), _ptr(wd), _ptr(sg), _ptr(su), _ptr(sd), _ptr(h_in),
                             _ptr(h_rows), _ptr(y_rows), _ptr(shared_y))
    return h_rows, y_rows, shared_y


def combine(y_rows, inv, topk_w, shared_y=None):
    y_rows = _f32(y_rows)
    topk_w = _f32(topk_w)
    T, k = topk_w.shape
    H = y_rows.shape[1]
    inv = _i32(inv)
    shared_y = _f32(shared_y)
    out = np.empty((T, H), dtype=np.uint16)
    lib().moe_ref_combine(H, k, T, _ptr(y_rows), _ptr(inv), _ptr(topk_w), _ptr(shared_y), _ptr(out))
    return out


def forward(x, w, k, ids=None, topk_w=None, exact=False, n_threads=0, want_f64=False,
            want_x_next=False):
    """The whole layer, token by token.

    ``w`` holds uint16 arrays w_router [E,H], w_gate, w_up [E,I,H], w_down [E,H,I], the
    optional shared-expert arrays, and an optional float32 b_router [E].  When ``ids`` and
    ``topk_w`` are given they replace the oracle's own routing.  Returns a dict with out
    (u16 [T,H]), ids, w and optionally out_f64 and x_next.
    """
    x = _u16(x)
    T, H = x.shape
    wr = _u16(w["w_router"])
    wg, wu, wd = _u16(w["w_gate"]), _u16(w["w_up"]), _u16(w["w_down"])
    E, I, _ = wg.shape
    sg, su, sd = _u16(w.get("ws_gate")), _u16(w.get("ws_up")), _u16(w.get("ws_down"))
    Is = 0 if sg is None else sg.shape[0]
    b = _f32(w.get("b_router"))
    ids_in, w_in = _i32(ids), _f32(topk_w)
    out = np.empty((T, H), dtype=np.uint16)
    out_f64 = np.empty((T, H), dtype=np.float64) if want_f64 else None
    x_next = np.empty((T, H), dtype=np.uint16) if want_x_next else None
    ids_out = np.empty((T, k), dtype=np.int32)
    w_out = np.empty((T, k), dtype=np.float32)
    lib().moe_ref_forward(H, E, k, I, Is, T, _ptr(x), _ptr(wr), _ptr(b), _ptr(wg), _ptr(wu),
                          _ptr(wd), _ptr(sg), _ptr(su), _ptr(sd), _ptr(ids_in), _ptr(w_in),
                          1 if exact else 0, int(n_threads), _ptr(out), _ptr(out_f64),
                          _ptr(x_next), _ptr(ids_out), _ptr(w_out))
    res = {"out": out, "ids": ids_out, "w": w_out}
    if want_f64:
        res["out_f64"] = out_f64
    if want_x_next:
        res["x_next"] = x_next
    return res


def dense_masked(x, w, ids, topk_w, exact=False):
    x = _u16(x)
    T, H = x.shape
    wg, wu, wd = _u16(w["w_gate"]), _u16(w["w_up"]), _u16(w["w_down"])
    E, I, _ = wg.shape
    sg, su, sd = _u16(w.get("ws_gate")), _u16(w.get("ws_up")), _u16(w.get("ws_down"))
    Is = 0 if sg is None else sg.shape[0]
    ids, topk_w = _i32(ids), _f32(topk_w)
    k = ids.shape[1]
    out = np.empty((T, H), dtype=np.float64)
    lib().moe_ref_dense_masked(H, E, k, I, Is, T, _ptr(x), _ptr(wg), _ptr(wu), _ptr(wd),
                               _ptr(sg), _ptr(su), _ptr(sd), _ptr(ids), _ptr(topk_w),
                               1 if exact else 0, _ptr(out))
    return out


def threads(n_threads=0):
    return lib().moe_ref_threads(int(n_threads))


# ---------------------------------------------------------- quantised expert weights --

def e4m3_to_f64(codes):
    """E4M3 byte codes -> float64 values (the C oracle's decoder, element by element)."""
    c = np.asarray(codes, dtype=np.uint8)
    f = lib().moe_ref_e4m3_to_double
    return np.array([f(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def float_to_e4m3(v):
    return int(lib().moe_ref_float_to_e4m3(float(v)))


def quantize_e4m3_rows(w):
    """bf16 bits [rows, cols] -> (E4M3 codes uint8 [rows, cols], fp32 scales [rows])."""
    w = _u16(w)
    rows, cols = w.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty(rows, dtype=np.float32)
    lib().moe_ref_quantize_e4m3_rows(rows, cols, _ptr(w), _ptr(q), _ptr(s))
    return q, s


def forward_q8(x, wq, k, ids, topk_w):
    """The layer with quantised expert weights on a given routing.  ``wq`` holds uint8 codes
    q_gate, q_up [E,I,H], q_down [E,H,I] with float32 scales s_gate, s_up [E,I], s_down [E,H],
    and optionally the shared expert's qs_gate, qs_up [Is,H], qs_down [H,Is] with ss_gate,
    ss_up [Is], ss_down [H].  Returns out (u16 [T,H])."""
    x = _u16(x)
    T, H = x.shape
    u8 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.uint8)
    qg, qu, qd = u8(wq["q_gate"]), u8(wq["q_up"]), u8(wq["q_down"])
    E, I, _ = qg.shape
    sg, su, sd = _f32(wq["s_gate"]), _f32(wq["s_up"]), _f32(wq["s_down"])
    qsg, qsu, qsd = u8(wq.get("qs_gate")), u8(wq.get("qs_up")), u8(wq.get("qs_down"))
    ssg, ssu, ssd = _f32(wq.get("ss_gate")), _f32(wq.get("ss_up")), _f32(wq.get("ss_down"))
    Is = 0 if qsg is None else qsg.shape[0]
    ids, topk_w = _i32(ids), _f32(topk_w)
    out = np.empty((T, H), dtype=np.uint16)
    lib().moe_ref_forward_q8(H, E, k, I, Is, T, _ptr(x), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su), _ptr(qd),
                             _ptr(sd), _ptr(qsg), _ptr(ssg), _ptr(qsu), _ptr(ssu), _ptr(qsd), _ptr(ssd),
                             _ptr(ids), _ptr(topk_w), _ptr(out))
    return out


def quantize_q4_rows(w):
    """bf16 bits [rows, cols] (cols % 32 == 0) -> (packed 4-bit codes uint8 [rows, cols/2], fp32
    block scales [rows, cols/32])."""
    w = _u16(w)
    rows, cols = w.shape
    q = np.empty((rows, cols // 2), dtype=np.uint8)
    s = np.empty((rows, cols // 32), dtype=np.float32)
    lib().moe_ref_quantize_q4_rows(rows, cols, _ptr(w), _ptr(q), _ptr(s))
    return q, s


def q4_codes(q_row):
    """The signed codes of one packed row (the C oracle's decoder, nibble by nibble)."""
    r = np.ascontiguousarray(q_row, dtype=np.uint8)
    f = lib().moe_ref_q4_code
    return np.array([f(_ptr(r), c) for c in range(2 * r.size)], dtype=np.int64)


def forward_q4(x, wq, k, ids, topk_w):
    """The layer with Q4 expert weights on a given routing.  ``wq`` holds packed codes q_gate,
    q_up [E,I,H/2], q_down [E,H,I/2] with float32 block scales s_gate, s_up [E,I,H/32], s_down
    [E,H,I/32], and optionally the shared expert's qs_gate, qs_up [Is,H/2], qs_down [H,Is/2]
    with ss_gate, ss_up [Is,H/32], ss_down [H,Is/32].  Returns out (u16 [T,H])."""
    x = _u16(x)
    T, H = x.shape
    u8 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.uint8)
    qg, qu, qd = u8(wq["q_gate"]), u8(wq["q_up"]), u8(wq["q_down"])
    E, I = qg.shape[0], qg.shape[1]
    sg, su, sd = _f32(wq["s_gate"]), _f32(wq["s_up"]), _f32(wq["s_down"])
    qsg, qsu, qsd = u8(wq.get("qs_gate")), u8(wq.get("qs_up")), u8(wq.get("qs_down"))
    ssg, ssu, ssd = _f32(wq.get("ss_gate")), _f32(wq.get("ss_up")), _f32(wq.get("ss_down"))
    Is = 0 if qsg is None else qsg.shape[0]
    ids, topk_w = _i32(ids), _f32(topk_w)
    out = np.empty((T, H), dtype=np.uint16)
    lib().moe_ref_forward_q4(H, E, k, I, Is, T, _ptr(x), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su), _ptr(qd),
                             _ptr(sd), _ptr(qsg), _ptr(ssg), _ptr(qsu), _ptr(ssu), _ptr(qsd), _ptr(ssd),
                             _ptr(ids), _ptr(topk_w), _ptr(out))
    return out
