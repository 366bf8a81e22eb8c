"""CPU-only checks of the C-ABI library: it loads, exports every symbol include/moe.h
declares, and validates arguments on the host before any device work.  No test here
launches a kernel or touches device memory."""
import ctypes
import os
import re
import subprocess

import pytest

from sparse_moe_router_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for fn in ("moe_route", "moe_route_from_logits", "moe_permute", "moe_expert_ffn", "moe_combine",
               "moe_forward", "moe_workspace_size", "moe_status_string"):
        assert fn in names
    assert sorted(abi.EXPORTS) == names


def test_library_exports_every_declared_symbol():
    L = abi.load()
    for fn in _declared():
        assert hasattr(L, fn), fn
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True, text=True)
    if out.returncode == 0:
        syms = set(line.split()[-1] for line in out.stdout.splitlines() if line.strip())
        for fn in _declared():
            assert fn in syms, fn


def _cfg(**kw):
    d = dict(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512)
    d.update(kw)
    return abi.config(**d)


def test_workspace_size_and_config_validation():
    L = abi.load()
    n1 = abi.workspace_size(_cfg(), 1)
    n8 = abi.workspace_size(_cfg(), 8192)
    assert 0 < n1 < n8
    # T*k*I*2 (h) + T*H*4 (acc) + T*Is*2 dominate
    assert n8 >= 8192 * 8 * 512 * 2 + 8192 * 2048 * 4
    for bad in (_cfg(top_k=0), _cfg(top_k=300), _cfg(hidden=0), _cfg(shared_inter=-1)):
        assert abi.workspace_size(bad, 16) == 0
    for unsup in (_cfg(hidden=100), _cfg(inter=96), _cfg(top_k=33, n_experts=64), _cfg(n_experts=2000)):
        assert abi.workspace_size(unsup, 16) == 0
    assert L.moe_workspace_size(None, 16) == 0
    assert abi.workspace_size(_cfg(), -1) == 0


def test_entry_points_reject_bad_arguments_without_device_work():
    L = abi.load()
    cfg = _cfg()
    w = abi.Weights()
    P = ctypes.c_void_p
    fake = P(0x10000)          # never dereferenced: validation fails first
    # null config / null pointers / negative T
    assert L.moe_forward(None, ctypes.byref(w), fake, 4, fake, None, None, fake, 1 << 30, None) == 1
    assert L.moe_forward(ctypes.byref(cfg), ctypes.byref(w), fake, 4, fake, None, None, fake, 1 << 30, None) == 1
    assert L.moe_forward(ctypes.byref(cfg), ctypes.byref(w), fake, -1, fake, None, None, fake, 1 << 30, None) == 1
    assert L.moe_route_from_logits(ctypes.byref(cfg), None, 5, fake, fake, None) == 1
    assert L.moe_permute(ctypes.byref(cfg), fake, 5, None, fake, fake, fake, 1 << 30, None) == 1
    assert L.moe_combine(ctypes.byref(cfg), None, fake, fake, None, 3, fake, None) == 1
    # unsupported shape
    assert L.moe_route_from_logits(ctypes.byref(_cfg(top_k=40, n_experts=64)), fake, 5, fake, fake, None) == 3
    # T == 0 is a no-op that succeeds, even with null tensors
    assert L.moe_forward(ctypes.byref(cfg), None, None, 0, None, None, None, None, 0, None) == 0
    assert L.moe_permute(ctypes.byref(cfg), None, 0, None, None, None, None, 0, None) == 0
    # workspace checks: misaligned, too small
    wt = abi.Weights(*(0x10000 for _ in range(8)))
    assert L.moe_forward(ctypes.byref(cfg), ctypes.byref(wt), fake, 4, fake, None, None, P(0x10010), 1 << 30, None) == 1
    assert L.moe_forward(ctypes.byref(cfg), ctypes.byref(wt), fake, 4, fake, None, None, fake, 1000, None) == 2
    # misaligned tensor
    assert L.moe_forward(ctypes.byref(cfg), ctypes.byref(wt), P(0x10002), 4, fake, None, None, fake, 1 << 30, None) == 1
    # missing shared-expert weights when Is > 0
    wn = abi.Weights(*(0x10000 for _ in range(5)), None, None, None)
    assert L.moe_forward(ctypes.byref(cfg), ctypes.byref(wn), fake, 4, fake, None, None, fake, 1 << 30, None) == 1


def test_plan_pieces():
    assert abi.moe_plan_pieces(13337) == [8192, 4096, 1024, 25]
    assert abi.moe_plan_pieces(8192) == [8192]
    assert abi.moe_plan_pieces(1) == [1]
    assert abi.moe_plan_pieces(0) == []
    assert abi.moe_plan_pieces(16383) == [8192, 4096, 2048, 1024, 1023]
    assert abi.moe_plan_pieces(3 * 8192 + 1024) == [8192, 8192, 8192, 1024]
    for T in range(0, 40000, 997):
        assert sum(abi.moe_plan_pieces(T)) == T
    with pytest.raises(ValueError):
        abi.moe_plan_pieces(-5)


def test_status_strings_and_timing_names():
    assert abi.status_string(0) == "ok"
    assert abi.status_string(2) == "workspace too small"
    names = abi.timing_classes()
    assert "gateup_gemm" in names and "decode_experts" in names
    with pytest.raises(abi.MoeError):
        abi.timing_read("no_such_kernel")


def test_graph_entry_points_validate_on_the_host():
    """moe_graph_*: argument errors are returned before any device work."""
    L = abi.load()
    cfg = _cfg()
    w = (abi.Weights * 2)()
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(0x1000)
    # no handle pointer, no layers, no layers counted, no tokens
    assert L.moe_graph_create(cfg, w, 1, 8, fake, None, fake, None, None, fake, 1 << 20, None, None) == 1
    assert L.moe_graph_create(cfg, None, 1, 8, fake, None, fake, None, None, fake, 1 << 20, None, ctypes.byref(h)) == 1
    assert L.moe_graph_create(cfg, w, 0, 8, fake, None, fake, None, None, fake, 1 << 20, None, ctypes.byref(h)) == 1
    assert L.moe_graph_create(cfg, w, 1, 0, fake, None, fake, None, None, fake, 1 << 20, None, ctypes.byref(h)) == 1
    # a stack needs x_last and scratch, distinct from each other and from x0 / out
    assert L.moe_graph_create(cfg, w, 2, 8, fake, None, fake, None, fake, fake, 1 << 20, None, ctypes.byref(h)) == 1
    a, b = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    assert L.moe_graph_create(cfg, w, 2, 8, fake, None, b, a, a, fake, 1 << 20, None, ctypes.byref(h)) == 1
    assert L.moe_graph_create(cfg, w, 2, 8, fake, None, b, fake, a, fake, 1 << 20, None, ctypes.byref(h)) == 1
    assert L.moe_graph_create(cfg, w, 65, 8, fake, None, b, a, ctypes.c_void_p(0x4000), fake, 1 << 20, None,
                              ctypes.byref(h)) == 3
    assert not h.value
    assert L.moe_graph_launch(None, None) == 1
    assert L.moe_graph_kernel_count(None) == -1
    assert L.moe_graph_destroy(None) == 0


def test_forward_q8_validates_on_the_host():
    """moe_forward_q8 rejects a bad call before any device work: null/incomplete weights, a
    missing shared expert's codes or scales, misaligned codes, a bad workspace; T == 0 succeeds."""
    L = abi.load()
    cfg = _cfg()
    P = ctypes.c_void_p
    fake = P(0x10000)
    full = abi.WeightsQ8(*(0x10000 for _ in range(14)))
    assert L.moe_forward_q8(ctypes.byref(cfg), None, fake, 4, fake, None, None, fake, 1 << 30, None) == 1
    assert L.moe_forward_q8(ctypes.byref(cfg), None, None, 0, None, None, None, None, 0, None) == 0
    assert L.moe_forward_q8(ctypes.byref(cfg), ctypes.byref(full), fake, -2, fake, None, None, fake, 1 << 30, None) == 1
    for field in ("q_gate", "s_down", "qs_up", "ss_down"):
        w = abi.WeightsQ8(*(0x10000 for _ in range(14)))
        setattr(w, field, None)
        assert L.moe_forward_q8(ctypes.byref(cfg), ctypes.byref(w), fake, 4, fake, None, None, fake, 1 << 30, None) == 1
    w = abi.WeightsQ8(*(0x10000 for _ in range(14)))
    w.q_down = 0x10008  # codes must be 16-byte aligned
    assert L.moe_forward_q8(ctypes.byref(cfg), ctypes.byref(w), fake, 4, fake, None, None, fake, 1 << 30, None) == 1
    assert L.moe_forward_q8(ctypes.byref(cfg), ctypes.byref(full), fake, 4, fake, None, None, fake, 1000, None) == 2
    assert L.moe_forward_q8(ctypes.byref(cfg), ctypes.byref(full), fake, 4, fake, None, None, P(0x10010),
                            1 << 30, None) == 1
    # no shared expert: its pointers may be NULL
    cfg0 = _cfg(shared_inter=0)
    w0 = abi.WeightsQ8(*(0x10000 for _ in range(8)), None, None, None, None, None, None)
    assert L.moe_forward_q8(ctypes.byref(cfg0), ctypes.byref(w0), fake, 4, fake, None, None, fake, 1000, None) == 2
