"""Seeded synthetic inputs for the MoE layer workloads.

This module draws random numbers and nothing else: it holds none of the layer's arithmetic
(no routing, no FFN, no rounding beyond storing fp32 draws as bf16).  Both the CUDA path and
the CPU oracle consume exactly the bytes it returns.

The pages measure only whole-model runs of a trained checkpoint (no layer-level workload and
no public dataset at layer level), so every workload here is synthetic, with the layer shape
of the pages' Qwen3.6-35B-A3B-class engines.

Recipe (per workload, one ``torch.Generator`` seeded with the workload's seed, on the device
the caller names):
  for each layer l, in this order:
    W_r [E,H]  ~ N(0, router_std)          (router_std = 0.02, or 1/sqrt(H) so logits ~ N(0,1))
    b   [E]    = -s * ln(rank_e)            (Zipf workloads only; rank = randperm(E) + 1;
                                             the last ``n_dead`` ranks get b = -30)
    W_g [E,I,H], W_u [E,I,H], W_d [E,H,I]  ~ N(0, 0.02)
    W_sg [Is,H], W_su [Is,H], W_sd [H,Is]  ~ N(0, 0.02)
  then x [T,H] ~ N(0, 1).
Every draw is fp32 rounded to bf16 (round to nearest even); the bias stays fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass(frozen=True)
class Shape:
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    T: int
    n_layers: int
    seed: int
    router_std: float
    zipf_s: Optional[float] = None
    n_dead: int = 0
    w_std: float = 0.02
    x_std: float = 1.0
    note: str = field(default="", compare=False)


_QWEN_MOE = Shape(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512)

WORKLOADS = {
    "tiny": Workload("tiny", Shape(256, 16, 4, 128, 128), T=64, n_layers=1, seed=0,
                     router_std=0.02, note="T=64, H=256, E=16, top-4, I=Is=128"),
    "decode": Workload("decode", _QWEN_MOE, T=1, n_layers=40, seed=1,
                       router_std=1.0 / math.sqrt(2048),
                       note="T=1, 40 distinct layers (~64.7 GB of weights)"),
    "prefill1k": Workload("prefill1k", _QWEN_MOE, T=1024, n_layers=1, seed=2,
                          router_std=1.0 / math.sqrt(2048), zipf_s=1.0,
                          note="T=1024, Zipf(1.0) expert popularity"),
    "prefill8k": Workload("prefill8k", _QWEN_MOE, T=8192, n_layers=4, seed=3,
                          router_std=1.0 / math.sqrt(2048),
                          note="T=8192, uniform routing, 4 distinct layers"),
    "prompt13337": Workload("prompt13337", _QWEN_MOE, T=13337, n_layers=4, seed=4,
                            router_std=1.0 / math.sqrt(2048), zipf_s=1.5, n_dead=4,
                            note="T=13337, Zipf(1.5), 4 experts never chosen, 4 layers"),
}


def _normal_bf16(gen, shape, std, device):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(mean=0.0, std=std, generator=gen)
    return t.to(torch.bfloat16)


def _make_router(w: Workload, gen: torch.Generator, device) -> dict:
    E, H = w.shape.n_experts, w.shape.hidden
    layer = {"w_router": _normal_bf16(gen, (E, H), w.router_std, device)}
    if w.zipf_s is not None:
        rank = torch.randperm(E, generator=gen, device=device).to(torch.float64) + 1.0
        b = -w.zipf_s * torch.log(rank)
        if w.n_dead:
            b[rank > E - w.n_dead] = -30.0
        layer["b_router"] = b.to(torch.float32)
    else:
        layer["b_router"] = None
    return layer


def make_layer(w: Workload, gen: torch.Generator, device) -> dict:
    """Draw one layer's weights (see the module docstring for the order)."""
    s = w.shape
    H, E, I, Is = s.hidden, s.n_experts, s.inter, s.shared_inter
    layer = _make_router(w, gen, device)
    layer["w_gate"] = _normal_bf16(gen, (E, I, H), w.w_std, device)
    layer["w_up"] = _normal_bf16(gen, (E, I, H), w.w_std, device)
    layer["w_down"] = _normal_bf16(gen, (E, H, I), w.w_std, device)
    if Is > 0:
        layer["ws_gate"] = _normal_bf16(gen, (Is, H), w.w_std, device)
        layer["ws_up"] = _normal_bf16(gen, (Is, H), w.w_std, device)
        layer["ws_down"] = _normal_bf16(gen, (H, Is), w.w_std, device)
    else:
        layer["ws_gate"] = layer["ws_up"] = layer["ws_down"] = None
    return layer


def make(w: Workload, device="cpu", n_layers: Optional[int] = None, T: Optional[int] = None):
    """All layers and the input x for a workload: (list of layer dicts, x [T,H] bf16).

    ``n_layers`` / ``T`` may shrink the workload (same recipe, same seed) for quick checks.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    L = w.n_layers if n_layers is None else n_layers
    layers = [make_layer(w, gen, device) for _ in range(L)]
    TT = w.T if T is None else T
    x = _normal_bf16(gen, (TT, w.shape.hidden), w.x_std, device)
    return layers, x


def _e4m3_codes(gen, shape, device):
    """Uniform draws over the 254 finite E4M3 bit patterns (0x7F and 0xFF, the NaNs, excluded).
    Bit patterns only: nothing here decodes them."""
    c = torch.randint(0, 254, shape, generator=gen, device=device, dtype=torch.int32)
    c = c + (c >= 0x7F).to(torch.int32)                # skip 0x7F
    return c.to(torch.uint8)


def _scales(gen, shape, base, device):
    s = torch.empty(shape, dtype=torch.float32, device=device)
    s.uniform_(0.5 * base, 1.5 * base, generator=gen)
    return s


def make_q8(w: Workload, device="cpu", n_layers: Optional[int] = None, T: Optional[int] = None,
            scale_base: float = 2e-4):
    """Layers with E4M3 expert weights and the input x, for the quantised-weight path.

    Per layer, in this order: W_r and b as in ``make_layer``; then for W_g, W_u, W_d and the shared
    expert's three matrices, the codes (uniform over the finite bit patterns) followed by one fp32
    scale per row, uniform in [0.5, 1.5] * scale_base.  Uniform codes have an RMS value near 100, so
    the default base puts the dequantised weights near the bf16 workloads' 0.02.  Then x ~ N(0, 1).
    Keys: w_router, b_router, q_gate/q_up/q_down with s_gate/s_up/s_down, and qs_*/ss_* for the
    shared expert (absent when I_s = 0).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    s = w.shape
    H, E, I, Is = s.hidden, s.n_experts, s.inter, s.shared_inter
    layers = []
    for _ in range(w.n_layers if n_layers is None else n_layers):
        layer = _make_router(w, gen, device)
        mats = [("q_gate", "s_gate", (E, I, H)), ("q_up", "s_up", (E, I, H)), ("q_down", "s_down", (E, H, I))]
        if Is > 0:
            mats += [("qs_gate", "ss_gate", (Is, H)), ("qs_up", "ss_up", (Is, H)), ("qs_down", "ss_down", (H, Is))]
        for qn, sn, shp in mats:
            layer[qn] = _e4m3_codes(gen, shp, device)
            layer[sn] = _scales(gen, shp[:-1], scale_base, device)
        layers.append(layer)
    TT = w.T if T is None else T
    x = _normal_bf16(gen, (TT, w.shape.hidden), w.x_std, device)
    return layers, x


def _q4_bytes(gen, shape, device):
    """Bytes of two 4-bit fields each uniform over the 15 patterns other than 8 (0b1000): bit
    patterns only, nothing here decodes them."""
    lo = torch.randint(0, 15, shape, generator=gen, device=device, dtype=torch.int32)
    hi = torch.randint(0, 15, shape, generator=gen, device=device, dtype=torch.int32)
    lo = lo + (lo >= 8).to(torch.int32)
    hi = hi + (hi >= 8).to(torch.int32)
    return (lo | (hi << 4)).to(torch.uint8)


def make_q4(w: Workload, device="cpu", n_layers: Optional[int] = None, T: Optional[int] = None,
            scale_base: float = 5e-3):
    """Layers with 4-bit expert weights and the input x, for the 4-bit path.

    Per layer, in this order: W_r and b as in ``make_layer``; then for W_g, W_u, W_d and the shared
    expert's three matrices, the packed codes (each 4-bit field uniform over the 15 patterns other
    than 0b1000) followed by one fp32 scale per block of 32 columns, uniform in [0.5, 1.5] *
    scale_base.  The default base puts the weights near the bf16 workloads' 0.02.  Then x ~ N(0, 1).
    Keys as in ``make_q8``: codes [rows, cols/2], scales [rows, cols/32].
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    s = w.shape
    H, E, I, Is = s.hidden, s.n_experts, s.inter, s.shared_inter
    layers = []
    for _ in range(w.n_layers if n_layers is None else n_layers):
        layer = _make_router(w, gen, device)
        mats = [("q_gate", "s_gate", (E, I, H)), ("q_up", "s_up", (E, I, H)), ("q_down", "s_down", (E, H, I))]
        if Is > 0:
            mats += [("qs_gate", "ss_gate", (Is, H)), ("qs_up", "ss_up", (Is, H)), ("qs_down", "ss_down", (H, Is))]
        for qn, sn, shp in mats:
            layer[qn] = _q4_bytes(gen, shp[:-1] + (shp[-1] // 2,), device)
            layer[sn] = _scales(gen, shp[:-1] + (shp[-1] // 32,), scale_base, device)
        layers.append(layer)
    TT = w.T if T is None else T
    x = _normal_bf16(gen, (TT, w.shape.hidden), w.x_std, device)
    return layers, x


def custom(shape: Shape, T: int, seed: int, router_std: float = 0.02, zipf_s=None,
           n_dead: int = 0, n_layers: int = 1, name: str = "custom") -> Workload:
    return Workload(name, shape, T=T, n_layers=n_layers, seed=seed, router_std=router_std,
                    zipf_s=zipf_s, n_dead=n_dead)


def to_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    import numpy as np
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def layer_to_host(layer: dict) -> dict:
    """Host copy of a layer dict in the oracle's representation (uint16 / float32)."""
    out = {}
    for k, v in layer.items():
        if v is None:
            continue
        if v.dtype == torch.bfloat16:
            out[k] = to_u16(v)
        else:
            out[k] = v.detach().cpu().numpy()
    return out
