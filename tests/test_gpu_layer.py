"""GPU parity of the expert FFNs, the combine and the whole layer (moe_forward) against the
CPU oracle, through the C-ABI.

Layer outputs: max |diff| <= 2e-2 and relative L2 <= 5e-3 (bf16 in, fp32 accumulate, bf16
out), with the oracle consuming the GPU's routing (whose ids are first checked bit-exact
against the oracle's selection on the GPU's own logits).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_moe_router_gb300 import abi, inputs

from helpers import (MAX_ABS, REL_L2, cfg_of, check_layer, compare_out, forward_gpu, host, make,
                     route_gpu, u16)

pytestmark = pytest.mark.gpu

TINY = inputs.Shape(256, 16, 4, 128, 128)


def _unfused(shape, layer, x):
    cfg = cfg_of(shape)
    T, k = x.shape[0], shape.top_k
    ws = abi.alloc_workspace(cfg, T)
    logits, ids, w = route_gpu(shape, layer, x, ws=ws)
    ids_d = torch.as_tensor(ids, device="cuda")
    offs = torch.empty(shape.n_experts + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    abi.moe_permute(cfg, ids_d, T, offs, perm, inv, ws)
    h_rows = torch.empty(T * k, shape.inter, dtype=torch.bfloat16, device="cuda")
    y_rows = torch.empty(T * k, shape.hidden, dtype=torch.float32, device="cuda")
    shared_y = torch.empty(T, shape.hidden, dtype=torch.float32, device="cuda") if shape.shared_inter else None
    abi.moe_expert_ffn(cfg, abi.weights(layer), x, T, offs, perm, h_rows, y_rows, shared_y, ws)
    out = torch.empty_like(x)
    w_d = torch.as_tensor(w, device="cuda")
    abi.moe_combine(cfg, y_rows, inv, w_d, shared_y, T, out)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    return dict(ids=ids, w=w, offs=offs.cpu().numpy(), perm=perm.cpu().numpy(), inv=inv.cpu().numpy(),
                h=u16(h_rows), y=y_rows.cpu().numpy(),
                shared_y=None if shared_y is None else shared_y.cpu().numpy(), out=u16(out))


@pytest.mark.parametrize("shape,T", [(TINY, 64), (TINY, 3), (inputs.Shape(512, 32, 4, 256, 0), 200),
                                     (inputs.Shape(1024, 64, 8, 384, 256), 70)])
def test_expert_ffn_and_combine_unfused(shape, T):
    layers, x = make(shape, T, seed=21)
    hl = host(layers[0])
    g = _unfused(shape, layers[0], x)
    o_offs, o_perm, o_inv = orc.permute(g["ids"], shape.n_experts)
    assert np.array_equal(g["offs"], o_offs) and np.array_equal(g["perm"], o_perm)
    assert np.array_equal(g["inv"], o_inv)
    # h rows: bf16 of the SwiGLU, within one bf16 step of the oracle (rounding of a value that
    # differs in the last fp32 bits can land one step apart)
    h_o, _, _ = orc.expert_ffn(u16(x), o_offs, o_perm, shape.top_k, hl, want_shared=False)
    hg, ho = orc.bf16_to_f64(g["h"]), orc.bf16_to_f64(h_o)
    assert np.all(np.abs(hg - ho) <= np.abs(ho) * 2 ** -7 + 1e-6)
    assert np.mean(g["h"] == h_o) > 0.97
    # y rows from the GPU's own h rows (isolates the down projection), shared_y from x
    _, y_o, s_o = orc.expert_ffn(u16(x), o_offs, o_perm, shape.top_k, hl, h_in=g["h"])
    np.testing.assert_allclose(g["y"], y_o, rtol=0, atol=1e-4 + 1e-4 * np.abs(y_o).max())
    if shape.shared_inter:
        np.testing.assert_allclose(g["shared_y"], s_o, rtol=0, atol=2e-3 * max(1.0, np.abs(s_o).max()))
    # combine of the GPU's rows: the fp32 slot-order sum rounds to bf16 once
    out_o = orc.combine(g["y"], g["inv"], g["w"], g["shared_y"])
    d = np.abs(orc.bf16_to_f64(g["out"]) - orc.bf16_to_f64(out_o))
    assert np.all(d <= np.abs(orc.bf16_to_f64(out_o)) * 2 ** -7 + 1e-6)
    compare_out(g["out"], orc.forward(u16(x), hl, shape.top_k, ids=g["ids"], topk_w=g["w"])["out"])


def test_forward_tiny_workload():
    wl = inputs.WORKLOADS["tiny"]
    layers, x = inputs.make(wl, device="cuda")
    ma, rl, mism = check_layer(wl.shape, layers[0], x)
    assert ma <= MAX_ABS and rl <= REL_L2


@pytest.mark.parametrize("T", [1, 2, 3, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 300, 1023, 1024, 1025])
def test_forward_length_sweep(T):
    layers, x = make(TINY, T, seed=100 + T)
    check_layer(TINY, layers[0], x)


@pytest.mark.parametrize("shape", [inputs.Shape(512, 8, 2, 256, 0), inputs.Shape(384, 1, 1, 128, 0),
                                   inputs.Shape(256, 16, 16, 128, 256), inputs.Shape(1024, 128, 1, 128, 128),
                                   # more than 256 experts: the decode top-k stages logits in shared memory
                                   inputs.Shape(256, 600, 8, 128, 128), inputs.Shape(256, 1024, 32, 128, 0)])
def test_forward_shapes(shape):
    layers, x = make(shape, 150, seed=7)
    check_layer(shape, layers[0], x)
    layers1, x1 = make(shape, 1, seed=8)
    check_layer(shape, layers1[0], x1)


@pytest.mark.parametrize("shape,T", [(inputs.Shape(256, 24, 3, 128, 128), 2100),
                                     (inputs.Shape(256, 40, 5, 128, 0), 1300),
                                     (inputs.Shape(512, 64, 6, 128, 128), 1111)])
def test_forward_top_k_not_dividing_the_chunk(shape, T):
    """k = 3, 5, 6: the permutation's chunks are whole tokens (680 / 408 / 336 tokens, 2040 / 2040 /
    2016 pairs), so chunk edges fall inside no token and the top-k kernel's 8-token blocks each land
    in one chunk; several chunks and a ragged last one, through moe_forward (top-k counts, one
    scan+scatter) and through moe_permute (three launches), both against the oracle."""
    layers, x = make(shape, T, seed=70 + shape.top_k)
    check_layer(shape, layers[0], x)
    _, ids, _ = route_gpu(shape, layers[0], x)
    cfg = cfg_of(shape)
    ws = abi.alloc_workspace(cfg, T)
    k = shape.top_k
    offs = torch.empty(shape.n_experts + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    abi.moe_permute(cfg, torch.as_tensor(ids, device="cuda"), T, offs, perm, inv, ws)
    torch.cuda.synchronize()
    for g, o in zip((offs, perm, inv), orc.permute(ids, shape.n_experts)):
        assert np.array_equal(g.cpu().numpy(), o)


def test_forward_single_expert_is_dense_swiglu_library():
    """E=1, k=1, no shared expert: the layer is a dense SwiGLU MLP; check against torch."""
    shape = inputs.Shape(512, 1, 1, 256, 0)
    layers, x = make(shape, 333, seed=3)
    out, _ = forward_gpu(shape, layers[0], x)
    L = layers[0]
    xf = x.float()
    g = xf @ L["w_gate"][0].float().T
    u = xf @ L["w_up"][0].float().T
    h = (torch.nn.functional.silu(g) * u).to(torch.bfloat16).float()
    ref = (h @ L["w_down"][0].float().T).to(torch.bfloat16)
    compare_out(u16(out), u16(ref))


def test_forward_x_next_and_alias():
    layers, x = make(TINY, 77, seed=9)
    out, xn = forward_gpu(TINY, layers[0], x, want_x_next=True)
    ref = orc.bf16_to_f64(u16(x)) + orc.bf16_to_f64(u16(out))
    want = torch.as_tensor(ref, dtype=torch.float32).to(torch.bfloat16)
    assert np.array_equal(u16(xn), u16(want))
    # a separate residual input: x_next = bf16(resid + out)
    cfg = cfg_of(TINY)
    resid = torch.randn_like(x.float()).to(torch.bfloat16)
    ws0 = abi.alloc_workspace(cfg, 77)
    out_r = torch.empty_like(x)
    xn_r = torch.empty_like(x)
    abi.moe_forward(cfg, abi.weights(layers[0]), x, 77, out_r, xn_r, ws0, resid=resid)
    torch.cuda.synchronize()
    assert torch.equal(xn_r, (resid.float() + out_r.float()).to(torch.bfloat16))
    compare_out(u16(out_r), u16(out))
    # x_next may alias x (resid defaults to x)
    ws = abi.alloc_workspace(cfg, 77)
    x2 = x.clone()
    out2 = torch.empty_like(x)
    abi.moe_forward(cfg, abi.weights(layers[0]), x2, 77, out2, x2, ws)
    torch.cuda.synchronize()
    assert np.array_equal(u16(x2), u16(xn))


def test_forward_zero_input_and_zero_tokens():
    layers, x = make(TINY, 40, seed=1)
    z = torch.zeros_like(x)
    out, _ = forward_gpu(TINY, layers[0], z)
    assert (u16(out) & 0x7FFF == 0).all()
    cfg = cfg_of(TINY)
    ws = abi.alloc_workspace(cfg, 1)
    assert abi.moe_forward_status(cfg, abi.weights(layers[0]), x, 0, out, None, ws) == 0


def test_forward_zero_routed_down_gives_shared_only():
    layers, x = make(TINY, 50, seed=2)
    L = dict(layers[0])
    L["w_down"] = torch.zeros_like(L["w_down"])
    out, _ = forward_gpu(TINY, L, x)
    hl = host(L)
    xf = x.float()
    h = (torch.nn.functional.silu(xf @ L["ws_gate"].float().T) * (xf @ L["ws_up"].float().T)).to(torch.bfloat16)
    ref = (h.float() @ L["ws_down"].float().T).to(torch.bfloat16)
    compare_out(u16(out), u16(ref))
    compare_out(u16(out), orc.forward(u16(x), hl, TINY.top_k)["out"])


def test_token_order_permutes_rows():
    layers, x = make(TINY, 90, seed=4)
    out, _ = forward_gpu(TINY, layers[0], x)
    p = torch.randperm(90, generator=torch.Generator().manual_seed(0)).cuda()
    out_p, _ = forward_gpu(TINY, layers[0], x[p].contiguous())
    compare_out(u16(out_p), u16(out[p]))


def test_piece_composition_matches_per_piece_calls():
    """moe_forward(T) is bit-identical to the concatenation of moe_forward over its planned
    pieces: every piece runs the same kernels on its own rows, and no kernel's arithmetic
    depends on the other pieces."""
    shape = inputs.Shape(256, 16, 4, 128, 128)
    T = 8192 + 4096 + 1024 + 25 + 1
    assert abi.moe_plan_pieces(T) == [8192, 4096, 1024, 26]
    layers, x = make(shape, T, seed=5)
    out, _ = forward_gpu(shape, layers[0], x)
    parts, t0 = [], 0
    for p in abi.moe_plan_pieces(T):
        o, _ = forward_gpu(shape, layers[0], x[t0:t0 + p].contiguous())
        parts.append(o)
        t0 += p
    assert torch.equal(out, torch.cat(parts))
    rows = np.r_[0:40, 8180:8210, 12280:12300, 13300:T]
    check_layer(shape, layers[0], x, rows=rows)


def test_launch_counter_and_timing():
    layers, x = make(TINY, 64, seed=6)
    n0 = abi.moe_launch_count()
    abi.timing_enable(True)
    forward_gpu(TINY, layers[0], x)
    abi.timing_enable(False)
    assert abi.moe_launch_count() - n0 >= 7
    n, ms = abi.timing_read("gateup_gemm")
    assert n == 1 and ms > 0
    assert "down_gemm" in abi.timing_classes()


def test_forward_is_bit_reproducible():
    """No atomics in the fused path: two runs on the same input give identical bits."""
    shape = inputs.Shape(512, 32, 4, 256, 256)
    layers, x = make(shape, 777, seed=13)
    a, _ = forward_gpu(shape, layers[0], x)
    b, _ = forward_gpu(shape, layers[0], x)
    assert torch.equal(a, b)


@pytest.mark.parametrize("T", [2, 3, 4, 5, 8])
def test_small_batch_decode_layer_shape(T):
    """2..4 tokens take the decode path (each selected expert's weights streamed once for every
    token that chose it), 5 and more the prefill path: parity at the 2048-wide, 256-expert top-8
    shape on both sides of the switch."""
    shape = inputs.Shape(2048, 256, 8, 512, 512)
    layers, x = make(shape, T, seed=40 + T)
    check_layer(shape, layers[0], x)


def test_small_batch_decode_repeated_tokens():
    """Identical token rows select identical experts: one block serves all of them."""
    shape = inputs.Shape(2048, 256, 8, 512, 512)
    layers, x = make(shape, 4, seed=47)
    x = x[torch.tensor([0, 1, 0, 0], device=x.device)].contiguous()
    check_layer(shape, layers[0], x)
    out, _ = forward_gpu(shape, layers[0], x)
    # rows 0, 2, 3 are the same token: the same output within the fp32 summation order
    compare_out(u16(out)[[2, 3]], u16(out)[[0, 0]])


@pytest.mark.parametrize("shape,T", [(inputs.Shape(256, 600, 8, 128, 128), 3), (TINY, 4), (TINY, 2),
                                     (inputs.Shape(256, 64, 32, 128, 128), 3)])
def test_small_batch_decode_other_shapes(shape, T):
    layers, x = make(shape, T, seed=60 + T)
    check_layer(shape, layers[0], x)
