"""GPU parity of moe_decode_chain (one token through a stack of layers in one launch) against
the CPU oracle, layer by layer, through the C-ABI.

A chain of n layers leaves x_n in x_last, so layer n of the chain can be checked on exactly the
input it saw: the oracle (consuming the GPU routing of that input) against the out of the
(n+1)-layer chain.  Bounds as for the layer: max |diff| <= 2e-2, relative L2 <= 5e-3.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_moe_router_gb300 import abi, inputs

from helpers import cfg_of, check_layer, compare_out, forward_gpu, host, make, check_x_last, route_gpu, u16

pytestmark = pytest.mark.gpu

DECODE = inputs.Shape(2048, 256, 8, 512, 512)
TINY = inputs.Shape(256, 16, 4, 128, 128)


def _chain(shape, layers, x0, n, resid=None, ws=None):
    cfg = cfg_of(shape)
    ws = abi.alloc_workspace(cfg, 1) if ws is None else ws
    out = torch.empty_like(x0)
    x_last = torch.empty_like(x0)
    abi.moe_decode_chain(cfg, [abi.weights(l) for l in layers[:n]], x0, out, x_last, ws, resid=resid)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    return out, x_last


def _layer_ref(shape, layer, x):
    """The oracle's out for one token x (bf16 [1, H]) on the GPU's routing of x."""
    logits, ids, w = route_gpu(shape, layer, x)
    ids_o, w_o = orc.route_from_logits(logits, shape.top_k)
    assert np.array_equal(ids, ids_o)
    return orc.forward(np.ascontiguousarray(u16(x)), host(layer), shape.top_k, ids=ids, topk_w=w)["out"]


@pytest.mark.parametrize("use_resid", [False, True])
@pytest.mark.parametrize("shape,L", [(DECODE, 4), (TINY, 5), (inputs.Shape(256, 600, 8, 128, 128), 3),
                                     (inputs.Shape(512, 32, 4, 256, 0), 3), (inputs.Shape(256, 64, 32, 128, 128), 3),
                                     # 2 and 4 chunks of the down-projection slice; the widest also
                                     # reads its router rows from global memory (no staging)
                                     (inputs.Shape(4096, 16, 4, 128, 128), 3), (inputs.Shape(8192, 16, 4, 128, 128), 2)])
def test_chain_layer_by_layer(shape, L, use_resid):
    layers, x0 = make(shape, 1, seed=500 + L + 7 * use_resid, n_layers=L)
    resid = x0.clone() if use_resid else None
    x_in = x0
    for n in range(1, L + 1):
        out, x_last = _chain(shape, layers, x0, n, resid)
        ref = _layer_ref(shape, layers[n - 1], x_in)
        compare_out(u16(out), ref, what="chain layer %d out" % (n - 1))
        r = u16(resid) if use_resid else u16(x_in)
        check_x_last(u16(x_last), r, u16(out), use_resid or n == 1)
        x_in = x_last


def test_chain_matches_layer_calls():
    """The chain and n_layers one-token moe_forward calls compute the same stack (the split-K
    atomics may differ in the last bit)."""
    L = 6
    layers, x0 = make(DECODE, 1, seed=610, n_layers=L)
    x = x0
    for l in range(L):
        out_l, x_next = forward_gpu(DECODE, layers[l], x, want_x_next=True)
        x = x_next
    out_c, x_c = _chain(DECODE, layers, x0, L)
    compare_out(u16(out_c), u16(out_l), what="chain vs per-layer calls")


def test_chain_more_items_than_blocks():
    """k * I / 32 + Is / 32 = 32 * 32 + 4 work items: more than the GPU holds at once, so every
    block walks several items (and keeps one top-k per layer)."""
    shape = inputs.Shape(256, 64, 32, 1024, 128)
    L = 3
    layers, x0 = make(shape, 1, seed=620, n_layers=L)
    x_in = x0
    for n in range(1, L + 1):
        out, x_last = _chain(shape, layers, x0, n)
        compare_out(u16(out), _layer_ref(shape, layers[n - 1], x_in), what="layer %d" % (n - 1))
        x_in = x_last


def test_chain_64_layers_and_reused_workspace():
    L = 64
    layers, x0 = make(TINY, 1, seed=630, n_layers=L)
    ws = abi.alloc_workspace(cfg_of(TINY), 1)
    r = x0.clone()  # a fixed residual keeps 64 random layers at unit scale
    out_a, x_a = _chain(TINY, layers, x0, L, resid=r, ws=ws)
    out_b, x_b = _chain(TINY, layers, x0, L, resid=r, ws=ws)  # the barrier words are re-armed per call
    compare_out(u16(out_b), u16(out_a), what="repeat")
    # the last layer against the oracle on its own input (x_63 from the 63-layer chain)
    _, x63 = _chain(TINY, layers, x0, L - 1, resid=r, ws=ws)
    compare_out(u16(out_a), _layer_ref(TINY, layers[L - 1], x63), what="layer 63")
    # and the one-token layer path on the same input agrees
    out_f, _ = forward_gpu(TINY, layers[L - 1], x63)
    compare_out(u16(out_a), u16(out_f), what="layer 63 vs moe_forward")


def test_chain_argument_errors():
    layers, x0 = make(TINY, 1, seed=640, n_layers=2)
    cfg = cfg_of(TINY)
    ws = abi.alloc_workspace(cfg, 1)
    out = torch.empty_like(x0)
    wts = [abi.weights(l) for l in layers]
    lib = abi.lib()
    arr = (abi.Weights * 65)(*(wts * 33)[:65])
    st = lib.moe_decode_chain(cfg, arr, 65, x0.data_ptr(), None, out.data_ptr(), None, ws.data_ptr(), ws.numel(),
                              None)
    assert st == 3  # more than 64 layers
    arr2 = (abi.Weights * 2)(*wts)
    assert lib.moe_decode_chain(cfg, arr2, 0, x0.data_ptr(), None, out.data_ptr(), None, ws.data_ptr(),
                                ws.numel(), None) == 1
    assert lib.moe_decode_chain(cfg, arr2, 2, x0.data_ptr() + 2, None, out.data_ptr(), None, ws.data_ptr(),
                                ws.numel(), None) == 1  # misaligned x0
    assert lib.moe_decode_chain(cfg, arr2, 2, x0.data_ptr(), None, out.data_ptr(), None, ws.data_ptr(),
                                256, None) == 2  # workspace too small
    big = inputs.Shape(16384, 16, 4, 128, 128)
    assert lib.moe_decode_chain(cfg_of(big), arr2, 2, x0.data_ptr(), None, out.data_ptr(), None, ws.data_ptr(),
                                ws.numel(), None) in (1, 2, 3)  # rejected before any launch
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
