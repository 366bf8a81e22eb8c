"""GPU parity of the 4-bit expert-weight path (codes in [-7, 7] with one fp32 scale per block of 32
columns) against the CPU oracle, through the C-ABI.

- moe_quantize_q4: packed codes and block scales bit-exact against the oracle's quantiser (both
  divide in fp32 with IEEE rounding and round the quotient half to even).
- moe_decode_chain_q4: layer by layer against the oracle's 4-bit layer on the GPU's routing of the
  input each layer saw (the chain of n layers leaves x_n in x_last), on synthetic codes and scales
  from the input module and on weights the GPU quantised; x_last bit-exact as bf16(r + out).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_moe_router_gb300 import abi, inputs

from helpers import cfg_of, compare_out, check_x_last, route_gpu, u16

pytestmark = pytest.mark.gpu

DECODE = inputs.Shape(2048, 256, 8, 512, 512)
TINY = inputs.Shape(256, 16, 4, 128, 128)


def _gpu_quantize(w):
    q = torch.empty(w.shape[:-1] + (w.shape[-1] // 2,), dtype=torch.uint8, device=w.device)
    s = torch.empty(w.shape[:-1] + (w.shape[-1] // 32,), dtype=torch.float32, device=w.device)
    abi.moe_quantize_q4(w, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _check_quantize(w):
    q, s = _gpu_quantize(w)
    cols = w.shape[-1]
    qo, so = orc.quantize_q4_rows(u16(w).reshape(-1, cols))
    np.testing.assert_array_equal(s.reshape(-1, cols // 32).view(np.uint32), so.view(np.uint32))
    np.testing.assert_array_equal(q.reshape(-1, cols // 2), qo)


def test_quantize_matches_oracle_on_weights():
    g = torch.Generator(device="cuda")
    g.manual_seed(950)
    w = torch.empty(4, 256, 512, device="cuda").normal_(0.0, 0.02, generator=g).to(torch.bfloat16)
    _check_quantize(w)


def test_quantize_edge_blocks():
    """Zero blocks (scale 1), signed zeros, one non-zero in a block, exact ties of the quotient
    (multiples of half the scale), a negative maximum, large and tiny magnitudes, a constant row."""
    g = torch.Generator(device="cuda")
    g.manual_seed(951)
    cols = 256
    w = torch.empty(9, cols, device="cuda").normal_(0.0, 1.0, generator=g)
    w[0] = 0.0
    w[1] = -0.0
    w[1, 37] = 3.0
    # scale 0.5 in every block (max 3.5): values k/4 give quotients k/2, half of them ties
    w[2] = (torch.arange(cols, device="cuda") % 29 - 14).float() * 0.25
    w[2, ::32] = 3.5
    w[3] = w[3].abs()
    w[3, 11] = -50.0
    w[4] *= 1e30
    w[5] *= 1e-30
    w[6] = torch.linspace(-1.0, 1.0, cols, device="cuda")
    w[7, :] = 1.0
    w[8, 64:96] = 0.0
    _check_quantize(w.to(torch.bfloat16))
    _check_quantize(w[:, :32].contiguous().to(torch.bfloat16))


def test_quantize_empty_and_errors():
    lib = abi.lib()
    assert lib.moe_quantize_q4(None, 0, 32, None, None, None) == 0
    assert lib.moe_quantize_q4(None, 3, 0, None, None, None) == 0
    assert lib.moe_quantize_q4(None, -1, 32, None, None, None) == 1
    assert lib.moe_quantize_q4(None, 2, 32, None, None, None) == 1
    w = torch.zeros(2, 48, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(2, 24, dtype=torch.uint8, device="cuda")
    s = torch.empty(2, 2, dtype=torch.float32, device="cuda")
    assert lib.moe_quantize_q4(w.data_ptr(), 2, 48, q.data_ptr(), s.data_ptr(), None) == 1  # 48 % 32 != 0


def _make_q4(shape, L, seed):
    w = inputs.custom(shape, T=1, seed=seed, router_std=0.02, n_layers=L)
    return inputs.make_q4(w, device="cuda")


def _chain_q4(shape, layers, x0, n, resid=None, ws=None):
    cfg = cfg_of(shape)
    ws = abi.alloc_workspace(cfg, 1) if ws is None else ws
    out = torch.empty_like(x0)
    x_last = torch.empty_like(x0)
    abi.moe_decode_chain_q4(cfg, [abi.weights_q4(l) for l in layers[:n]], x0, out, x_last, ws, resid=resid)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    return out, x_last


def _host_q4(layer):
    return {k: v.cpu().numpy() for k, v in layer.items() if v is not None and k not in ("w_router", "b_router")}


def _layer_ref_q4(shape, layer, x):
    logits, ids, w = route_gpu(shape, layer, x)
    ids_o, _ = orc.route_from_logits(logits, shape.top_k)
    assert np.array_equal(ids, ids_o)
    return orc.forward_q4(np.ascontiguousarray(u16(x)), _host_q4(layer), shape.top_k, ids, w)


@pytest.mark.parametrize("use_resid", [False, True])
@pytest.mark.parametrize("shape,L", [(DECODE, 3), (TINY, 4), (inputs.Shape(256, 600, 8, 128, 128), 2),
                                     (inputs.Shape(512, 32, 4, 256, 0), 2),
                                     (inputs.Shape(256, 64, 32, 128, 128), 2),
                                     # 2 chunks of the down slice; router rows not staged
                                     (inputs.Shape(4096, 16, 4, 128, 128), 2),
                                     (inputs.Shape(8192, 16, 4, 128, 128), 2)])
def test_chain_q4_layer_by_layer(shape, L, use_resid):
    layers, x0 = _make_q4(shape, L, seed=760 + L + 5 * use_resid)
    resid = x0.clone() if use_resid else None
    x_in = x0
    for n in range(1, L + 1):
        out, x_last = _chain_q4(shape, layers, x0, n, resid)
        compare_out(u16(out), _layer_ref_q4(shape, layers[n - 1], x_in), what="q4 chain layer %d" % (n - 1))
        r = u16(resid) if use_resid else u16(x_in)
        check_x_last(u16(x_last), r, u16(out), use_resid or n == 1)
        x_in = x_last


def test_chain_q4_more_items_than_blocks():
    """k * I / 32 + Is / 32 = 32 * 32 + 4 work items: every block walks several items."""
    shape = inputs.Shape(256, 64, 32, 1024, 128)
    layers, x0 = _make_q4(shape, 2, seed=770)
    x_in = x0
    for n in range(1, 3):
        out, x_last = _chain_q4(shape, layers, x0, n)
        compare_out(u16(out), _layer_ref_q4(shape, layers[n - 1], x_in), what="layer %d" % (n - 1))
        x_in = x_last


def test_chain_q4_on_gpu_quantised_weights():
    """The whole 4-bit path: bf16 weights through moe_quantize_q4, then the chain, against the
    oracle on the same codes (which the quantiser test pins against the oracle's own)."""
    shape = DECODE
    w = inputs.custom(shape, T=1, seed=780, router_std=0.02, n_layers=2)
    layers_bf, x0 = inputs.make(w, device="cuda")
    layers = [abi.quantize_layer_q4(l) for l in layers_bf]
    del layers_bf
    torch.cuda.synchronize()
    out1, x1 = _chain_q4(shape, layers, x0, 1)
    compare_out(u16(out1), _layer_ref_q4(shape, layers[0], x0), what="layer 0")
    out2, _ = _chain_q4(shape, layers, x0, 2)
    compare_out(u16(out2), _layer_ref_q4(shape, layers[1], x1), what="layer 1")


def test_chain_q4_argument_errors():
    layers, x0 = _make_q4(TINY, 2, seed=790)
    cfg = cfg_of(TINY)
    ws = abi.alloc_workspace(cfg, 1)
    out = torch.empty_like(x0)
    lib = abi.lib()

    def call(lw, n=2, x=x0.data_ptr()):
        arr = (abi.WeightsQ4 * len(lw))(*lw)
        return lib.moe_decode_chain_q4(cfg, arr, n, x, None, out.data_ptr(), None, ws.data_ptr(), ws.numel(), None)

    good = [abi.weights_q4(l) for l in layers]
    assert call(good, n=0) == 1
    assert call(good, x=x0.data_ptr() + 2) == 1
    bad = [abi.weights_q4(l) for l in layers]
    bad[1].s_down = None
    assert call(bad) == 1
    bad = [abi.weights_q4(l) for l in layers]
    bad[0].ss_gate = None  # the shared expert is present (Is > 0)
    assert call(bad) == 1
    bad = [abi.weights_q4(l) for l in layers]
    bad[0].q_up = bad[0].q_up + 8
    assert call(bad) == 1
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    assert call(good) == 0
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
