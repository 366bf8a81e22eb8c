"""GPU parity of the quantised-weight path (E4M3 expert weights with fp32 row scales) against the
CPU oracle, through the C-ABI.

- moe_quantize_e4m3: codes and scales bit-exact against the oracle's row quantiser (both divide
  in fp32 with IEEE rounding; the code is the nearest E4M3 value, ties to even).
- moe_decode_chain_q8: layer by layer against the oracle's quantised layer on the GPU's routing
  of the input each layer saw (the chain of n layers leaves x_n in x_last), on synthetic codes
  and scales from the input module; x_last bit-exact as bf16(r + out).
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
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    s = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    abi.moe_quantize_e4m3(w, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _check_quantize(w):
    q, s = _gpu_quantize(w)
    cols = w.shape[-1]
    qo, so = orc.quantize_e4m3_rows(u16(w).reshape(-1, cols))
    np.testing.assert_array_equal(s.reshape(-1).view(np.uint32), so.view(np.uint32))
    np.testing.assert_array_equal(q.reshape(-1, cols), qo)


def test_quantize_matches_oracle_on_weights():
    g = torch.Generator(device="cuda")
    g.manual_seed(900)
    w = torch.empty(4, 256, 512, device="cuda").normal_(0.0, 0.02, generator=g).to(torch.bfloat16)
    _check_quantize(w)


def test_quantize_edge_rows():
    """A zero row (scale 1), signed zeros, a single non-zero, a row spanning the subnormal range
    and beyond (values that round to zero of either sign), a negative maximum, large and tiny
    magnitudes, and a ragged column count."""
    g = torch.Generator(device="cuda")
    g.manual_seed(901)
    cols = 300
    w = torch.empty(10, cols, device="cuda").normal_(0.0, 1.0, generator=g)
    w[0] = 0.0
    w[1] = -0.0
    w[1, 7] = 3.0
    w[2] = torch.logspace(-24, 0, cols, base=2.0, device="cuda") * torch.where(
        torch.arange(cols, device="cuda") % 2 == 0, 1.0, -1.0)
    w[3] = w[3].abs()
    w[3, 11] = -50.0
    w[4] *= 1e30
    w[5] *= 1e-30
    w[6] = torch.linspace(-1.0, 1.0, cols, device="cuda")
    w[7, :] = 1.0
    _check_quantize(w.to(torch.bfloat16))
    _check_quantize(w[:, :16].contiguous().to(torch.bfloat16))
    _check_quantize(w[:1, :1].contiguous().to(torch.bfloat16))


def test_quantize_empty_and_errors():
    lib = abi.lib()
    assert lib.moe_quantize_e4m3(None, 0, 5, None, None, None) == 0
    assert lib.moe_quantize_e4m3(None, 3, 0, None, None, None) == 0
    assert lib.moe_quantize_e4m3(None, -1, 5, None, None, None) == 1
    assert lib.moe_quantize_e4m3(None, 2, 5, None, None, None) == 1


def _make_q8(shape, L, seed):
    w = inputs.custom(shape, T=1, seed=seed, router_std=0.02, n_layers=L)
    return inputs.make_q8(w, device="cuda")


def _chain_q8(shape, layers, x0, n, resid=None, ws=None):
    cfg = cfg_of(shape)
    ws = abi.alloc_workspace(cfg, 1) if ws is None else ws
    out = torch.empty_like(x0)
    x_last = torch.empty_like(x0)
    abi.moe_decode_chain_q8(cfg, [abi.weights_q8(l) for l in layers[:n]], x0, out, x_last, ws, resid=resid)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    return out, x_last


def _host_q8(layer):
    return {k: v.cpu().numpy() for k, v in layer.items() if v is not None and k not in ("w_router", "b_router")}


def _layer_ref_q8(shape, layer, x):
    logits, ids, w = route_gpu(shape, layer, x)
    ids_o, _ = orc.route_from_logits(logits, shape.top_k)
    assert np.array_equal(ids, ids_o)
    return orc.forward_q8(np.ascontiguousarray(u16(x)), _host_q8(layer), shape.top_k, ids, w)


@pytest.mark.parametrize("use_resid", [False, True])
@pytest.mark.parametrize("shape,L", [(DECODE, 3), (TINY, 4), (inputs.Shape(256, 600, 8, 128, 128), 2),
                                     (inputs.Shape(512, 32, 4, 256, 0), 2),
                                     (inputs.Shape(4096, 16, 4, 128, 128), 2)])
def test_chain_q8_layer_by_layer(shape, L, use_resid):
    layers, x0 = _make_q8(shape, L, seed=700 + L + 5 * use_resid)
    resid = x0.clone() if use_resid else None
    x_in = x0
    for n in range(1, L + 1):
        out, x_last = _chain_q8(shape, layers, x0, n, resid)
        compare_out(u16(out), _layer_ref_q8(shape, layers[n - 1], x_in), what="q8 chain layer %d" % (n - 1))
        r = u16(resid) if use_resid else u16(x_in)
        check_x_last(u16(x_last), r, u16(out), use_resid or n == 1)
        x_in = x_last


def test_chain_q8_on_gpu_quantised_weights():
    """The whole quantised path: bf16 weights through moe_quantize_e4m3, then the chain, against
    the oracle on the same codes (which the quantiser test pins against the oracle's own)."""
    shape = TINY
    w = inputs.custom(shape, T=1, seed=710, router_std=0.02, n_layers=2)
    layers_bf, x0 = inputs.make(w, device="cuda")
    layers = [abi.quantize_layer(l) for l in layers_bf]
    torch.cuda.synchronize()
    out1, x1 = _chain_q8(shape, layers, x0, 1)
    compare_out(u16(out1), _layer_ref_q8(shape, layers[0], x0), what="layer 0")
    out2, _ = _chain_q8(shape, layers, x0, 2)
    compare_out(u16(out2), _layer_ref_q8(shape, layers[1], x1), what="layer 1")


def test_chain_q8_argument_errors():
    layers, x0 = _make_q8(TINY, 2, seed=720)
    cfg = cfg_of(TINY)
    ws = abi.alloc_workspace(cfg, 1)
    out = torch.empty_like(x0)
    lib = abi.lib()

    def call(lw, n=2, x=x0.data_ptr()):
        arr = (abi.WeightsQ8 * len(lw))(*lw)
        return lib.moe_decode_chain_q8(cfg, arr, n, x, None, out.data_ptr(), None, ws.data_ptr(), ws.numel(), None)

    good = [abi.weights_q8(l) for l in layers]
    assert call(good, n=0) == 1
    assert call(good, x=x0.data_ptr() + 2) == 1
    bad = [abi.weights_q8(l) for l in layers]
    bad[1].s_down = None
    assert call(bad) == 1
    bad = [abi.weights_q8(l) for l in layers]
    bad[0].ss_gate = None  # the shared expert is present (Is > 0)
    assert call(bad) == 1
    bad = [abi.weights_q8(l) for l in layers]
    bad[0].q_up = bad[0].q_up + 8
    assert call(bad) == 1
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    # and the good call still runs
    assert call(good) == 0
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0


# ------------------------------------------------------------ prefill with E4M3 weights --

def _forward_q8(shape, layer, x):
    cfg = cfg_of(shape)
    T = x.shape[0]
    ws = abi.alloc_workspace(cfg, min(T, 8192))
    out, xn = torch.empty_like(x), torch.empty_like(x)
    abi.moe_forward_q8(cfg, abi.weights_q8(layer), x, T, out, xn, ws)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    return out, xn


@pytest.mark.parametrize("shape,T", [(TINY, 64), (TINY, 1), (TINY, 3), (TINY, 5), (TINY, 300), (TINY, 1025),
                                     (inputs.Shape(512, 32, 4, 256, 0), 200),
                                     (inputs.Shape(1024, 64, 8, 384, 256), 70),
                                     (inputs.Shape(256, 16, 16, 128, 256), 40),
                                     (inputs.Shape(384, 1, 1, 128, 0), 33)])
def test_forward_q8_matches_oracle(shape, T):
    """moe_forward_q8 (the grouped GEMMs widening E4M3 codes to bf16 in shared memory, row scales
    in the epilogue) against the oracle's quantised layer on the GPU's routing: every row."""
    layers, x = inputs.make_q8(inputs.custom(shape, T=T, seed=800 + T, router_std=0.02), device="cuda")
    out, xn = _forward_q8(shape, layers[0], x)
    compare_out(u16(out), _layer_ref_q8(shape, layers[0], x), what="forward_q8")
    assert torch.equal(xn, (x.float() + out.float()).to(torch.bfloat16))


@pytest.mark.parametrize("T", [8192, 1000])
def test_forward_q8_layer_shape_sampled(T):
    """The 2048-wide, 256-expert top-8 layer with E4M3 weights quantised on the device from a bf16
    layer (moe_quantize_e4m3, pinned bit-exact against the oracle's quantiser above), checked on
    sampled rows (every piece edge included) against the oracle on the same codes."""
    shape = DECODE
    wl = inputs.custom(shape, T=T, seed=820 + T % 7, router_std=1.0 / np.sqrt(shape.hidden))
    layers_bf, x = inputs.make(wl, device="cuda")
    layer = abi.quantize_layer(layers_bf[0])
    del layers_bf
    torch.cuda.synchronize()
    out, _ = _forward_q8(shape, layer, x)
    logits, ids, w = route_gpu(shape, layer, x)
    ids_o, _ = orc.route_from_logits(logits, shape.top_k)
    assert np.array_equal(ids, ids_o)
    rng = np.random.default_rng(T)
    rows = np.unique(np.concatenate([[0, 1, T - 2, T - 1], rng.choice(T, size=64, replace=False)]))
    ref = orc.forward_q8(np.ascontiguousarray(u16(x)[rows]), _host_q8(layer), shape.top_k,
                         np.ascontiguousarray(ids[rows]), np.ascontiguousarray(w[rows]))
    compare_out(u16(out)[rows], ref, what="forward_q8 layer shape")
