"""GPU checks of moe_graph_* (a layer stack captured once as a CUDA graph and replayed): the
replay computes what the same moe_forward calls compute eagerly, on the buffers' contents at
launch time, and the first layer matches the CPU oracle."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_moe_router_gb300 import abi, inputs

from helpers import cfg_of, compare_out, host, make, route_gpu, u16

pytestmark = pytest.mark.gpu

TINY = inputs.Shape(256, 16, 4, 128, 128)
MID = inputs.Shape(512, 32, 4, 256, 256)


def _eager(shape, layers, x0, T, resid=None):
    """The stack as plain moe_forward calls: (out of the last layer, x_n)."""
    cfg = cfg_of(shape)
    ws = abi.alloc_workspace(cfg, min(T, 8192))
    out = torch.empty_like(x0)
    x = x0
    for l in layers:
        nxt = torch.empty_like(x0)
        abi.moe_forward(cfg, abi.weights(l), x, T, out, nxt, ws, resid=resid)
        x = nxt
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    return out, x


def _graph(shape, layers, x0, T, resid=None):
    cfg = cfg_of(shape)
    ws = abi.alloc_workspace(cfg, min(T, 8192))
    out, x_last, scratch = torch.empty_like(x0), torch.empty_like(x0), torch.empty_like(x0)
    g = abi.Graph(cfg, [abi.weights(l) for l in layers], T, x0, out, x_last, scratch, ws, resid=resid,
                  keep=layers)
    return g, out, x_last, ws


@pytest.mark.parametrize("shape,T,L,use_resid", [(TINY, 64, 1, False), (TINY, 300, 3, True), (MID, 1100, 2, False),
                                                  (MID, 2077, 4, True),
                                                  (inputs.Shape(256, 16, 4, 128, 256), 200, 2, False)])
def test_graph_replay_equals_eager_calls(shape, T, L, use_resid):
    layers, x0 = make(shape, T, seed=800 + T, n_layers=L)
    resid = x0.clone() if use_resid else None
    out_e, x_e = _eager(shape, layers, x0, T, resid)
    g, out, x_last, ws = _graph(shape, layers, x0, T, resid)
    out.zero_()
    x_last.zero_()
    n0 = abi.moe_launch_count()
    g.launch()
    g.launch()
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    assert g.kernels > 0 and abi.moe_launch_count() - n0 == 2 * g.kernels
    # the prefill path has no atomics: bit-identical to the eager calls
    np.testing.assert_array_equal(u16(out), u16(out_e))
    np.testing.assert_array_equal(u16(x_last), u16(x_e))


def test_graph_reads_inputs_at_launch_and_matches_the_oracle():
    shape, T = TINY, 64
    layers, x0 = make(shape, T, seed=820, n_layers=1)
    g, out, _, ws = _graph(shape, layers, x0, T)
    _, x_new = make(shape, T, seed=821, n_layers=0)
    x0.copy_(x_new)  # new contents, same buffer
    g.launch()
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    logits, ids, w = route_gpu(shape, layers[0], x_new)
    ids_o, _ = orc.route_from_logits(logits, shape.top_k)
    assert np.array_equal(ids, ids_o)
    ref = orc.forward(u16(x_new), host(layers[0]), shape.top_k, ids=ids, topk_w=w)["out"]
    compare_out(u16(out), ref, what="graph out on a new input")


def test_graph_of_decode_path_tokens():
    """T = 2 runs the decode kernels (fp32 atomics): the replay agrees with eager calls within
    the layer tolerance."""
    shape, T = TINY, 2
    layers, x0 = make(shape, T, seed=830, n_layers=2)
    out_e, _ = _eager(shape, layers, x0, T)
    g, out, _, ws = _graph(shape, layers, x0, T)
    g.launch()
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    compare_out(u16(out), u16(out_e), what="decode-path graph")


def test_graph_create_errors_leave_no_graph():
    shape, T = TINY, 64
    layers, x0 = make(shape, T, seed=840, n_layers=2)
    cfg = cfg_of(shape)
    ws = abi.alloc_workspace(cfg, T)
    out = torch.empty_like(x0)
    with pytest.raises(abi.MoeError):
        abi.Graph(cfg, [abi.weights(l) for l in layers], T, x0, out, None, None, ws)  # a stack needs x_last
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    xl, sc = torch.empty_like(x0), torch.empty_like(x0)
    with pytest.raises(abi.MoeError):
        abi.Graph(cfg, [abi.weights(l) for l in layers], T, x0, out, xl, sc, small)  # workspace too small
    torch.cuda.synchronize()
