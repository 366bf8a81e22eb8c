"""GPU parity of the routing steps through the C-ABI: top-k from logits, router GEMM, permute.

Integer outputs (ids, offsets, perm, inv) must be bit-exact against the oracle; weights
within a few fp32 ulps; router logits within 1e-5*(1+|l|) of the oracle's fp64 sum.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_moe_router_gb300 import abi, inputs

from helpers import cfg_of, host, logits_tol, make, u16

pytestmark = pytest.mark.gpu


def _route_from_logits(E, k, logits_np):
    cfg = abi.config(128, E, k, 128, 0)
    T = logits_np.shape[0]
    lg = torch.as_tensor(logits_np, device="cuda")
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    abi.moe_route_from_logits(cfg, lg, T, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,E,k,scale", [(1000, 16, 4, 0.25), (777, 256, 8, 0.5), (300, 64, 6, 0.125),
                                         (50, 1024, 32, 0.25), (33, 16, 16, 1.0), (64, 16, 1, 0.25),
                                         (5, 40, 7, 0.25)])
def test_topk_bitexact_with_ties(T, E, k, scale):
    rng = np.random.default_rng(T + E + k)
    # coarse grid: many equal logits, so the lower-index tie-break is exercised
    logits = (np.round(rng.standard_normal((T, E)) / scale) * scale).astype(np.float32)
    ids, w = _route_from_logits(E, k, logits)
    ids_o, w_o = orc.route_from_logits(logits, k)
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=2e-6, atol=1e-7)


def test_topk_all_equal_and_k1():
    ids, w = _route_from_logits(256, 8, np.full((9, 256), -1.5, dtype=np.float32))
    assert (ids == np.arange(8)).all() and (w == np.float32(0.125)).all()
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((100, 256)).astype(np.float32)
    ids, w = _route_from_logits(256, 1, lg)
    assert (w == 1.0).all() and np.array_equal(ids[:, 0], np.argmax(lg, axis=1))


@pytest.mark.parametrize("shape,T,router_std,zipf", [
    (inputs.Shape(256, 16, 4, 128, 128), 64, 0.02, None),
    (inputs.Shape(256, 16, 4, 128, 128), 3, 0.02, None),
    (inputs.Shape(2048, 256, 8, 512, 512), 300, 2048 ** -0.5, 1.0),
    (inputs.Shape(512, 200, 6, 128, 0), 130, 512 ** -0.5, None),
])
def test_router_gemm_logits_and_selection(shape, T, router_std, zipf):
    layers, x = make(shape, T, seed=11, router_std=router_std, zipf_s=zipf)
    hl = host(layers[0])
    cfg = cfg_of(shape)
    ws = abi.alloc_workspace(cfg, T)
    logits = torch.empty(T, shape.n_experts, dtype=torch.float32, device="cuda")
    ids = torch.empty(T, shape.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, shape.top_k, dtype=torch.float32, device="cuda")
    abi.moe_route(cfg, abi.weights(layers[0]), x, T, logits, ids, w, ws)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    ref = orc.router_logits(u16(x), hl["w_router"], hl.get("b_router"))
    assert np.all(np.abs(lg - ref) <= logits_tol(ref))
    ids_o, w_o = orc.route_from_logits(lg, shape.top_k)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    np.testing.assert_allclose(w.cpu().numpy(), w_o, rtol=2e-6, atol=1e-7)


def _permute_gpu(E, k, ids_np):
    cfg = abi.config(128, E, k, 128, 0)
    T = ids_np.shape[0]
    ws = abi.alloc_workspace(cfg, T)
    ids = torch.as_tensor(ids_np, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    abi.moe_permute(cfg, ids, T, offs, perm, inv, ws)
    torch.cuda.synchronize()
    st = abi.moe_check_status(ws)
    return offs.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy(), st


def _distinct_ids(rng, T, E, k, p=None):
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(1, 16, 4), (64, 16, 4), (1023, 256, 8), (1025, 256, 8),
                                   (8192, 256, 8), (4097, 64, 2), (333, 1024, 32), (100, 8, 8)])
def test_permute_bitexact(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    ids = _distinct_ids(rng, T, E, k)
    offs, perm, inv, st = _permute_gpu(E, k, ids)
    o, p, i = orc.permute(ids, E)
    assert st == 0
    assert np.array_equal(offs, o) and np.array_equal(perm, p) and np.array_equal(inv, i)


def test_permute_skewed_and_empty_experts():
    rng = np.random.default_rng(5)
    E, k, T = 256, 8, 3000
    pop = 1.0 / np.arange(1, E + 1) ** 1.5
    pop[-20:] = 0.0
    ids = _distinct_ids(rng, T, E, k, p=pop / pop.sum())
    offs, perm, inv, st = _permute_gpu(E, k, ids)
    o, p, i = orc.permute(ids, E)
    assert st == 0 and np.array_equal(offs, o) and np.array_equal(perm, p) and np.array_equal(inv, i)
    assert (np.diff(o)[-20:] == 0).all()
    # every pair on one expert (k = 1)
    ids1 = np.full((500, 1), 7, dtype=np.int32)
    offs, perm, inv, st = _permute_gpu(16, 1, ids1)
    o, p, i = orc.permute(ids1, 16)
    assert st == 0 and np.array_equal(offs, o) and np.array_equal(perm, p) and np.array_equal(inv, i)


def test_permute_flags_out_of_range_ids():
    ids = np.array([[0, 3], [1, 16]], dtype=np.int32)
    offs, perm, inv, st = _permute_gpu(16, 2, ids)
    assert st == 1  # MOE_ERR_INVALID_ARG recorded by the kernel
    assert inv[3] == -1 and offs[-1] == 3
    # the status word was cleared by the read
    _, _, _, st2 = _permute_gpu(16, 2, np.array([[0, 3]], dtype=np.int32))
    assert st2 == 0
