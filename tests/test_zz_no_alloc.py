"""moe_permute_noalloc: the permutation for callers that cannot allocate device memory where
they route tokens (a process that reserves all device memory at start-up, host code with no
allocator).  It takes no workspace: its scratch table is a fixed array inside the library.

This file is collected last, so a run that stops at the first failure has already run every
other test.  The checks pass alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_moe_router_gb300 import abi

pytestmark = pytest.mark.gpu


def _ids(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


def _with_workspace(cfg, ids):
    T, k = ids.shape
    ws = abi.alloc_workspace(cfg, T)
    offs = torch.empty(cfg.n_experts + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    abi.moe_permute(cfg, torch.as_tensor(ids, device="cuda"), T, offs, perm, inv, ws)
    torch.cuda.synchronize()
    return offs.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy()


def _no_alloc(cfg, ids):
    T, k = ids.shape
    offs = torch.full((cfg.n_experts + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    abi.moe_permute_noalloc(cfg, torch.as_tensor(ids, device="cuda"), T, offs, perm, inv)
    torch.cuda.synchronize()
    return offs.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy()


@pytest.mark.parametrize("T,E,k", [(8192, 256, 8), (1000, 64, 6), (3, 16, 4)])
def test_no_alloc_permute_matches_workspace_permute_twice(T, E, k):
    """Two calls in a row (different inputs, so the second reuses the table the first left
    behind) each match moe_permute and the oracle's permutation exactly (integer outputs: the
    tolerance is zero)."""
    cfg = abi.config(2048, E, k, 512, 512)
    for seed in (1, 2):
        ids = _ids(T, E, k, seed + T)
        want = _with_workspace(cfg, ids)
        got = _no_alloc(cfg, ids)
        for g, w in zip(got, want):
            assert np.array_equal(g, w)
        # and against the CPU oracle's stable counting sort
        for g, o in zip(got, orc.permute(ids, E)):
            assert np.array_equal(g, o)


def test_no_alloc_permute_rejects_oversize_problems():
    L = abi.load()
    cfg = abi.config(2048, 256, 8, 512, 512)
    fake = ctypes.c_void_p(0x10000)   # never touched: the size check fails first
    assert L.moe_permute_noalloc(ctypes.byref(cfg), fake, 8193, fake, fake, fake, None) == 3
    big_e = abi.config(2048, 1025, 8, 512, 512)
    assert L.moe_permute_noalloc(ctypes.byref(big_e), fake, 16, fake, fake, fake, None) == 3
