"""Device-side failure reporting, without faulting, trapping or hanging the GPU.

Every wait in the library's kernels is bounded: a wait that runs out records MOE_ERR_TIMEOUT in
the workspace status word and the kernel returns.  moe_selftest_wait runs that same wait on a
barrier nothing ever arrives at (a flag nothing sets), with a short limit, so the failure path
runs for real; the context must stay usable afterwards.  (Out-of-range expert ids, the other
device-reported error, are covered with the permutation tests.)"""
import time

import pytest

from sparse_moe_router_gb300 import abi, inputs

from helpers import check_layer, make

pytestmark = pytest.mark.gpu

TIMEOUT = 5


def _ws():
    return abi.alloc_workspace(abi.config(hidden=256, n_experts=16, top_k=4, inter=128, shared_inter=128), 4)


def test_wait_that_runs_out_reports_timeout_and_returns():
    ws = _ws()
    t0 = time.perf_counter()
    abi.moe_selftest_wait(ws, 2_000_000, arrive=False)     # 2 ms, nothing arrives
    assert abi.moe_check_status(ws) == TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert abi.moe_check_status(ws) == 0                    # read and cleared


def test_wait_that_completes_reports_nothing():
    ws = _ws()
    abi.moe_selftest_wait(ws, 2_000_000, arrive=True)
    assert abi.moe_check_status(ws) == 0


def test_context_usable_after_a_timeout():
    ws = _ws()
    for _ in range(3):
        abi.moe_selftest_wait(ws, 1_000_000, arrive=False)
        assert abi.moe_check_status(ws) == TIMEOUT
    shape = inputs.Shape(256, 16, 4, 128, 128)
    layers, x = make(shape, 64, seed=3)
    check_layer(shape, layers[0], x)


def test_selftest_rejects_bad_arguments():
    ws = _ws()
    with pytest.raises(abi.MoeError):
        abi.moe_selftest_wait(ws, 2_000_000_000, arrive=False)  # limit above 1 s
    with pytest.raises(abi.MoeError):
        abi.moe_selftest_wait(ws[:64], 1000, arrive=False)      # smaller than the status area

