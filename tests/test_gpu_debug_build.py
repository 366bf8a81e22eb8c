"""The MOE_DEBUG build of the library (libmoe_debug.so): the same layer results, and indices read
from device data that fall outside their buffers reported in the status word instead of used.

Runs in a child process, which loads the debug library alone; the bad inputs below are only
ever given to that library (its checks skip every access they would make out of bounds)."""
import os
import subprocess
import sys
import textwrap

import pytest

from sparse_moe_router_gb300 import build as lib_build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys
    sys.path.insert(0, sys.argv[2])
    import numpy as np
    import torch
    from oracle import moe_oracle as orc
    from sparse_moe_router_gb300 import abi, inputs
    sys.path.insert(0, sys.argv[2] + "/tests")
    from helpers import compare_out, route_gpu, u16

    L = abi.load(sys.argv[1])
    assert L.moe_debug_build() == 1, "not the debug build"
    shape = inputs.Shape(256, 16, 4, 128, 128)
    T, k = 64, 4
    P = T * k
    layers, x = inputs.make(inputs.custom(shape, T=T, seed=31), device="cuda")
    cfg = abi.config_of(shape)
    ws = abi.alloc_workspace(cfg, T)
    w = abi.weights(layers[0])

    # 1. a valid layer: the checks change nothing
    out = torch.empty_like(x)
    abi.moe_forward(cfg, w, x, T, out, None, ws)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    logits, ids, tw = route_gpu(shape, layers[0], x, ws=ws)
    ref = orc.forward(u16(x), inputs.layer_to_host(layers[0]), k, ids=ids, topk_w=tw)["out"]
    compare_out(u16(out), ref, what="debug build layer")

    # 2. moe_expert_ffn on a permutation naming pairs past T*k and offsets past T*k: reported
    offs, perm, inv = (torch.as_tensor(a, device="cuda") for a in orc.permute(ids, shape.n_experts))
    bad_perm = perm.clone()
    bad_perm[::7] = 10 ** 7
    bad_offs = offs.clone()
    bad_offs[-1] = P + 64
    h = torch.empty(P, shape.inter, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(P, shape.hidden, dtype=torch.float32, device="cuda")
    for po, pp in ((offs, bad_perm), (bad_offs, perm)):
        abi.moe_expert_ffn(cfg, w, x, T, po, pp, h, y, None, ws)
        torch.cuda.synchronize()
        assert abi.moe_check_status(ws) == 1, "bad index not reported"

    # 3. moe_combine with rows past the y rows it was given: skipped (this call has no status word)
    abi.moe_expert_ffn(cfg, w, x, T, offs, perm, h, y, None, ws)
    bad_inv = inv.clone()
    bad_inv[::5] = 10 ** 7
    out2 = torch.empty_like(x)
    abi.moe_combine(cfg, y, bad_inv, torch.as_tensor(tw, device="cuda"), None, T, out2)
    torch.cuda.synchronize()
    assert torch.isfinite(out2.float()).all()

    # 4. the context is still usable: the valid layer again, bit-identical
    out3 = torch.empty_like(x)
    abi.moe_forward(cfg, w, x, T, out3, None, ws)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0 and torch.equal(out3, out)
    print("debug build ok")
""")


def test_debug_build_checks_indices():
    path = lib_build.build(debug=True)
    r = subprocess.run([sys.executable, "-c", SCRIPT, path, ROOT], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "debug build ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
