"""Pins of the CPU oracle against what the mathematics and library routines fix.

Each test checks one oracle function against something other than itself: a hand-worked
closed form, a library routine (numpy / torch / scipy), an invariant, a special case that
reduces to a textbook operation, or brute force on tiny inputs.  Chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe_oracle as orc
from sparse_moe_router_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(a):
    """float array (exactly representable or not) -> bf16 bits via torch's RNE cast of fp32."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _tiny(seed=0, T=24, shape=None, **kw):
    shape = shape or inputs.Shape(64, 8, 3, 32, 32)
    w = inputs.custom(shape, T=T, seed=seed, **kw)
    layers, x = inputs.make(w, device="cpu")
    return inputs.layer_to_host(layers[0]), inputs.to_u16(x), shape


# ------------------------------------------------------------------ rounding helpers --

def test_bf16_rounding_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1.0, -1.0, 3.3895e38, 1e-40, -1e-42]]).astype(np.float32)
    want = _bf16_bits(v)
    got = np.array([orc.double_to_bf16(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rounding_ties_and_single_rounding():
    # Exact ties round to even.
    assert orc.double_to_bf16(1.0 + 2 ** -8) == 0x3F80          # between 0x3F80 and 0x3F81
    assert orc.double_to_bf16(1.0 + 3 * 2 ** -8) == 0x3F82      # between 0x3F81 and 0x3F82
    assert orc.double_to_bf16(-(1.0 + 2 ** -8)) == 0xBF80
    # Just above a tie must round up: a conversion through fp32 would lose the 2^-40 and
    # round the resulting tie to even (0x3F80): one rounding step is required.
    assert orc.double_to_bf16(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert orc.double_to_bf16(float("inf")) == 0x7F80
    assert orc.double_to_bf16(3.5e38) == 0x7F80                  # above max finite -> inf
    assert orc.double_to_bf16(2 ** -133) == 0x0001               # smallest subnormal
    assert orc.double_to_bf16(2 ** -134) == 0x0000               # tie with 0 -> even (0)
    for b in (0x0001, 0x3F80, 0x4049, 0xC2F7, 0x7F7F, 0x8000):
        assert orc.double_to_bf16(orc.bf16_to_f64(np.array([b]))[0]) == b


def test_silu_matches_library():
    g = np.linspace(-30, 30, 1201)
    want = torch.nn.functional.silu(torch.as_tensor(g, dtype=torch.float64)).numpy()
    got = np.array([orc.silu(v) for v in g])
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-300)
    assert orc.silu(0.0) == 0.0


# -------------------------------------------------------------- worked closed form --

def test_worked_example_closed_form():
    with open(os.path.join(GOLDEN, "worked_tiny.json")) as f:
        g = json.load(f)
    inp, exp_ = g["inputs"], g["expected"]
    w = {k: _bf16_bits(v) for k, v in inp.items() if k != "x"}
    for k, v in inp.items():
        if k != "x":   # every input is exactly representable: check the fixture itself
            assert np.array_equal(orc.bf16_to_f64(w[k]), np.asarray(v, dtype=np.float64))
    x = _bf16_bits(inp["x"])
    k = g["shape"]["top_k"]
    logits = orc.router_logits(x, w["w_router"])
    assert np.array_equal(logits, np.asarray(exp_["logits"], dtype=np.float32))
    ids, wt = orc.route_from_logits(logits, k)
    assert ids.tolist() == exp_["ids"]
    e = math.e
    assert wt[0, 0] == np.float32(e / (e + 1)) and wt[0, 1] == np.float32(1 / (e + 1))
    assert wt.tolist() == exp_["w_fp32"]
    res = orc.forward(x, w, k, want_f64=True)
    assert [[hex(b) for b in row] for row in res["out"]] == exp_["out_bits"]
    np.testing.assert_allclose(res["out_f64"], exp_["out_unrounded"], rtol=1e-13)
    # h rows: the permuted order holds expert 1 (row 0) then expert 2 (row 1).
    offs, perm, inv = orc.permute(ids, 4)
    h_rows, y_rows, shared_y = orc.expert_ffn(x, offs, perm, k, w)
    assert hex(h_rows[inv[1], 0]) == exp_["h_bits_by_expert"]["1"]
    assert hex(h_rows[inv[0], 0]) == exp_["h_bits_by_expert"]["2"]
    assert np.allclose(shared_y, 187 * 2 ** -9)


# ------------------------------------------------------------------- router logits --

def test_router_logits_match_library_matmul():
    w, x, s = _tiny(seed=3, T=17)
    b = np.random.default_rng(0).standard_normal(s.n_experts).astype(np.float32)
    got = orc.router_logits(x, w["w_router"], b)
    ref = (orc.bf16_to_f64(x) @ orc.bf16_to_f64(w["w_router"]).T).astype(np.float32) + b
    assert np.array_equal(got, ref)
    got0 = orc.router_logits(x, w["w_router"], None)
    assert np.array_equal(got0, (orc.bf16_to_f64(x) @ orc.bf16_to_f64(w["w_router"]).T).astype(np.float32))


# ------------------------------------------------------------------------ top-k --

def _stable_topk(l, k):
    # Library routine: stable sort of -l keeps the lower index first among equal logits.
    return np.argsort(-l.astype(np.float64), kind="stable")[:k]


def test_topk_matches_stable_sort_with_many_ties():
    rng = np.random.default_rng(7)
    T, E, k = 10000, 16, 4
    # Logits on a coarse grid so equal values are frequent.
    logits = (np.round(rng.standard_normal((T, E)) * 4) / 4).astype(np.float32)
    ids, w = orc.route_from_logits(logits, k)
    ref = np.stack([_stable_topk(l, k) for l in logits])
    assert np.array_equal(ids, ref)
    # Weights: softmax over the selected logits (the full denominator cancels).
    sel = np.take_along_axis(logits.astype(np.float64), ref, axis=1)
    ref_w = scipy.special.softmax(sel, axis=1).astype(np.float32)
    np.testing.assert_allclose(w, ref_w, rtol=3e-7, atol=0)


def test_topk_brute_force_tiny():
    # Every assignment of values {0,1,2} to E=4 logits, every k: brute force over subsets.
    import itertools
    for vals in itertools.product([0.0, 1.0, 2.0], repeat=4):
        l = np.asarray(vals, dtype=np.float32)[None]
        for k in range(1, 5):
            ids, _ = orc.route_from_logits(l, k)
            # brute force: the lexicographically best subset by (sum of ranks in sorted order)
            order = sorted(range(4), key=lambda e: (-vals[e], e))
            assert ids[0].tolist() == order[:k]


def test_topk_all_equal_logits():
    for E, k in [(16, 4), (16, 3), (256, 8), (7, 7)]:
        ids, w = orc.route_from_logits(np.full((3, E), 0.375, dtype=np.float32), k)
        assert (ids == np.arange(k)).all()
        assert (w == np.float32(1.0 / k)).all()


def test_topk_k1_weight_is_one():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((500, 16)).astype(np.float32)
    ids, w = orc.route_from_logits(logits, 1)
    assert (w == 1.0).all()
    assert np.array_equal(ids[:, 0], np.argmax(logits, axis=1))


def test_topk_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(4)
    logits = (rng.standard_normal((300, 16)) * 3).astype(np.float32)
    ids, w = orc.route_from_logits(logits, 16)
    ref_ids = np.stack([_stable_topk(l, 16) for l in logits])
    assert np.array_equal(ids, ref_ids)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    ref_w = np.take_along_axis(p, ref_ids, axis=1).astype(np.float32)
    np.testing.assert_allclose(w, ref_w, rtol=3e-7, atol=1e-30)


def test_weights_sum_to_one_and_lie_in_unit_interval():
    rng = np.random.default_rng(5)
    for E, k in [(16, 4), (256, 8), (64, 6)]:
        logits = (rng.standard_normal((400, E)) * rng.uniform(0.1, 8)).astype(np.float32)
        _, w = orc.route_from_logits(logits, k)
        assert (w > 0).all() and (w <= 1).all()
        s = w.astype(np.float64).sum(axis=1)
        assert np.all(np.abs(s - 1.0) <= 4 * 2 ** -23)


# ---------------------------------------------------------------------- permute --

def test_permute_is_stable_sort_by_expert():
    rng = np.random.default_rng(11)
    for T, E, k in [(64, 16, 4), (1, 8, 3), (333, 32, 8), (50, 4, 4)]:
        logits = rng.standard_normal((T, E)).astype(np.float32)
        ids, _ = orc.route_from_logits(logits, k)
        offs, perm, inv = orc.permute(ids, E)
        flat = ids.ravel()
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        assert np.array_equal(offs, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        assert offs[-1] == T * k and np.all(np.diff(offs) >= 0)
        assert np.array_equal(inv[perm], np.arange(T * k))
        assert np.array_equal(perm[inv], np.arange(T * k))
        # each token appears in exactly k distinct expert groups
        groups = np.searchsorted(offs, np.arange(T * k), side="right") - 1
        tok_groups = {}
        for row, p in enumerate(perm):
            tok_groups.setdefault(p // k, set()).add(groups[row])
        assert all(len(v) == k for v in tok_groups.values()) and len(tok_groups) == T


def test_permute_empty_and_single_expert():
    ids = np.zeros((10, 1), dtype=np.int32) + 3
    offs, perm, inv = orc.permute(ids, 5)
    assert offs.tolist() == [0, 0, 0, 0, 10, 10]
    assert perm.tolist() == list(range(10))
    with pytest.raises(ValueError):
        orc.permute(np.array([[5]], dtype=np.int32), 5)


# --------------------------------------------------------------- FFN and combine --

def _torch_swiglu(x64, wg64, wu64, wd64, round_h):
    g = x64 @ wg64.T
    u = x64 @ wu64.T
    a = torch.nn.functional.silu(g) * u
    if round_h:
        a = a.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    return a @ wd64.T


def test_single_expert_reduces_to_dense_swiglu():
    shape = inputs.Shape(64, 1, 1, 48, 0)
    w, x, _ = _tiny(seed=9, T=20, shape=shape)
    res = orc.forward(x, w, 1, exact=True, want_f64=True)
    t = lambda a: torch.as_tensor(orc.bf16_to_f64(a))
    ref = _torch_swiglu(t(x), t(w["w_gate"][0]), t(w["w_up"][0]), t(w["w_down"][0]), False)
    np.testing.assert_allclose(res["out_f64"], ref.numpy(), rtol=1e-12, atol=1e-14)
    assert (res["w"] == 1.0).all() and (res["ids"] == 0).all()
    # rounded-h mode: within one bf16 spacing of the library evaluation
    res_r = orc.forward(x, w, 1, want_f64=True)
    ref_r = _torch_swiglu(t(x), t(w["w_gate"][0]), t(w["w_up"][0]), t(w["w_down"][0]), True)
    np.testing.assert_allclose(res_r["out_f64"], ref_r.numpy(), rtol=1e-6, atol=1e-7)


def test_zero_input_gives_zero_output():
    w, x, _ = _tiny(seed=1)
    res = orc.forward(np.zeros_like(x), w, 3)
    assert (res["out"] & 0x7FFF == 0).all()


def test_zero_routed_down_leaves_shared_expert():
    w, x, s = _tiny(seed=2)
    w0 = dict(w)
    w0["w_down"] = np.zeros_like(w["w_down"])
    res = orc.forward(x, w0, s.top_k, exact=True, want_f64=True)
    t = lambda a: torch.as_tensor(orc.bf16_to_f64(a))
    ref = _torch_swiglu(t(x), t(w["ws_gate"]), t(w["ws_up"]), t(w["ws_down"]), False)
    np.testing.assert_allclose(res["out_f64"], ref.numpy(), rtol=1e-12, atol=1e-14)


def test_sparse_equals_dense_masked_library():
    """Sparse top-k evaluation == dense all-experts evaluation masked to the chosen k.

    The dense form is evaluated twice: by the oracle's expert-major loop and by torch
    float64 matmuls over all experts (library routines)."""
    w, x, s = _tiny(seed=5, T=16)
    res = orc.forward(x, w, s.top_k, exact=True, want_f64=True)
    dm = orc.dense_masked(x, w, res["ids"], res["w"], exact=True)
    np.testing.assert_allclose(res["out_f64"], dm, rtol=1e-12, atol=1e-13)
    t = lambda a: torch.as_tensor(orc.bf16_to_f64(a))
    xt = t(x)
    mask = torch.zeros(x.shape[0], s.n_experts, dtype=torch.float64)
    mask.scatter_(1, torch.as_tensor(res["ids"], dtype=torch.int64),
                  torch.as_tensor(res["w"], dtype=torch.float64))
    ref = torch.zeros(x.shape[0], s.hidden, dtype=torch.float64)
    for e in range(s.n_experts):
        y = _torch_swiglu(xt, t(w["w_gate"][e]), t(w["w_up"][e]), t(w["w_down"][e]), False)
        ref += mask[:, e:e + 1] * y
    ref += _torch_swiglu(xt, t(w["ws_gate"]), t(w["ws_up"]), t(w["ws_down"]), False)
    np.testing.assert_allclose(res["out_f64"], ref.numpy(), rtol=1e-11, atol=1e-13)
    # Routing with the oracle's own logits equals the stable-sort top-k of library logits.
    lib_logits = (orc.bf16_to_f64(x) @ orc.bf16_to_f64(w["w_router"]).T).astype(np.float32)
    assert np.array_equal(res["ids"], np.stack([_stable_topk(l, s.top_k) for l in lib_logits]))


def test_token_permutation_permutes_rows():
    w, x, s = _tiny(seed=6, T=19)
    res = orc.forward(x, w, s.top_k)
    p = np.random.default_rng(0).permutation(x.shape[0])
    res_p = orc.forward(np.ascontiguousarray(x[p]), w, s.top_k)
    assert np.array_equal(res_p["out"], res["out"][p])


def test_unfused_pieces_match_whole_layer():
    w, x, s = _tiny(seed=8, T=21)
    res = orc.forward(x, w, s.top_k, want_f64=True)
    logits = orc.router_logits(x, w["w_router"])
    ids, wt = orc.route_from_logits(logits, s.top_k)
    assert np.array_equal(ids, res["ids"]) and np.array_equal(wt, res["w"])
    offs, perm, inv = orc.permute(ids, s.n_experts)
    h_rows, y_rows, shared_y = orc.expert_ffn(x, offs, perm, s.top_k, w)
    out = orc.combine(y_rows, inv, wt, shared_y)
    # y rows and shared_y are rounded to fp32 before the combine: at most one bf16 step apart
    a, b = orc.bf16_to_f64(out), orc.bf16_to_f64(res["out"])
    assert np.all(np.abs(a - b) <= np.abs(b) * 2 ** -7 + 1e-30)
    assert np.mean(out == res["out"]) > 0.99


def test_expert_ffn_given_h_rows():
    """The h_in path of expert_ffn (the GPU down-projection check feeds it the GPU's h rows):
    (a) fed its own h rows it reproduces its own y rows, which equal the whole layer's per-pair
    y (the combine of those rows gives forward's output); (b) fed arbitrary bf16 rows in a
    shuffled row order, row r's y is W_d[e(r)] @ h_in[r] (torch float64 matmul), so a slip of
    the row index, a transposed W_d or a wrong expert base fails."""
    w, x, s = _tiny(seed=14, T=23)
    logits = orc.router_logits(x, w["w_router"])
    ids, wt = orc.route_from_logits(logits, s.top_k)
    offs, perm, inv = orc.permute(ids, s.n_experts)
    h_rows, y_rows, shared_y = orc.expert_ffn(x, offs, perm, s.top_k, w)
    _, y_again, _ = orc.expert_ffn(x, offs, perm, s.top_k, w, h_in=h_rows)
    assert np.array_equal(y_again, y_rows)
    out = orc.combine(y_again, inv, wt, shared_y)
    ref = orc.forward(x, w, s.top_k)["out"]
    a, b = orc.bf16_to_f64(out), orc.bf16_to_f64(ref)
    assert np.all(np.abs(a - b) <= np.abs(b) * 2 ** -7 + 1e-30)
    # (b) shuffled, arbitrary h rows
    rng = np.random.default_rng(3)
    h_any = _bf16_bits(rng.standard_normal(h_rows.shape))
    h_any = np.ascontiguousarray(h_any[rng.permutation(h_any.shape[0])])
    _, y_any, _ = orc.expert_ffn(x, offs, perm, s.top_k, w, h_in=h_any)
    wd = torch.as_tensor(orc.bf16_to_f64(w["w_down"]))
    hv = torch.as_tensor(orc.bf16_to_f64(h_any))
    expert_of_row = np.repeat(np.arange(s.n_experts), np.diff(offs))
    want = torch.stack([wd[int(e)] @ hv[r] for r, e in enumerate(expert_of_row)])
    np.testing.assert_allclose(y_any, want.to(torch.float32).numpy(), rtol=1e-6, atol=1e-7)


def test_x_next_is_rounded_residual():
    w, x, s = _tiny(seed=10, T=9)
    res = orc.forward(x, w, s.top_k, want_x_next=True)
    ref = _bf16_bits(orc.bf16_to_f64(x) + orc.bf16_to_f64(res["out"]))
    # fp32 cast of the fp64 sum is exact here (two bf16 values), so one rounding either way
    assert np.array_equal(res["x_next"], ref)


def test_bias_shifts_selection():
    w, x, s = _tiny(seed=12, T=30)
    b = np.zeros(s.n_experts, dtype=np.float32)
    b[5] = 100.0
    w_b = dict(w, b_router=b)
    res = orc.forward(x, w_b, s.top_k)
    assert (res["ids"][:, 0] == 5).all()


def test_threads_reports_count():
    assert orc.threads(3) == 3 and orc.threads(0) >= 1
