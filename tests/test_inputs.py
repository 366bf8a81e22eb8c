"""The seeded input generators (CPU): reproducible draws of the documented shapes and ranges."""
import numpy as np
import torch

from sparse_moe_router_gb300 import inputs

TINY = inputs.Shape(256, 16, 4, 128, 128)


def test_make_is_reproducible_and_shaped():
    w = inputs.custom(TINY, T=12, seed=5, n_layers=2, zipf_s=1.0)
    a_layers, a_x = inputs.make(w)
    b_layers, b_x = inputs.make(w)
    assert torch.equal(a_x, b_x) and a_x.shape == (12, 256) and a_x.dtype == torch.bfloat16
    for la, lb in zip(a_layers, b_layers):
        for k in la:
            if la[k] is None:
                assert lb[k] is None
            else:
                assert torch.equal(la[k], lb[k])
    l0 = a_layers[0]
    assert l0["w_gate"].shape == (16, 128, 256) and l0["w_down"].shape == (16, 256, 128)
    assert l0["ws_down"].shape == (256, 128) and l0["b_router"].dtype == torch.float32
    # Zipf bias: -s ln(rank) over a permutation of 1..E
    ranks = np.exp(-l0["b_router"].numpy().astype(np.float64))
    assert sorted(np.round(ranks).astype(int).tolist()) == list(range(1, 17))


def test_make_q8_codes_scales_and_router():
    w = inputs.custom(TINY, T=3, seed=9, n_layers=2)
    layers, x = inputs.make_q8(w)
    bf_layers, bf_x = inputs.make(w)
    for l, bl in zip(layers, [bf_layers[0], None]):
        for q, sc, shp in (("q_gate", "s_gate", (16, 128, 256)), ("q_up", "s_up", (16, 128, 256)),
                           ("q_down", "s_down", (16, 256, 128)), ("qs_gate", "ss_gate", (128, 256)),
                           ("qs_up", "ss_up", (128, 256)), ("qs_down", "ss_down", (256, 128))):
            codes = l[q].numpy()
            assert l[q].dtype == torch.uint8 and codes.shape == shp
            assert not np.any((codes & 0x7F) == 0x7F)  # no NaN pattern
            s = l[sc].numpy()
            assert s.shape == shp[:-1] and s.dtype == np.float32
            assert np.all(s >= 0.5 * 2e-4) and np.all(s <= 1.5 * 2e-4)
        if bl is not None:  # the router is drawn first, exactly as in the bf16 recipe
            assert torch.equal(l["w_router"], bl["w_router"])
    # all 254 finite codes occur in a large enough draw
    assert len(np.unique(layers[0]["q_gate"].numpy())) == 254
    assert x.shape == (3, 256) and x.dtype == torch.bfloat16


def test_make_q8_without_shared_expert():
    shape = inputs.Shape(256, 16, 4, 128, 0)
    layers, _ = inputs.make_q8(inputs.custom(shape, T=2, seed=1))
    assert "qs_gate" not in layers[0] and "q_gate" in layers[0]
