"""Pins of the oracle's 4-bit integer block quantisation (Q4: blocks of 32 columns, one fp32
scale per block, codes in [-7, 7] as two's-complement nibbles) against what the format and the
mathematics fix: codes and scales worked out by hand, the nibble packing, ties to even, the
all-zero block, the reconstruction error bound, and the layer on exactly representable weights
equal to the bf16 oracle's layer.  CPU only."""
import numpy as np
import pytest

from oracle import moe_oracle as orc


def _bf16(v):
    """float values that are bf16 values -> bf16 bits (checked exact)."""
    f = np.asarray(v, dtype=np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(orc.bf16_to_f64(bits), f.astype(np.float64))
    return bits


def test_hand_worked_block():
    # amax 3.5 -> scale 0.5 (3.5 / 7 is exact); w / 0.5 = 2 w, rounded half to even
    vals = np.zeros(32, dtype=np.float32)
    vals[:12] = [3.5, -3.5, 0.25, 0.75, -0.25, 1.0, 0.0, -1.25, 1.75, 2.25, -0.75, 0.5]
    q, s = orc.quantize_q4_rows(_bf16(vals)[None, :])
    assert q.shape == (1, 16) and s.shape == (1, 1)
    assert s[0, 0] == np.float32(0.5)
    # 2w = 7, -7, 0.5 -> 0 (even), 1.5 -> 2, -0.5 -> -0 = 0, 2, 0, -2.5 -> -2, 3.5 -> 4, 4.5 -> 4,
    #      -1.5 -> -2, 1
    want = [7, -7, 0, 2, 0, 2, 0, -2, 4, 4, -2, 1] + [0] * 20
    np.testing.assert_array_equal(orc.q4_codes(q[0]), want)
    # packing: column 2j in the low nibble of byte j, 2j+1 in the high nibble; two's complement
    assert q[0, 0] == ((-7 & 15) << 4 | 7)
    assert q[0, 1] == (2 << 4 | 0)
    assert q[0, 3] == ((-2 & 15) << 4 | 0)


def test_zero_block_and_block_independence():
    rng = np.random.default_rng(5)
    vals = (rng.standard_normal((3, 96)) * 0.1).astype(np.float32)
    vals[1, 32:64] = 0.0                                    # an all-zero block: scale 1, codes 0
    vals[2, :32] *= 1000.0                                  # one large block does not touch the others
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    q, s = orc.quantize_q4_rows(bits)
    assert s[1, 1] == np.float32(1.0)
    np.testing.assert_array_equal(orc.q4_codes(q[1])[32:64], np.zeros(32))
    q_small, s_small = orc.quantize_q4_rows(bits[2:3, 32:])
    np.testing.assert_array_equal(q[2, 16:], q_small[0])
    np.testing.assert_array_equal(s[2, 1:], s_small[0])


def test_codes_are_nearest_and_error_bounded():
    rng = np.random.default_rng(9)
    vals = (rng.standard_normal((8, 64)) * 0.03).astype(np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    wb = orc.bf16_to_f64(bits).astype(np.float32)
    q, s = orc.quantize_q4_rows(bits)
    for r in range(8):
        codes = orc.q4_codes(q[r])
        for b in range(2):
            blk = wb[r, 32 * b:32 * b + 32]
            amax = np.float32(np.abs(blk).max())
            sc = np.float32(amax / np.float32(7.0))
            assert s[r, b] == sc
            c = codes[32 * b:32 * b + 32]
            assert np.abs(c).max() == 7                      # the block's largest magnitude takes +-7
            ratio = (blk / sc).astype(np.float64)           # the fp32 quotient the code rounds
            # nearest integer: no other code in [-7, 7] is closer
            assert np.all(np.abs(ratio - c) <= 0.5 + 1e-6)
            # reconstruction within half a step of the block's scale
            assert np.all(np.abs(c * np.float64(sc) - blk) <= 0.5 * np.float64(sc) * (1 + 1e-6))


@pytest.mark.parametrize("Is", [0, 32])
def test_q4_layer_equals_bf16_layer_on_exact_weights(Is):
    """Power-of-two scales make scale * code a bf16 value exactly (codes have 3 significant bits);
    the bf16 oracle on those weights must give the same bits.  The blocks are built so that
    quantising the bf16 weights reproduces the codes and scales (each block reaches +-7)."""
    rng = np.random.default_rng(21 + Is)
    H, E, k, I, T = 64, 5, 2, 32, 4

    def qmat(rows, cols):
        codes = rng.integers(-7, 8, size=(rows, cols))
        codes[:, ::32] = 7 * np.where(rng.random((rows, cols // 32)) < 0.5, 1, -1)  # each block reaches +-7
        s = (2.0 ** rng.integers(-9, -5, size=(rows, cols // 32))).astype(np.float32)
        v = codes * np.repeat(s, 32, axis=1).astype(np.float64)
        bits = _bf16(v.astype(np.float32))
        q, sq = orc.quantize_q4_rows(bits)
        np.testing.assert_array_equal(sq, s)
        for r in range(rows):
            np.testing.assert_array_equal(orc.q4_codes(q[r]), codes[r])
        return q, sq, bits

    wq, wb = {}, {}
    for name, (rows, cols) in (("gate", (I, H)), ("up", (I, H)), ("down", (H, I))):
        qs, ss, bs = [], [], []
        for _ in range(E):
            q, s, b = qmat(rows, cols)
            qs.append(q); ss.append(s); bs.append(b)
        wq["q_" + name], wq["s_" + name] = np.stack(qs), np.stack(ss)
        wb["w_" + name] = np.stack(bs)
    if Is:
        for name, (rows, cols) in (("gate", (Is, H)), ("up", (Is, H)), ("down", (H, Is))):
            q, s, b = qmat(rows, cols)
            wq["qs_" + name], wq["ss_" + name] = q, s
            wb["ws_" + name] = b
    wb["w_router"] = np.zeros((E, H), dtype=np.uint16)
    x = (rng.standard_normal((T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    got = orc.forward_q4(x, wq, k, ids, w)
    want = orc.forward(x, wb, k, ids=ids, topk_w=w)["out"]
    np.testing.assert_array_equal(got, want)
