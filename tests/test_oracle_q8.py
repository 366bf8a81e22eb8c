"""Pins of the oracle's quantised-weight functions (E4M3 codes with fp32 row scales) against
what the format and the mathematics fix: decoded values worked out by hand from the format's
definition, encoding as the nearest code by brute force over all finite codes, and the layer
on exactly representable weights equal to the bf16 oracle's layer.  CPU only."""
import numpy as np
import pytest

from oracle import moe_oracle as orc

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)  # NaN excluded


def test_e4m3_decoding_fixed_values():
    # (code, value) from sign / exponent (bias 7) / 3 fraction bits; exponent 0 is subnormal
    table = [(0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
             (0x30, 0.5), (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x48, 4.0),
             (0x77, 240.0), (0x78, 256.0), (0x7E, 448.0), (0xB8, -1.0), (0xFE, -448.0)]
    got = orc.e4m3_to_f64([c for c, _ in table])
    np.testing.assert_array_equal(got, [v for _, v in table])
    assert np.isnan(orc.e4m3_to_f64([0x7F])[0]) and np.isnan(orc.e4m3_to_f64([0xFF])[0])
    assert np.signbit(orc.e4m3_to_f64([0x80])[0])


def test_e4m3_decoding_is_monotone_and_symmetric():
    pos = orc.e4m3_to_f64(np.arange(0x00, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    np.testing.assert_array_equal(orc.e4m3_to_f64(np.arange(0x80, 0xFF, dtype=np.uint8)), -pos)


def _nearest_code(v, vals):
    """Brute force: the finite code nearest to v; on a tie the one with the even fraction."""
    v = max(min(v, 448.0), -448.0)
    d = np.abs(vals - v)
    best = np.flatnonzero(d == d.min())
    if len(best) > 1:
        even = [b for b in best if (FINITE[b] & 1) == 0]
        best = even
    # +0 and -0 are both exact for v == 0: take the code with v's sign
    cands = FINITE[best]
    if len(cands) > 1:
        cands = [c for c in cands if bool(c & 0x80) == bool(np.signbit(v))]
    return int(cands[0])


def test_e4m3_encoding_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(7)
    vals = orc.e4m3_to_f64(FINITE)
    tests = list(rng.standard_normal(400) * 3.0) + list(rng.standard_normal(200) * 200.0)
    tests += list(rng.uniform(-2.0 ** -6, 2.0 ** -6, 200))               # subnormal range
    tests += [1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 464.0, 470.0, 1000.0, -1000.0, 0.0]
    midpoints = (vals[1:128][:-1] + vals[1:128][1:]) / 2                # exact ties between codes
    tests += list(midpoints[::3])
    for v in tests:
        v32 = float(np.float32(v))
        assert orc.float_to_e4m3(v32) == _nearest_code(v32, vals), v32


def test_row_quantisation_scales_and_codes():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((6, 40)) * 0.05).astype(np.float32)
    w[2] = 0.0                                                          # an all-zero row: scale 1
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)                  # bf16 (truncation is fine: any bf16 data)
    q, s = orc.quantize_e4m3_rows(bits)
    wb = orc.bf16_to_f64(bits).astype(np.float32)
    for r in range(6):
        amax = np.float32(np.abs(wb[r]).max())
        want = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        assert s[r] == want
        for c in range(40):
            assert q[r, c] == orc.float_to_e4m3(float(np.float32(wb[r, c] / s[r])))
    # the row's largest magnitude maps to the largest code, and reconstruction is within half a
    # code step of each value (relative 2^-4 for normal codes)
    rec = orc.e4m3_to_f64(q) * s[:, None].astype(np.float64)
    err = np.abs(rec - wb.astype(np.float64))
    assert np.all(err <= np.maximum(np.abs(wb) * 2.0 ** -4, s[:, None] * 2.0 ** -9 * 0.5 + 1e-30))


@pytest.mark.parametrize("Is", [0, 32])
def test_quantised_layer_equals_bf16_layer_on_exact_weights(Is):
    """Scales that are powers of two make scale * code a bf16 value exactly (4 significant bits);
    the bf16 oracle on those bf16 weights must then give the same bits."""
    rng = np.random.default_rng(11 + Is)
    H, E, k, I, T = 64, 6, 2, 32, 5
    codes = FINITE[np.abs(orc.e4m3_to_f64(FINITE)) <= 8.0]              # moderate magnitudes

    def qmat(rows, cols):
        q = rng.choice(codes, size=(rows, cols)).astype(np.uint8)
        s = (2.0 ** rng.integers(-9, -5, size=rows)).astype(np.float32)
        return q, s

    def to_bf16(q, s):
        v = orc.e4m3_to_f64(q) * s[:, None].astype(np.float64)
        bits = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal(orc.bf16_to_f64(bits), v)                 # exactly representable
        return bits

    wq, wb = {}, {}
    for name, (rows, cols) in (("gate", (I, H)), ("up", (I, H)), ("down", (H, I))):
        qs, ss, bs = [], [], []
        for _ in range(E):
            q, s = qmat(rows, cols)
            qs.append(q); ss.append(s); bs.append(to_bf16(q, s))
        wq["q_" + name], wq["s_" + name] = np.stack(qs), np.stack(ss)
        wb["w_" + name] = np.stack(bs)
    if Is:
        for name, (rows, cols) in (("gate", (Is, H)), ("up", (Is, H)), ("down", (H, Is))):
            q, s = qmat(rows, cols)
            wq["qs_" + name], wq["ss_" + name] = q, s
            wb["ws_" + name] = to_bf16(q, s)
    wb["w_router"] = np.zeros((E, H), dtype=np.uint16)
    x = (rng.standard_normal((T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    got = orc.forward_q8(x, wq, k, ids, w)
    want = orc.forward(x, wb, k, ids=ids, topk_w=w)["out"]
    np.testing.assert_array_equal(got, want)
