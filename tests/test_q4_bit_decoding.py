"""The 4-bit decode kernels' code widening, restated on the CPU against the format's definition
(two's-complement nibbles, column 2j in the low nibble of byte j, 8 columns a little-endian
32-bit word): flip bit 3 of every nibble, mask the nibble pair (s, s + 4) of a word into
0x43004300, subtract 136 from both bf16 halves.  Each half must be the code of its column."""
import numpy as np


def _bf16_value(bits):
    return float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0])


def _code(nibble):
    return nibble - 16 if nibble >= 8 else nibble


def test_every_nibble_value():
    for n in range(16):
        u = n ^ 8
        v = _bf16_value(0x4300 | u)
        assert v == 128.0 + u                       # 7 fraction bits at exponent 7: steps of 1
        assert v - 136.0 == _code(n)                # the subtraction is exact (integers below 256)


def test_pairs_of_a_word_map_to_columns():
    rng = np.random.default_rng(11)
    for _ in range(200):
        codes = rng.integers(-7, 8, size=8)        # columns 0..7 of one word
        nib = [int(c) & 15 for c in codes]
        byts = [nib[2 * j] | (nib[2 * j + 1] << 4) for j in range(4)]  # column 2j low, 2j+1 high
        w = int.from_bytes(bytes(byts), "little") ^ 0x88888888
        for s in range(4):
            t = ((w >> (4 * s)) & 0x000F000F) | 0x43004300
            lo, hi = t & 0xFFFF, t >> 16
            assert _bf16_value(lo) - 136.0 == codes[s]
            assert _bf16_value(hi) - 136.0 == codes[s + 4]
