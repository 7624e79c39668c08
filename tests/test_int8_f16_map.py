"""The int8 decode of the 8-bit decode kernel, restated on the host and pinned to the format.

The kernel's dequant warps turn four int8 codes (one 32-bit word) into two f16x2 words:
flip each byte's top bit (code + 128, as an unsigned byte u), place u under the f16 bit
pattern 0x64 (the f16 value 1024 + u, exact: u < 1024 needs no rounding) with two byte
permutes (selector 0x5140 for codes 0 and 1, 0x7362 for codes 2 and 3, second source
0x64646464), then subtract 1152 in f16 (exact: the difference is a small integer).  The
result must equal the two's-complement value of every code, lanes in code order.
"""
import numpy as np


def byte_perm(x, y, sel):
    """Byte permute of two 32-bit words (result byte i = byte (sel >> 4i) & 7 of y:x)."""
    src = [(x >> (8 * k)) & 0xFF for k in range(4)] + [(y >> (8 * k)) & 0xFF for k in range(4)]
    return sum(src[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def halves(word):
    pair = np.array([word & 0xFFFF, word >> 16], dtype=np.uint16)
    return pair.view(np.float16)


def test_int8_map_is_exact_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    want = codes.view(np.int8).astype(np.float64)
    for c0 in range(0, 256, 4):
        w = int(c0) | (int(c0 + 1) << 8) | (int(c0 + 2) << 16) | (int(c0 + 3) << 24)
        x = w ^ 0x80808080
        lo = halves(byte_perm(x, 0x64646464, 0x5140))
        hi = halves(byte_perm(x, 0x64646464, 0x7362))
        got = (np.concatenate([lo, hi]) - np.float16(1152.0)).astype(np.float64)  # f16 arithmetic
        np.testing.assert_array_equal(got, want[c0:c0 + 4])


def test_magic_constant_values():
    assert np.array([0x6400], dtype=np.uint16).view(np.float16)[0] == 1024.0
    assert np.array([0x6480], dtype=np.uint16).view(np.float16)[0] == 1152.0
