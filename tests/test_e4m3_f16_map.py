"""The e4m3 decode of the FP8 decode kernel, restated on the host and pinned to the format.

The kernel's dequant warps turn four e4m3 codes (one 32-bit word) into two f16x2 words in two
ways and mix them: (a) a byte permute that puts code 0 in bits 8-15 and code 1 in bits
24-31 (selector 0x1404; 0x3424 for codes 2 and 3), then sign bits kept and the 7 exponent +
mantissa bits shifted right by one into f16's fields; (b) the conversion unit, whose exact
result is multiplied by 2^-8.  Both must equal the code's value times 2^-8 exactly, lanes in
code order.  Here (a) is re-derived in numpy (independently of the kernel source) and checked
against the oracle's e4m3 decoder, which is written from the format definition (OCP e4m3fn:
bias 7, subnormals m/8 * 2^-6, S.1111.111 = NaN); (b) is the definition itself times 2^-8,
so the check is that every finite code times 2^-8 is an f16 value.
"""
import numpy as np


def byte_perm(x, y, sel):
    """Byte permute of two 32-bit words (result byte i = byte (sel >> 4i) & 7 of y:x)."""
    src = [(x >> (8 * k)) & 0xFF for k in range(4)] + [(y >> (8 * k)) & 0xFF for k in range(4)]
    return sum(src[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def f16_pair_from_word(w):
    h0 = byte_perm(w, 0, 0x1404)
    h1 = byte_perm(w, 0, 0x3424)
    lo = (h0 & 0x80008000) | ((h0 >> 1) & 0x3F803F80)
    hi = (h1 & 0x80008000) | ((h1 >> 1) & 0x3F803F80)
    return lo, hi


def halves(word):
    pair = np.array([word & 0xFFFF, word >> 16], dtype=np.uint16)
    return pair.view(np.float16).astype(np.float64)


def test_integer_map_is_exact_for_every_finite_code(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    want = oracle_mod.e4m3_to_double(codes)
    for c0 in range(0, 256, 4):
        w = int(c0) | (int(c0 + 1) << 8) | (int(c0 + 2) << 16) | (int(c0 + 3) << 24)
        lo, hi = f16_pair_from_word(w)
        got = np.concatenate([halves(lo), halves(hi)])
        for k in range(4):
            v = want[c0 + k]
            if np.isnan(v):
                continue  # NaN codes do not occur in a quantised cache
            assert got[k] == v * 2.0 ** -8, (hex(c0 + k), got[k], v)


def test_scaled_values_are_f16_values(oracle_mod):
    vals = oracle_mod.e4m3_to_double(np.arange(256, dtype=np.uint8))
    vals = vals[~np.isnan(vals)] * 2.0 ** -8
    assert np.array_equal(vals.astype(np.float16).astype(np.float64), vals)
    assert np.max(np.abs(vals)) == 1.75  # 448 * 2^-8
