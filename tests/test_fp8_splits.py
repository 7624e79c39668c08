"""The two 8-bit splits of the e4m3 decode kernel, restated on the host and pinned to the
number formats.

The kernel feeds both GEMMs 8-bit operands (tcgen05 kind::f8f6f4):
  * each bf16 query row, scaled by a power of two that puts its largest |q| in [128, 256),
    becomes q_hi = e4m3(x) and q_lo = e4m3(x - q_hi);
  * P, formed times 2^6 (so at most 2^8), becomes p_hi = e4m3(x) and p_lo = e5m2(x - p_hi).
Its header claims: the Q split is exact for every element within 2^9 of the row's largest
|q| and otherwise off by at most 2^-17 of it; the P split is within 2^-8 relative from
x = 2^-6 up, within 2^-14 absolute below, and loses no x >= 2^-16 (2^-22 of P = 1).  The
conversions round to nearest, ties to even, saturating.  Here both formats are enumerated
from their definitions (OCP e4m3fn: bias 7, no infinities, S.1111.111 = NaN, max 448; OCP
e5m2: bias 15, IEEE-style specials, max 57344), rounding is done on those value grids, and
the claims are checked over every bf16 value in range (Q) and a dense grid (P).
"""
import numpy as np
import pytest
import torch


def _grid(ebits, mbits, bias, e4m3):
    vals, parity = [], []
    for e in range(2 ** ebits):
        for m in range(2 ** mbits):
            if e4m3 and e == 2 ** ebits - 1 and m == 2 ** mbits - 1:
                continue  # e4m3fn: S.1111.111 is NaN; the rest of the top binade is finite
            if not e4m3 and e == 2 ** ebits - 1:
                continue  # e5m2: exponent all ones is Inf / NaN
            if e == 0:
                v = (m / 2 ** mbits) * 2.0 ** (1 - bias)
            else:
                v = (1 + m / 2 ** mbits) * 2.0 ** (e - bias)
            vals.append(v)
            parity.append(m & 1)
    order = np.argsort(vals)
    return np.asarray(vals)[order], np.asarray(parity)[order]


E4M3 = _grid(4, 3, 7, True)
E5M2 = _grid(5, 2, 15, False)


def _round(x, fmt):
    """Round to nearest on the format's finite grid, ties to the even significand,
    saturating at the largest finite value."""
    v, par = fmt
    ax = np.abs(np.asarray(x, dtype=np.float64))
    i = np.clip(np.searchsorted(v, ax), 1, len(v) - 1)
    lo, hi = v[i - 1], v[i]
    pick = np.where(ax - lo < hi - ax, lo, np.where(hi - ax < ax - lo, hi, np.where(par[i - 1] == 0, lo, hi)))
    pick = np.where(ax >= v[-1], v[-1], pick)
    return np.sign(x) * pick


def _bf16_values(lo_exp, hi_exp):
    """Every positive bf16 value in [2^lo_exp, 2^hi_exp)."""
    out = []
    for e in range(lo_exp, hi_exp):
        out.append((1 + np.arange(128) / 128.0) * 2.0 ** e)
    return np.concatenate(out)


def test_format_grids():
    assert E4M3[0].max() == 448.0 and E5M2[0].max() == 57344.0
    assert E4M3[0][1] == 2.0 ** -9 and E5M2[0][1] == 2.0 ** -16  # smallest subnormals
    assert len(E4M3[0]) == 127 and len(E5M2[0]) == 124  # finite non-negative codes (+0 once each)


@pytest.mark.parametrize("name,fmt,dtype", [("e4m3", E4M3, torch.float8_e4m3fn), ("e5m2", E5M2, torch.float8_e5m2)])
def test_rounding_matches_torch_cast(name, fmt, dtype):
    g = np.random.default_rng(3)
    x = g.standard_normal(200000) * np.exp2(g.uniform(-18, 8, 200000))
    x = x[np.abs(x) < fmt[0].max()]
    ref = torch.from_numpy(x).float().to(dtype).double().numpy()
    np.testing.assert_array_equal(_round(x.astype(np.float32).astype(np.float64), fmt), ref)


def test_query_split_exact_within_2e9_of_row_max():
    x = _bf16_values(-2, 8)  # the row max is in [128, 256): 2^9 below it is >= 2^-2
    x = np.concatenate([x, -x])
    hi = _round(x, E4M3)
    lo = _round(x - hi, E4M3)
    np.testing.assert_array_equal(hi + lo, x)


def test_query_split_floor_below():
    x = _bf16_values(-40, -2)
    x = np.concatenate([x, -x])
    hi = _round(x, E4M3)
    lo = _round(x - hi, E4M3)
    assert np.abs(hi + lo - x).max() <= 2.0 ** -17 * 128.0  # 2^-17 of the smallest row max


def test_p_split_bounds():
    x = np.exp2(np.linspace(-24.0, 8.0, 320001))
    hi = _round(x, E4M3)
    lo = _round(x - hi, E5M2)
    err = np.abs(hi + lo - x)
    normal = x >= 2.0 ** -6
    assert (err[normal] / x[normal]).max() <= 2.0 ** -8
    assert err[~normal].max() <= 2.0 ** -14
    assert (hi + lo)[x >= 2.0 ** -16].min() > 0.0
    assert np.abs(hi).max() <= 256.0  # x <= 2^8: no saturation


def test_p_split_with_e4m3_low_part_would_flush_the_tail():
    """The reason p_lo is e5m2: with an e4m3 low part, x < 2^-10 rounds to zero."""
    x = np.exp2(np.linspace(-16.0, -10.5, 1001))
    hi = _round(x, E4M3)
    assert (hi + _round(x - hi, E4M3)).max() == 0.0
    assert (hi + _round(x - hi, E5M2)).min() > 0.0
