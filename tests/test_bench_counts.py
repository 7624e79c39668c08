"""The algorithmic counts behind bench.py's rooflines, checked by brute force on small
shapes: the decode flops and bytes count each visible (query row, key) pair and each
latent row, page-table entry and q/out/lse row once; the prefill flops count the keys each
new token sees under the prefix-offset causal mask."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mla_attention_paged_gb300.inputs import DecodeWorkload, PrefillWorkload  # noqa: E402


@pytest.mark.parametrize("T,H,lens,P,kv", [(1, 16, [1024], 64, "bf16"), (4, 2, [4, 70, 129], 16, "bf16"),
                                          (8, 3, [8, 9, 300], 8, "e4m3"), (5, 1, [64, 65], 64, "int8")])
def test_decode_counts_by_enumeration(T, H, lens, P, kv):
    wl = DecodeWorkload("count", len(lens), T, H, lens, kv_dtype=kv, page_size=P)
    pairs = 0
    for L in lens:
        for t in range(T):
            for h in range(H):
                pairs += sum(1 for j in range(L) if j <= L - T + t)
    assert bench.decode_flops(wl) == 2 * pairs * (576 + 512)
    e = 2 if kv == "bf16" else 1
    kv_bytes, total = bench.decode_bytes(wl)
    assert kv_bytes == sum(L for L in lens) * 576 * e
    pages = sum(len(range(0, L, P)) for L in lens)
    assert total == kv_bytes + 4 * pages + len(lens) * T * H * (576 * 2 + 512 * 2 + 4)


@pytest.mark.parametrize("prefix,new,H", [([0], [5], 1), ([7, 0], [3, 64], 2), ([100, 3], [0, 17], 4)])
def test_prefill_flops_by_enumeration(prefix, new, H):
    wl = PrefillWorkload("count", prefix, new, H, seed=0)
    pairs = 0
    for p, n in zip(prefix, new):
        for i in range(n):
            pairs += sum(1 for j in range(p + n) if j <= p + i)
    assert bench.prefill_flops(wl) == 2 * H * (192 + 128) * pairs
