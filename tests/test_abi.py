"""C-ABI checks that need no GPU: the library loads, exports every function declared in
include/*.h, and its host-side planning and argument validation behave as documented.
No compute call is made here."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mla():
    from mla_attention_paged_gb300 import build
    build.build()
    from mla_attention_paged_gb300 import mla as m
    return m


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(inc, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(mla_[A-Za-z0-9_]+)\s*\(", text, re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["mla_decode_plan", "mla_decode", "mla_prefill_varlen", "mla_get_status", "mla_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol(mla):
    lib = ctypes.CDLL(mla.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), f"libmla.so does not export {name}"


def test_binding_covers_the_header(mla):
    """The Python binding lists exactly the functions the header declares, and gives each
    its C signature."""
    assert sorted(mla.EXPORTED) == _declared_functions()
    for name in mla.EXPORTED:
        fn = getattr(mla.lib, name)
        if name != "mla_version":  # the one function without arguments
            assert fn.argtypes, f"{name} has no argument types set"


def test_plan_struct_layout(mla):
    assert ctypes.sizeof(mla.DecodePlan) == 72
    assert mla.DecodePlan.workspace_bytes.offset == 64 and mla.DecodePlan.split_major.offset == 56


def test_status_strings(mla):
    assert mla.status_string(0) == "MLA_OK"
    assert mla.status_string(3) == "MLA_ERR_WORKSPACE_TOO_SMALL"
    assert mla.status_string(99) == "MLA_ERR_UNKNOWN"
    assert mla.lib.mla_version() >= 100


def test_plan_fills_one_wave_and_sizes_workspace(mla):
    """16 requests of 1024 tiles on 152 SMs.  A bf16 pool (fixed cost 3 tile-times per CTA)
    takes the chunk that shares the tiles evenly over the SMs: 108 tiles, 144 CTAs of 108
    and 16 remainders of 52 launched last, two of them on each of the 8 SMs left free
    (111 + 2 for the combine, against 117 + 2 for the one-wave plan of 114).  An e4m3 pool
    (fixed cost 10) would tie there (two remainders of 52 + 10 on an SM: 124 + 2, as the
    one-wave plan) and takes 109: remainders of 43, 2 x 53 < 119.  A batch that fits one
    wave at the balanced chunk keeps the one-wave plan: the smallest chunk that fits."""
    lens = [65536] * 16
    bf = mla.decode_plan(lens, q_len=4, num_heads=16, page_size=64, max_pages_per_seq=1024,
                         num_pages=16 * 1024, num_sms=152)
    assert bf.rows == 64 and bf.head_groups == 1
    assert bf.chunk_tokens == 108 * 64 and bf.max_splits == 10 and bf.split_major == 1
    parts = 16 * bf.max_splits * 64
    assert bf.workspace_bytes == 256 + parts * 512 * 2 + parts * 4  # bf16 partial rows + fp32 lse
    assert _plan_cost([1024] * 16, 1, 108, 152) == 113 < _plan_cost([1024] * 16, 1, 114, 152) == 119
    f8 = mla.decode_plan(lens, q_len=4, num_heads=16, page_size=64, max_pages_per_seq=1024,
                         num_pages=16 * 1024, kv_dtype=mla.MLA_KV_E4M3, num_sms=152)
    assert f8.chunk_tokens == 109 * 64 and f8.max_splits == 10 and f8.split_major == 1
    assert (_plan_cost([1024] * 16, 1, 109, 152, fixed=10) == 121
            < _plan_cost([1024] * 16, 1, 108, 152, fixed=10) == 126 == _plan_cost([1024] * 16, 1, 114, 152, fixed=10))
    lens = [60000] * 8  # 938 tiles: 8 x 19 = 152 CTAs of 50 fill one wave exactly
    plan = mla.decode_plan(lens, q_len=4, num_heads=16, page_size=64, max_pages_per_seq=938,
                           num_pages=8 * 938, num_sms=152)
    ctas = sum((L + plan.chunk_tokens - 1) // plan.chunk_tokens for L in lens) * plan.head_groups
    assert ctas <= 152 and plan.split_major == 0
    # the next smaller chunk would overflow one wave
    smaller = plan.chunk_tokens - 64
    assert sum((L + smaller - 1) // smaller for L in lens) > 152


def test_plan_single_split_needs_no_workspace(mla):
    plan = mla.decode_plan([300] * 200, q_len=1, num_heads=16, page_size=64, max_pages_per_seq=5,
                           num_pages=1000, num_sms=152)
    assert plan.max_splits == 1 and plan.workspace_bytes == 0


def test_plan_head_groups_for_many_heads(mla):
    plan = mla.decode_plan([8192, 131072], q_len=2, num_heads=128, page_size=64, max_pages_per_seq=2048,
                           num_pages=4096, num_sms=152)
    assert plan.rows == 256 and plan.head_groups == 4


def _plan_cost(tiles, groups, ct, sms, fixed=3):
    """The planner's cost model, restated: CTAs in launch order (group fastest; with one
    row group split by split, every request's split s before any split s + 1; with several
    request by request) dispatched onto the SM that frees first, each costing its tiles + a
    fixed part (3 tile-times, 10 for an e4m3 pool); a plan with more than one split adds 2
    for the combine."""
    import heapq
    splits = [-(-t // ct) for t in tiles]
    n_ctas = groups * sum(splits)
    if n_ctas <= sms:
        span = max(min(t, ct) for t in tiles) + fixed
    else:
        free = [0] * sms
        span = 0
        if groups == 1:
            order = [(t, s) for s in range(max(splits)) for t, ns in zip(tiles, splits) if s < ns]
        else:
            order = [(t, s) for t, ns in zip(tiles, splits) for s in range(ns)]
        for t, s in order:
            cost = min(ct, t - s * ct) + fixed
            for _ in range(groups):
                start = heapq.heappop(free)
                heapq.heappush(free, start + cost)
                span = max(span, start + cost)
    return span + (2 if max(splits) > 1 else 0)


def test_plan_splits_a_multi_wave_absorbed_prefill(mla):
    """4 requests x 512 new tokens x 16 heads on 32K keys: 128 row groups per request, 512
    CTAs unsplit (3.4 waves of 152 SMs: 4 x 515 = 2060 tile-times).  Two splits of 256
    tiles: 1024 CTAs in 6.7 waves, 7 x 259 + 2 = 1815 (three: 1536 CTAs of ~174, four:
    2048 CTAs of 131, 14 x 131 + 2 = 1836).  1815 is within 1.1 x the work spread over the
    SMs (4 x 128 x 515 / 152 = 1735), so the wider scan of 5-32 splits does not run."""
    plan = mla.decode_plan([32768] * 4, q_len=512, num_heads=16, page_size=64, max_pages_per_seq=512,
                           num_pages=2048, num_sms=152)
    assert plan.head_groups == 128 and plan.split_major == 0
    assert plan.chunk_tokens == 256 * 64 and plan.max_splits == 2
    assert plan.workspace_bytes == 256 + 4 * 2 * 512 * 16 * (512 * 2 + 4)
    assert _plan_cost([512] * 4, 128, 256, 152) == 1815 and _plan_cost([512] * 4, 128, 512, 152) == 2060
    assert 10 * 1815 <= 11 * -(-4 * 128 * 515 // 152)


def test_plan_evens_out_a_ragged_many_head_batch(mla):
    """16 requests of 8K-128K keys at q_len 2 x 128 heads (four row groups): the one-wave
    plan (4 splits of the longest request, 152 CTAs) leaves the SMs far less work on
    average than its longest CTA, over 1.1 x the spread, so the planner also tries 5-32
    splits; one of those wins, its shorter CTAs evened out over several waves."""
    rng = np.random.default_rng(2026)
    lens = [int(x) for x in rng.integers(8192, 131073, 16)]
    tiles = [(L + 63) // 64 for L in lens]
    mp = max(tiles)
    plan = mla.decode_plan(lens, q_len=2, num_heads=128, page_size=64, max_pages_per_seq=mp, num_pages=16 * mp,
                           num_sms=152)
    ct = plan.chunk_tokens // 64
    assert plan.head_groups == 4 and plan.split_major == 0
    one_wave = min(c for c in range(4, mp + 1) if 4 * sum(-(-t // c) for t in tiles) <= 152)
    spread = -(-sum((t + 3) * 4 for t in tiles) // 152)
    assert 10 * _plan_cost(tiles, 4, one_wave, 152) > 11 * spread
    assert -(-mp // ct) > 4 and _plan_cost(tiles, 4, ct, 152) < _plan_cost(tiles, 4, one_wave, 152)
    assert _plan_cost(tiles, 4, ct, 152) == min(_plan_cost(tiles, 4, -(-mp // k), 152) for k in range(1, 33))


def test_plan_one_sm_never_splits(mla):
    """On one SM every CTA runs after the previous one, so a split only adds per-CTA fixed
    cost and a combine: the plan keeps one split per request, whatever the lengths.  (The
    ragged batch [5000, 130, 2999]: 79 + 3 + 47 tiles; three-way splits of 27 tiles would
    cost 147 + 2 tile-times against 138.)"""
    plan = mla.decode_plan([5000, 130, 2999], q_len=4, num_heads=16, page_size=64, max_pages_per_seq=79,
                           num_pages=300, num_sms=1)
    assert plan.max_splits == 1 and plan.workspace_bytes == 0
    assert _plan_cost([79, 3, 47], 1, 79, 1) == 138 < _plan_cost([79, 3, 47], 1, 27, 1) == 149
    rng = np.random.default_rng(7)
    for _ in range(30):
        B = int(rng.integers(1, 12))
        T = int(rng.choice([1, 2, 4, 8, 64]))
        H = int(rng.choice([16, 128]))
        lens = [int(x) for x in rng.integers(T, 300000, B)]
        mp = (max(lens) + 63) // 64
        plan = mla.decode_plan(lens, q_len=T, num_heads=H, page_size=64, max_pages_per_seq=mp,
                               num_pages=B * mp, num_sms=1)
        assert plan.max_splits == 1 and plan.chunk_tokens == mp * 64


def test_plan_invariants_on_random_batches(mla):
    """Seeded random batches (ragged lengths, 1-8 drafts or a long absorbed prefill, 16 or
    128 heads, several SM counts): the split chunk is whole 64-key tiles, at least four of
    them (or the whole of the longest request), or fewer where the longest request still
    takes at most 32 splits (one round of the combine); the plan's estimated duration is the
    lowest over its candidates (1-4 splits of the longest request, 1-32 with several row
    groups when the others cost over 1.1 x the work spread over the SMs, the smallest chunk
    that keeps the call in one wave when the unsplit call fits one, and with one row group
    the
    chunks that share all tiles evenly over one or two waves), so it is never longer
    than the unsplit call's; a split that fits one wave is the smallest such chunk; and the
    workspace fits every split."""
    rng = np.random.default_rng(12)
    for _ in range(60):
        B = int(rng.integers(1, 40))
        T = int(rng.choice([1, 2, 4, 8, 300]))
        H = int(rng.choice([16, 128]))
        if T * H > 131072:
            continue
        sms = int(rng.choice([1, 3, 16, 100, 152]))
        lens = [int(x) for x in rng.integers(T, 200000, B)]
        mp = (max(lens) + 63) // 64
        plan = mla.decode_plan(lens, q_len=T, num_heads=H, page_size=64, max_pages_per_seq=mp,
                               num_pages=B * mp, num_sms=sms)
        tiles = [(L + 63) // 64 for L in lens]
        mt = max(tiles)
        ct = plan.chunk_tokens // 64
        lo = min(4, max(1, -(-mt // 32)))
        assert plan.chunk_tokens % 64 == 0 and ct >= lo
        groups = (T * H + 63) // 64
        assert plan.head_groups == groups
        n_ctas = lambda c: groups * sum((t + c - 1) // c for t in tiles)
        assert plan.max_splits == (max(lens) + plan.chunk_tokens - 1) // plan.chunk_tokens
        cands = [c for c in (-(-mt // k) for k in range(1, 5)) if c >= lo]
        one_wave = None
        if n_ctas(mt) <= sms:
            one_wave = min(c for c in range(lo, mt + 1) if n_ctas(c) <= sms)
            cands.append(one_wave)
        if groups == 1:
            base1, base2 = -(-sum(tiles) // sms), -(-sum(tiles) // (2 * sms))
            cands += [c for c in [base1 + d for d in range(9)] + [base2] if lo <= c < mt]
        cost = lambda c: _plan_cost(tiles, groups, c, sms)
        if groups > 1:
            spread = -(-sum((t + 3) * groups for t in tiles) // sms)
            if 10 * min(cost(c) for c in cands + [mt]) > 11 * spread:
                cands += [c for c in (-(-mt // k) for k in range(5, 33)) if c >= lo]
        assert ct in cands + [mt]
        assert cost(ct) == min(cost(c) for c in cands)
        assert cost(ct) <= cost(mt)
        if plan.max_splits > 1 and n_ctas(ct) <= sms and one_wave is not None:
            assert ct == one_wave
        if plan.max_splits > 1:
            parts = B * plan.max_splits * T * H
            assert plan.workspace_bytes == 256 + parts * 512 * 2 + parts * 4
        else:
            assert plan.workspace_bytes == 0


def test_plan_is_memoised_and_deterministic(mla):
    a = mla.decode_plan([1000, 5000], 2, 16, 64, 100, 200, num_sms=152)
    b = mla.decode_plan([1000, 5000], 2, 16, 64, 100, 200, num_sms=152)
    assert a.as_dict() == b.as_dict()


@pytest.mark.parametrize("kw,code", [
    (dict(seq_lens=[3], q_len=4), 1),                 # fewer cached tokens than drafts
    (dict(seq_lens=[10000], max_pages=10), 1),        # beyond the table
    (dict(seq_lens=[10000], q_len=8193), 2),          # more new tokens than the absorbed prefill takes
    (dict(seq_lens=[10000], q_len=2048, heads=128), 2),  # more than 131072 folded rows
    (dict(page_size=48), 2),                          # unsupported page size
    (dict(kv_dtype=7), 1),
])
def test_plan_rejects_bad_arguments(mla, kw, code):
    args = dict(seq_lens=[100], q_len=1, heads=16, page_size=64, max_pages=200, pages=200, kv_dtype=0)
    args.update(kw)
    lens = torch.tensor(args["seq_lens"], dtype=torch.int32)
    plan = mla.DecodePlan()
    rc = mla.lib.mla_decode_plan(len(args["seq_lens"]), ctypes.c_void_p(lens.data_ptr()), args["q_len"], args["heads"],
                                 args["page_size"], args["max_pages"], args["pages"], args["kv_dtype"], 152,
                                 ctypes.byref(plan))
    assert rc == code


def test_decode_validates_before_touching_the_device(mla):
    plan = mla.decode_plan([65536] * 4, 4, 16, 64, 1024, 4096, num_sms=152)
    assert plan.workspace_bytes > 0
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation
    P = ctypes.c_void_p
    # null pointer
    rc = mla.lib.mla_decode(ctypes.byref(plan), None, fake, fake, fake, 4, 16, 0.07, 1.0, fake, fake, fake,
                            plan.workspace_bytes, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    # q_len differs from the plan
    rc = mla.lib.mla_decode(ctypes.byref(plan), fake, fake, fake, fake, 2, 16, 0.07, 1.0, fake, fake, fake,
                            plan.workspace_bytes, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    # workspace too small
    rc = mla.lib.mla_decode(ctypes.byref(plan), fake, fake, fake, fake, 4, 16, 0.07, 1.0, fake, fake, fake,
                            plan.workspace_bytes - 1, None)
    assert rc == mla.MLA_ERR_WORKSPACE_TOO_SMALL
    # misaligned q
    rc = mla.lib.mla_decode(ctypes.byref(plan), P((1 << 20) + 2), fake, fake, fake, 4, 16, 0.07, 1.0, fake, fake,
                            fake, plan.workspace_bytes, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    # non-positive scale
    rc = mla.lib.mla_decode(ctypes.byref(plan), fake, fake, fake, fake, 4, 16, 0.0, 1.0, fake, fake, fake,
                            plan.workspace_bytes, None)
    assert rc == mla.MLA_ERR_INVALID_ARG


def test_int8_paged_entry_validates_before_touching_the_device(mla):
    """A pool with a scale per page goes through mla_decode_int8_paged only, with its scales;
    no other pool takes scales.  Every call below fails validation on the host."""
    paged = mla.decode_plan([4096] * 2, 2, 16, 64, 64, 256, mla.MLA_KV_INT8_PAGE, num_sms=152)
    plain = mla.decode_plan([4096] * 2, 2, 16, 64, 64, 256, mla.MLA_KV_INT8, num_sms=152)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced
    ws = max(paged.workspace_bytes, plain.workspace_bytes)
    # mla_decode has no scales for a per-page pool
    rc = mla.lib.mla_decode(ctypes.byref(paged), fake, fake, fake, fake, 2, 16, 0.07, 1.0, fake, fake, fake, ws, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    rc = mla.lib.mla_decode_partial(ctypes.byref(paged), fake, fake, fake, fake, 2, 16, 0.07, 1.0, fake, fake, fake,
                                    ws, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    # the per-page entry point refuses other plans, null scales and misaligned scales
    rc = mla.lib.mla_decode_int8_paged(ctypes.byref(plain), fake, fake, fake, fake, fake, 2, 16, 0.07, 1.0, fake,
                                       fake, fake, ws, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    rc = mla.lib.mla_decode_int8_paged(ctypes.byref(paged), fake, fake, None, fake, fake, 2, 16, 0.07, 1.0, fake,
                                       fake, fake, ws, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    rc = mla.lib.mla_decode_int8_paged(ctypes.byref(paged), fake, fake, ctypes.c_void_p((1 << 20) + 2), fake, fake,
                                       2, 16, 0.07, 1.0, fake, fake, fake, ws, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
