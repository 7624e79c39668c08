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
    assert ctypes.sizeof(mla.DecodePlan) == 64


def test_status_strings(mla):
    assert mla.status_string(0) == "MLA_OK"
    assert mla.status_string(3) == "MLA_ERR_WORKSPACE_TOO_SMALL"
    assert mla.status_string(99) == "MLA_ERR_UNKNOWN"
    assert mla.lib.mla_version() >= 100


def test_plan_fills_one_wave_and_sizes_workspace(mla):
    lens = [65536] * 16
    plan = mla.decode_plan(lens, q_len=4, num_heads=16, page_size=64, max_pages_per_seq=1024,
                           num_pages=16 * 1024, num_sms=152)
    assert plan.rows == 64 and plan.head_groups == 1
    assert plan.chunk_tokens % 64 == 0
    ctas = sum((L + plan.chunk_tokens - 1) // plan.chunk_tokens for L in lens) * plan.head_groups
    assert ctas <= 152
    # the next smaller chunk would overflow one wave
    smaller = plan.chunk_tokens - 64
    assert sum((L + smaller - 1) // smaller for L in lens) > 152
    assert plan.max_splits == (65536 + plan.chunk_tokens - 1) // plan.chunk_tokens
    parts = 16 * plan.max_splits * 64
    assert plan.workspace_bytes == 256 + parts * 512 * 2 + parts * 4  # bf16 partial rows + fp32 lse


def test_plan_single_split_needs_no_workspace(mla):
    plan = mla.decode_plan([300] * 200, q_len=1, num_heads=16, page_size=64, max_pages_per_seq=5,
                           num_pages=1000, num_sms=152)
    assert plan.max_splits == 1 and plan.workspace_bytes == 0


def test_plan_head_groups_for_many_heads(mla):
    plan = mla.decode_plan([8192, 131072], q_len=2, num_heads=128, page_size=64, max_pages_per_seq=2048,
                           num_pages=4096, num_sms=152)
    assert plan.rows == 256 and plan.head_groups == 4


def test_plan_splits_a_multi_wave_absorbed_prefill(mla):
    """4 requests x 512 new tokens x 16 heads on 32K keys: 128 row groups per request, 512
    CTAs unsplit (3.4 waves of 152).  Two splits of 256 tiles give 7 waves x 259 = 1813
    tile-times against 4 x 515 = 2060 unsplit (three: 11 x 174; four: 14 x 131)."""
    plan = mla.decode_plan([32768] * 4, q_len=512, num_heads=16, page_size=64, max_pages_per_seq=512,
                           num_pages=2048, num_sms=152)
    assert plan.head_groups == 128
    assert plan.chunk_tokens == 256 * 64 and plan.max_splits == 2
    assert plan.workspace_bytes == 256 + 4 * 2 * 512 * 16 * (512 * 2 + 4)


def test_plan_invariants_on_random_batches(mla):
    """Seeded random batches (ragged lengths, 1-8 drafts or a long absorbed prefill, 16 or
    128 heads, several SM counts): the split chunk is whole 64-key tiles and at least four
    of them (or the whole of the longest request); while one split per request fits in one
    wave of CTAs, one wave whenever a request is split and the smallest chunk with that
    property; beyond one wave, the whole request or 2-4 splits, whichever has the lowest
    waves x (tiles per CTA + 3); and a workspace that fits every split."""
    rng = np.random.default_rng(12)
    for _ in range(60):
        B = int(rng.integers(1, 40))
        T = int(rng.choice([1, 2, 4, 8, 300]))
        H = int(rng.choice([16, 128]))
        if T * H > 131072:
            continue
        sms = int(rng.choice([16, 100, 152]))
        lens = [int(x) for x in rng.integers(T, 200000, B)]
        mp = (max(lens) + 63) // 64
        plan = mla.decode_plan(lens, q_len=T, num_heads=H, page_size=64, max_pages_per_seq=mp,
                               num_pages=B * mp, num_sms=sms)
        tiles = [(L + 63) // 64 for L in lens]
        ct = plan.chunk_tokens // 64
        assert plan.chunk_tokens % 64 == 0 and ct >= min(4, max(tiles))
        groups = (T * H + 63) // 64
        assert plan.head_groups == groups
        n_ctas = lambda c: groups * sum((t + c - 1) // c for t in tiles)
        ctas = n_ctas(ct)
        assert plan.max_splits == (max(lens) + plan.chunk_tokens - 1) // plan.chunk_tokens
        if n_ctas(max(tiles)) > sms:  # more than one wave even unsplit
            cost = lambda c: -(-n_ctas(c) // sms) * (c + 3)
            cands = [max(tiles)] + [c for c in (-(-max(tiles) // k) for k in (2, 3, 4)) if c >= 4]
            assert ct in cands and cost(ct) == min(cost(c) for c in cands)
        elif plan.max_splits > 1:
            assert ctas <= sms
            if ct > min(4, max(tiles)):
                assert groups * sum((t + ct - 2) // (ct - 1) for t in tiles) > sms
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
