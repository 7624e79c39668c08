"""GPU parity of mla_prefill_varlen and mla_prefill_paged (through the C ABI) against the
fp64 CPU oracle.

Tolerances: max-abs 2e-2 and relative L2 5e-3 over the compared outputs, LSE within 1e-3
absolute.  Small ragged batches are compared element by element; the full-size workload
(5 requests, 20K-100K prefix, 256-2048 new tokens, 16 heads) on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

from mla_attention_paged_gb300.inputs import PrefillWorkload, make_prefill_inputs, page_prefill_kv, prefill_workloads

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from mla_attention_paged_gb300 import build
    build.build()
    from mla_attention_paged_gb300 import mla as m
    return m


def run_gpu(mla, inp):
    d = "cuda"
    out, lse = mla.prefill_varlen(inp.q.to(d), inp.k.to(d), inp.v.to(d), inp.cu_seqlens_q.to(d),
                                  inp.cu_seqlens_kv.to(d), inp.prefix_lens.to(d), inp.max_seqlen_q, inp.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(out, lse, ref_out, ref_lse):
    out = out.reshape(ref_out.shape)
    lse = lse.reshape(ref_lse.shape)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    err = np.abs(out - ref_out).max()
    assert err <= MAX_ABS, f"max-abs {err:.3e}"
    rel = np.linalg.norm(out - ref_out) / max(np.linalg.norm(ref_out), 1e-30)
    assert rel <= REL_L2, f"rel-L2 {rel:.3e}"
    lerr = np.abs(lse - ref_lse).max()
    assert lerr <= LSE_ABS, f"lse abs {lerr:.3e}"


SMALL = [
    ("no_prefix", [0], [5], 1),
    ("one_block", [7], [128], 2),
    ("block_plus_one", [64], [129], 2),
    ("ragged", [1, 63, 65, 300], [300, 1, 64, 17], 3),
    ("empty_request", [10, 40], [0, 77], 16),
    ("long_prefix", [5000], [260], 16),
    ("many_heads", [100], [200], 32),
    # q blocks with at least 8 key tiles run as two CTAs over the two halves of their keys
    ("causal_split", [0], [1300], 4),          # no prefix: the causal diagonal in both halves
    ("prefix_split", [1500, 3000], [200, 40], 8),
]


@pytest.mark.parametrize("name,prefix,new,H", SMALL, ids=[c[0] for c in SMALL])
def test_prefill_small(mla, oracle_mod, name, prefix, new, H):
    wl = PrefillWorkload(name, prefix, new, H, seed=200 + len(name))
    inp = make_prefill_inputs(wl, "cpu")
    out, lse = run_gpu(mla, inp)
    ref_out, ref_lse = oracle_mod.mla_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_kv,
                                              inp.prefix_lens, inp.scale)
    check(out, lse, ref_out, ref_lse)


def test_prefill_peaked_scores(mla, oracle_mod):
    """Large scores (q scaled by 8): the running max moves by more than the lazy-rescale
    threshold, so the O-row rescale path runs."""
    wl = PrefillWorkload("peaked", [700, 90], [150, 333], 4, seed=11)
    inp = make_prefill_inputs(wl, "cpu")
    inp.q = (inp.q.float() * 8).to(torch.bfloat16)
    out, lse = run_gpu(mla, inp)
    ref_out, ref_lse = oracle_mod.mla_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_kv,
                                              inp.prefix_lens, inp.scale)
    check(out, lse, ref_out, ref_lse)


def test_prefill_split_halves_are_deterministic(mla):
    """Two CTAs share a q block's keys and the one that finishes second merges: the result
    must not depend on which that is.  Five runs of a prefill whose q blocks all split
    give the same bits."""
    wl = PrefillWorkload("split_repeat", [2000, 4000], [300, 700], 8, seed=21)
    inp = make_prefill_inputs(wl, "cpu")
    dev = "cuda"
    outs = []
    for _ in range(5):
        out, lse = mla.prefill_varlen(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens_q.to(dev),
                                      inp.cu_seqlens_kv.to(dev), inp.prefix_lens.to(dev), inp.max_seqlen_q, inp.scale)
        torch.cuda.synchronize()
        assert mla.get_status() == mla.MLA_OK
        outs.append((out.view(torch.int16).cpu(), lse.view(torch.int32).cpu()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_prefill_more_q_blocks_than_split_slots(mla, oracle_mod):
    """128 heads x 9 q blocks = 1152 (request, head, q block) slots, past the 1024 scratch
    slots of the key-range split: the first 1024 q blocks of 8+ key tiles split, the rest
    run whole, in one launch.  Sampled rows of heads on both sides of the boundary (slots
    are numbered head-major, so heads 113 and up hold slots past 1024) against the oracle."""
    wl = PrefillWorkload("slots", [900], [1100], 128, seed=23)
    inp = make_prefill_inputs(wl, "cuda")
    out, lse = run_gpu(mla, inp)
    H = wl.heads
    rows = [t * H + h for t in (0, 127, 128, 700, 1023, 1024, 1099) for h in (0, 64, 112, 113, 127)]
    ref_out, ref_lse = oracle_mod.mla_prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.cu_seqlens_q.cpu(),
                                              inp.cu_seqlens_kv.cpu(), inp.prefix_lens.cpu(), inp.scale, rows=rows)
    check(out.reshape(-1, 128)[rows], lse.reshape(-1)[rows], ref_out, ref_lse)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_prefill_no_new_tokens_is_a_no_op(mla):
    wl = PrefillWorkload("none", [10], [0], 2, seed=1)
    inp = make_prefill_inputs(wl, "cpu")
    out, lse = run_gpu(mla, inp)
    assert out.size == 0 and lse.size == 0


@pytest.mark.parametrize("name", list(prefill_workloads().keys()))
def test_prefill_full_size_sampled(mla, oracle_mod, name):
    wl = prefill_workloads()[name]
    inp = make_prefill_inputs(wl, "cuda")
    out, lse = run_gpu(mla, inp)
    H = wl.heads
    g = np.random.default_rng(5)
    rows = []
    off = 0
    for n in wl.new_lens:
        toks = {off, off + n - 1, off + min(n - 1, 127), off + min(n - 1, 128)}
        toks |= set(int(x) for x in g.integers(off, off + n, 6))
        for t in sorted(toks):
            for h in (0, H - 1, int(g.integers(H))):
                rows.append(t * H + h)
        off += n
    rows = sorted(set(rows))
    ref_out, ref_lse = oracle_mod.mla_prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.cu_seqlens_q.cpu(),
                                              inp.cu_seqlens_kv.cpu(), inp.prefix_lens.cpu(), inp.scale, rows=rows)
    check(out.reshape(-1, 128)[rows], lse.reshape(-1)[rows], ref_out, ref_lse)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


# ------------------------------------------------------------------------------------
# paged K/V: the same prefill reading every key (prefix and new tokens) through a page table
# ------------------------------------------------------------------------------------
def run_gpu_paged(mla, inp, pk):
    d = "cuda"
    out, lse = mla.prefill_paged(inp.q.to(d), pk.k_pages.to(d), pk.v_pages.to(d), pk.page_table.to(d),
                                 inp.cu_seqlens_q.to(d), pk.kv_lens.to(d), inp.max_seqlen_q, inp.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    return out.float().cpu().numpy(), lse.cpu().numpy()


PAGED = [
    ("ragged_p16", [1, 63, 65, 300], [300, 1, 64, 17], 3, 16),
    ("ragged_p64", [1, 63, 65, 300], [300, 1, 64, 17], 3, 64),
    ("empty_request_p32", [10, 40], [0, 77], 8, 32),
    ("long_prefix_p128", [5000], [260], 16, 128),
    ("tile_crossing_p256", [200, 700], [129, 333], 4, 256),
]


@pytest.mark.parametrize("name,prefix,new,H,P", PAGED, ids=[c[0] for c in PAGED])
def test_prefill_paged_small(mla, oracle_mod, name, prefix, new, H, P):
    """Every output against the oracle run on the contiguous rows the pages were built from."""
    wl = PrefillWorkload(name, prefix, new, H, seed=300 + len(name))
    inp = make_prefill_inputs(wl, "cpu")
    pk = page_prefill_kv(inp, P, seed=7, extra_pages=3)
    out, lse = run_gpu_paged(mla, inp, pk)
    ref_out, ref_lse = oracle_mod.mla_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_kv,
                                              inp.prefix_lens, inp.scale)
    check(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("P", [16, 64, 256])
def test_prefill_paged_equals_contiguous_bitwise(mla, P):
    """The paged call gives the contiguous call's bits: the same keys in the same tiles, and
    the rows a tile holds past a request's end are masked either way (P = 0 times finite
    values)."""
    wl = PrefillWorkload("paged_vs_contiguous", [700, 90, 1500], [150, 333, 64], 4, seed=12)
    inp = make_prefill_inputs(wl, "cpu")
    pk = page_prefill_kv(inp, P, seed=8)
    out_c, lse_c = run_gpu(mla, inp)
    out_p, lse_p = run_gpu_paged(mla, inp, pk)
    np.testing.assert_array_equal(out_c, out_p)
    np.testing.assert_array_equal(lse_c, lse_p)


def test_prefill_paged_full_size_sampled(mla, oracle_mod):
    """The 5-request workload (prefix 20K-100K, 256-2048 new tokens, 16 heads) with its K/V in
    64-token pages, sampled rows against the oracle."""
    wl = prefill_workloads()["prefill_b5_h16_prefix"]
    inp = make_prefill_inputs(wl, "cuda")
    pk = page_prefill_kv(inp, 64, seed=9)
    out, lse = run_gpu_paged(mla, inp, pk)
    H = wl.heads
    g = np.random.default_rng(6)
    rows = []
    off = 0
    for n in wl.new_lens:
        toks = {off, off + n - 1} | set(int(x) for x in g.integers(off, off + n, 6))
        for t in sorted(toks):
            for h in (0, H - 1, int(g.integers(H))):
                rows.append(t * H + h)
        off += n
    rows = sorted(set(rows))
    ref_out, ref_lse = oracle_mod.mla_prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.cu_seqlens_q.cpu(),
                                              inp.cu_seqlens_kv.cpu(), inp.prefix_lens.cpu(), inp.scale, rows=rows)
    check(out.reshape(-1, 128)[rows], lse.reshape(-1)[rows], ref_out, ref_lse)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_prefill_paged_bad_page_id_is_reported(mla):
    """A page id outside [0, num_pages) is reported as MLA_ERR_DEVICE_ARG.  The pools given to
    the call are views into larger allocations (8 spare pages on each side), so the id used
    here still names allocated memory."""
    wl = PrefillWorkload("paged_bad", [300, 40], [100, 20], 2, seed=13)
    inp = make_prefill_inputs(wl, "cuda")
    pk = page_prefill_kv(inp, 64, seed=10)
    n = pk.k_pages.shape[0]
    kb = torch.zeros((n + 16,) + tuple(pk.k_pages.shape[1:]), dtype=torch.bfloat16, device="cuda")
    vb = torch.zeros((n + 16,) + tuple(pk.v_pages.shape[1:]), dtype=torch.bfloat16, device="cuda")
    kb[8:8 + n] = pk.k_pages
    vb[8:8 + n] = pk.v_pages
    pt = pk.page_table.clone()
    pt[0, 2] = n + 3
    mla.prefill_paged(inp.q, kb[8:8 + n], vb[8:8 + n], pt, inp.cu_seqlens_q, pk.kv_lens, inp.max_seqlen_q, inp.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_ERR_DEVICE_ARG
    mla.prefill_paged(inp.q, kb[8:8 + n], vb[8:8 + n], pk.page_table, inp.cu_seqlens_q, pk.kv_lens,
                      inp.max_seqlen_q, inp.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
