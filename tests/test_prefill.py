"""GPU parity of mla_prefill_varlen (through the C ABI) against the fp64 CPU oracle.

Tolerances: max-abs 2e-2 and relative L2 5e-3 over the compared outputs, LSE within 1e-3
absolute.  Small ragged batches are compared element by element; the full-size workload
(5 requests, 20K-100K prefix, 256-2048 new tokens, 16 heads) on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

from mla_attention_paged_gb300.inputs import PrefillWorkload, make_prefill_inputs, prefill_workloads

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
