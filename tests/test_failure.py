"""Failure detection on the GPU without faulting or hanging it.

* The bounded mbarrier wait every kernel uses gives up after its limit and records
  MLA_ERR_TIMEOUT in the status word (a self-test kernel waits on a barrier that nothing
  arrives on); the context stays usable afterwards.
* Device-side argument checks are caught by the kernels before any access that depends
  on them and reported as MLA_ERR_DEVICE_ARG: a decode request longer than the plan
  allows, a page id outside the pool (on the bf16 path, whose TMA reads zero-fill outside
  the pool even without the check), and a prefill request with more new tokens than the
  host's max_seqlen_q sized the grid for.
"""
import time

import numpy as np
import pytest
import torch

from mla_attention_paged_gb300.inputs import DecodeWorkload, make_decode_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from mla_attention_paged_gb300 import build
    build.build()
    from mla_attention_paged_gb300 import mla as m
    return m


def test_bounded_wait_times_out_and_context_survives(mla, oracle_mod):
    assert mla.get_status() == mla.MLA_OK
    t0 = time.perf_counter()
    mla.selftest_wait_timeout()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert mla.get_status() == mla.MLA_ERR_TIMEOUT
    assert 0.5 < waited < 30.0
    assert mla.get_status() == mla.MLA_OK  # read-and-clear
    # the context still runs real work correctly
    wl = DecodeWorkload("after_timeout", 1, 2, 16, [333], seed=3)
    inp = make_decode_inputs(wl, "cpu")
    plan = mla.decode_plan(inp.seq_lens, 2, 16, 64, inp.page_table.shape[1], inp.kv_pool.shape[0])
    out, lse = mla.decode(plan, inp.q.cuda(), inp.kv_pool.cuda(), inp.page_table.cuda(), inp.seq_lens.cuda(),
                          inp.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    ref, _ = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale)
    assert np.abs(out.float().cpu().numpy() - ref).max() < 2e-2


def test_length_beyond_plan_is_reported(mla):
    wl = DecodeWorkload("too_long", 2, 1, 16, [500, 500], seed=4)
    inp = make_decode_inputs(wl, "cpu")
    plan = mla.decode_plan([500, 500], 1, 16, 64, inp.page_table.shape[1], inp.kv_pool.shape[0])
    bad = torch.tensor([500, 600], dtype=torch.int32)  # 600 > planned maximum 500
    mla.decode(plan, inp.q.cuda(), inp.kv_pool.cuda(), inp.page_table.cuda(), bad.cuda(), inp.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_ERR_DEVICE_ARG
    assert mla.get_status() == mla.MLA_OK


@pytest.mark.parametrize("bad_id", [-1, 10**6], ids=["negative", "past_pool"])
def test_page_id_outside_pool_is_reported(mla, bad_id):
    wl = DecodeWorkload("bad_page", 2, 2, 16, [700, 300], seed=6)
    inp = make_decode_inputs(wl, "cpu")
    plan = mla.decode_plan([700, 300], 2, 16, 64, inp.page_table.shape[1], inp.kv_pool.shape[0])
    pt = inp.page_table.clone()
    pt[0, 3] = bad_id
    mla.decode(plan, inp.q.cuda(), inp.kv_pool.cuda(), pt.cuda(), inp.seq_lens.cuda(), inp.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_ERR_DEVICE_ARG
    # the valid table runs clean afterwards
    mla.decode(plan, inp.q.cuda(), inp.kv_pool.cuda(), inp.page_table.cuda(), inp.seq_lens.cuda(), inp.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK


def test_prefill_request_beyond_max_seqlen_is_reported(mla):
    """max_seqlen_q below a request's new-token count: the grid covers only its first
    query block, so the kernel reports the request instead of leaving rows unwritten."""
    from mla_attention_paged_gb300.inputs import PrefillWorkload, make_prefill_inputs
    pi = make_prefill_inputs(PrefillWorkload("too_many_new", [100, 50], [300, 40], 2, seed=7), "cuda")
    mla.prefill_varlen(pi.q, pi.k, pi.v, pi.cu_seqlens_q, pi.cu_seqlens_kv, pi.prefix_lens, 128, pi.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_ERR_DEVICE_ARG
    mla.prefill_varlen(pi.q, pi.k, pi.v, pi.cu_seqlens_q, pi.cu_seqlens_kv, pi.prefix_lens, 300, pi.scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
