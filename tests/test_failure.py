"""Failure detection on the GPU without faulting or hanging it.

* The bounded mbarrier wait every kernel uses gives up after its limit and records
  MLA_ERR_TIMEOUT in the status word (a self-test kernel waits on a barrier that nothing
  arrives on); the context stays usable afterwards.
* Device-side argument checks are caught by the kernels before any access that depends
  on them and reported as MLA_ERR_DEVICE_ARG: a decode request longer than the plan
  allows, a page id outside the pool (bf16, e4m3 and int8 pools), and a prefill request
  with more new tokens than the host's max_seqlen_q sized the grid for.
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


def _decode_any(mla, plan, q, pool, scales, pt, sl, scale, kv_scale):
    if scales is not None:
        return mla.decode_int8_paged(plan, q, pool, scales, pt, sl, scale, kv_scale)
    return mla.decode(plan, q, pool, pt, sl, scale, kv_scale)


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "int8", "int8page"])
@pytest.mark.parametrize("bad", ["negative", "past_pool"])
def test_page_id_outside_pool_is_reported(mla, kv, bad):
    """A page id outside [0, num_pages) is reported as MLA_ERR_DEVICE_ARG.  The pool given
    to the call is a view into a larger allocation (16 spare pages on each side), so the
    ids used here (-1 and num_pages + 5) still name allocated memory: the test checks the
    report without any read outside an allocation, whatever the kernel does."""
    wl = DecodeWorkload("bad_page", 2, 2, 16, [700, 300], kv_dtype=kv, seed=6)
    inp = make_decode_inputs(wl, "cpu")
    n = inp.kv_pool.shape[0]
    big = torch.zeros((n + 32,) + tuple(inp.kv_pool.shape[1:]), dtype=inp.kv_pool.dtype, device="cuda")
    big[16:16 + n] = inp.kv_pool.cuda()
    pool = big[16:16 + n]
    kvd = {"e4m3": mla.MLA_KV_E4M3, "int8": mla.MLA_KV_INT8,
           "int8page": mla.MLA_KV_INT8_PAGE}.get(kv, mla.MLA_KV_BF16)
    plan = mla.decode_plan([700, 300], 2, 16, 64, inp.page_table.shape[1], n, kvd)
    scales = inp.page_scales.cuda().float() if inp.page_scales is not None else None
    pt = inp.page_table.clone()
    pt[0, 3] = -1 if bad == "negative" else n + 5
    _decode_any(mla, plan, inp.q.cuda(), pool, scales, pt.cuda(), inp.seq_lens.cuda(), inp.scale, inp.kv_scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_ERR_DEVICE_ARG
    # the valid table runs clean afterwards
    _decode_any(mla, plan, inp.q.cuda(), pool, scales, inp.page_table.cuda(), inp.seq_lens.cuda(), inp.scale,
                inp.kv_scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK


@pytest.mark.parametrize("bad", [-1.0, float("nan"), 300.0])
def test_page_scale_outside_range_is_reported(mla, bad):
    """A page scale (relative to kv_scale) that is negative, not finite or above 255, on a
    page a request reads, is reported as MLA_ERR_DEVICE_ARG; valid scales run clean after."""
    wl = DecodeWorkload("bad_scale", 2, 2, 16, [700, 300], kv_dtype="int8page", seed=8)
    inp = make_decode_inputs(wl, "cuda")
    n = inp.kv_pool.shape[0]
    plan = mla.decode_plan([700, 300], 2, 16, 64, inp.page_table.shape[1], n, mla.MLA_KV_INT8_PAGE)
    scales = inp.page_scales.float().clone()
    scales[int(inp.page_table[1, 2])] = bad * inp.kv_scale
    mla.decode_int8_paged(plan, inp.q, inp.kv_pool, scales, inp.page_table, inp.seq_lens, inp.scale, inp.kv_scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_ERR_DEVICE_ARG
    mla.decode_int8_paged(plan, inp.q, inp.kv_pool, inp.page_scales.float(), inp.page_table, inp.seq_lens,
                          inp.scale, inp.kv_scale)
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
