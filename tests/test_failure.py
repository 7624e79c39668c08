"""Failure detection on the GPU without faulting or hanging it.

* The bounded mbarrier wait every kernel uses gives up after its limit and records
  MLA_ERR_TIMEOUT in the status word (a self-test kernel waits on a barrier that nothing
  arrives on); the context stays usable afterwards.
* A device-side argument check (a request longer than the plan allows) is caught by the
  kernel before any access that depends on it and reported as MLA_ERR_DEVICE_ARG.
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
