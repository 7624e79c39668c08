"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (an engine whose memory manager owns every free byte
of the device, a plugin given no allocator), so this entry point keeps its split-KV
scratch in a fixed 32 MiB buffer inside the library instead of taking a workspace.  The
test calls it through the C ABI twice in a row, on two different batches, and checks
each result against mla_decode with a caller-provided workspace, within the tolerances
the other decode tests use.  It lives in its own file so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from mla_attention_paged_gb300.inputs import DecodeWorkload, make_decode_inputs

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


def _noalloc_fn(mla):
    lib = ctypes.CDLL(mla.LIB_PATH)
    fn = lib.mla_decode_noalloc
    P = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(mla.DecodePlan), P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                   ctypes.c_float, P, P, P]
    return fn


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row(mla):
    fn = _noalloc_fn(mla)
    stream = torch.cuda.current_stream()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    cases = [DecodeWorkload("noalloc_a", 4, 4, 16, [32768, 32000, 20000, 12345], seed=501, peaked=True),
             DecodeWorkload("noalloc_b", 3, 2, 16, [4096, 60000, 333], seed=502)]
    for wl in cases:
        inp = make_decode_inputs(wl, "cuda")
        plan = mla.decode_plan(inp.seq_lens.cpu(), wl.q_len, wl.heads, wl.page_size, inp.page_table.shape[1],
                               inp.kv_pool.shape[0])
        assert plan.max_splits > 1 and 0 < plan.workspace_bytes <= (32 << 20)
        ref_out, ref_lse = mla.decode(plan, inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale)
        out = torch.empty_like(ref_out)
        lse = torch.empty_like(ref_lse)
        rc = fn(ctypes.byref(plan), p(inp.q), p(inp.kv_pool), p(inp.page_table), p(inp.seq_lens), wl.q_len,
                wl.heads, inp.scale, 1.0, p(out), p(lse), ctypes.c_void_p(stream.cuda_stream))
        assert rc == mla.MLA_OK, mla.status_string(rc)
        torch.cuda.synchronize()
        assert mla.get_status() == mla.MLA_OK
        a = out.float().cpu().numpy()
        r = ref_out.float().cpu().numpy()
        assert np.isfinite(a).all()
        assert np.abs(a - r).max() <= MAX_ABS
        assert np.linalg.norm(a - r) / np.linalg.norm(r) <= REL_L2
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= LSE_ABS
        # the binding's wrapper makes the same call
        out2, lse2 = mla.decode_noalloc(plan, inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale)
        torch.cuda.synchronize()
        assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
        assert torch.equal(lse2.view(torch.int32), lse.view(torch.int32))


def test_noalloc_rejects_plans_beyond_its_buffer(mla):
    fn = _noalloc_fn(mla)
    plan = mla.decode_plan([131072] * 16, 2, 128, 64, 2048, 16 * 2048, num_sms=100000)
    assert plan.workspace_bytes > (32 << 20)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = fn(ctypes.byref(plan), fake, fake, fake, fake, 2, 128, 0.07, 1.0, fake, fake, None)
    assert rc == mla.MLA_ERR_WORKSPACE_TOO_SMALL
