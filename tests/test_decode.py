"""GPU parity of mla_decode (through the C ABI) against the fp64 CPU oracle.

Tolerances (bf16 output): max-abs 2e-2 and relative L2 5e-3 over the compared outputs,
LSE within 1e-3 absolute; 8-bit KV (e4m3 or int8): the same relative-L2 and LSE bounds,
with max-abs 6e-2, against the oracle run on the same codes and scale.  Small cases are compared element by element over every output; the
full-size workloads are compared on sampled rows the oracle computes one by one, in the
same launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

from mla_attention_paged_gb300.inputs import DecodeWorkload, decode_workloads, make_decode_inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3
MAX_ABS_FP8 = 6e-2


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from mla_attention_paged_gb300 import build
    build.build()
    from mla_attention_paged_gb300 import mla as m
    return m


def run_gpu(mla, inp, num_sms=0, dev="cuda"):
    wl = inp.wl
    q = inp.q.to(dev)
    pool = inp.kv_pool.to(dev)
    pt = inp.page_table.to(dev)
    sl = inp.seq_lens.to(dev)
    kvd = {torch.uint8: mla.MLA_KV_E4M3, torch.int8: mla.MLA_KV_INT8}.get(pool.dtype, mla.MLA_KV_BF16)
    if inp.page_scales is not None:
        kvd = mla.MLA_KV_INT8_PAGE
    plan = mla.decode_plan(inp.seq_lens.cpu(), wl.q_len, wl.heads, wl.page_size, pt.shape[1], pool.shape[0],
                           kvd, num_sms)
    if inp.page_scales is not None:
        out, lse = mla.decode_int8_paged(plan, q, pool, inp.page_scales.to(dev).float(), pt, sl, inp.scale,
                                         inp.kv_scale)
    else:
        out, lse = mla.decode(plan, q, pool, pt, sl, inp.scale, inp.kv_scale)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    return out.float().cpu().numpy(), lse.cpu().numpy(), plan


def check(out, lse, ref_out, ref_lse, fp8=False):
    out = out.reshape(ref_out.shape)
    lse = lse.reshape(ref_lse.shape)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    err = np.abs(out - ref_out)
    assert err.max() <= (MAX_ABS_FP8 if fp8 else MAX_ABS), f"max-abs {err.max():.3e}"
    rel = np.linalg.norm(out - ref_out) / max(np.linalg.norm(ref_out), 1e-30)
    assert rel <= REL_L2, f"rel-L2 {rel:.3e}"
    lerr = np.abs(lse - ref_lse).max()
    assert lerr <= LSE_ABS, f"lse abs {lerr:.3e}"


def _full_check(mla, oracle_mod, wl, num_sms=0):
    inp = make_decode_inputs(wl, "cpu")
    out, lse, plan = run_gpu(mla, inp, num_sms)
    ref_out, ref_lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                                             kv_scale=inp.kv_scale, page_scales=inp.page_scales)
    check(out, lse, ref_out, ref_lse, fp8=(wl.kv_dtype != "bf16"))
    return out, lse, plan


# ------------------------------------------------------------------------------------
# small cases, every output compared
# ------------------------------------------------------------------------------------
SMALL = [
    # name, B, T, H, lens, page, kv
    ("one_key", 1, 1, 16, [1], 64, "bf16"),
    ("ragged_tails", 6, 1, 16, [1, 63, 64, 65, 127, 200], 64, "bf16"),
    ("drafts4", 3, 4, 16, [4, 70, 333], 64, "bf16"),
    ("drafts2_h8", 2, 2, 8, [129, 1000], 64, "bf16"),
    ("rows_not_mult16", 2, 3, 5, [90, 257], 64, "bf16"),
    ("two_groups", 2, 3, 40, [300, 77], 64, "bf16"),
    ("h128", 2, 2, 128, [520, 1999], 64, "bf16"),
    ("page8", 2, 4, 16, [45, 300], 8, "bf16"),
    ("page16", 2, 2, 16, [500, 17], 16, "bf16"),
    ("page32", 1, 4, 16, [1025], 32, "bf16"),
    ("page128", 2, 1, 16, [700, 129], 128, "bf16"),
    ("page256", 1, 4, 16, [2000], 256, "bf16"),
    ("long_single", 1, 1, 16, [20000], 64, "bf16"),
    # at most 32 folded rows (the bf16 kernel with Q in tensor memory and a three-tile ring):
    # page geometries, 1-4 tiles (the first tile in the stage Q arrived in is tile 2), 24
    # rows (the second row warp half full), 32 rows over many tiles
    ("narrow_page8", 2, 2, 16, [45, 300], 8, "bf16"),
    ("narrow_page32", 1, 2, 16, [1025], 32, "bf16"),
    ("narrow_page256", 1, 1, 16, [2000], 256, "bf16"),
    ("narrow_tails", 7, 2, 16, [2, 64, 127, 128, 129, 192, 193], 64, "bf16"),
    ("narrow_rows24", 2, 3, 8, [500, 1300], 64, "bf16"),
    ("narrow_rows32", 2, 2, 16, [4000, 9000], 64, "bf16"),
    ("narrow_one_row", 2, 1, 1, [100, 7], 64, "bf16"),   # one folded row: BMM2 N = 16
    ("narrow_rows17", 2, 1, 17, [300, 65], 64, "bf16"),  # the second row warp holds one row
    # 33-64 folded rows in one group: pages of 16 and 128 keys, lengths around tile
    # boundaries, 40 and 48 rows, long requests over many splits
    ("rows64_page16", 2, 4, 16, [300, 97], 16, "bf16"),
    ("rows64_page128", 2, 4, 16, [700, 129], 128, "bf16"),
    ("rows64_tails", 8, 4, 16, [4, 47, 48, 49, 96, 97, 191, 240], 64, "bf16"),
    ("rows40", 2, 5, 8, [500, 1300], 64, "bf16"),
    ("rows48", 2, 3, 16, [777, 2049], 32, "bf16"),
    ("rows64_long", 2, 4, 16, [9000, 17000], 64, "bf16"),
    ("fp8_drafts4", 2, 4, 16, [300, 1000], 64, "e4m3"),
    ("fp8_ragged", 3, 1, 16, [1, 65, 130], 64, "e4m3"),
    ("fp8_page16", 2, 2, 16, [77, 500], 16, "e4m3"),
    ("fp8_page128", 1, 3, 16, [700], 128, "e4m3"),
    ("fp8_page8", 2, 4, 16, [45, 300], 8, "e4m3"),      # eight page boxes per tile
    ("fp8_page32", 1, 4, 16, [1025], 32, "e4m3"),
    ("fp8_page256", 1, 2, 16, [2000], 256, "e4m3"),
    ("fp8_tails", 5, 1, 16, [2, 64, 127, 128, 129], 64, "e4m3"),  # tile counts 1-3 and full tails
    ("fp8_h128", 1, 2, 128, [900], 64, "e4m3"),
    ("mtp8", 2, 8, 16, [700, 2000], 64, "bf16"),   # q_len 8: 128 folded rows, two row groups
    ("fp8_mtp8", 2, 8, 16, [333, 1500], 64, "e4m3"),
    ("int8_drafts4", 2, 4, 16, [300, 1000], 64, "int8"),
    ("int8_ragged", 3, 1, 16, [1, 65, 130], 64, "int8"),
    ("int8_page16", 2, 2, 16, [77, 500], 16, "int8"),
    ("int8_page128", 1, 3, 16, [700], 128, "int8"),
    ("int8_h128", 1, 2, 128, [900], 64, "int8"),
    ("int8_page8", 2, 4, 16, [45, 300], 8, "int8"),
    ("int8_page32", 1, 4, 16, [1025], 32, "int8"),
    ("int8_page256", 1, 2, 16, [2000], 256, "int8"),
    ("int8_tails", 5, 1, 16, [2, 64, 127, 128, 129], 64, "int8"),
    ("int8page_drafts4", 2, 4, 16, [300, 1000], 64, "int8page"),
    ("int8page_ragged", 3, 1, 16, [1, 65, 130], 64, "int8page"),
    ("int8page_page16", 2, 2, 16, [77, 500], 16, "int8page"),
    ("int8page_page128", 1, 3, 16, [700], 128, "int8page"),
    ("int8page_page8", 2, 4, 16, [45, 300], 8, "int8page"),
]


@pytest.mark.parametrize("name,B,T,H,lens,P,kv", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("peaked", [False, True], ids=["plain", "peaked"])
def test_decode_small(mla, oracle_mod, name, B, T, H, lens, P, kv, peaked):
    wl = DecodeWorkload(name, B, T, H, lens, page_size=P, kv_dtype=kv, seed=100 + len(name), peaked=peaked,
                        extra_pages=2)
    _full_check(mla, oracle_mod, wl)


@pytest.mark.parametrize("q_len", [4, 2], ids=["rows64", "rows32"])
@pytest.mark.parametrize("num_sms", [1, 3, 16, 152, 100000])
def test_decode_split_counts_agree(mla, oracle_mod, num_sms, q_len):
    """Different split counts (one split per request up to the minimum chunk) give the
    oracle's result; the LSE merge of the partials is exercised whenever splits > 1.  On 1
    and 3 SMs the plans take more than one wave and launch split by split; q_len 2 x 16
    heads runs the kernel with Q in tensor memory."""
    wl = DecodeWorkload("splits", 3, q_len, 16, [3000, 65, 9000], seed=77, peaked=True)
    _, _, plan = _full_check(mla, oracle_mod, wl, num_sms=num_sms)
    if num_sms >= 152:
        assert plan.max_splits > 1
    assert plan.split_major == (1 if num_sms <= 3 else 0)


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "int8"])
def test_decode_combine_many_splits(mla, oracle_mod, kv):
    """More than 64 splits per request: the combine takes its splits in several batches and
    rescales the running sum between them; a ragged batch mixes 2 to ~80 splits."""
    wl = DecodeWorkload("manysplits", 3, 2, 16, [20000, 300, 17000], kv_dtype=kv, seed=78, peaked=True)
    _, _, plan = _full_check(mla, oracle_mod, wl, num_sms=100000)
    assert plan.max_splits > 64


@pytest.mark.parametrize("kv,num_sms,q_len", [("bf16", 0, 4), ("e4m3", 0, 4), ("int8", 0, 4), ("bf16", 1, 4),
                                              ("bf16", 0, 2), ("bf16", 1, 2)],
                         ids=["bf16", "e4m3", "int8", "one_split", "bf16_rows32", "one_split_rows32"])
def test_decode_stages_equal_decode_bitwise(mla, kv, num_sms, q_len):
    """mla_decode_partial then mla_decode_combine gives mla_decode's bits (multi-split and
    single-split plans; the combine enqueues nothing for the latter).  q_len 2 x 16 heads
    runs the kernel that keeps Q in tensor memory."""
    wl = DecodeWorkload("stages", 3, q_len, 16, [5000, 130, 2999], kv_dtype=kv, seed=79, peaked=True)
    inp = make_decode_inputs(wl, "cuda")
    kvd = {"e4m3": mla.MLA_KV_E4M3, "int8": mla.MLA_KV_INT8}.get(kv, mla.MLA_KV_BF16)
    plan = mla.decode_plan(wl.seq_lens, wl.q_len, wl.heads, wl.page_size, inp.page_table.shape[1],
                           inp.kv_pool.shape[0], kvd, num_sms)
    assert (plan.max_splits > 1) == (num_sms == 0)
    out1, lse1 = mla.decode(plan, inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale, inp.kv_scale)
    out2, lse2, ws = mla.decode_partial(plan, inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                                        inp.kv_scale)
    mla.decode_combine(plan, inp.seq_lens, out2, lse2, workspace=ws)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1.view(torch.int32), lse2.view(torch.int32))


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "int8"])
def test_decode_one_million_keys_sampled(mla, oracle_mod, kv):
    """A 2^20-key context (16384 pages of 64): the planner's split count and the kernels at
    the long end, checked on sampled rows the oracle computes one by one."""
    wl = DecodeWorkload("l1m", 1, 2, 16, [1 << 20], kv_dtype=kv, seed=80)
    inp = make_decode_inputs(wl, "cuda")
    out, lse, plan = run_gpu(mla, inp)
    assert plan.max_splits > 1
    rows = [0, 5, 16, 31]
    ref_out, ref_lse = oracle_mod.mla_decode(inp.q.cpu(), inp.kv_pool.cpu(), inp.page_table.cpu(),
                                             inp.seq_lens.cpu(), inp.scale, kv_scale=inp.kv_scale, rows=rows)
    check(out.reshape(-1, 512)[rows], lse.reshape(-1)[rows], ref_out, ref_lse, fp8=(kv != "bf16"))
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_decode_maximum_rows_sampled(mla, oracle_mod):
    """The largest call the plan accepts: q_len 8192 new tokens x 16 heads = 131072 folded
    rows (2048 row groups, more than one wave of CTAs) over a 640-token paged prefix;
    sampled rows at the first and last tokens and at row-group boundaries against the
    oracle, every output finite."""
    T, H = 8192, 16
    wl = DecodeWorkload("max_rows", 1, T, H, [T + 640], seed=83)
    inp = make_decode_inputs(wl, "cuda")
    out, lse, plan = run_gpu(mla, inp)
    assert plan.rows == T * H == 131072 and plan.head_groups == 2048
    rows = [0, 1, 15, 16, 63, 64, 65, 4095, 4096, 65535, 65536, 100000, 131007, 131008, 131070, 131071]
    ref_out, ref_lse = oracle_mod.mla_decode(inp.q.cpu(), inp.kv_pool.cpu(), inp.page_table.cpu(),
                                             inp.seq_lens.cpu(), inp.scale, kv_scale=inp.kv_scale, rows=rows)
    check(out.reshape(-1, 512)[rows], lse.reshape(-1)[rows], ref_out, ref_lse, fp8=False)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("kv,T,lens", [("bf16", 64, [200, 1000]), ("bf16", 300, [4400]), ("e4m3", 128, [129, 3000])],
                         ids=["bf16_t64", "bf16_t300", "e4m3_t128"])
def test_decode_absorbed_prefill_over_paged_prefix(mla, oracle_mod, kv, T, lens):
    """Prefill of T new tokens over a paged prefix in absorbed form: the decode call with
    q_len = T (new token t sees the prefix and new tokens 0..t), T*H folded rows in many
    64-row groups; every output compared."""
    wl = DecodeWorkload("absorbed_prefill", len(lens), T, 16, lens, kv_dtype=kv, seed=81 + T)
    _full_check(mla, oracle_mod, wl)


def _wide_range_queries(seed, outlier):
    wl = DecodeWorkload("wide_q", 2, 4, 16, [700, 1500], kv_dtype="e4m3", seed=91)
    inp = make_decode_inputs(wl, "cpu")
    g = torch.Generator().manual_seed(seed)
    q = inp.q.float()
    q = q * torch.pow(2.0, torch.randint(-16, 5, q.shape, generator=g).float())
    q[0, 0, 0] = 0.0
    q[0, 1, 3, 17] = outlier
    inp.q = q.to(torch.bfloat16)
    return inp


def test_decode_e4m3_queries_over_many_binades(mla, oracle_mod):
    """The e4m3 kernel splits each bf16 query row into two e4m3 parts under a per-row
    power-of-two scale.  Rows whose elements span 2^-16 .. 2^4 of their typical size, an
    all-zero row and a row with one element 1000x its neighbours: parity with the oracle
    (on the same bf16 queries) within the usual bounds."""
    inp = _wide_range_queries(5, 40.0)
    out, lse, _ = run_gpu(mla, inp)
    ref_out, ref_lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                                             kv_scale=inp.kv_scale)
    check(out, lse, ref_out, ref_lse, fp8=True)


def test_decode_e4m3_query_split_error_bound(mla, oracle_mod):
    """The split is exact for elements within 2^9 of their row's largest |q|; smaller
    elements carry an absolute error of at most 2^-17 of it (e4m3's subnormal floor under
    the row scale).  A row with one element of 3e4 among elements near 1e-2 has scores in
    the thousands: its log-sum-exp stays within scale * 2^-17 * max|q| * max_j sum_i |k_ji|
    of the oracle's, every other row within 1e-3, and the outputs within the usual bounds."""
    inp = _wide_range_queries(5, 3.0e4)
    out, lse, _ = run_gpu(mla, inp)
    ref_out, ref_lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                                             kv_scale=inp.kv_scale)
    out = out.reshape(ref_out.shape)
    lse = lse.reshape(ref_lse.shape)
    rel = np.linalg.norm(out - ref_out) / np.linalg.norm(ref_out)
    assert np.isfinite(out).all() and rel <= REL_L2 and np.abs(out - ref_out).max() <= MAX_ABS_FP8
    keys = inp.kv_pool.view(torch.float8_e4m3fn).double().abs().sum(-1).max().item() * inp.kv_scale
    qmax = inp.q.float().abs().amax(-1).double().numpy()
    bound = np.maximum(inp.scale * 2.0 ** -17 * qmax * keys, LSE_ABS)
    assert (np.abs(lse - ref_lse) <= bound).all()


def test_decode_e4m3_dominant_key_over_long_tail(mla, oracle_mod):
    """The e4m3 kernel feeds P to its second GEMM in two 8-bit parts (e4m3 hi, e5m2 lo).
    Each head's query points at one key of its request, so that key's score stands 12 to
    19.5 above the others in the log2 domain (head h: 12 + h/2) and thousands of keys sit
    near 2^-12 .. 2^-19.5 of the row max: a tail that holds up to a few percent of the row's
    mass, which an e4m3 low part would flush to zero below 2^-15.  Every row's output
    within the relative-L2 bound of the oracle's, and the usual bounds overall."""
    wl = DecodeWorkload("long_tail", 2, 2, 16, [4096, 3000], kv_dtype="e4m3", seed=97)
    inp = make_decode_inputs(wl, "cpu")
    P = wl.page_size
    keys = inp.kv_pool.view(torch.float8_e4m3fn).double() * inp.kv_scale
    q = torch.empty(2, 2, 16, 576, dtype=torch.float64)
    for b, L in enumerate(wl.seq_lens):
        pos = L // 3
        kd = keys[int(inp.page_table[b, pos // P]), pos % P]
        for h in range(16):
            gap_log2 = 12.0 + 0.5 * h
            q[b, :, h] = kd * (gap_log2 * math.log(2.0) / (inp.scale * float(kd @ kd)))
    inp.q = q.to(torch.bfloat16)
    out, lse, _ = run_gpu(mla, inp)
    ref_out, ref_lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                                             kv_scale=inp.kv_scale)
    check(out, lse, ref_out, ref_lse, fp8=True)
    o = out.reshape(-1, 512)
    r = ref_out.reshape(-1, 512)
    row_rel = np.linalg.norm(o - r, axis=1) / np.linalg.norm(r, axis=1)
    assert row_rel.max() <= REL_L2, f"worst row rel-L2 {row_rel.max():.3e}"


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "int8", "int8page"])
def test_decode_running_max_rises_every_tile(mla, oracle_mod, kv):
    """Keys built so that each row's scores climb 4 to 7 (head h: 4 (1 + h/20)) in the log2
    domain every 64 keys: the running max moves on every tile of the e4m3 kernel (threshold
    2) and every second or third tile of the others (threshold 8), so O is rescaled again and
    again while BMM2s are in flight.  The climb lives in the 64 rope columns, which take part
    in the scores but not in V, so the outputs keep the usual size.  Parity with the oracle
    on every output."""
    wl = DecodeWorkload("rising", 2, 2, 16, [1000, 2100], kv_dtype=kv, seed=61)
    inp = make_decode_inputs(wl, "cpu")
    n_pages, P, _ = inp.kv_pool.shape
    g = torch.Generator().manual_seed(62)
    u = torch.zeros(576, dtype=torch.float64)
    u[512:] = torch.randn(64, generator=g, dtype=torch.float64)
    u /= u.norm()
    x = torch.randn(n_pages, P, 576, generator=g, dtype=torch.float64) * 0.5
    for b, L in enumerate(wl.seq_lens):
        idx = torch.arange(L)
        pages = inp.page_table[b, idx // P].long()
        x[pages, idx % P] += (4.0 * idx.double() / 64.0)[:, None] * u
    if kv == "bf16":
        inp.kv_pool, inp.kv_scale = x.to(torch.bfloat16), 1.0
    elif kv == "e4m3":
        inp.kv_scale = float(x.abs().max()) / 448.0
        inp.kv_pool = (x / inp.kv_scale).clamp(-448.0, 448.0).float().to(torch.float8_e4m3fn).view(torch.uint8)
    elif kv == "int8":
        inp.kv_scale = float(x.abs().max()) / 127.0
        inp.kv_pool = torch.round(x / inp.kv_scale).clamp(-127.0, 127.0).to(torch.int8)
    else:
        inp.page_scales = x.abs().amax(dim=(1, 2)).clamp(min=1e-30) / 127.0
        inp.kv_scale = float(inp.page_scales.max())
        inp.kv_pool = torch.round(x / inp.page_scales[:, None, None]).clamp(-127.0, 127.0).to(torch.int8)
    c = math.log(2.0) / inp.scale  # a key's score in the log2 domain is then its k . u
    q = torch.empty(2, 2, 16, 576, dtype=torch.float64)
    for h in range(16):
        q[:, :, h] = c * (1.0 + h / 20.0) * u
    inp.q = q.to(torch.bfloat16)
    out, lse, _ = run_gpu(mla, inp)
    ref_out, ref_lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                                             kv_scale=inp.kv_scale, page_scales=inp.page_scales)
    check(out, lse, ref_out, ref_lse, fp8=(kv != "bf16"))


def test_decode_page_shuffle_invariance_bitwise(mla):
    wl = DecodeWorkload("shuffle", 2, 4, 16, [1500, 777], seed=5, extra_pages=7)
    inp = make_decode_inputs(wl, "cpu")
    out1, lse1, _ = run_gpu(mla, inp)
    n = inp.kv_pool.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    pool2 = torch.empty_like(inp.kv_pool)
    pool2[perm] = inp.kv_pool
    inp.kv_pool = pool2
    inp.page_table = perm[inp.page_table.long()].to(torch.int32)
    out2, lse2, _ = run_gpu(mla, inp)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)


def test_decode_fold_neutrality(mla):
    """T drafts folded into one launch equal T single-token launches whose cache ends at
    each draft's own position.  Peaked inputs (a few keys dominate each row, outputs of
    the size of a value row) so that a row mixed up between the folded and the separate
    launches shows far above the relative-L2 bound."""
    wl = DecodeWorkload("fold", 2, 4, 16, [700, 1300], seed=9, peaked=True)
    inp = make_decode_inputs(wl, "cpu")
    out, lse, _ = run_gpu(mla, inp)
    out = out.reshape(2, 4, 16, 512)
    lse = lse.reshape(2, 4, 16)
    assert np.linalg.norm(out) > 1.0  # outputs are dominated by planted rows, not ~1e-4 means
    for t in range(4):
        w1 = DecodeWorkload("fold1", 2, 1, 16, [700 - 3 + t, 1300 - 3 + t], seed=9)
        one = make_decode_inputs(w1, "cpu")
        one.q = inp.q[:, t:t + 1].contiguous()
        one.kv_pool, one.page_table = inp.kv_pool, inp.page_table
        o1, l1, _ = run_gpu(mla, one)
        a = o1.reshape(2, 16, 512)
        b = out[:, t]
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= REL_L2
        assert np.abs(l1.reshape(2, 16) - lse[:, t]).max() <= LSE_ABS


# ------------------------------------------------------------------------------------
# full-size workloads, sampled rows
# ------------------------------------------------------------------------------------
def _sample_rows(wl, per_request=8, seed=0):
    g = np.random.default_rng(seed)
    rows = []
    for b in range(wl.batch):
        picks = {(0, 0), (wl.q_len - 1, wl.heads - 1)}
        while len(picks) < per_request:
            picks.add((int(g.integers(wl.q_len)), int(g.integers(wl.heads))))
        for t, h in sorted(picks):
            rows.append((b * wl.q_len + t) * wl.heads + h)
    return rows


@pytest.mark.parametrize("name", list(decode_workloads().keys()))
def test_decode_full_size_sampled(mla, oracle_mod, name):
    wl = decode_workloads()[name]
    inp = make_decode_inputs(wl, "cuda")
    out, lse, plan = run_gpu(mla, inp)
    rows = _sample_rows(wl, per_request=16 if wl.batch <= 4 else 6)
    ref_out, ref_lse = oracle_mod.mla_decode(inp.q.cpu(), inp.kv_pool.cpu(), inp.page_table.cpu(),
                                             inp.seq_lens.cpu(), inp.scale, kv_scale=inp.kv_scale, rows=rows,
                                             page_scales=inp.page_scales)
    check(out.reshape(-1, 512)[rows], lse.reshape(-1)[rows], ref_out, ref_lse, fp8=(wl.kv_dtype != "bf16"))
    # every output finite, including rows not sampled
    assert np.isfinite(out).all() and np.isfinite(lse).all()
