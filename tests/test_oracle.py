"""Pins for the CPU fp64 oracle (no GPU).

The pages print no worked example, so the oracle is pinned to things outside itself:
  * library routines for the textbook formula: torch's float64 scaled_dot_product_attention
    with an explicit boolean mask, and torch.logsumexp, on tiny shapes;
  * closed forms: equal scores give the mean of the visible values with
    lse = s + ln(n_visible); a single visible key returns that value row;
  * invariants of the method: physical page order does not matter, split + LSE merge
    equals the unsplit result, folding draft tokens into rows is result-neutral;
  * the e4m3 decode table against torch's float8_e4m3fn conversion on all 256 codes and
    against points the format definition fixes;
  * int8 codes: with a power-of-two scale the decoded values are exact in bf16, so the
    int8 pool must give bit-for-bit the bf16 pool's result; the extreme codes decode to
    -128 and 127 times the scale;
  * int8 codes with a scale per page: library SDPA on the rows dequantised page by page;
    equal page scales give bit-for-bit the per-tensor result; one visible key in a page
    whose id differs from its table slot returns its codes times that page's scale.
Each is chosen so that a plausible slip (dropped term, wrong causal index, wrong value
columns, transposed operand, wrong log base) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from mla_attention_paged_gb300.inputs import DecodeWorkload, make_decode_inputs

D, DV = 576, 512


def _paged(B, T, H, lens, P, seed, kv="bf16", extra_pages=3, peaked=False):
    wl = DecodeWorkload("tiny", B, T, H, list(lens), page_size=P, kv_dtype=kv, seed=seed,
                        extra_pages=extra_pages, peaked=peaked)
    return make_decode_inputs(wl, "cpu")


def _dense_kv(inp, b, L):
    """Gather request b's first L latent rows from the pool (indexing only) as float64."""
    P = inp.kv_pool.shape[1]
    idx = torch.arange(L)
    pages = inp.page_table[b, idx // P].long()
    rows = inp.kv_pool[pages, idx % P]
    if rows.dtype == torch.uint8:
        rows = rows.view(torch.float8_e4m3fn).to(torch.float64) * inp.kv_scale
    elif rows.dtype == torch.int8:
        if inp.page_scales is not None:
            rows = rows.to(torch.float64) * inp.page_scales.double()[pages][:, None]
        else:
            rows = rows.to(torch.float64) * inp.kv_scale
    else:
        rows = rows.to(torch.float64)
    return rows


def _sdpa_decode(inp, lens_include_drafts=True):
    B, T, H, _ = inp.q.shape
    out = torch.zeros(B, T, H, DV, dtype=torch.float64)
    lse = torch.zeros(B, T, H, dtype=torch.float64)
    for b in range(B):
        L = int(inp.seq_lens[b]) + (0 if lens_include_drafts else T)
        kv = _dense_kv(inp, b, L)                      # [L, 576]
        q = inp.q[b].to(torch.float64).permute(1, 0, 2)  # [H, T, 576]
        mask = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]  # [T, L]
        o = F.scaled_dot_product_attention(q, kv[None].expand(H, L, D), kv[None, :, :DV].expand(H, L, DV),
                                           attn_mask=mask[None], scale=inp.scale)
        out[b] = o.permute(1, 0, 2)
        s = torch.matmul(q, kv.T) * inp.scale
        s = s.masked_fill(~mask[None], float("-inf"))
        lse[b] = torch.logsumexp(s, dim=-1).T
    return out.numpy(), lse.numpy()


CASES = [
    # B, T, H, lens, P, kv
    (1, 1, 1, [1], 1, "bf16"),
    (1, 1, 2, [5], 4, "bf16"),
    (2, 4, 3, [4, 70], 16, "bf16"),
    (2, 2, 4, [65, 64], 64, "bf16"),
    (2, 3, 2, [33, 9], 4, "e4m3"),
    (1, 4, 4, [70], 64, "e4m3"),
    (2, 3, 2, [33, 9], 4, "int8"),
    (1, 4, 4, [70], 64, "int8"),
    (2, 3, 2, [33, 9], 4, "int8page"),
    (2, 2, 3, [70, 130], 64, "int8page"),
    (2, 2, 2, [300, 129], 128, "bf16"),   # pages larger than one tile, a request ending inside one
    (1, 1, 2, [600], 256, "e4m3"),
]


@pytest.mark.parametrize("B,T,H,lens,P,kv", CASES)
@pytest.mark.parametrize("peaked", [False, True])
def test_decode_matches_library_sdpa(oracle_mod, B, T, H, lens, P, kv, peaked):
    inp = _paged(B, T, H, lens, P, seed=7 + B + T + P, kv=kv, peaked=peaked)
    out, lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                                     kv_scale=inp.kv_scale, page_scales=inp.page_scales)
    ref_out, ref_lse = _sdpa_decode(inp)
    np.testing.assert_allclose(out, ref_out, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_decode_other_draft_reading_matches_sdpa(oracle_mod):
    inp = _paged(2, 3, 2, [10, 17], 4, seed=11)
    out, lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens - 3, inp.scale,
                                     lens_include_drafts=False)
    ref_out, ref_lse = _sdpa_decode(inp)
    np.testing.assert_allclose(out, ref_out, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_equal_scores_give_mean_of_visible_values(oracle_mod):
    """Query non-zero only on the rope columns, every key sharing its rope columns: all
    scores are equal, so out is the plain mean of the visible value rows (first 512
    columns) and lse = s + ln(n_visible)."""
    B, T, H, L, P = 1, 4, 2, 37, 8
    inp = _paged(B, T, H, [L], P, seed=3)
    q = torch.zeros(B, T, H, D)
    q[..., DV:] = torch.randn(B, T, H, D - DV, generator=torch.Generator().manual_seed(5))
    q = q.to(torch.bfloat16)
    rope = torch.randn(D - DV, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    pool = inp.kv_pool.clone()
    pool[:, :, DV:] = rope
    out, lse = oracle_mod.mla_decode(q, pool, inp.page_table, inp.seq_lens, inp.scale)
    vals = torch.stack([pool[int(inp.page_table[0, j // P]), j % P, :DV] for j in range(L)]).to(torch.float64)
    for t in range(T):
        n_vis = L - T + t + 1
        mean = vals[:n_vis].mean(0).numpy()
        for h in range(H):
            s = inp.scale * float(torch.dot(q[0, t, h].double(), pool[0, 0].double()))
            np.testing.assert_allclose(out[0, t, h], mean, rtol=1e-12, atol=1e-15)
            assert abs(lse[0, t, h] - (s + math.log(n_vis))) < 1e-12


def test_single_visible_key_returns_that_value_row(oracle_mod):
    """L_b = T: draft 0 sees only key 0, so out = V row 0 exactly, lse = scale * q . k_0."""
    B, T, H, P = 2, 4, 3, 4
    inp = _paged(B, T, H, [T] * B, P, seed=9, peaked=True)
    out, lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale)
    for b in range(B):
        k0 = inp.kv_pool[int(inp.page_table[b, 0]), 0].double()
        for h in range(H):
            np.testing.assert_array_equal(out[b, 0, h], k0[:DV].numpy())
            s = inp.scale * float(np.dot(inp.q[b, 0, h].double().numpy(), k0.numpy()))
            assert abs(lse[b, 0, h] - s) < 1e-13


def test_page_shuffle_invariance_bitwise(oracle_mod):
    B, T, H, P = 2, 2, 4, 4
    inp = _paged(B, T, H, [23, 41], P, seed=13, extra_pages=5)
    out1, lse1 = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale)
    n = inp.kv_pool.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(99))
    pool2 = torch.empty_like(inp.kv_pool)
    pool2[perm] = inp.kv_pool                     # physical page p moves to slot perm[p]
    pt2 = perm[inp.page_table.long()].to(torch.int32)
    out2, lse2 = oracle_mod.mla_decode(inp.q, pool2, pt2, inp.seq_lens, inp.scale)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)


def test_split_plus_lse_merge_equals_unsplit(oracle_mod):
    """softmax over keys [0, L) from the two halves [0, c) and [c, L) merged by LSE."""
    B, T, H, P, L, c = 1, 1, 3, 8, 96, 40
    inp = _paged(B, T, H, [L], P, seed=17)
    full_o, full_l = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale)
    o1, l1 = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, torch.tensor([c]), inp.scale)
    pt2 = inp.page_table[:, c // P:]
    o2, l2 = oracle_mod.mla_decode(inp.q, inp.kv_pool, pt2, torch.tensor([L - c]), inp.scale)
    lse = np.logaddexp(l1, l2)
    merged = np.exp(l1 - lse)[..., None] * o1 + np.exp(l2 - lse)[..., None] * o2
    np.testing.assert_allclose(merged, full_o, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse, full_l, rtol=1e-13, atol=1e-13)


def test_fold_neutrality(oracle_mod):
    """T draft rows computed together equal T single-token calls whose cache ends at the
    draft's own position (the causal limit of draft t is L - T + t)."""
    B, T, H, P = 2, 4, 3, 8
    lens = [29, 50]
    inp = _paged(B, T, H, lens, P, seed=19)
    out, lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale)
    for t in range(T):
        lt = inp.seq_lens - T + 1 + t
        o, l = oracle_mod.mla_decode(inp.q[:, t:t + 1].contiguous(), inp.kv_pool, inp.page_table, lt, inp.scale)
        np.testing.assert_array_equal(o[:, 0], out[:, t])
        np.testing.assert_array_equal(l[:, 0], lse[:, t])


def test_row_selection_matches_full(oracle_mod):
    inp = _paged(2, 2, 4, [31, 12], 4, seed=23)
    out, lse = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale)
    rows = [0, 5, 9, 15, 3]
    o, l = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale, rows=rows)
    np.testing.assert_array_equal(o, out.reshape(-1, DV)[rows])
    np.testing.assert_array_equal(l, lse.reshape(-1)[rows])


def test_decode_rejects_bad_arguments(oracle_mod):
    inp = _paged(1, 4, 1, [8], 4, seed=1)
    with pytest.raises(ValueError):   # fewer cached tokens than drafts
        oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, torch.tensor([3]), inp.scale)
    bad = inp.page_table.clone()
    bad[0, 0] = inp.kv_pool.shape[0]
    with pytest.raises(ValueError):   # page id outside the pool
        oracle_mod.mla_decode(inp.q, inp.kv_pool, bad, inp.seq_lens, inp.scale)


# ------------------------------------------------------------------------------------
# e4m3 table
# ------------------------------------------------------------------------------------

def test_e4m3_table_matches_torch_on_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle_mod.e4m3_to_double(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))


def test_e4m3_format_points(oracle_mod):
    f = lambda c: float(oracle_mod.e4m3_to_double([c])[0])
    assert f(0x7E) == 448.0 and f(0xFE) == -448.0          # largest finite
    assert math.isnan(f(0x7F)) and math.isnan(f(0xFF))     # the only NaNs
    assert f(0x01) == 2.0 ** -9                            # smallest subnormal
    assert f(0x08) == 2.0 ** -6                            # smallest normal
    assert f(0x38) == 1.0 and f(0x40) == 2.0 and f(0x39) == 1.125
    assert f(0x00) == 0.0 and math.copysign(1.0, f(0x80)) == -1.0
    finite = [c for c in range(256) if not math.isnan(f(c))]
    assert len(finite) == 254


def test_int8_pool_equals_bf16_pool_of_its_values(oracle_mod):
    inp = _paged(2, 3, 4, [70, 13], 16, seed=21, kv="int8")
    scale = 2.0 ** -5  # codes * 2^-5 (|code| <= 127, seven bits) are exact in bf16
    vals = (inp.kv_pool.to(torch.float64) * scale).to(torch.bfloat16)
    assert torch.equal(vals.to(torch.float64), inp.kv_pool.to(torch.float64) * scale)
    o8, l8 = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale, kv_scale=scale)
    ob, lb = oracle_mod.mla_decode(inp.q, vals, inp.page_table, inp.seq_lens, inp.scale)
    np.testing.assert_array_equal(o8, ob)
    np.testing.assert_array_equal(l8, lb)


def test_int8_extreme_codes(oracle_mod):
    # one visible key: the output is that key's value row, i.e. the decoded codes
    q = torch.zeros(1, 1, 1, D, dtype=torch.bfloat16)
    pool = torch.zeros(1, 1, D, dtype=torch.int8)
    pool[0, 0, :4] = torch.tensor([-128, 127, -1, 1], dtype=torch.int8)
    out, lse = oracle_mod.mla_decode(q, pool, torch.zeros(1, 1, dtype=torch.int32), torch.ones(1, dtype=torch.int32),
                                     0.1, kv_scale=0.5)
    assert out[0, 0, 0, :4].tolist() == [-64.0, 63.5, -0.5, 0.5]
    assert lse[0, 0, 0] == 0.0


def test_int8_equal_page_scales_equal_per_tensor_bitwise(oracle_mod):
    inp = _paged(2, 3, 4, [70, 13], 16, seed=23, kv="int8")
    n_pages = inp.kv_pool.shape[0]
    o1, l1 = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale, kv_scale=0.037)
    o2, l2 = oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                                   page_scales=torch.full((n_pages,), 0.037, dtype=torch.float64))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_int8_page_scale_is_that_of_the_rows_page(oracle_mod):
    # one visible key, in physical page 1 named by table slot 0: the output is its codes
    # times page 1's scale (not slot 0's, not page 0's)
    q = torch.zeros(1, 1, 1, D, dtype=torch.bfloat16)
    pool = torch.zeros(2, 1, D, dtype=torch.int8)
    pool[1, 0, :4] = torch.tensor([-128, 127, -1, 1], dtype=torch.int8)
    pool[0, 0, :4] = torch.tensor([5, 5, 5, 5], dtype=torch.int8)
    table = torch.tensor([[1, 0]], dtype=torch.int32)
    out, lse = oracle_mod.mla_decode(q, pool, table, torch.ones(1, dtype=torch.int32), 0.1,
                                     page_scales=torch.tensor([0.5, 0.25], dtype=torch.float64))
    assert out[0, 0, 0, :4].tolist() == [-32.0, 31.75, -0.25, 0.25]
    assert lse[0, 0, 0] == 0.0


def test_page_scales_rejected_for_non_int8_pools(oracle_mod):
    inp = _paged(1, 1, 2, [5], 4, seed=3)
    with pytest.raises(TypeError):
        oracle_mod.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                              page_scales=torch.ones(inp.kv_pool.shape[0]))


# ------------------------------------------------------------------------------------
# prefill
# ------------------------------------------------------------------------------------

def _prefill_case(prefix, new, H, dqk, dv, seed):
    g = torch.Generator().manual_seed(seed)
    nq, nkv = sum(new), sum(p + n for p, n in zip(prefix, new))
    q = torch.randn(nq, H, dqk, generator=g).to(torch.bfloat16)
    k = torch.randn(nkv, H, dqk, generator=g).to(torch.bfloat16)
    v = torch.randn(nkv, H, dv, generator=g).to(torch.bfloat16)
    cq, ck = [0], [0]
    for p, n in zip(prefix, new):
        cq.append(cq[-1] + n)
        ck.append(ck[-1] + p + n)
    return q, k, v, torch.tensor(cq, dtype=torch.int32), torch.tensor(ck, dtype=torch.int32), \
        torch.tensor(prefix, dtype=torch.int32)


def _sdpa_prefill(q, k, v, cq, ck, prefix, scale):
    out = torch.zeros(q.shape[0], q.shape[1], v.shape[2], dtype=torch.float64)
    lse = torch.zeros(q.shape[0], q.shape[1], dtype=torch.float64)
    for b in range(len(prefix)):
        qb = q[cq[b]:cq[b + 1]].double().permute(1, 0, 2)
        kb = k[ck[b]:ck[b + 1]].double().permute(1, 0, 2)
        vb = v[ck[b]:ck[b + 1]].double().permute(1, 0, 2)
        n, L = qb.shape[1], kb.shape[1]
        if n == 0:
            continue
        mask = torch.arange(L)[None, :] <= (int(prefix[b]) + torch.arange(n))[:, None]
        out[cq[b]:cq[b + 1]] = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask[None], scale=scale).permute(1, 0, 2)
        s = (qb @ kb.transpose(1, 2) * scale).masked_fill(~mask[None], float("-inf"))
        lse[cq[b]:cq[b + 1]] = torch.logsumexp(s, -1).T
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("prefix,new,H", [([0], [5], 1), ([7, 0, 33], [3, 6, 1], 2), ([130, 5], [0, 70], 3)])
def test_prefill_matches_library_sdpa(oracle_mod, prefix, new, H):
    q, k, v, cq, ck, pl = _prefill_case(prefix, new, H, 192, 128, seed=len(prefix) + H)
    scale = 1 / math.sqrt(192)
    out, lse = oracle_mod.mla_prefill(q, k, v, cq, ck, pl, scale)
    ref_out, ref_lse = _sdpa_prefill(q, k, v, cq, ck, pl, scale)
    np.testing.assert_allclose(out, ref_out, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_prefill_without_prefix_is_plain_causal(oracle_mod):
    q, k, v, cq, ck, pl = _prefill_case([0, 0], [9, 17], 2, 192, 128, seed=31)
    scale = 0.1
    out, _ = oracle_mod.mla_prefill(q, k, v, cq, ck, pl, scale)
    for b in range(2):
        qb = q[cq[b]:cq[b + 1]].double().permute(1, 0, 2)
        kb = k[ck[b]:ck[b + 1]].double().permute(1, 0, 2)
        vb = v[ck[b]:ck[b + 1]].double().permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(qb, kb, vb, is_causal=True, scale=scale).permute(1, 0, 2)
        np.testing.assert_allclose(out[cq[b]:cq[b + 1]], ref.numpy(), rtol=1e-10, atol=1e-13)


def test_prefill_single_new_token_equals_decode(oracle_mod):
    """One new token per request, one head, qk = the 576 latent row and v = its first
    512 columns: the prefill row is the decode row with q_len 1 over the same keys."""
    prefix = [40, 3]
    new = [1, 1]
    g = torch.Generator().manual_seed(37)
    nkv = sum(prefix) + 2
    lat = torch.randn(nkv, 1, D, generator=g).to(torch.bfloat16)
    q = torch.randn(2, 1, D, generator=g).to(torch.bfloat16)
    cq = torch.tensor([0, 1, 2], dtype=torch.int32)
    ck = torch.tensor([0, 41, 45], dtype=torch.int32)
    pl = torch.tensor(prefix, dtype=torch.int32)
    scale = 0.05
    out_p, lse_p = oracle_mod.mla_prefill(q, lat, lat[:, :, :DV].contiguous(), cq, ck, pl, scale)
    # the same rows as a paged decode with page size 1: pool row = kv row
    pool = lat.reshape(nkv, 1, D)
    pt = torch.zeros(2, 41, dtype=torch.int32)
    pt[0, :41] = torch.arange(0, 41)
    pt[1, :4] = torch.arange(41, 45)
    out_d, lse_d = oracle_mod.mla_decode(q.reshape(2, 1, 1, D), pool, pt, torch.tensor([41, 4]), scale)
    np.testing.assert_array_equal(out_p[:, 0], out_d[:, 0, 0])
    np.testing.assert_array_equal(lse_p[:, 0], lse_d[:, 0, 0])


def test_prefill_rejects_inconsistent_lengths(oracle_mod):
    q, k, v, cq, ck, pl = _prefill_case([4], [3], 1, 192, 128, seed=1)
    with pytest.raises(ValueError):
        oracle_mod.mla_prefill(q, k, v, cq, ck, pl + 1, 0.1)
