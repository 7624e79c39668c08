"""Seeded synthetic inputs for MLA decode and prefill.

This module draws random numbers and lays them out; it holds none of the attention
arithmetic.  Both the CUDA path and the CPU oracle consume what it returns.

Workload shapes follow the coding-agent serving pattern the TokenSpeed pages describe
(long cached prefixes, a handful of speculative draft tokens per decode step, ragged
prefill appends of a few hundred to a few thousand tokens on top of a long prefix; see
"构建面向 Agentic 推理的下一代 LLM 推理引擎", sections "为什么 Agentic 推理需要新推理引擎"
and "Kernel：让 MLA 真正跑满 GPU").  The public SWE-smith traffic those pages measure on
is not available; these synthetic draws stand in for it.

Recipe (all draws from one torch.Generator seeded per workload):
  * decode Q and latent KV: N(0, 1) / sqrt(576), bf16; scale 1/sqrt(192).
  * FP8 KV: latent N(0, 1), kv_scale = amax|x| / 448, codes = e4m3fn(x / kv_scale).
  * INT8 KV: latent N(0, 1), kv_scale = amax|x| / 127, codes = round(x / kv_scale) as int8.
  * INT8 KV with a scale per page: each page's N(0, 1) latents times 2^U(-2, 0), encoded with
    that page's amax / 127; kv_scale = the largest page scale.
  * pages: 64-token pages; each request owns ceil(L_b / 64) pages taken from one shared
    pool in a random permutation.
  * "peaked" variants multiply Q by 30 and plant near-copies of a query direction into
    random key rows so that attention concentrates (exercises max/rescale logic).
  * prefill Q/K/V: N(0, 1) bf16, 16 heads, qk 192, v 128, scale 1/sqrt(192).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D_LATENT = 576   # 512 latent + 64 rope columns
D_V = 512        # value = first 512 latent columns
D_QK_PREFILL = 192
D_V_PREFILL = 128


@dataclass
class DecodeWorkload:
    name: str
    batch: int
    q_len: int
    heads: int
    seq_lens: list            # per request, drafts included
    page_size: int = 64
    kv_dtype: str = "bf16"    # "bf16", "e4m3", "int8" or "int8page"
    seed: int = 0
    peaked: bool = False
    extra_pages: int = 0      # unused pool pages (pool larger than needed)


@dataclass
class PrefillWorkload:
    name: str
    prefix_lens: list
    new_lens: list
    heads: int = 16
    seed: int = 0


def _ragged_lens(batch, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g)]


def decode_workloads():
    """The decode workloads: small, speculative, ragged (16 and 128 heads), FP8 (q_len 4, and the
    ragged shape) and its bf16 twin."""
    return {
        "decode_b1_q1_h16_l1024": DecodeWorkload("decode_b1_q1_h16_l1024", 1, 1, 16, [1024], seed=1000),
        "decode_b4_q4_h16_l32k": DecodeWorkload("decode_b4_q4_h16_l32k", 4, 4, 16, [32768] * 4, seed=1001),
        "decode_b16_q2_h16_ragged": DecodeWorkload(
            "decode_b16_q2_h16_ragged", 16, 2, 16, _ragged_lens(16, 8192, 131072, 1002), seed=1002),
        "decode_b16_q2_h128_ragged": DecodeWorkload(
            "decode_b16_q2_h128_ragged", 16, 2, 128, _ragged_lens(16, 8192, 131072, 1002), seed=1002),
        "decode_fp8_b8_q4_h16_l64k": DecodeWorkload(
            "decode_fp8_b8_q4_h16_l64k", 8, 4, 16, [65536] * 8, kv_dtype="e4m3", seed=1003),
        "decode_fp8_b16_q4_h16_l64k": DecodeWorkload(
            "decode_fp8_b16_q4_h16_l64k", 16, 4, 16, [65536] * 16, kv_dtype="e4m3", seed=1003),
        # the headline's shape over an e4m3 pool (32 folded rows per request)
        "decode_fp8_b16_q2_h16_ragged": DecodeWorkload(
            "decode_fp8_b16_q2_h16_ragged", 16, 2, 16, _ragged_lens(16, 8192, 131072, 1002), kv_dtype="e4m3",
            seed=1002),
        "decode_bf16_b16_q4_h16_l64k": DecodeWorkload(
            "decode_bf16_b16_q4_h16_l64k", 16, 4, 16, [65536] * 16, seed=1003),
        "decode_int8_b16_q4_h16_l64k": DecodeWorkload(
            "decode_int8_b16_q4_h16_l64k", 16, 4, 16, [65536] * 16, kv_dtype="int8", seed=1003),
        "decode_int8page_b16_q4_h16_l64k": DecodeWorkload(
            "decode_int8page_b16_q4_h16_l64k", 16, 4, 16, [65536] * 16, kv_dtype="int8page", seed=1003),
        # prefill in absorbed form over a paged prefix: 512 new tokens on 32K cached ones
        "decode_b4_q512_h16_l32k": DecodeWorkload(
            "decode_b4_q512_h16_l32k", 4, 512, 16, [32768 + 512] * 4, seed=1005),
    }


def prefill_workloads():
    g = torch.Generator().manual_seed(1004)
    prefix = [int(x) for x in torch.randint(20000, 100001, (5,), generator=g)]
    new = [int(x) for x in torch.randint(256, 2049, (5,), generator=g)]
    return {"prefill_b5_h16_prefix": PrefillWorkload("prefill_b5_h16_prefix", prefix, new, 16, seed=1004),
            # a smaller case of the same kernel (K/V ~1 GB, above L2) for profiler captures
            "prefill_b2_h16_prefix24k": PrefillWorkload("prefill_b2_h16_prefix24k", [24000, 23000], [1024, 1024], 16,
                                                        seed=1006)}


@dataclass
class DecodeInputs:
    q: torch.Tensor            # [B, T, H, 576] bf16
    kv_pool: torch.Tensor      # [n_pages, page, 576] bf16, uint8 e4m3 codes or int8 codes
    page_table: torch.Tensor   # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    kv_scale: float
    scale: float
    wl: DecodeWorkload = field(repr=False, default=None)
    page_scales: torch.Tensor = None  # [n_pages] float32 (int8 pools with a scale per page)


def make_decode_inputs(wl: DecodeWorkload, device="cpu", max_pages=None) -> DecodeInputs:
    """Draw the inputs of one decode workload on ``device`` from its seed."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    B, T, H, P = wl.batch, wl.q_len, wl.heads, wl.page_size
    pages_per = [(L + P - 1) // P for L in wl.seq_lens]
    n_pages = sum(pages_per) + wl.extra_pages
    mp = max(pages_per) if max_pages is None else max_pages
    q = torch.randn(B, T, H, D_LATENT, generator=g, device=dev, dtype=torch.float32) / math.sqrt(D_LATENT)
    if wl.peaked:
        q = q * 30.0
    perm = torch.randperm(n_pages, generator=g, device=dev).to(torch.int32)
    page_table = torch.zeros(B, mp, dtype=torch.int32, device=dev)
    off = 0
    for b, n in enumerate(pages_per):
        page_table[b, :n] = perm[off:off + n]
        off += n
    # latent pool, drawn page by page range to bound the fp32 temporary
    kv_scale = 1.0
    if wl.kv_dtype == "bf16":
        pool = torch.empty(n_pages, P, D_LATENT, dtype=torch.bfloat16, device=dev)
        step = max(1, (1 << 27) // (P * D_LATENT))
        for s in range(0, n_pages, step):
            e = min(n_pages, s + step)
            pool[s:e] = (torch.randn(e - s, P, D_LATENT, generator=g, device=dev) / math.sqrt(D_LATENT)).to(torch.bfloat16)
    elif wl.kv_dtype == "e4m3":
        raw = torch.empty(n_pages, P, D_LATENT, dtype=torch.float32, device=dev)
        step = max(1, (1 << 27) // (P * D_LATENT))
        for s in range(0, n_pages, step):
            e = min(n_pages, s + step)
            raw[s:e] = torch.randn(e - s, P, D_LATENT, generator=g, device=dev)
        amax = float(raw.abs().max())
        kv_scale = amax / 448.0
        pool = torch.empty(n_pages, P, D_LATENT, dtype=torch.uint8, device=dev)
        for s in range(0, n_pages, step):
            e = min(n_pages, s + step)
            pool[s:e] = (raw[s:e] / kv_scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        del raw
    elif wl.kv_dtype == "int8":
        raw = torch.empty(n_pages, P, D_LATENT, dtype=torch.float32, device=dev)
        step = max(1, (1 << 27) // (P * D_LATENT))
        for s in range(0, n_pages, step):
            e = min(n_pages, s + step)
            raw[s:e] = torch.randn(e - s, P, D_LATENT, generator=g, device=dev)
        amax = float(raw.abs().max())
        kv_scale = amax / 127.0
        pool = torch.empty(n_pages, P, D_LATENT, dtype=torch.int8, device=dev)
        for s in range(0, n_pages, step):
            e = min(n_pages, s + step)
            pool[s:e] = torch.round(raw[s:e] / kv_scale).clamp_(-127.0, 127.0).to(torch.int8)
        del raw
    elif wl.kv_dtype == "int8page":
        # a scale per page: each page's N(0,1) latents times a spread factor 2^U(-2,0), so
        # that pages differ in range (up to 4x) while values keep the other pools' size,
        # encoded as round(x / s_page) with s_page = its amax / 127
        raw = torch.empty(n_pages, P, D_LATENT, dtype=torch.float32, device=dev)
        step = max(1, (1 << 27) // (P * D_LATENT))
        spread = torch.pow(2.0, torch.rand(n_pages, generator=g, device=dev) * 2.0 - 2.0)
        for s in range(0, n_pages, step):
            e = min(n_pages, s + step)
            raw[s:e] = torch.randn(e - s, P, D_LATENT, generator=g, device=dev) * spread[s:e, None, None]
        page_scales = (raw.abs().amax(dim=(1, 2)) / 127.0).clamp_(min=1e-30)
        pool = torch.empty(n_pages, P, D_LATENT, dtype=torch.int8, device=dev)
        for s in range(0, n_pages, step):
            e = min(n_pages, s + step)
            pool[s:e] = torch.round(raw[s:e] / page_scales[s:e, None, None]).clamp_(-127.0, 127.0).to(torch.int8)
        kv_scale = float(page_scales.max())
        del raw
    else:
        raise ValueError(wl.kv_dtype)
    if wl.peaked:
        _plant_near_duplicates(q, pool, page_table, wl, g, kv_scale,
                               page_scales if wl.kv_dtype == "int8page" else None)
    seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
    return DecodeInputs(q.to(torch.bfloat16), pool, page_table, seq_lens, kv_scale,
                        1.0 / math.sqrt(D_QK_PREFILL), wl,
                        page_scales if wl.kv_dtype == "int8page" else None)


def _plant_near_duplicates(q, pool, page_table, wl, g, kv_scale, page_scales=None):
    """Overwrite a few random key rows of each request with a scaled copy of one of its
    query directions plus noise, so that a handful of keys dominate the softmax.  (int8
    rows are encoded with their page's scale when the pool has one per page.)"""
    dev = q.device
    B, T, H, P = wl.batch, wl.q_len, wl.heads, wl.page_size
    for b in range(B):
        L = wl.seq_lens[b]
        n_plant = min(4, L)
        pos = torch.randint(0, L, (n_plant,), generator=g, device=dev)
        heads = torch.randint(0, H, (n_plant,), generator=g, device=dev)
        for i in range(n_plant):
            j = int(pos[i])
            h = int(heads[i])
            direction = q[b, T - 1, h].float()
            row = direction / direction.norm() * 4.0
            row = row + 0.05 * torch.randn(D_LATENT, generator=g, device=dev)
            page = int(page_table[b, j // P])
            if pool.dtype == torch.uint8:
                pool[page, j % P] = (row / kv_scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            elif pool.dtype == torch.int8:
                sc = float(page_scales[page]) if page_scales is not None else kv_scale
                pool[page, j % P] = torch.round(row / sc).clamp(-127.0, 127.0).to(torch.int8)
            else:
                pool[page, j % P] = row.to(torch.bfloat16)


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    cu_seqlens_q: torch.Tensor
    cu_seqlens_kv: torch.Tensor
    prefix_lens: torch.Tensor
    max_seqlen_q: int
    scale: float
    wl: PrefillWorkload = field(repr=False, default=None)


def make_prefill_inputs(wl: PrefillWorkload, device="cpu") -> PrefillInputs:
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    H = wl.heads
    n_q = sum(wl.new_lens)
    n_kv = sum(p + n for p, n in zip(wl.prefix_lens, wl.new_lens))
    q = torch.randn(n_q, H, D_QK_PREFILL, generator=g, device=dev).to(torch.bfloat16)
    k = torch.empty(n_kv, H, D_QK_PREFILL, dtype=torch.bfloat16, device=dev)
    v = torch.empty(n_kv, H, D_V_PREFILL, dtype=torch.bfloat16, device=dev)
    step = 1 << 16
    for s in range(0, n_kv, step):
        e = min(n_kv, s + step)
        k[s:e] = torch.randn(e - s, H, D_QK_PREFILL, generator=g, device=dev).to(torch.bfloat16)
        v[s:e] = torch.randn(e - s, H, D_V_PREFILL, generator=g, device=dev).to(torch.bfloat16)
    cq = [0]
    ck = [0]
    for p, n in zip(wl.prefix_lens, wl.new_lens):
        cq.append(cq[-1] + n)
        ck.append(ck[-1] + p + n)
    return PrefillInputs(q, k, v,
                         torch.tensor(cq, dtype=torch.int32, device=dev),
                         torch.tensor(ck, dtype=torch.int32, device=dev),
                         torch.tensor(wl.prefix_lens, dtype=torch.int32, device=dev),
                         max(wl.new_lens) if wl.new_lens else 0,
                         1.0 / math.sqrt(D_QK_PREFILL), wl)


@dataclass
class PagedKV:
    k_pages: torch.Tensor      # [num_pages, page_size, H, 192] bf16
    v_pages: torch.Tensor      # [num_pages, page_size, H, 128] bf16
    page_table: torch.Tensor   # [B, max_pages] int32
    kv_lens: torch.Tensor      # [B] int32: prefix + new tokens


def page_prefill_kv(inp: PrefillInputs, page_size: int, seed: int, extra_pages: int = 0) -> PagedKV:
    """Lay a prefill batch's contiguous per-request K/V rows out in a paged cache (layout
    only): request b's p_b + n_b rows fill ceil((p_b + n_b) / page_size) pages taken from
    one shared pool in a random permutation; the rest of each request's last page and
    ``extra_pages`` unused pages hold random values."""
    dev = inp.k.device
    g = torch.Generator(device=dev).manual_seed(seed)
    H = inp.k.shape[1]
    P = page_size
    cu = [int(x) for x in inp.cu_seqlens_kv.cpu()]
    lens = [cu[b + 1] - cu[b] for b in range(len(cu) - 1)]
    pages_per = [(L + P - 1) // P for L in lens]
    n_pages = sum(pages_per) + extra_pages
    mp = max(1, max(pages_per))
    k_pages = torch.randn(n_pages, P, H, D_QK_PREFILL, generator=g, device=dev).to(torch.bfloat16)
    v_pages = torch.randn(n_pages, P, H, D_V_PREFILL, generator=g, device=dev).to(torch.bfloat16)
    perm = torch.randperm(n_pages, generator=g, device=dev).to(torch.int32)
    page_table = torch.zeros(len(lens), mp, dtype=torch.int32, device=dev)
    kf = k_pages.view(n_pages * P, H, D_QK_PREFILL)
    vf = v_pages.view(n_pages * P, H, D_V_PREFILL)
    off = 0
    for b, (L, n) in enumerate(zip(lens, pages_per)):
        page_table[b, :n] = perm[off:off + n]
        off += n
        if L == 0:
            continue
        j = torch.arange(L, device=dev)
        dst = page_table[b, j // P].long() * P + j % P
        kf[dst] = inp.k[cu[b]:cu[b + 1]]
        vf[dst] = inp.v[cu[b]:cu[b + 1]]
    return PagedKV(k_pages, v_pages, page_table, torch.tensor(lens, dtype=torch.int32, device=dev))
