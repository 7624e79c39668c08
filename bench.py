"""Benchmark of the MLA hot path on GB300 (one JSON line on rank 0).

Headline workload: absorbed MLA speculative decode, batch 16, q_len 2, 16 heads, per-request
cached lengths drawn uniformly from [8192, 131072] (seeded), 64-token pages shuffled in a
shared pool, bf16 (synthetic, seeded): the largest decode configuration on one GPU, 1.28 GB
of latent KV, which exceeds L2, so every step streams its KV from HBM.  One step = one
mla_decode call (plan cached; split-KV partial kernel + LSE combine kernel).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --profile-case <workload>     (three calls, for a profiler capture;
                                                   paged_p64:<prefill workload> for the paged prefill)

Timing: `value` = KV bytes / time of one CUDA graph holding the K steps (no event nodes
inside); the roofline's kernel time = one pair of CUDA events around a second graph of
back-to-back launches of the split-KV partial kernel alone (mla_decode_partial); `e2e` =
wall clock of K end-to-end steps (one packed H2D copy of q / page table / lengths, the
decode call, one packed D2H copy of out / lse, copies on their own streams) replayed from
one graph.  The extra lines (the other decode workloads, the absorbed prefill over a paged
prefix, the varlen prefill over a paged cache and over contiguous K/V) are graph-timed the
same way and printed last, compactly.

N > 1 runs under torchrun: every rank runs an independent replica (the path has no
exchange step); value = all ranks' KV bytes / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_attention_paged_gb300.inputs import decode_workloads, make_decode_inputs  # noqa: E402

METRIC = "MLA decode KV-read GB/s & µs/call vs 8 TB/s; varlen prefill TFLOP/s"
WORKLOAD = "decode_b16_q2_h16_ragged"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def decode_bytes(wl):
    """Algorithmic bytes of one decode call: each request's latent rows once, its page-table
    entries, and the query / output / lse rows."""
    e = 1 if wl.kv_dtype in ("e4m3", "int8", "int8page") else 2
    kv = sum(L * 576 * e for L in wl.seq_lens)
    # page-table entries (and, for a pool with a scale per page, the pages' fp32 scales)
    per_page = 8 if wl.kv_dtype == "int8page" else 4
    pt = sum(((L + wl.page_size - 1) // wl.page_size) * per_page for L in wl.seq_lens)
    io = wl.batch * wl.q_len * wl.heads * (576 * 2 + 512 * 2 + 4)
    return kv, kv + pt + io


def decode_flops(wl):
    """2 * H * (576 + 512) * sum over query tokens of the keys each one sees (token t of a
    request of L keys sees keys 0 .. L - T + t)."""
    T = wl.q_len
    keys = sum(T * (L - T) + T * (T + 1) // 2 for L in wl.seq_lens)
    return 2 * wl.heads * (576 + 512) * keys


def prefill_flops(wl):
    """2 * H * (192 + 128) * sum over new tokens of the keys each one sees."""
    keys = sum(n * p + n * (n + 1) // 2 for p, n in zip(wl.prefix_lens, wl.new_lens))
    return 2 * wl.heads * (192 + 128) * keys


def graph_ms_per_call(fn, n, stream):
    """Capture fn(0..n-1) into one CUDA graph, replay it once to warm up, then time one
    replay between two CUDA events on `stream`; returns milliseconds per call.  (Events
    between kernels inside a graph were measured to add ~6 us each on this part, so a
    kernel's duration is taken over n back-to-back launches instead.)"""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            fn(i)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        a.record(stream)
        g.replay()
        b.record(stream)
    stream.synchronize()
    ms = a.elapsed_time(b) / n
    del g
    return ms


# Workloads whose decode sits above the tensor ridge (flops per KV byte): their fraction is
# taken against the bf16 tensor peak, the others against HBM bandwidth.
TENSOR_BOUND = ("decode_b16_q2_h128_ragged", "decode_b4_q512_h16_l32k")
# The extra lines, in print order: the last ones are the configurations the targets are
# quoted on (batch 16 / 64K prefix, and the varlen prefill), so they end the JSON line.
EXTRA_DECODE = ["decode_b4_q4_h16_l32k", "decode_b1_q1_h16_l1024", "decode_b16_q2_h128_ragged",
                "decode_b4_q512_h16_l32k", "decode_int8_b16_q4_h16_l64k", "decode_int8page_b16_q4_h16_l64k",
                "decode_fp8_b8_q4_h16_l64k", "decode_fp8_b16_q2_h16_ragged",
                "decode_bf16_b16_q4_h16_l64k", "decode_fp8_b16_q4_h16_l64k"]


def decode_sets(name, dev, rank=0):
    """Input sets of one decode workload: enough independent sets that their KV exceeds 2.5x
    L2 (rotated between calls so that every call reads its KV from HBM), or one set when the
    workload alone is larger than that."""
    wl = decode_workloads()[name]
    kv_bytes, _ = decode_bytes(wl)
    n_sets = 1 if kv_bytes >= 2.5 * L2_BYTES else max(2, math.ceil(2.5 * L2_BYTES / kv_bytes) + 1)
    sets = []
    for i in range(n_sets):
        w = decode_workloads()[name]
        w.seed = replica_seed(wl.seed, i, rank)
        sets.append(make_decode_inputs(w, dev))
    return wl, sets


def measure_decode_extra(mla, name, dev, steps=200):
    """Secondary decode line: device time per call (graph of back-to-back calls) and the
    partial kernel's own rate (graph of back-to-back partial launches), as a fraction of the
    binding roofline."""
    wl, sets = decode_sets(name, dev)
    n_sets = len(sets)
    kv_bytes, alg_bytes = decode_bytes(wl)
    kvd = {"e4m3": mla.MLA_KV_E4M3, "int8": mla.MLA_KV_INT8,
           "int8page": mla.MLA_KV_INT8_PAGE}.get(wl.kv_dtype, mla.MLA_KV_BF16)
    plan = mla.decode_plan(wl.seq_lens, wl.q_len, wl.heads, wl.page_size, sets[0].page_table.shape[1],
                           sets[0].kv_pool.shape[0], kvd)
    ws_buf = mla.workspace_for(plan, dev)
    out = torch.empty(wl.batch, wl.q_len, wl.heads, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(wl.batch, wl.q_len, wl.heads, dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(device=dev)

    def call(i):
        s = sets[i % n_sets]
        if s.page_scales is not None:
            mla.decode_int8_paged(plan, s.q, s.kv_pool, s.page_scales, s.page_table, s.seq_lens, s.scale,
                                  s.kv_scale, out=out, lse=lse, workspace=ws_buf, stream=st)
        else:
            mla.decode(plan, s.q, s.kv_pool, s.page_table, s.seq_lens, s.scale, s.kv_scale, out=out, lse=lse,
                       workspace=ws_buf, stream=st)

    def partial(i):
        # (a pool with a scale per page has no partial-only entry point: its line times whole calls)
        s = sets[i % n_sets]
        if s.page_scales is not None:
            call(i)
            return
        mla.decode_partial(plan, s.q, s.kv_pool, s.page_table, s.seq_lens, s.scale, s.kv_scale, out=out, lse=lse,
                           workspace=ws_buf, stream=st)

    with torch.cuda.stream(st):
        for i in range(5):
            call(i)
    st.synchronize()
    call_ms = graph_ms_per_call(call, steps, st)
    part_ms = graph_ms_per_call(partial, steps, st)
    assert mla.get_status(st) == mla.MLA_OK
    peak = _peaks()
    del sets
    rec = {"us": round(call_ms * 1e3, 2), "kernel_us": round(part_ms * 1e3, 2), "splits": plan.max_splits}
    if name in TENSOR_BOUND:
        tf = decode_flops(wl) / (part_ms / 1e3) / 1e12
        rec.update(bound="tensor", tflops=round(tf, 1), frac=round(tf / peak["bf16_tflops"], 3))
    else:
        gbs = alg_bytes / (part_ms / 1e3) / 1e9
        rec.update(bound="hbm", gbs=round(gbs, 1), frac=round(gbs / peak["hbm_gbs"], 3))
    return rec


def measure_prefill(mla, dev, steps=10, page_size=None):
    """The varlen prefill line (5 requests, prefix 20K-100K, 256-2048 new tokens, 16 heads):
    contiguous K/V, or (page_size given) the same K/V laid out in a shuffled paged cache and
    read through the page table."""
    from mla_attention_paged_gb300.inputs import make_prefill_inputs, page_prefill_kv, prefill_workloads
    wl = prefill_workloads()["prefill_b5_h16_prefix"]
    inp = make_prefill_inputs(wl, dev)
    out = torch.empty(inp.q.shape[0], wl.heads, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(inp.q.shape[0], wl.heads, dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(device=dev)
    if page_size:
        pk = page_prefill_kv(inp, page_size, seed=wl.seed + 1)
        inp.k = inp.v = None  # only the paged copy is read

        def call(i=0):
            mla.prefill_paged(inp.q, pk.k_pages, pk.v_pages, pk.page_table, inp.cu_seqlens_q, pk.kv_lens,
                              inp.max_seqlen_q, inp.scale, out=out, lse=lse, stream=st)
    else:
        def call(i=0):
            mla.prefill_varlen(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_kv, inp.prefix_lens,
                               inp.max_seqlen_q, inp.scale, out=out, lse=lse, stream=st)

    with torch.cuda.stream(st):
        for _ in range(2):
            call()
    st.synchronize()
    ms = graph_ms_per_call(call, steps, st)
    assert mla.get_status(st) == mla.MLA_OK
    tf = prefill_flops(wl) / (ms / 1e3) / 1e12
    peak = _peaks()
    return {"us": round(ms * 1e3, 1), "bound": "tensor", "tflops": round(tf, 1),
            "frac": round(tf / peak["bf16_tflops"], 3)}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def replica_seed(base_seed, set_index, rank):
    """Seed of input set `set_index` on replica `rank`: every rank and set draws its own data."""
    return base_seed + 97 * set_index + 100003 * rank


TRAFFIC_SOURCES = ("mla_decode_narrow_sm103a.cu", "sm103a_ptx.cuh")  # the headline's partial kernel


def _sources_sha256(names):
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "mla_attention_paged_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic_record(workload):
    """DRAM bytes per launch of the partial kernel on `workload` from the committed ncu
    summary, if it was taken on the current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "decode_partial_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_sha256") != _sources_sha256(TRAFFIC_SOURCES) or rec.get("workload") != workload:
            return None
        return rec
    except Exception:
        return None


def _oracle_rows_for(inp_cpu, rows_total, seconds, seed):
    """Run the oracle on random row subsets of one decode workload until about `seconds` of
    oracle time are spent; returns (rows done, seconds)."""
    import numpy as np

    import oracle
    rng = np.random.default_rng(seed)
    n = 1
    done_rows, elapsed = 0, 0.0
    while elapsed < seconds:
        rows = rng.choice(rows_total, size=min(n, rows_total), replace=False)
        t0 = time.perf_counter()
        oracle.mla_decode(inp_cpu.q, inp_cpu.kv_pool, inp_cpu.page_table, inp_cpu.seq_lens, inp_cpu.scale,
                          kv_scale=inp_cpu.kv_scale, rows=rows)
        elapsed += time.perf_counter() - t0
        done_rows += len(rows)
        per_row = elapsed / done_rows
        n = int(max(1, min(rows_total, (seconds - elapsed) / max(per_row, 1e-9))))
    return done_rows, elapsed


def cpu_baseline(wl, inp_cpu, seconds=10.0, single_seconds=4.0):
    """The fp64 oracle, as it stands, on a bounded sample of this workload's rows: random
    row subsets until about `seconds` of oracle time on every host thread, then about
    `single_seconds` on one thread.  Each figure is the workload's KV bytes over the time a
    whole pass would take at the sampled rate (rows of one workload cost about the same)."""
    import oracle
    oracle.build()
    rows_total = wl.batch * wl.q_len * wl.heads
    kv_bytes, _ = decode_bytes(wl)
    threads = oracle.num_threads()
    done, el = _oracle_rows_for(inp_cpu, rows_total, seconds, 0)
    oracle.set_num_threads(1)
    try:
        done1, el1 = _oracle_rows_for(inp_cpu, rows_total, single_seconds, 1)
    finally:
        oracle.set_num_threads(threads)
    return {"value": kv_bytes / (el * rows_total / done) / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} of the {rows_total} (request, draft, head) rows of {wl.name}, fp64, {el:.1f} s; "
                      f"pass time scaled by rows",
            "single_thread": {"value": kv_bytes / (el1 * rows_total / done1) / 1e9, "unit": "GB/s",
                              "rows": done1, "seconds": round(el1, 2)}}


def run_reference(args, ws, rank):
    """Reference arm: the CPU fp64 oracle, as it stands, on the host cores.  Each step is a
    bounded sample of the headline workload's rows (sized so the whole run takes about a
    minute); ms_per_step is the sample's measured time and value the workload's KV bytes
    over the time a whole pass would take at that rate."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    oracle.build()
    wl = decode_workloads()[WORKLOAD]
    inp = make_decode_inputs(wl, "cpu")
    rows_total = wl.batch * wl.q_len * wl.heads
    rng = np.random.default_rng(1)
    threads = oracle.num_threads()
    t0 = time.perf_counter()
    oracle.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                      rows=rng.choice(rows_total, min(threads, rows_total), replace=False))
    per_row = max((time.perf_counter() - t0) / threads, 1e-5)
    budget = 60.0 / max(1, args.steps + args.warmup)
    rows_per_step = int(max(1, min(rows_total, budget / per_row)))
    for _ in range(args.warmup):
        oracle.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                          rows=rng.choice(rows_total, rows_per_step, replace=False))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.mla_decode(inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale,
                          rows=rng.choice(rows_total, rows_per_step, replace=False))
    el = time.perf_counter() - t0
    kv_bytes, _ = decode_bytes(wl)
    step_s = el / args.steps
    val = kv_bytes * rows_per_step / rows_total / step_s / 1e9
    sample = (f"each step: {rows_per_step} of the {rows_total} (request, draft, head) rows of {WORKLOAD}, fp64; "
              f"value = KV bytes x sampled fraction / step time")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": wl.batch, "q_len": wl.q_len, "heads": wl.heads,
                       "kv_len": "U[8192,131072]", "page_size": wl.page_size, "kv_dtype": wl.kv_dtype},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile_case(name):
    """Three calls of one workload, for a profiler to capture (no timing, no JSON line)."""
    from mla_attention_paged_gb300 import build
    from mla_attention_paged_gb300.inputs import make_prefill_inputs, prefill_workloads
    build.build()
    from mla_attention_paged_gb300 import mla
    if name.startswith("paged_p64:") and name.split(":", 1)[1] in prefill_workloads():
        from mla_attention_paged_gb300.inputs import page_prefill_kv
        wl = prefill_workloads()[name.split(":", 1)[1]]
        inp = make_prefill_inputs(wl, "cuda")
        pk = page_prefill_kv(inp, 64, seed=wl.seed + 1)
        for _ in range(3):
            mla.prefill_paged(inp.q, pk.k_pages, pk.v_pages, pk.page_table, inp.cu_seqlens_q, pk.kv_lens,
                              inp.max_seqlen_q, inp.scale)
    elif name in prefill_workloads():
        inp = make_prefill_inputs(prefill_workloads()[name], "cuda")
        for _ in range(3):
            mla.prefill_varlen(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_kv, inp.prefix_lens,
                               inp.max_seqlen_q, inp.scale)
    else:
        wl = decode_workloads()[name]
        inp = make_decode_inputs(wl, "cuda")
        kvd = {"e4m3": mla.MLA_KV_E4M3, "int8": mla.MLA_KV_INT8,
               "int8page": mla.MLA_KV_INT8_PAGE}.get(wl.kv_dtype, mla.MLA_KV_BF16)
        plan = mla.decode_plan(wl.seq_lens, wl.q_len, wl.heads, wl.page_size, inp.page_table.shape[1],
                               inp.kv_pool.shape[0], kvd)
        for _ in range(3):
            if inp.page_scales is not None:
                mla.decode_int8_paged(plan, inp.q, inp.kv_pool, inp.page_scales, inp.page_table, inp.seq_lens,
                                      inp.scale, inp.kv_scale)
            else:
                mla.decode(plan, inp.q, inp.kv_pool, inp.page_table, inp.seq_lens, inp.scale, inp.kv_scale)
    torch.cuda.synchronize()
    status = mla.get_status()
    if status != mla.MLA_OK:
        raise RuntimeError(f"device status {mla.status_string(status)}")
    print(f"profile case {name}: ok", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary decode / prefill lines")
    ap.add_argument("--profile-case", default=None,
                    help="run three calls of one named workload (a profiler target) and exit without timing")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    args.warmup = max(args.warmup, 3)
    ws, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    from mla_attention_paged_gb300 import build
    if rank == 0 or ws == 1:
        build.build()
    _barrier(ws)
    from mla_attention_paged_gb300 import mla

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl, sets = decode_sets(WORKLOAD, dev, rank)
    n_sets = len(sets)
    kv_bytes, alg_bytes = decode_bytes(wl)
    s0 = sets[0]
    plan = mla.decode_plan(wl.seq_lens, wl.q_len, wl.heads, wl.page_size, s0.page_table.shape[1],
                           s0.kv_pool.shape[0], mla.MLA_KV_BF16)
    ws_buf = mla.workspace_for(plan, dev)
    outs = [torch.empty(wl.batch, wl.q_len, wl.heads, 512, dtype=torch.bfloat16, device=dev) for _ in sets]
    lses = [torch.empty(wl.batch, wl.q_len, wl.heads, dtype=torch.float32, device=dev) for _ in sets]
    stream = torch.cuda.Stream(device=dev)

    def step(i, st):
        s = sets[i % n_sets]
        mla.decode(plan, s.q, s.kv_pool, s.page_table, s.seq_lens, s.scale, 1.0, out=outs[i % n_sets],
                   lse=lses[i % n_sets], workspace=ws_buf, stream=st)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, stream)
    stream.synchronize()
    assert mla.get_status(stream) == mla.MLA_OK

    # Timed region: one CUDA graph holding exactly K steps (no event nodes inside it: an
    # event recorded between two kernels of a graph was measured to add ~6 us per call).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(args.steps):
            step(i, stream)
    stream.synchronize()

    # Duration of the dominant kernel: the split-KV partial kernel alone, launched back to
    # back (same inputs) in a second graph, timed between one pair of CUDA events on the
    # launch stream, right after the timed replay and under the same clock sampling.
    n_k = max(20, min(args.steps, 400))

    def partial_step(i):
        s = sets[i % n_sets]
        mla.decode_partial(plan, s.q, s.kv_pool, s.page_table, s.seq_lens, s.scale, 1.0, out=outs[i % n_sets],
                           lse=lses[i % n_sets], workspace=ws_buf, stream=stream)

    kgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(kgraph, stream=stream):
        for i in range(n_k):
            partial_step(i)
    stream.synchronize()
    # pre-roll under the clock sampler, then the timed replay
    sampler = ClockSampler(local)
    t_end = time.perf_counter() + 1.0
    with torch.cuda.stream(stream):
        while time.perf_counter() < t_end:
            graph.replay()
            stream.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kstart, kstop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(ws)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        start.record(stream)
        graph.replay()
        stop.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    _barrier(ws)
    with torch.cuda.stream(stream):
        kgraph.replay()  # warm
        kstart.record(stream)
        kgraph.replay()
        kstop.record(stream)
    stream.synchronize()
    clocks = sampler.stop()
    status = mla.get_status(stream)
    if status != mla.MLA_OK:
        raise RuntimeError(f"device status {mla.status_string(status)}")
    ms = start.elapsed_time(stop)
    ms_max = _max_over_ranks(ms, ws, dev)
    total_bytes = _sum_over_ranks(kv_bytes * args.steps, ws, dev)
    value = total_bytes / (ms_max / 1e3) / 1e9
    part_ms = kstart.elapsed_time(kstop) / n_k
    peaks = _peaks()
    achieved = alg_bytes / (part_ms / 1e3) / 1e9
    traffic = _traffic_record(WORKLOAD)

    # End to end through the public API: each step copies that step's q, page table and
    # lengths from pinned host memory to the device (packed in one buffer: one copy), calls
    # mla_decode, and copies out + lse back to pinned host memory (one packed buffer, one
    # copy).  The latent cache is device-resident.  Two I/O slots (or one per input set)
    # alternate, so that step i+1's inputs and step i-1's results move while step i computes.
    def _packed(tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    def _view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    n_io = max(2, n_sets)
    in_offs, in_bytes = _packed([sets[0].q, sets[0].page_table, sets[0].seq_lens])
    out_offs, out_bytes = _packed([outs[0], lses[0]])
    host_in, dev_in, host_out, dev_out = [], [], [], []
    for k in range(n_io):
        s = sets[k % n_sets]
        hb = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        for t, off in zip((s.q, s.page_table, s.seq_lens), in_offs):
            _view(hb, off, t).copy_(t.cpu())
        host_in.append(hb)
        db = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        dev_in.append((db, _view(db, in_offs[0], s.q), _view(db, in_offs[1], s.page_table),
                       _view(db, in_offs[2], s.seq_lens)))
        ob = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        dev_out.append((ob, _view(ob, out_offs[0], outs[0]), _view(ob, out_offs[1], lses[0])))
        host_out.append(torch.empty(out_bytes, dtype=torch.uint8).pin_memory())
    h2d = sum(t.numel() * t.element_size() for t in (sets[0].q, sets[0].page_table, sets[0].seq_lens))
    d2h = sum(t.numel() * t.element_size() for t in (outs[0], lses[0]))
    e2e_steps = min(args.steps, 500)

    s_h2d = torch.cuda.Stream(device=dev)
    s_d2h = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(n_io)]
    ev_done = [torch.cuda.Event() for _ in range(n_io)]
    ev_read = [torch.cuda.Event() for _ in range(n_io)]

    def e2e_step(i):
        k = i % n_io
        s = sets[k % n_sets]
        db, q_d, pt_d, sl_d = dev_in[k]
        ob, out_d, lse_d = dev_out[k]
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(ev_done[k])       # the last step on this slot has consumed its inputs
            db.copy_(host_in[k], non_blocking=True)
            ev_in[k].record(s_h2d)
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_read[k])          # its results have been copied out
        mla.decode(plan, q_d, s.kv_pool, pt_d, sl_d, s.scale, 1.0, out=out_d, lse=lse_d, workspace=ws_buf,
                   stream=stream)
        ev_done[k].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_done[k])
            host_out[k].copy_(ob, non_blocking=True)
            ev_read[k].record(s_d2h)

    def e2e_steps_in(graph_, n):
        # one CUDA graph holding n end-to-end steps: the copy streams fork from the capture
        # stream at the start and join it at the end
        ev_start, ev_h, ev_d = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        with torch.cuda.graph(graph_, stream=stream):
            ev_start.record(stream)
            s_h2d.wait_event(ev_start)
            s_d2h.wait_event(ev_start)
            for k in range(n_io):  # nothing pending on any slot at the start
                ev_done[k].record(stream)
                ev_read[k].record(s_d2h)
            for i in range(n):
                e2e_step(i)
            ev_h.record(s_h2d)
            ev_d.record(s_d2h)
            stream.wait_event(ev_h)
            stream.wait_event(ev_d)

    e2e_graph = torch.cuda.CUDAGraph()
    e2e_steps_in(e2e_graph, e2e_steps)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e2e_graph.replay()  # warm
    torch.cuda.synchronize(dev)
    _barrier(ws)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e2e_graph.replay()
    enqueue_s = time.perf_counter() - t0
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    del e2e_graph
    e2e_s = _max_over_ranks(e2e_s, ws, dev)
    e2e_val = _sum_over_ranks(kv_bytes * e2e_steps, ws, dev) / e2e_s / 1e9

    launches_per_step = 1 + (1 if plan.max_splits > 1 else 0)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "us_per_call": ms_max / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)/sqrt(576) latents, shuffled 64-token pages)",
        "config": {"workload": WORKLOAD, "batch": wl.batch, "q_len": wl.q_len, "heads": wl.heads,
                   "kv_len": "U[8192,131072]", "page_size": wl.page_size, "kv_dtype": wl.kv_dtype,
                   "parallelism": f"replicas x{ws}",
                   "l2": (f"inputs rotated over {n_sets} sets" if n_sets > 1 else
                          f"inputs larger than L2 ({kv_bytes / 2**20:.0f} MiB KV)"),
                   "splits": plan.max_splits},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": (traffic["dram_bytes_per_launch"] if traffic else None),
                     "kernel": "decode_partial_narrow_kernel", "kernel_us": part_ms * 1e3,
                     "alg_bytes_per_launch": alg_bytes, "peak_source": peaks["source"] + " copy bandwidth"},
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "us_per_call": e2e_s / e2e_steps * 1e6,
                "host_enqueue_us_per_call": enqueue_s / e2e_steps * 1e6},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "timing": "value: one CUDA graph of K steps between CUDA events on the launch stream; kernel: "
                  f"{n_k} back-to-back partial-kernel launches in one graph; e2e: wall clock of one graph of "
                  "steps with packed H2D/D2H copies on copy streams",
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        inp_cpu = make_decode_inputs(decode_workloads()[WORKLOAD], "cpu")
        line["cpu_baseline"] = cpu_baseline(wl, inp_cpu)
        del inp_cpu
    if not args.no_extra:
        # the other hot-path rows, each measured on its own (not part of `value`): per call
        # (us), partial kernel alone (kernel_us) and its fraction of the binding roofline
        del sets, host_in, dev_in, host_out, dev_out, graph, kgraph
        torch.cuda.empty_cache()
        extra = {}
        for name in EXTRA_DECODE:
            extra[name] = measure_decode_extra(mla, name, dev)
            torch.cuda.empty_cache()
        extra["prefill_paged_p64_b5_h16_prefix"] = measure_prefill(mla, dev, page_size=64)
        torch.cuda.empty_cache()
        extra["prefill_b5_h16_prefix"] = measure_prefill(mla, dev)
        line["extra"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
