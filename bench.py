#!/usr/bin/env python3
"""Benchmark one sparse MLA decode step on synthetic fp8_ds_mla inputs; prints ONE JSON line.

Metric: gathered KV tokens/s (valid (token, entry) rows attended per second) for one
decode step = index conversion + fused gather/dequant/tcgen05 attention + LSE combine,
all in libsmd's CUDA kernels.  Inputs are resident in HBM when the timed region starts;
L2 is flushed (a 512 MiB write) between timed steps, outside the per-step CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl ours|reference]

--config picks the headline workload among the five decode shapes (0 tiny, 1 single
request, 2 mid batch, 3 large batch [default: the largest single-GPU step], 4 long
context); --extra-configs lists the others measured in the same run and reported under
``extra_workloads``.  Each step is one CUDA-graph replay of the smd_sparse_mla_decode call.  Under torchrun each rank runs its own
replica of the workload on its own GPU (weak scaling, no data-path collective); the
timed region is bracketed by barriers and the max time over ranks is reported.
``--impl reference`` times the float64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "gathered KV tokens/s and achieved HBM GB/s (fraction of roofline) per decode step"
UNIT = "tokens/s"
FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--extra-configs", default="2,4,1", help="other workloads measured in the same run")
    ap.add_argument("--extra-steps", type=int, default=300)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-oracle sample length")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bf16-steps", type=int, default=100,
                    help="steps of the headline step over a bf16 latent cache; 0 skips it")
    ap.add_argument("--indexer-steps", type=int, default=100,
                    help="steps of the indexer workloads (logits + top-k) measured in the same run; 0 skips them")
    ap.add_argument("--num-splits", type=int, default=None,
                    help="split request for the main workload (as num_splits of the C API; default: the workload's)")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def roofline(H: int, rows: int, seconds: float, peaks: dict, source: str, traffic=None) -> dict:
    """Roofline of the attention kernel: 584 gathered bytes and 4*512*H flops per valid row."""
    bytes_ = 584.0 * rows
    flops = 4.0 * 512 * H * rows
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    gbs = bytes_ / seconds / 1e9
    tflops = flops / seconds / 1e12
    if flops / bytes_ > ridge:
        r = {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["traffic"] = traffic
    r["peak_source"] = f"{source} (MEASURED_PEAKS.json burst)" if source == "measured" else "fallback"
    r["algorithmic_bytes_per_launch"] = bytes_
    r["algorithmic_flops_per_launch"] = flops
    r["hbm_gbs_achieved"] = gbs
    r["hbm_frac"] = gbs / peaks["hbm_gbs"]
    r["tensor_tflops_achieved"] = tflops
    r["tensor_frac"] = tflops / peaks["bf16_tflops"]
    return r


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i",
                 str(self.index), "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(config: int, rank: int) -> int:
    """Each replica draws its own inputs (same shapes, different values)."""
    from sparse_mla_decode_req_gb300 import synth
    return synth.SEED_BASE + config + 1000 * rank


def max_over_ranks(pg, seconds: float, device) -> float:
    """The slowest replica's time (the job finishes when the last rank does)."""
    if pg is None:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_rate(rows_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job throughput: every replica processes rows_per_step per step."""
    return rows_per_step * steps * world / seconds


def cpu_oracle_rate(inp, seconds: float, max_steps: int | None = None):
    """Time the float64 oracle on whole tokens of the workload (cycling) for ~`seconds`."""
    import numpy as np

    import oracle
    w = inp.workload
    q = oracle.decode_bf16(inp.q.cpu().contiguous().view(__import__("torch").int16).numpy().view(np.uint16))
    cache = inp.kv_cache.cpu().numpy()
    bt = inp.block_table.cpu().numpy()
    rid = inp.req_id.cpu().numpy()
    topk = inp.topk_idx.cpu().numpy()
    swa = inp.swa_idx.cpu().numpy()
    sink = inp.sink.cpu().double().numpy()
    valid = ((topk >= 0).sum(axis=1) + (swa >= 0).sum(axis=1)) if w.n_entries else np.zeros(w.num_tokens)
    rows = 0
    steps = 0
    t0 = time.perf_counter()
    t = 0
    while True:
        oracle.sparse_mla_decode(q, cache, bt, rid, topk, swa, sink, inp.scale, w.block_size, tokens=[t])
        rows += int(valid[t])
        steps += 1
        t = (t + 1) % w.num_tokens
        el = time.perf_counter() - t0
        if (max_steps is not None and steps >= max_steps) or (max_steps is None and el >= seconds):
            break
    el = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return rows / el, el, steps, rows, cores


def run_reference(args, world, rank):
    """The reference arm: the float64 CPU oracle, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return 0
    import torch

    from sparse_mla_decode_req_gb300 import synth
    w = synth.WORKLOADS[args.config]
    inp = synth.make_inputs(w, device="cpu")
    cpu_oracle_rate(inp, 0.0, max_steps=max(1, args.warmup))
    rate, el, steps, rows, cores = cpu_oracle_rate(inp, 0.0, max_steps=max(1, args.steps))
    sample = f"{steps} oracle steps of one token each (cycling over the {w.num_tokens} tokens), {rows} valid rows"
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    del torch
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    """The workload both arms run (the split count, an implementation choice of the GPU
    path, is reported beside it as `num_splits`)."""
    return {"workload": w.name, "description": w.description, "batch": w.num_tokens, "heads": w.num_heads,
            "topk": w.topk, "swa": w.swa, "context": [w.ctx_lo, w.ctx_hi], "block_size": w.block_size,
            "l2": "flushed between timed steps (512 MiB write)"}


# The roofline at the GB300 spec figures: max(gathered bytes / 8 TB/s, FLOPs / 2.25 PFLOP/s
# dense bf16) (the measured peaks are the `roofline` object's denominators).
SPEC_HBM_GBS = 8000.0
SPEC_BF16_TFLOPS = 2250.0


def step_bytes(inp, S: int) -> dict:
    """Bytes one decode step must move (algorithmic): the gathered 584-byte rows, q read, out
    written, lse written, the index lists, request ids and block table read.  The converted
    slots and split partials are the implementation's own traffic and are listed apart."""
    w = inp.workload
    T, H, N = w.num_tokens, w.num_heads, w.n_entries
    gathered = 584 * inp.n_valid
    qo = 2 * T * H * 512 * 2
    lse = T * H * 4
    idx = T * N * 4 + T * 4 + inp.block_table.numel() * 4
    impl = 2 * T * N * 4 + ((T * S * H * 512 * 4 + T * S * H * 4) * 2 if S > 1 else 0)
    return {"gathered": gathered, "full": gathered + qo + lse + idx, "q_and_out": qo, "lse": lse, "indices": idx,
            "implementation_scratch": impl}


def fractions(H: int, rows: int, nbytes: dict, seconds: float, peaks: dict) -> dict:
    """Roofline fractions of `seconds` for one step's work."""
    flops = 4.0 * 512 * H * rows
    t_spec = max(nbytes["gathered"] / (SPEC_HBM_GBS * 1e9), flops / (SPEC_BF16_TFLOPS * 1e12))
    t_meas = max(nbytes["gathered"] / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    t_full = nbytes["full"] / (peaks["hbm_gbs"] * 1e9)
    return {"spec_peak_frac": t_spec / seconds, "spec_roofline_us": t_spec * 1e6,
            "measured_peak_frac": t_meas / seconds, "full_bytes_frac": t_full / seconds,
            "full_bytes_floor_us": t_full * 1e6, "full_bytes_gbs": nbytes["full"] / seconds / 1e9}


def measure(api, lib, synth, torch, w, seed, dev, flush, K: int, W: int, KP: int, sampler=None, pg=None):
    """Times one workload: K CUDA-graph replays of the product call smd_sparse_mla_decode (L2
    flushed between them, events around each replay), then KP staged steps with events
    between the three kernels for the per-kernel breakdown and the attention roofline."""
    import ctypes

    inp = synth.make_inputs(w, seed=seed, device=dev)
    T, H, N = w.num_tokens, w.num_heads, w.n_entries
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    topk = inp.topk_idx if w.topk else None
    swa = inp.swa_idx if w.swa else None
    dims = api.make_dims(inp.q, inp.kv_cache, inp.block_table, inp.req_id, topk, swa, w.block_size)
    S = api.select_num_splits(dims, w.max_splits, sms)
    out = torch.empty(T, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = torch.zeros(api.workspace_size(dims, w.max_splits, sms), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def call():
        api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id, topk, swa, inp.sink, inp.scale,
                              out=out, lse=lse, num_splits=w.max_splits, workspace=ws, block_size=w.block_size,
                              stream=stream)

    with torch.cuda.stream(stream):
        call()  # per-device set-up outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            call()
        for _ in range(max(W, 3)):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        if sampler is not None:
            sampler.start()
            time.sleep(0.1)
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if pg is not None:
            pg.barrier()
        clocks = sampler.stop() if sampler is not None else None
    step_ms = [a.elapsed_time(b) for a, b in ev]
    status = api.read_status(ws)  # raises on a recorded timeout

    # staged pass: convert | attention | combine with events between them
    gidx = torch.empty(T, N, dtype=torch.int32, device=dev)
    o_part = torch.empty(T, S, H, 512, dtype=torch.float32, device=dev) if S > 1 else None
    lse_part = torch.empty(T, S, H, dtype=torch.float32, device=dev) if S > 1 else None
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    P = api._ptr
    sp = ctypes.c_void_p(stream.cuda_stream)
    conv_args = (ctypes.byref(dims), P(inp.block_table), P(inp.req_id), P(topk), P(swa), P(gidx), sp)
    attn_dims = api.attention_dims(T, H, N, inp.num_pages, w.block_size)
    attn_args = (ctypes.byref(attn_dims), None, P(inp.q), P(inp.kv_cache), P(gidx), None, P(inp.sink),
                 ctypes.c_float(inp.scale), int(w.max_splits), P(out), P(lse), P(o_part), P(lse_part), P(st), sp)
    comb_args = (T, S, H, P(o_part), P(lse_part), P(inp.sink), P(out), P(lse), sp)
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(KP)]
    with torch.cuda.stream(stream):
        for i in range(KP + 3):
            flush.zero_()
            e = evk[i - 3] if i >= 3 else None
            if e:
                e[0].record(stream)
            api._check(lib.smd_convert_req_index(*conv_args))
            if e:
                e[1].record(stream)
            api._check(lib.smd_sparse_mla_attention(*attn_args))
            if e:
                e[2].record(stream)
            if S > 1:
                api._check(lib.smd_lse_combine(*comb_args))
            if e:
                e[3].record(stream)
        torch.cuda.synchronize()
    assert int(st.item()) == 0, "a kernel's bounded wait gave up during the benchmark"
    return {"inp": inp, "S": S, "step_ms": step_ms, "wall": wall, "clocks": clocks, "status": status,
            "attn_ms": [e[1].elapsed_time(e[2]) for e in evk], "conv_ms": [e[0].elapsed_time(e[1]) for e in evk],
            "comb_ms": [e[2].elapsed_time(e[3]) for e in evk], "out": out, "stream": stream}


def measure_bf16_cache(api, torch, synth, w, seed, dev, flush, steps: int, peaks: dict, src: str) -> dict:
    """The same decode step over a bf16 latent cache (1024-byte rows, no dequantisation):
    `steps` CUDA-graph replays of the product call (L2 flushed between them) and `steps`
    attention-only launches over the converted slots, events around each.  Its roofline
    counts 1024 bytes per valid row; set beside the fp8 step it bounds what dequantising
    the fp8 rows costs."""
    inp = synth.make_inputs(w, seed=seed, device=dev)
    cache = synth.make_cache_bf16(inp.num_pages, w.block_size, seed * 4 + 9, dev)
    T, H, N = w.num_tokens, w.num_heads, w.n_entries
    topk = inp.topk_idx if w.topk else None
    swa = inp.swa_idx if w.swa else None
    out = torch.empty(T, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    dims = api.make_dims(inp.q, cache, inp.block_table, inp.req_id, topk, swa, w.block_size, api.CACHE_BF16)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ws = torch.zeros(api.workspace_size(dims, w.max_splits, sms), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def call():
        api.sparse_mla_decode(inp.q, cache, inp.block_table, inp.req_id, topk, swa, inp.sink, inp.scale, out=out,
                              lse=lse, num_splits=w.max_splits, workspace=ws, block_size=w.block_size, stream=stream,
                              cache_format=api.CACHE_BF16)

    gidx = api.convert_req_index(inp.block_table, inp.req_id, topk, swa, inp.num_pages, w.block_size)
    with torch.cuda.stream(stream):
        call()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        eva = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(3 + steps):
            flush.zero_()
            e = ev[i - 3] if i >= 3 else None
            if e:
                e[0].record(stream)
            graph.replay()
            if e:
                e[1].record(stream)
        for i in range(3 + steps):
            flush.zero_()
            e = eva[i - 3] if i >= 3 else None
            if e:
                e[0].record(stream)
            api.sparse_mla_attention(inp.q, cache, gidx, inp.sink, inp.scale, num_pages=inp.num_pages,
                                     num_splits=w.max_splits, block_size=w.block_size, stream=stream,
                                     cache_format=api.CACHE_BF16)
            if e:
                e[1].record(stream)
        torch.cuda.synchronize()
    api.read_status(ws)
    step_us = [a.elapsed_time(b) * 1e3 for a, b in ev]
    attn_us = [a.elapsed_time(b) * 1e3 for a, b in eva]
    rows = inp.n_valid
    attn_s = statistics.mean(attn_us) / 1e6
    gbs = rows * 1024.0 / attn_s / 1e9
    del inp, cache, gidx
    return {
        "workload": w.name, "cache_format": "bf16 (1024-byte rows)", "steps": steps,
        "step_us_median": statistics.median(step_us), "attention_us_mean": statistics.mean(attn_us),
        "rows_per_s": rows / (statistics.median(step_us) / 1e6),
        "roofline_attention": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": rows * 1024.0,
                               "peak_source": f"{src} (MEASURED_PEAKS.json burst)" if src == "measured" else "fallback"},
        "timing": "CUDA-graph replays of smd_sparse_mla_decode and attention-only launches, events around each, "
                  "512 MiB L2 flush before each",
    }


def measure_indexer(api, torch, si, wi, dev, flush, steps: int, peaks: dict, src: str) -> dict:
    """The indexer step on one of its workloads: `steps` pairs of launches (fp8 paged MQA
    logits, then top-k), L2 flushed before each pair, CUDA events around each launch on the
    launching stream.  The logits kernel's roofline: per position its 128 key bytes and
    float32 scale from HBM, plus the query heads, weights and the float32 logits row, at
    the measured copy bandwidth (2 * 128 * H flops per position sit far below the fp8
    tensor ridge)."""
    inp = si.make_indexer_inputs(wi, device=dev)
    T, H, D, K = wi.num_tokens, wi.num_heads, wi.head_dim, wi.topk
    L = inp.max_len
    logits = torch.empty(T, L, dtype=torch.float32, device=dev)
    topk = torch.empty(T, K, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    # the key gather of every cached position of every request as one ragged batch
    lens = torch.tensor(inp.ctx, dtype=torch.int64)
    cu = torch.zeros(T + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    n_all = int(cu[-1])
    tts = torch.repeat_interleave(torch.arange(T, dtype=torch.int32), lens).to(dev)
    cu = cu.to(dev)
    k_all = torch.empty(n_all, D, dtype=torch.uint8, device=dev)
    s_all = torch.empty(n_all, dtype=torch.float32, device=dev)
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(3 + steps):
            flush.zero_()
            e = gev[i - 3] if i >= 3 else None
            if e:
                e[0].record(stream)
            api.indexer_gather_k(inp.cache, inp.block_table, cu, tts, T, wi.block_size, D, 0, k_out=k_all,
                                 scale_out=s_all, stream=stream)
            if e:
                e[1].record(stream)
        torch.cuda.synchronize()
    g_us = [a.elapsed_time(b) * 1e3 for a, b in gev]
    g_bytes = 2 * n_all * (D + 4) + n_all * 4 * 2  # key bytes and scales read and written, cu/seq ids
    del k_all, s_all, tts
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(3 + steps):
            flush.zero_()
            e = ev[i - 3] if i >= 3 else None
            if e:
                e[0].record(stream)
            api.indexer_mqa_logits(inp.q, inp.weights, inp.cache, inp.block_table, inp.req_id, inp.ctx_lens, L,
                                   block_size=wi.block_size, logits=logits, stream=stream)
            if e:
                e[1].record(stream)
            api.indexer_topk(logits, inp.ctx_lens, K, out=topk, stream=stream)
            if e:
                e[2].record(stream)
        torch.cuda.synchronize()
    lg_us = [a.elapsed_time(b) * 1e3 for a, b, _ in ev]
    tk_us = [b.elapsed_time(c) * 1e3 for _, b, c in ev]
    # the pair as one CUDA-graph replay, the top-k launched as a programmatic dependent of the
    # logits kernel (no event between them), L2 flushed before each replay
    def pair():
        api.indexer_mqa_logits(inp.q, inp.weights, inp.cache, inp.block_table, inp.req_id, inp.ctx_lens, L,
                               block_size=wi.block_size, logits=logits, stream=stream)
        api.indexer_topk(logits, inp.ctx_lens, K, out=topk, stream=stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        pair()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            pair()
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(3 + steps):
            flush.zero_()
            e = pev[i - 3] if i >= 3 else None
            if e:
                e[0].record(stream)
            graph.replay()
            if e:
                e[1].record(stream)
        torch.cuda.synchronize()
    pair_us = [a.elapsed_time(b) * 1e3 for a, b in pev]
    del graph
    positions = int(sum(inp.ctx))
    key_bytes = positions * (D + 4)
    alg = key_bytes + T * H * D + T * H * 4 + T * L * 4
    flops = 2.0 * H * D * positions
    lg_s = statistics.mean(lg_us) / 1e6
    gbs = alg / lg_s / 1e9
    del inp, logits, topk
    return {
        "workload": wi.name, "tokens": T, "heads": H, "head_dim": D, "topk": K, "positions": positions,
        "max_len": L, "steps": steps,
        "logits_us": {"mean": statistics.mean(lg_us), "median": statistics.median(lg_us)},
        "topk_us": {"mean": statistics.mean(tk_us), "median": statistics.median(tk_us)},
        "positions_per_s": positions / ((statistics.median(lg_us) + statistics.median(tk_us)) / 1e6),
        "pair_us": {"mean": statistics.mean(pair_us), "median": statistics.median(pair_us),
                    "method": "logits + top-k captured in one CUDA graph (the top-k a programmatic dependent "
                              "of the logits kernel), events around each replay, L2 flushed before each"},
        "pair_positions_per_s": positions / (statistics.median(pair_us) / 1e6),
        "roofline_logits": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": alg,
                            "key_bytes_per_launch": key_bytes,
                            "tensor_tflops_achieved": flops / lg_s / 1e12,
                            "traffic": load_traffic(wi.name, "indexer_traffic.json", "k_indexer_logits.cu"),
                            "peak_source": f"{src} (MEASURED_PEAKS.json burst)" if src == "measured" else "fallback",
                            "kernel": "smd::indexer_logits_kernel"},
        "gather_us": {"mean": statistics.mean(g_us), "median": statistics.median(g_us)},
        "gather_gbs": g_bytes / (statistics.mean(g_us) / 1e6) / 1e9,
        "gather_frac": g_bytes / (statistics.mean(g_us) / 1e6) / 1e9 / peaks["hbm_gbs"],
        "timing": "events around each launch, L2 flushed before each logits + top-k pair and each gather",
    }


def summary(w, r, peaks, src) -> dict:
    """Per-workload numbers shared by the headline and the extra workloads."""
    inp, S = r["inp"], r["S"]
    rows = inp.n_valid
    nb = step_bytes(inp, S)
    mean_s = statistics.mean(r["step_ms"]) / 1e3
    med_s = statistics.median(r["step_ms"]) / 1e3
    attn_s = statistics.mean(r["attn_ms"]) / 1e3
    roof = roofline(w.num_heads, rows, attn_s, peaks, src, load_traffic(w.name))
    roof["kernel"] = "smd::attn_kernel"
    roof["launch_us_mean"] = attn_s * 1e6
    roof.update({k: v for k, v in fractions(w.num_heads, rows, nb, attn_s, peaks).items()})
    return {
        "workload": w.name, "splits": S, "valid_rows": rows, "bytes_per_step": nb,
        "step_us_mean": mean_s * 1e6, "step_us_median": med_s * 1e6,
        "step_us_p90": sorted(r["step_ms"])[int(0.9 * (len(r["step_ms"]) - 1))] * 1e3,
        "rows_per_s": rows / mean_s, "roofline_attention": roof,
        "roofline_step": fractions(w.num_heads, rows, nb, med_s, peaks),
        "kernels_us_mean": {"convert": statistics.mean(r["conv_ms"]) * 1e3, "attention": attn_s * 1e6,
                            "combine": statistics.mean(r["comb_ms"]) * 1e3 if S > 1 else 0.0},
    }


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch

    from sparse_mla_decode_req_gb300 import api, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    lib = api.load()
    peaks, src = load_peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    w = synth.WORKLOADS[args.config]
    if args.num_splits is not None:
        w = dataclasses.replace(w, max_splits=args.num_splits)
    K = args.steps
    sampler = ClockSampler(local)
    r = measure(api, lib, synth, torch, w, rank_seed(args.config, rank), dev, flush, K, args.warmup,
                min(K, 200), sampler, pg)
    inp, S = r["inp"], r["S"]
    rows_per_step = inp.n_valid
    total_s = max_over_ranks(pg, sum(r["step_ms"]) / 1e3, dev)
    value = job_rate(rows_per_step, K, world, total_s)
    head = summary(w, r, peaks, src)
    roof = {k: head["roofline_attention"][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof.update({k: v for k, v in head["roofline_attention"].items() if k not in roof})

    # end to end through the public call with host buffers: h2d of the step's inputs,
    # decode, d2h of out + lse, per step (out still holds the device path's result)
    try:
        e2e = run_e2e(api, inp, w, dev, r["stream"], flush, min(args.e2e_steps, K), rows_per_step,
                      device_out=r["out"], seed=rank_seed(args.config, rank) + 7)
    except Exception as exc:  # keep the device-timed line; the failure is reported in it
        e2e = {"seconds": None, "steps": 0, "h2d": 0, "d2h": 0, "error": repr(exc)[:300]}
        print(f"e2e leg failed: {exc!r}", file=sys.stderr)
    secs = max_over_ranks(pg, e2e["seconds"] if e2e["seconds"] is not None else float("inf"), dev)
    e2e_val = job_rate(rows_per_step, e2e["steps"], world, secs) if secs != float("inf") else None
    ssecs = max_over_ranks(pg, e2e.get("serial_seconds") or float("inf"), dev)
    serial_e2e = None
    if ssecs != float("inf") and e2e["steps"]:
        serial_e2e = {"value": job_rate(rows_per_step, e2e["steps"], world, ssecs),
                      "us_per_step": ssecs / e2e["steps"] * 1e6,
                      "method": "one stream: copy in, decode, copy out; each step timed alone after an L2 flush"}

    link_e2e = None
    if e2e.get("link_seconds") and e2e["steps"] and secs != float("inf"):
        pair_us = e2e["link_seconds"] / e2e["steps"] * 1e6
        step_us = secs / e2e["steps"] * 1e6
        link_e2e = {"copy_pair_us": pair_us, "step_us": step_us, "frac": pair_us / step_us,
                    "method": "the step's copy in and copy out alone, both directions at once on their "
                              "two streams, no decode: the host link's bound on the pipelined step"}

    # the other target workloads (mid batch, long context; the single-request latency case)
    # measured the same way in the same run, on rank 0's replica only
    extras = {}
    if rank == 0 and world == 1 and args.extra_configs:
        for ci in [int(x) for x in args.extra_configs.split(",") if x.strip() != ""]:
            if ci == args.config:
                continue
            we = synth.WORKLOADS[ci]
            re_ = measure(api, lib, synth, torch, we, rank_seed(ci, 0), dev, flush, args.extra_steps, 3,
                          min(args.extra_steps, 200))
            extras[we.name] = summary(we, re_, peaks, src)
            del re_
            torch.cuda.empty_cache()

    # the same headline step over a bf16 latent cache
    bf16_cache = None
    if rank == 0 and world == 1 and args.bf16_steps > 0:
        bf16_cache = measure_bf16_cache(api, torch, synth, w, rank_seed(args.config, 0), dev, flush,
                                        args.bf16_steps, peaks, src)
        torch.cuda.empty_cache()

    # the indexer step (the top-k source of the decode) on its two workloads
    indexer = {}
    if rank == 0 and world == 1 and args.indexer_steps > 0:
        from sparse_mla_decode_req_gb300 import synth_indexer as si
        for wi in si.INDEXER_WORKLOADS:
            indexer[wi.name] = measure_indexer(api, torch, si, wi, dev, flush, args.indexer_steps, peaks, src)
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, el, steps_done, rows_done, cores = cpu_oracle_rate(inp, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{steps_done} oracle steps of one token each ({rows_done} valid rows, {el:.1f} s, "
                         f"numpy BLAS on all host cores)"}

    S_launches = 2 + (1 if S > 1 else 0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_s / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; fp8_ds_mla rows quantised from N(0,1))",
        "config": workload_config(w),
        "num_splits": S,
        "roofline": roof,
        "roofline_step": head["roofline_step"],
        "bytes_per_step": head["bytes_per_step"],
        "step_timing": {"us_mean": head["step_us_mean"], "us_median": head["step_us_median"],
                        "us_p90": head["step_us_p90"],
                        "method": "CUDA-graph replay of the smd_sparse_mla_decode call (convert, attention, "
                                  "combine), events around each replay, 512 MiB L2 flush between replays"},
        "step_breakdown_us": {**head["kernels_us_mean"],
                              "timing": f"{min(K, 200)} staged steps with events between the kernels "
                                        "(no launch overlap)"},
        "extra_workloads": extras,
        "bf16_cache": bf16_cache,
        "indexer": indexer,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "steps": e2e["steps"], "transfers": "one h2d of the packed inputs, one d2h of out + lse, per step",
                "method": "pipelined over three streams (step i+1's copy in and step i-1's copy out overlap "
                          "step i's decode), two device buffer sets, three rotating input sets (no L2 reuse "
                          "between consecutive steps); timed from the first copy in to the last copy out",
                "serial": serial_e2e,
                "link": link_e2e,
                "matches_device_path": e2e.get("matches_device_path"), **({"error": e2e["error"]} if "error" in e2e else {})},
        "gpu_launches": K * S_launches,
        "clocks": r["clocks"],
        "wall_s_timed_region": r["wall"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def kernel_code_hash(path: str) -> str:
    """Hash of a CUDA source with // comments and blank lines removed: a comment edit
    leaves the compiled kernel, and so a traffic capture of it, valid."""
    import hashlib
    import re
    lines = []
    with open(path) as f:
        for line in f:
            code = re.sub(r"//.*", "", line).rstrip()
            if code:
                lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def load_traffic(name: str, profile: str = "attn_traffic.json", source: str = "k_attn.cu"):
    """DRAM bytes per launch of a kernel from a committed ncu summary, if the kernel's source
    is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", profile)
    src = os.path.join(ROOT, "sparse_mla_decode_req_gb300", "csrc", source)
    key = "k_" + source.split("_", 1)[1].split(".")[0] + "_code_hash"
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(name)
        if e and e.get(key) == kernel_code_hash(src):
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


def pack_layout(named):
    """Byte layout of (name, tensor) pairs packed back to back at 256-byte offsets:
    ({name: (offset, nbytes, dtype, shape)}, total bytes)."""
    lay, off = {}, 0
    for k, t in named:
        n = t.numel() * t.element_size()
        lay[k] = (off, n, t.dtype, tuple(t.shape))
        off = (off + n + 255) // 256 * 256
    return lay, max(off, 256)


def pack_views(buf, lay):
    """Typed, shaped views into a flat uint8 buffer laid out by pack_layout."""
    return {k: buf[o:o + n].view(dt).view(shape) for k, (o, n, dt, shape) in lay.items()}


def e2e_names(w):
    """The per-step host inputs of the public call, in packing order."""
    return [k for k in ("q", "block_table", "req_id", "topk_idx", "swa_idx")
            if not (k == "topk_idx" and not w.topk) and not (k == "swa_idx" and not w.swa)]


def e2e_input_sets(inp, w, n, seed):
    """n host input sets of the step's shapes: set 0 is the step's own inputs; each other set
    draws a fresh q and fresh top-k positions in every token's context (the same -1 entries,
    window and block table), so that consecutive steps of the pipelined leg gather
    different rows and find nothing of the previous step in L2."""
    import torch
    base = {k: getattr(inp, k).cpu() for k in e2e_names(w)}
    sets = [base]
    g = torch.Generator().manual_seed(seed)
    for _ in range(1, n):
        d = dict(base)
        d["q"] = torch.randn(base["q"].shape, generator=g).to(torch.bfloat16)
        if "topk_idx" in d:
            tk = base["topk_idx"].clone()
            for t in range(tk.shape[0]):
                valid = tk[t] >= 0
                nv = int(valid.sum())
                if nv:
                    tk[t, valid] = torch.randperm(int(inp.ctx_lens[t]), generator=g)[:nv].to(torch.int32)
            d["topk_idx"] = tk
        sets.append(d)
    return sets


def run_e2e(api, inp, w, dev, stream, flush, steps, rows_per_step, device_out=None, seed=0):
    """The step through the public call with host-resident inputs.  Every step copies its
    inputs (packed in one pinned buffer) to the device in one transfer, runs
    sparse_mla_decode on views of that buffer, and reads out and lse (one device buffer)
    back in one transfer.

    Pipelined (the reported value): the copies in, the decode and the copies out run on
    three streams over two device input and two result buffers, so step i + 1's inputs
    travel while step i decodes and step i - 1's results come back, as a serving loop
    would run; the timed region spans all steps from the first copy in to the last copy
    out.  Three input sets rotate (see e2e_input_sets), so no step finds its rows in L2.
    Serial (reported beside it): one stream, copy in, decode, copy out, each step timed
    alone after an L2 flush."""
    import torch
    names = e2e_names(w)
    sets = e2e_input_sets(inp, w, 3, seed)
    lay_in, nb_in = pack_layout([(k, sets[0][k]) for k in names])
    h_in = []
    for st in sets:
        h = torch.zeros(nb_in, dtype=torch.uint8).pin_memory()
        for k, v in pack_views(h, lay_in).items():
            v.copy_(st[k])
        h_in.append(h)
    T, H = w.num_tokens, w.num_heads
    lay_out, nb_out = pack_layout([("out", torch.empty(T, H, 512, dtype=torch.bfloat16)),
                                   ("lse", torch.empty(T, H, dtype=torch.float32))])
    d_in = [torch.empty(nb_in, dtype=torch.uint8, device=dev) for _ in range(2)]
    dbuf = [pack_views(x, lay_in) for x in d_in]
    d_res = [torch.empty(nb_out, dtype=torch.uint8, device=dev) for _ in range(2)]
    res = [pack_views(x, lay_out) for x in d_res]
    h_res = [torch.empty(nb_out, dtype=torch.uint8).pin_memory() for _ in range(2)]
    dims = api.make_dims(dbuf[0]["q"], inp.kv_cache, dbuf[0]["block_table"], dbuf[0]["req_id"],
                         dbuf[0].get("topk_idx"), dbuf[0].get("swa_idx"), w.block_size)
    ws = torch.empty(api.workspace_size(dims, w.max_splits, 0), dtype=torch.uint8, device=dev)

    def decode(b):
        api.sparse_mla_decode(dbuf[b]["q"], inp.kv_cache, dbuf[b]["block_table"], dbuf[b]["req_id"],
                              dbuf[b].get("topk_idx"), dbuf[b].get("swa_idx"), inp.sink, inp.scale,
                              out=res[b]["out"], lse=res[b]["lse"], num_splits=w.max_splits, workspace=ws,
                              block_size=w.block_size, stream=stream)

    # ---- serial: every copy, call and event on one stream
    def one():
        d_in[0].copy_(h_in[0], non_blocking=True)
        decode(0)
        h_res[0].copy_(d_res[0], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            one()
            b.record(stream)
        torch.cuda.synchronize()
    serial_s = sum(a.elapsed_time(b) for a, b in evs) / 1e3
    matches = None
    if device_out is not None:  # same inputs, same kernels: the results must agree bit for bit
        matches = bool(torch.equal(pack_views(h_res[0], lay_out)["out"], device_out.cpu()))

    # ---- pipelined: copies in on s_in, decode on `stream`, copies out on s_out
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i & 1
        if i >= 2:
            s_in.wait_event(ev_done[b])  # decode i - 2 has read d_in[b]
        with torch.cuda.stream(s_in):
            d_in[b].copy_(h_in[i % len(h_in)], non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # the copy out of step i - 2 has read d_res[b]
        decode(b)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            h_res[b].copy_(d_res[b], non_blocking=True)
        ev_out[b].record(s_out)

    torch.cuda.synchronize()
    i = 0
    for _ in range(6):  # warm-up
        step(i)
        i += 1
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for _ in range(steps):
        step(i)
        i += 1
    t1.record(s_out)
    torch.cuda.synchronize()
    pipe_s = t0.elapsed_time(t1) / 1e3
    if device_out is not None:  # one more step on set 0: the pipelined path gives the same result
        while i % len(h_in) != 0:
            i += 1
        step(i)
        torch.cuda.synchronize()
        matches = bool(matches and torch.equal(pack_views(h_res[i & 1], lay_out)["out"], device_out.cpu()))

    # the host link's own bound on this schedule: the same copies in and out, both directions
    # at once on their two streams, with no decode between them
    torch.cuda.synchronize()
    l0, l1, l_in = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                    torch.cuda.Event())
    l0.record(s_in)
    s_out.wait_event(l0)
    for j in range(steps):
        with torch.cuda.stream(s_in):
            d_in[j & 1].copy_(h_in[j % len(h_in)], non_blocking=True)
        with torch.cuda.stream(s_out):
            h_res[j & 1].copy_(d_res[j & 1], non_blocking=True)
    l_in.record(s_in)
    s_out.wait_event(l_in)
    l1.record(s_out)
    torch.cuda.synchronize()
    link_s = l0.elapsed_time(l1) / 1e3
    return {"seconds": pipe_s, "steps": steps, "h2d": nb_in, "d2h": nb_out, "matches_device_path": matches,
            "serial_seconds": serial_s, "link_seconds": link_s}


if __name__ == "__main__":
    sys.exit(main())
