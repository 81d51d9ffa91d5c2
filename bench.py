#!/usr/bin/env python
"""Benchmark of one ragged continuous-batching attention step on GB300.

A step is the whole hot path over one packed batch: the step's K/V appended
to the paged cache (cb_append_kv), then attention of every packed query row
(cb_ragged_attention: split-KV decode rows on CUDA cores and prefill chunks
on tcgen05 tensor cores, concurrently).  The default workload is the decode
step (256 sequences, one query each, cached contexts uniform in [512, 4096],
32 heads x 128, bf16, block 16, blocks randomly permuted in the pool);
--workload picks the others.  Inputs are seeded synthetic values generated
in HBM before timing; the KV cache (9.7 GB for the decode step) is far larger
than L2, so no flush is needed between steps.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ragged-attention step tokens/s on 1 GB300; % HBM / tensor roofline per step"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BELOW = 512 * 2 ** 20      # steps moving fewer bytes get an L2 flush between timed steps


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def make_workload(name: str, decode_seqs: int = 256):
    from continuous_batching_ragged_gb300 import workloads as W
    if name == "decode":
        return W.decode_step(num_seqs=decode_seqs), f"decode_{decode_seqs}seq_ctx512-4096_bf16_H32_A128_B16"
    if name == "mixed":
        return W.mixed_step(), "mixed_m2048_64decode_ctx256-4096_chunks661-661-662_bf16_H32_A128_B16"
    if name == "long":
        return W.long_prompt_chunk(15), "long_prompt_32768_last_chunk_2048_bf16_H32_A128_B16"
    if name == "tiny":
        return W.tiny_fp32(), "tiny_fp32_H4_A64_B4_T6"
    if name == "decode_gqa":
        return (W.decode_step(num_seqs=decode_seqs, num_kv_heads=8),
                f"decode_gqa_{decode_seqs}seq_ctx512-4096_bf16_Hq32_Hkv8_A128_B16")
    if name == "decode_gqa_kv4":
        return (W.decode_step(num_seqs=decode_seqs, num_kv_heads=4),
                f"decode_gqa_{decode_seqs}seq_ctx512-4096_bf16_Hq32_Hkv4_A128_B16")
    if name == "decode_mqa":
        return (W.decode_step(num_seqs=decode_seqs, num_kv_heads=1),
                f"decode_mqa_{decode_seqs}seq_ctx512-4096_bf16_Hq32_Hkv1_A128_B16")
    if name == "mixed_gqa":
        return (W.mixed_step(num_kv_heads=8),
                "mixed_gqa_m2048_64decode_ctx256-4096_chunks661-661-662_bf16_Hq32_Hkv8_A128_B16")
    if name == "mixed_padded":
        return W.left_padded(W.mixed_step()), "mixed_m2048_left_padded_to_67x662_masked_bf16_H32_A128_B16"
    if name == "insertion":
        return W.page_insertion_example(), "insertion_B8_n100_ragged_bf16_H32_A128_B16"
    if name == "insertion_padded":
        return (W.left_padded(W.page_insertion_example()),
                "insertion_B8_n100_left_padded_8x100_masked_bf16_H32_A128_B16")
    raise SystemExit(f"unknown workload {name}")


def algorithmic_work(b):
    """Bytes and flops counted once (each KV byte read once, masked pairs not counted)."""
    e = b.elem_bytes
    H, A = b.num_heads, b.head_dim
    Hkv = b.kv_heads                   # keys and values have Hkv heads (grouped-query attention)
    kv_read = int(np.sum(b.context_lens.astype(np.int64))) * 2 * Hkv * A * e
    qo = b.T * H * A * e * 2
    append = 2 * 2 * b.T * Hkv * A * e
    pairs = sum(int(q) * int(p) + int(q) * (int(q) + 1) // 2 for p, q in zip(b.p, b.q_len))
    flops = 4 * A * H * pairs
    decode = b.q_len == 1
    dec_bytes = (int(np.sum(b.context_lens[decode].astype(np.int64))) * 2 * Hkv * A * e
                 + int(np.sum(decode)) * H * A * e * 2)
    pre = b.q_len > 1
    pre_bytes = (int(np.sum(b.context_lens[pre].astype(np.int64))) * 2 * Hkv * A * e
                 + int(np.sum(b.q_len[pre])) * H * A * e * 2)
    return {"bytes": kv_read + qo + append, "flops": flops, "decode_bytes": dec_bytes,
            "prefill_bytes": pre_bytes,
            "append_bytes": append,
            "prefill_flops": 4 * A * H * sum(int(q) * int(p) + int(q) * (int(q) + 1) // 2
                                             for p, q in zip(b.p, b.q_len) if q > 1)}


def profiled_traffic_ratio(profile: str):
    """DRAM bytes per algorithmic byte recorded from an ncu capture of the
    kernel (dram__bytes_read.sum + dram__bytes_write.sum over the same
    algorithmic bytes model), or None if no summary records it."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.startswith("dram_bytes_per_algorithmic_byte:"):
            return float(line.split(":", 1)[1])
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# device staging (inputs generated in HBM by the seeded device generator)
# ---------------------------------------------------------------------------

class Staged:
    """One step's inputs in HBM.  With `cache` given, the step runs on that
    cache as it stands (its cached prefix is not regenerated)."""

    def __init__(self, b, torch, api, W, cache=None):
        dt = torch.bfloat16 if b.dtype == "bf16" else torch.float32
        self.b = b
        fill = cache is None
        if cache is None:
            cache = api.KVCache.empty(b.num_blocks, b.kv_heads, b.block_size, b.head_dim, dt)
            cache.k.zero_()
            cache.v.zero_()
        self.cache = cache
        sid = torch.from_numpy(b.seq_ids).cuda()
        if fill and int(b.p.max()) > 0:
            pl = torch.from_numpy(b.p.astype(np.int32)).cuda()
            bt = torch.from_numpy(b.block_tables).cuda()
            for kind, pool in ((W.KIND_K, self.cache.k), (W.KIND_V, self.cache.v)):
                api.cb_synth_fill_cache(pool, b.seed, kind, b.layer, sid, pl, bt, int(b.p.max()))
        rows = torch.from_numpy(np.repeat(b.seq_ids, b.q_len)).cuda()
        pos = torch.from_numpy(np.concatenate(
            [b.gen_positions(s, np.arange(b.p[s], b.p[s] + b.q_len[s])) for s in range(b.num_seqs)])
            .astype(np.int32)).cuda()
        self.q, self.k_new, self.v_new = (torch.empty((b.T, b.heads_of(kind), b.head_dim), dtype=dt, device="cuda")
                                          for kind in (W.KIND_Q, W.KIND_K, W.KIND_V))
        for kind, t in ((W.KIND_Q, self.q), (W.KIND_K, self.k_new), (W.KIND_V, self.v_new)):
            api.cb_synth_tokens(t, b.seed, kind, b.layer, rows, pos)
        self.cu = torch.from_numpy(b.cu_seqlens_q).cuda()
        self.ctx = torch.from_numpy(b.context_lens).cuda()
        self.bt = torch.from_numpy(b.block_tables).cuda()
        self.slots = torch.from_numpy(b.slot_mapping).cuda()
        self.out = torch.empty_like(self.q)
        self.grouped = b.num_heads != b.kv_heads
        ws = (api.cb_attention_workspace_size_gqa(self.cache, b.num_heads, b.num_seqs, b.T, b.max_context_len)
              if self.grouped else api.cb_attention_workspace_size(self.cache, b.num_seqs, b.T, b.max_context_len))
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device="cuda")
        self.scale = 1.0 / math.sqrt(b.head_dim)
        self.api = api
        self.pads = None if b.pad_lens is None else torch.from_numpy(b.pad_lens.astype(np.int32)).cuda()

    def append(self, stream=None, k=None, v=None, slots=None):
        self.api.cb_append_kv(self.k_new if k is None else k, self.v_new if v is None else v,
                              self.slots if slots is None else slots, self.cache, stream)

    def attend(self, stream=None, q=None, cu=None, ctx=None, bt=None, out=None):
        b = self.b
        args = (self.q if q is None else q, self.cache, self.cu if cu is None else cu,
                self.ctx if ctx is None else ctx, self.bt if bt is None else bt)
        kw = dict(max_q_len=b.max_q_len, max_context_len=b.max_context_len, scale=self.scale,
                  out=self.out if out is None else out, workspace=self.ws, stream=stream)
        if self.pads is not None:
            self.api.cb_padded_attention(*args, self.pads, **kw)
        elif self.grouped:
            self.api.cb_ragged_attention_gqa(*args, **kw)
        else:
            self.api.cb_ragged_attention(*args, **kw)


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------

_RANDOM_CACHE = {}


def _random_inputs(n_max, c_max, H, A, Hkv=None):
    Hkv = H if Hkv is None else Hkv
    key = (n_max, c_max, H, A, Hkv)
    if key not in _RANDOM_CACHE:
        rng = np.random.default_rng(0)
        _RANDOM_CACHE.clear()
        _RANDOM_CACHE[key] = (rng.standard_normal((n_max, H, A)), rng.standard_normal((c_max, Hkv, A)),
                              rng.standard_normal((c_max, Hkv, A)))
    return _RANDOM_CACHE[key]


def time_oracle(b, budget_s: float, detail: bool = False, repeat: bool = False):
    """Time the oracle (as it stands) on a bounded sample of the workload's
    sequences, with random inputs of the workload's shapes (drawn once and
    sliced per sequence; drawing them is not timed).  Returns (tokens/s,
    sample description, cores, seconds spent), plus the query tokens and
    sequences processed with detail."""
    from oracle import attention as oa
    H, A = b.num_heads, b.head_dim
    scale = 1.0 / math.sqrt(A)
    qbuf, kbuf, vbuf = _random_inputs(b.max_q_len, b.max_context_len, H, A, b.kv_heads)
    order = np.argsort(-b.q_len, kind="stable")          # prefill chunks first, then decodes
    done_tokens, done_seqs, spent, passes = 0, 0, 0.0, 0
    while True:                                         # repeat: whole passes until the budget is spent
        for s in order:
            n, c = int(b.q_len[s]), int(b.context_lens[s])
            t0 = time.perf_counter()
            oa.attend_sequence(qbuf[:n], kbuf[:c], vbuf[:c], c - n, scale)
            spent += time.perf_counter() - t0
            done_tokens += n
            done_seqs += 1
            if spent >= budget_s:
                break
        passes += 1
        if not repeat or spent >= budget_s:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"{done_seqs} of {b.num_seqs} sequences ({done_tokens} of {b.T} query tokens, all "
              f"{H} heads), fp64 numpy, random inputs of the workload's shapes")
    if passes > 1:
        sample = (f"{passes} passes over all {b.num_seqs} sequences ({done_tokens} query tokens, all {H} heads), "
                  "fp64 numpy, random inputs of the workload's shapes")
    if detail:
        return done_tokens / spent, sample, cores, spent, done_tokens, done_seqs
    return done_tokens / spent, sample, cores, spent


# ---------------------------------------------------------------------------
# serving trace: the scheduler drives every step
# ---------------------------------------------------------------------------

def run_trace_graph(torch, api, W, requests, *, num_layers, num_heads, head_dim, block_size,
                    token_budget, num_blocks, seed, max_steps=100000, admission="reserve_lifetime",
                    stats_out=None, num_kv_heads=None, on_step=None, per_layer_outs=False):
    """run_trace with each step captured once as a CUDA graph (StepGraph):
    per step the host builds the batch, the device generator writes every
    layer's Q/K/V (not timed), the metadata is copied into the graph's fixed
    buffers, and the timed region is one graph replay -- the step plan, then
    cb_append_kv_dims + cb_ragged_attention_planned for every layer.
    per_layer_outs gives every layer its own output buffer (default: one
    shared buffer); on_step(step, batch, outs) runs after each replay."""
    from continuous_batching_ragged_gb300.step_graph import StepGraph
    dt = torch.bfloat16
    hkv = num_kv_heads or num_heads
    caches = [api.KVCache.empty(num_blocks, hkv, block_size, head_dim, dt) for _ in range(num_layers)]
    for c in caches:
        c.k.zero_()
        c.v.zero_()
    longest = max(r.prompt_len + r.output_len for r in requests)
    max_blocks = (longest + block_size - 1) // block_size + 1
    shape, kv_shape = (token_budget, num_heads, head_dim), (token_budget, hkv, head_dim)
    q = [torch.zeros(shape, dtype=dt, device="cuda") for _ in range(num_layers)]
    k, v = ([torch.zeros(kv_shape, dtype=dt, device="cuda") for _ in range(num_layers)] for _ in range(2))
    out = [torch.zeros(shape, dtype=dt, device="cuda") for _ in range(num_layers if per_layer_outs else 1)]
    sg = StepGraph(caches, q, k, v, out, max_seqs=token_budget, max_blocks_per_seq=max_blocks,
                   scale=1.0 / math.sqrt(head_dim))
    sched = api.Scheduler(token_budget, block_size, num_blocks, admission=admission)
    for r in requests:
        sched.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
    steps = []
    stream = torch.cuda.current_stream()
    for step in range(max_steps):
        t0 = time.perf_counter()
        bt = sched.build_batch()
        t_sched = time.perf_counter() - t0
        S, T = bt.num_seqs, bt.T
        if S == 0:
            t0 = time.perf_counter()
            sched.complete_step()
            t_sched += time.perf_counter() - t0
            if sched.idle:
                break
            steps.append({"T": 0, "sched_s": t_sched, "gpu_ms": 0.0})
            continue
        rows = torch.from_numpy(np.repeat(bt.request_ids, bt.q_lens).astype(np.int64)).cuda()
        pos = torch.from_numpy(np.concatenate([np.arange(c - n, c) for c, n in
                                               zip(bt.context_lens, bt.q_lens)]).astype(np.int32)).cuda()
        for layer in range(num_layers):
            for kind, t in ((W.KIND_Q, q[layer]), (W.KIND_K, k[layer]), (W.KIND_V, v[layer])):
                api.cb_synth_tokens(t[:T], seed, kind, layer, rows, pos)
        sg.load(bt.cu_seqlens_q, bt.context_lens, bt.block_tables, bt.slot_mapping, bt.max_q_len,
                bt.max_context_len)
        if sg.graph is None:
            sg.run_eager()                 # resolves per-device state; the replay below redoes the step
            torch.cuda.synchronize()
            sg.capture()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        sg.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        api.cb_check_device_errors()
        if on_step is not None:
            on_step(step, bt, [o[:T] for o in out])
        t0 = time.perf_counter()
        sched.complete_step()
        t_sched += time.perf_counter() - t0
        steps.append({"T": T, "S": S, "decode": bt.num_decode, "sched_s": t_sched,
                      "gpu_ms": e0.elapsed_time(e1), "kv_tokens": int(np.sum(bt.context_lens)),
                      "q_lens": bt.q_lens, "max_q_len": bt.max_q_len, "ctx": bt.context_lens})
    if stats_out is not None:
        st = sched.stats()
        stats_out.update(num_preempted=st.num_preempted, recomputed_tokens=st.recomputed_tokens)
    del sg, caches
    torch.cuda.empty_cache()
    return steps


def run_trace(torch, api, W, requests, *, num_layers, num_heads, head_dim, block_size,
              token_budget, num_blocks, seed, on_layer=None, max_steps=100000,
              admission="reserve_lifetime", stats_out=None, num_kv_heads=None):
    """Serve ``requests`` to completion.  Each step: cb_build_batch on the host,
    metadata to the device, then per layer the step's Q/K/V (device generator,
    keyed by request id and position, not timed) followed by the timed
    cb_append_kv + cb_ragged_attention on that layer's cache.  Returns per-step
    records (tokens, host scheduler seconds, device attention milliseconds)."""
    dt = torch.bfloat16
    hkv = num_kv_heads or num_heads
    grouped = hkv != num_heads
    caches = [api.KVCache.empty(num_blocks, hkv, block_size, head_dim, dt)
              for _ in range(num_layers)]
    for c in caches:
        c.k.zero_()
        c.v.zero_()
    sched = api.Scheduler(token_budget, block_size, num_blocks, admission=admission)
    for r in requests:
        sched.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
    scale = 1.0 / math.sqrt(head_dim)
    ws = torch.empty(0, dtype=torch.uint8, device="cuda")
    qkv = None
    steps = []
    stream = torch.cuda.current_stream()
    for step in range(max_steps):
        t0 = time.perf_counter()
        bt = sched.build_batch()
        t_sched = time.perf_counter() - t0
        S, T = bt.num_seqs, bt.T
        if S == 0:
            t0 = time.perf_counter()
            sched.complete_step()
            t_sched += time.perf_counter() - t0
            if sched.idle:
                break
            steps.append({"T": 0, "sched_s": t_sched, "gpu_ms": 0.0})
            continue
        q_lens = bt.q_lens
        rows = np.repeat(bt.request_ids, q_lens)
        pos = np.concatenate([np.arange(c - q, c) for c, q in zip(bt.context_lens, q_lens)])
        d_rows = torch.from_numpy(rows.astype(np.int64)).cuda()
        d_pos = torch.from_numpy(pos.astype(np.int32)).cuda()
        cu = torch.from_numpy(bt.cu_seqlens_q).cuda()
        ctx = torch.from_numpy(bt.context_lens).cuda()
        btab = torch.from_numpy(bt.block_tables).cuda()
        slots = torch.from_numpy(bt.slot_mapping).cuda()
        need = (api.cb_attention_workspace_size_gqa(caches[0], num_heads, S, T, bt.max_context_len) if grouped
                else api.cb_attention_workspace_size(caches[0], S, T, bt.max_context_len))
        if need > ws.numel():
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        if qkv is None or qkv[0].shape[0] < T:
            rows_cap = max(T, token_budget)
            qkv = [torch.empty((rows_cap, h, head_dim), dtype=dt, device="cuda")
                   for h in (num_heads, hkv, hkv, num_heads)]
        q, k, v, out = (t[:T] for t in qkv)
        events = []
        for layer in range(num_layers):
            for kind, t in ((W.KIND_Q, q), (W.KIND_K, k), (W.KIND_V, v)):
                api.cb_synth_tokens(t, seed, kind, layer, d_rows, d_pos)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            api.cb_append_kv(k, v, slots, caches[layer])
            attend = api.cb_ragged_attention_gqa if grouped else api.cb_ragged_attention
            attend(q, caches[layer], cu, ctx, btab, max_q_len=bt.max_q_len,
                   max_context_len=bt.max_context_len, scale=scale, out=out, workspace=ws)
            e1.record(stream)
            events.append((e0, e1))
            if on_layer is not None:       # runs in stream order, before the next layer reuses `out`
                on_layer(step, layer, bt, out)
        torch.cuda.synchronize()
        gpu_ms = sum(e0.elapsed_time(e1) for e0, e1 in events)
        api.cb_check_device_errors()
        t0 = time.perf_counter()
        sched.complete_step()
        t_sched += time.perf_counter() - t0
        steps.append({"T": T, "S": S, "decode": bt.num_decode, "sched_s": t_sched, "gpu_ms": gpu_ms,
                      "kv_tokens": int(np.sum(bt.context_lens)), "q_lens": q_lens,
                      "max_q_len": bt.max_q_len,
                      "ctx": bt.context_lens})
    if stats_out is not None:
        st = sched.stats()
        stats_out.update(num_preempted=st.num_preempted, recomputed_tokens=st.recomputed_tokens)
    del caches
    torch.cuda.empty_cache()
    return steps


def attention_launches(num_seqs, num_tokens, max_q_len, dtype="bf16"):
    """Kernels cb_ragged_attention launches for one call, by its routing: fp32
    runs one row-mode kernel; bf16 runs the step plan, then the decode kernel
    (max_q_len == 1), the prefill kernel (one sequence, all prefill) or both."""
    if dtype != "bf16":
        return 1
    if max_q_len == 1 or (num_seqs == 1 and max_q_len == num_tokens):
        return 2
    return 3


def launches_per_layer(st):
    """Kernels cb_append_kv + cb_ragged_attention launch for one layer of a step."""
    return 1 + attention_launches(st["S"], st["T"], st["max_q_len"])


def trace_step_roofline(step, num_layers, num_heads, head_dim, peaks, num_kv_heads=None):
    """Roofline time of one step over all layers (algorithmic bytes and flops):
    each cached K/V byte once, q and out, the append; flops over query heads."""
    e = 2
    H, A = num_heads, head_dim
    Hkv = num_kv_heads or num_heads
    ctx = step["ctx"].astype(np.int64)
    q = step["q_lens"].astype(np.int64)
    p = ctx - q
    bytes_ = int(ctx.sum()) * 2 * Hkv * A * e + step["T"] * H * A * e * 2 + 4 * step["T"] * Hkv * A * e
    flops = 4 * A * H * int(np.sum(q * p + q * (q + 1) // 2))
    t = max(bytes_ / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops_sustained"] * 1e12))
    return num_layers * t * 1e3, num_layers * bytes_, num_layers * flops


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def max_over_ranks(x: float) -> float:
    """The slowest rank's value (identity without a process group).  Uses the
    group's own device: CUDA tensors under NCCL, CPU tensors under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank: int, slowest_ms: float, world: int) -> float:
    """Whole-job tokens/s of N independent replicas (weak scaling): every rank
    serves the same step, so the job completes world * tokens in the slowest
    rank's time."""
    return world * tokens_per_rank / (slowest_ms * 1e-3)


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_config(b, label, work, world=1):
    """The `config` object of a step workload's line (the same in both arms)."""
    useful = b.useful_tokens if b.useful_tokens is not None else b.T
    return {"workload": label, "num_seqs": b.num_seqs, "tokens_per_step": useful, "computed_query_rows": b.T,
            "kv_bytes_read": int(work["bytes"] - work["append_bytes"]),
            "l2": ("inputs larger than L2 (KV cache read per step >> 129 MB)" if work["bytes"] > L2_FLUSH_BELOW
                   else "L2 flushed between timed steps (a 512 MB write outside the step's events)"),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args, b, label):
    """The reference arm: the oracle, as it stands, on the host cores.  Each
    step processes the workload's sequences in order until the step's budget
    (about 150 s over all steps) is spent; when the budget covers every
    sequence the step is the whole workload.  value = query tokens processed /
    seconds spent, ms_per_step = seconds spent per step."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    work = algorithmic_work(b)
    budget = max(0.2, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    spent_steps, tokens_steps, seqs_steps = [], [], []
    cores, sample = 1, ""
    for i in range(args.warmup + args.steps):
        tps, sample, cores, spent, done_tokens, done_seqs = time_oracle(b, budget, detail=True)
        if i >= args.warmup:
            spent_steps.append(spent)
            tokens_steps.append(done_tokens)
            seqs_steps.append(done_seqs)
    value = sum(tokens_steps) / sum(spent_steps)
    whole = min(seqs_steps) == b.num_seqs
    cfg = workload_config(b, label, work)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(spent_steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "reference_step": ("the whole workload per step" if whole else
                               f"a bounded sample per step: {min(seqs_steps)}-{max(seqs_steps)} of "
                               f"{b.num_seqs} sequences; value is the sample's rate"),
            "sampled_tokens_per_step": statistics.mean(tokens_steps),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_trace_bench(args, graph=False, print_line=True):
    """The serving trace end to end: 2000 requests, 32 layers, budget 4096
    (graph: each step one CUDA-graph replay).  Returns the line (ours arm)."""
    from continuous_batching_ragged_gb300 import workloads as W
    cfg = dict(W.SERVING_TRACE)
    if args.trace_blocks:
        cfg["num_blocks"] = args.trace_blocks
    cfg["num_kv_heads"] = args.kv_heads or cfg["num_heads"]
    reqs = W.serving_trace()
    label = (f"serving_trace_{len(reqs)}req_{cfg['num_layers']}layers_m{cfg['token_budget']}_"
             f"{cfg['num_blocks']}blocks_bf16_H{cfg['num_heads']}_A128_B16")
    if cfg["num_kv_heads"] != cfg["num_heads"]:
        label += f"_Hkv{cfg['num_kv_heads']}"
    if args.admission != "reserve_lifetime":
        label += "_" + args.admission
    rank, world, local = dist_info()
    if args.impl == "reference":
        if rank != 0:
            return
        # the oracle on one mid-trace step's batch (one layer), as a bounded sample
        from oracle.scheduler import Scheduler as OS
        o = OS(cfg["token_budget"], cfg["block_size"], cfg["num_blocks"], admission=args.admission)
        for r in reqs:
            o.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
        batch = None
        for _ in range(60):
            batch = o.build_batch()
            o.complete_step()
        b = W.RaggedBatch(num_heads=cfg["num_heads"], head_dim=cfg["head_dim"],
                          num_kv_heads=cfg["num_kv_heads"],
                          block_size=cfg["block_size"], dtype="bf16", seed=4, layer=0,
                          seq_ids=batch.request_ids, p=(batch.context_lens - batch.q_lens).astype(np.int64),
                          q_len=batch.q_lens.astype(np.int64), block_tables=batch.block_tables,
                          num_blocks=cfg["num_blocks"])
        run_reference(args, b, label)
        return
    import torch
    from continuous_batching_ragged_gb300 import build as _build
    _build.build()
    from continuous_batching_ragged_gb300 import api
    torch.cuda.set_device(local)
    peaks = load_peaks()
    kw = dict(num_layers=cfg["num_layers"], num_heads=cfg["num_heads"], head_dim=cfg["head_dim"],
              block_size=cfg["block_size"], token_budget=cfg["token_budget"],
              num_blocks=cfg["num_blocks"], seed=4, num_kv_heads=cfg["num_kv_heads"])
    runner = run_trace_graph if graph else run_trace
    kw["admission"] = args.admission
    # warm-up: a short trace of the first requests
    runner(torch, api, W, reqs[:16], max_steps=max(3, args.warmup), **kw)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    t0 = time.perf_counter()
    sched_stats = {}
    steps = runner(torch, api, W, reqs, stats_out=sched_stats, **kw)
    wall = time.perf_counter() - t0
    clocks = sampler.stop()
    busy = [st for st in steps if st["T"] > 0]
    tokens = sum(st["T"] for st in busy)
    gpu_ms = sum(st["gpu_ms"] for st in busy)
    roof = [trace_step_roofline(st, cfg["num_layers"], cfg["num_heads"], cfg["head_dim"], peaks,
                                cfg["num_kv_heads"]) for st in busy]
    fracs = np.array([r[0] / st["gpu_ms"] for r, st in zip(roof, busy)])
    sched_us = 1e6 * np.mean([st["sched_s"] for st in steps])
    line = {"metric": METRIC, "value": tokens / (gpu_ms * 1e-3), "unit": UNIT, "n_gpus": 1,
            "steps": len(steps), "warmup": max(3, args.warmup), "ms_per_step": gpu_ms / len(busy),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": label, "requests": len(reqs), "layers": cfg["num_layers"],
                       "tokens_total": tokens,
                       "l2": "inputs larger than L2 (%.0f GB of KV pools)" % (
                           cfg["num_blocks"] * cfg["block_size"] * cfg["num_kv_heads"] * cfg["head_dim"] * 2 * 2
                           * cfg["num_layers"] / 1e9),
                       "timed": "cb_append_kv + cb_ragged_attention of every layer of every step; "
                                "Q/K/V generation between layers not timed"},
            "step_roofline": {"frac_total": sum(r[0] for r in roof) / gpu_ms,
                              "frac_p10": float(np.percentile(fracs, 10)),
                              "frac_p50": float(np.percentile(fracs, 50)),
                              "frac_p90": float(np.percentile(fracs, 90)),
                              "bytes_total": sum(r[1] for r in roof), "flops_total": sum(r[2] for r in roof)},
            "scheduler_us_per_step": sched_us, "wall_s": wall,
            "admission": args.admission, "preemptions": sched_stats.get("num_preempted", 0),
            "recomputed_tokens": sched_stats.get("recomputed_tokens", 0),
            "useful_tokens_per_s": (tokens - sched_stats.get("recomputed_tokens", 0)) / (gpu_ms * 1e-3),
            "gpu_ms_total": gpu_ms,
            "mean_decode_per_step": float(np.mean([st["decode"] for st in busy])),
            "clocks": clocks,
            "gpu_launches": (sum(1 + 3 * cfg["num_layers"] for st in busy) if graph else
                             sum(cfg["num_layers"] * launches_per_layer(st) for st in busy))}
    if graph:
        line["config"]["workload"] = label + "_graph"
        line["config"]["timed"] = ("one CUDA-graph replay per step: the step plan, then cb_append_kv_dims + "
                                   "cb_ragged_attention_planned of every layer; Q/K/V generation not timed")
    line["roofline"] = {"kernel": "whole step (append + attention, all layers)", "bound": "hbm or tensor per step",
                        "achieved": None, "peak": None, "unit": None,
                        "frac": line["step_roofline"]["frac_total"], "traffic": None,
                        "note": "sum over steps of max(bytes / HBM, flops / sustained bf16) over measured time"}
    if print_line:
        print(json.dumps(line), flush=True)
    return line


def _sm_count() -> int:
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152


def dominant_roofline(b, work, attn_ms, peaks):
    """Roofline of the step's dominant kernel: the larger of the decode rows'
    HBM time and the prefill chunks' tensor time.  Both kernels run inside the
    one attention call, so in a mixed step the call's time bounds the dominant
    kernel's time from above (the fraction is then a lower bound)."""
    t_dec = work["decode_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_pre = work["prefill_flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_dec >= t_pre:
        group = b.num_heads // b.kv_heads
        # the library's routing: groups of 5..32 heads on tensor cores, groups
        # of four too unless the step is decode-only with at least 10 units
        # (sequence, key/value head) per SM
        tensor_decode = b.dtype == "bf16" and (4 < group <= 32 or (group == 4 and (
            b.max_q_len > 1 or b.num_seqs * b.kv_heads < 10 * _sm_count())))
        dom = {"kernel": ("decode_tc_kernel (grouped decode rows on tensor cores)" if tensor_decode else
                          "split_kv_persistent_kernel (decode rows)" if b.dtype == "bf16" else "split_kv_kernel"),
               "bound": "hbm", "achieved": work["decode_bytes"] / (attn_ms * 1e-3) / 1e9,
               "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        prof = ("decode_tc_mqa_64seq.md" if tensor_decode else
                "split_kv_persistent_gqa_decode_200seq.md" if group > 1 else "split_kv_persistent_decode_64seq.md")
        alg = work["decode_bytes"]
    else:
        dom = {"kernel": "prefill_tc_kernel (prefill chunks)", "bound": "tensor",
               "achieved": work["prefill_flops"] / (attn_ms * 1e-3) / 1e12,
               "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
        prof, alg = "prefill_tc_persistent_long_prompt_last_chunk.md", work["prefill_bytes"]
    dom["frac"] = dom["achieved"] / dom["peak"]
    ratio = profiled_traffic_ratio(prof) if b.dtype == "bf16" else None
    dom["traffic"] = None if ratio is None else ratio * alg
    if ratio is not None:
        dom["traffic_source"] = (f"profiles/{prof}: dram bytes per algorithmic byte of an ncu capture "
                                 f"({ratio}), times this launch's {alg} algorithmic bytes")
    dom["peak_source"] = f"of {peaks['source']}"
    return dom


def step_roofline_of(work, ms, append_ms, attn_ms, peaks):
    t_hbm = work["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = work["flops"] / (peaks["bf16_tflops"] * 1e12)
    return {"bytes": work["bytes"], "flops": work["flops"], "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "roofline_ms": max(t_hbm, t_tc) * 1e3, "measured_ms": ms,
            "frac": max(t_hbm, t_tc) * 1e3 / ms,
            "frac_vs_nominal_8tbs": (work["bytes"] / (NOMINAL_HBM_GBS * 1e9)) * 1e3 / ms,
            "append_ms": append_ms, "attention_ms": attn_ms}


def time_steps(torch, st, steps, stream, flush_buf=None, barrier=False):
    """Time `steps` steps (append + attention) with CUDA events on `stream`.
    Without flush_buf: back to back, ms = (end - start) / steps.  With it:
    the buffer is rewritten before each step, outside the step's events, and
    ms = the mean of the steps' own event times.  Returns (ms per step, mean
    append ms, mean attention ms)."""
    import torch.distributed as dist
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    if barrier:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        if flush_buf is not None:
            flush_buf.add_(1)
        ev[i][0].record(stream)
        st.append()
        ev[i][1].record(stream)
        st.attend()
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if barrier:
        dist.barrier()
    append_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    if flush_buf is None:
        ms = t_start.elapsed_time(t_end) / steps
    else:
        ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)
    return ms, append_ms, attn_ms


def measure_config(torch, api, W, b, label, peaks, steps, warmup, world=1, barrier=False, min_seconds=0.0):
    """Stage one step workload in HBM and time `steps` steps after `warmup`
    untimed ones (more steps when min_seconds asks for a longer timed region,
    so that the clock sampler sees it).  Returns (result dict, staged step)."""
    st = Staged(b, torch, api, W)
    stream = torch.cuda.current_stream()
    work = algorithmic_work(b)
    flush = torch.empty(L2_FLUSH_BELOW // 4, dtype=torch.float32, device="cuda").zero_() \
        if work["bytes"] < L2_FLUSH_BELOW else None
    for _ in range(warmup):
        st.append()
        st.attend()
    api.cb_check_device_errors()
    torch.cuda.synchronize()
    if min_seconds > 0:
        est, _, _ = time_steps(torch, st, 3, stream, flush)
        steps = max(steps, int(math.ceil(min_seconds / (est * 1e-3))))
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    ms, append_ms, attn_ms = time_steps(torch, st, steps, stream, flush, barrier)
    clocks = sampler.stop()
    api.cb_check_device_errors()
    cfg = workload_config(b, label, work, world)
    useful = cfg["tokens_per_step"]
    res = {"config": cfg, "steps": steps, "ms_per_step": ms, "tokens_per_s": useful / (ms * 1e-3),
           "roofline": dominant_roofline(b, work, attn_ms, peaks),
           "step_roofline": step_roofline_of(work, ms, append_ms, attn_ms, peaks),
           "clocks": clocks,
           "gpu_launches": (1 + attention_launches(b.num_seqs, b.T, b.max_q_len, b.dtype)) * steps}
    return res, st


def measure_e2e(torch, api, st, steps, world):
    """The same step through the public API with host buffers: pinned H2D of
    the step's inputs and metadata, the two calls, D2H of the output."""
    stream = torch.cuda.current_stream()
    host = {name: getattr(st, name).cpu().pin_memory() for name in
            ("q", "k_new", "v_new", "cu", "ctx", "bt", "slots")}
    dev_in = {name: torch.empty_like(getattr(st, name)) for name in host}
    out_host = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        for name, t in host.items():
            dev_in[name].copy_(t, non_blocking=True)
        st.append(k=dev_in["k_new"], v=dev_in["v_new"], slots=dev_in["slots"])
        st.attend(q=dev_in["q"], cu=dev_in["cu"], ctx=dev_in["ctx"], bt=dev_in["bt"])
        out_host.copy_(st.out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / steps)
    api.cb_check_device_errors()
    useful = st.b.useful_tokens if st.b.useful_tokens is not None else st.b.T
    return {"value": replica_throughput(useful, e2e_ms, world), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}


def oracle_one_thread(workload, decode_seqs, budget):
    """The oracle timed with one BLAS/OpenMP thread, in a child process (the
    thread count of numpy's BLAS is fixed when it loads)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, bench; b, _ = bench.make_workload(%r, %d); "
            "tps, sample, cores, spent = bench.time_oracle(b, %f, repeat=True); "
            "print(json.dumps([tps, sample]))" % (workload, decode_seqs, budget))
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=120)
        tps, sample = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:            # a baseline only: never fail the bench over it
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    return {"value": tps, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
            "threads": "OMP/OPENBLAS/MKL_NUM_THREADS=1"}


def measure_long_prompt(torch, api, W, peaks, steps, warmup):
    """The long-prompt config as specified: one 32768-token prompt processed in
    16 chunks of 2048, each appended to the one paged cache and attended over
    it in turn.  A step is all 16 chunks; tokens/s counts the prompt's tokens."""
    chunks = [W.long_prompt_chunk(k) for k in range(16)]
    b0 = chunks[0]
    cache = api.KVCache.empty(b0.num_blocks, b0.kv_heads, b0.block_size, b0.head_dim, torch.bfloat16)
    cache.k.zero_()
    cache.v.zero_()
    staged = [Staged(b, torch, api, W, cache=cache) for b in chunks]
    stream = torch.cuda.current_stream()
    works = [algorithmic_work(b) for b in chunks]

    def one_prompt(ev=None):
        for i, st in enumerate(staged):
            if ev is not None:
                ev[i][0].record(stream)
            st.append()
            if ev is not None:
                ev[i][1].record(stream)
            st.attend()
            if ev is not None:
                ev[i][2].record(stream)

    for _ in range(warmup):
        one_prompt()
    api.cb_check_device_errors()
    torch.cuda.synchronize()
    evs = [[tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in staged] for _ in range(steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        one_prompt(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    api.cb_check_device_errors()
    ms = t0.elapsed_time(t1) / steps
    chunk_attn_ms = [statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for ev in evs) for i in range(16)]
    attn_ms = sum(chunk_attn_ms)
    append_ms = sum(statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for ev in evs) for i in range(16))
    flops = sum(w["prefill_flops"] for w in works)
    bytes_ = sum(w["bytes"] for w in works)
    achieved = flops / (attn_ms * 1e-3) / 1e12
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = bytes_ / (peaks["hbm_gbs"] * 1e9)
    ratio = profiled_traffic_ratio("prefill_tc_persistent_long_prompt_last_chunk.md")
    del staged, cache
    torch.cuda.empty_cache()
    return {"config": {"workload": "long_prompt_32768_in_16_chunks_of_2048_bf16_H32_A128_B16",
                       "tokens_per_step": 32768, "chunks": 16,
                       "l2": "inputs larger than L2 (each chunk reads up to 537 MB of KV)"},
            "steps": steps, "ms_per_step": ms, "tokens_per_s": 32768 / (ms * 1e-3),
            "roofline": {"kernel": "prefill_tc_kernel (16 launches, one per chunk)", "bound": "tensor",
                         "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"],
                         "frac_vs_sustained": achieved / peaks["bf16_tflops_sustained"],
                         "traffic": None if ratio is None else ratio * sum(w["prefill_bytes"] for w in works),
                         "peak_source": f"of {peaks['source']}"},
            "step_roofline": {"flops": flops, "bytes": bytes_, "roofline_ms": max(t_tc, t_hbm) * 1e3,
                              "measured_ms": ms, "frac": max(t_tc, t_hbm) * 1e3 / ms,
                              "append_ms": append_ms, "attention_ms": attn_ms,
                              "chunk_attention_ms": [round(x, 4) for x in chunk_attn_ms],
                              "chunk_tensor_frac": [round(w["prefill_flops"] / (x * 1e-3) / 1e12 / peaks["bf16_tflops"], 3)
                                                    for w, x in zip(works, chunk_attn_ms)]},
            "clocks": clocks, "gpu_launches": 16 * 3 * steps}


def measure_per_config(torch, api, W, peaks, args):
    """Every other config, each timed in its own region with its own clock
    samples: the tiny fp32 step, the mixed step, the long prompt (last chunk
    alone and all 16 chunks), and the serving trace (eager and graph)."""
    out = {}
    warm = max(3, args.warmup)
    for name in ("tiny", "mixed", "long"):
        b, label = make_workload(name)
        res, st = measure_config(torch, api, W, b, label, peaks, max(10, min(args.steps, 100)), warm,
                                 min_seconds=0.5)
        del st
        torch.cuda.empty_cache()
        if name == "tiny" and not args.no_cpu_baseline:
            # the tiny step is the oracle's own scale: time it on all host cores and on one
            tps, sample, cores, _ = time_oracle(b, 2.0, repeat=True)
            res["cpu_baseline"] = {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
            res["cpu_baseline_1thread"] = oracle_one_thread("tiny", 256, 2.0)
        out[label] = res
    res = measure_long_prompt(torch, api, W, peaks, max(5, min(args.steps, 30)), warm)
    out[res["config"]["workload"]] = res
    for graph in (False, True):
        line = run_trace_bench(argparse.Namespace(**dict(vars(args), impl="ours", kv_heads=0, trace_blocks=0,
                                                         admission="reserve_lifetime")),
                               graph=graph, print_line=False)
        keep = ("steps", "ms_per_step", "config", "roofline", "step_roofline", "clocks", "gpu_launches",
                "gpu_ms_total", "wall_s", "scheduler_us_per_step", "mean_decode_per_step")
        res = {k: line[k] for k in keep}
        res["tokens_per_s"] = line["value"]
        out[line["config"]["workload"]] = res
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=["decode", "mixed", "long", "tiny", "trace", "trace_graph",
                                                             "decode_gqa", "decode_gqa_kv4", "decode_mqa", "mixed_gqa",
                                                             "mixed_padded", "insertion",
                                                             "insertion_padded"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="default workload only: skip the other configs (mixed, long prompt, trace)")
    ap.add_argument("--admission", default="reserve_lifetime", choices=["reserve_lifetime", "prompt_preempt"],
                    help="scheduler admission policy of the trace workloads")
    ap.add_argument("--trace-blocks", type=int, default=0, help="KV pool blocks of the trace workloads")
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="key/value heads of the trace workloads (grouped-query attention; 0: one per query head)")
    ap.add_argument("--decode-seqs", type=int, default=256,
                    help="sequences of the decode workload (smaller cases for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    if args.workload in ("trace", "trace_graph"):
        run_trace_bench(args, graph=args.workload == "trace_graph")
        return
    b, label = make_workload(args.workload, args.decode_seqs)
    if args.impl == "reference":
        run_reference(args, b, label)
        return

    import torch
    import torch.distributed as dist
    from continuous_batching_ragged_gb300 import build as _build
    _build.build()
    from continuous_batching_ragged_gb300 import api
    from continuous_batching_ragged_gb300 import workloads as W

    rank, world, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    peaks = load_peaks()

    res, st = measure_config(torch, api, W, b, label, peaks, args.steps, args.warmup, world=world,
                             barrier=world > 1)
    ms = max_over_ranks(res["ms_per_step"])
    useful = res["config"]["tokens_per_step"]
    value = replica_throughput(useful, ms, world)
    e2e = measure_e2e(torch, api, st, max(10, args.steps // 3), world)

    cpu = cpu_1t = None
    if rank == 0 and not args.no_cpu_baseline:
        tps, sample, cores, _ = time_oracle(b, args.cpu_budget)
        cpu = {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
        if args.workload in ("decode", "tiny"):
            cpu_1t = oracle_one_thread(args.workload, args.decode_seqs, min(8.0, args.cpu_budget))
    del st
    torch.cuda.empty_cache()

    per_config = None
    if args.workload == "decode" and world == 1 and not args.no_per_config:
        per_config = measure_per_config(torch, api, W, peaks, args)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": b.dtype, "data": "synthetic",
                "config": res["config"], "roofline": res["roofline"], "step_roofline": res["step_roofline"],
                "cpu_baseline": cpu, "e2e": e2e, "clocks": res["clocks"], "gpu_launches": res["gpu_launches"]}
        if cpu_1t is not None:
            line["cpu_baseline_1thread"] = cpu_1t
        if per_config is not None:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
