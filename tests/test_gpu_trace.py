"""The serving trace end to end: the C++ scheduler drives every step, each
layer appends and attends over its own paged cache, and sampled rows of
sampled (step, layer, sequence, head) are checked against the oracle, which
regenerates each request's history from the seeded definition."""
import numpy as np
import pytest
import torch

import bench
from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run_and_check(reqs, *, num_layers, num_blocks, token_budget, check_every, seed=4,
                   admission="reserve_lifetime", stats_out=None):
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import assert_tolerance, oracle_rows
    rng = np.random.default_rng(0)
    samples = []
    checked_layers = []

    def on_layer(step, layer, bt, out):
        # every layer of a checked step: one random sequence, plus the step's
        # last sequence (a prefill chunk when there is one) on the first and
        # last layers
        if step % check_every:
            return
        q_lens = bt.q_lens
        seqs = {int(rng.integers(bt.num_seqs))}
        if layer in (0, num_layers - 1):
            seqs.add(bt.num_seqs - 1)
        for s in seqs:
            q, c = int(q_lens[s]), int(bt.context_lens[s])
            rows = sorted(set(rng.choice(q, min(q, 3), replace=False).tolist()) | {q - 1})
            h = int(rng.integers(32))
            idx = torch.tensor([int(bt.cu_seqlens_q[s]) + r for r in rows], device="cuda")
            got = out.index_select(0, idx)[:, h].float().cpu().numpy()
            samples.append((layer, int(bt.request_ids[s]), c, q, rows, h, got))
        checked_layers.append((step, layer))

    steps = bench.run_trace(torch, api, W, reqs, num_layers=num_layers, num_heads=32, head_dim=128,
                            block_size=16, token_budget=token_budget, num_blocks=num_blocks,
                            seed=seed, on_layer=on_layer, admission=admission, stats_out=stats_out)
    recomputed = stats_out["recomputed_tokens"] if stats_out is not None else 0
    assert sum(st["T"] for st in steps) == sum(r.prompt_len + r.output_len - 1 for r in reqs) + recomputed
    got, exp = [], []
    for layer, rid, c, q, rows, h, g in samples:
        b = W.RaggedBatch(num_heads=32, head_dim=128, block_size=16, dtype="bf16", seed=seed,
                          layer=layer, seq_ids=np.array([rid]), p=np.array([c - q]),
                          q_len=np.array([q]), block_tables=np.zeros((1, 1), np.int32),
                          num_blocks=1)
        exp.append(oracle_rows(b, 0, [h], rows)[:, 0])
        got.append(g)
    assert len(samples) >= 4
    by_step = {}
    for st, layer in checked_layers:
        by_step.setdefault(st, set()).add(layer)
    assert by_step and all(layers == set(range(num_layers)) for layers in by_step.values())
    assert_tolerance(np.concatenate(got).astype(np.float64), np.concatenate(exp))
    return steps


def test_serving_trace_reduced(native_lib):
    reqs = W.serving_trace(num_requests=120, prompt_median=200, prompt_cap=2048, out_median=30,
                           out_min=5, out_max=60)
    _run_and_check(reqs, num_layers=2, num_blocks=3000, token_budget=1024, check_every=7)


def test_serving_trace_full_size(native_lib):
    """2000 requests, 32 layers, budget 4096, 10240 blocks (86 GB of pools)."""
    cfg = W.SERVING_TRACE
    steps = _run_and_check(W.serving_trace(), num_layers=cfg["num_layers"],
                           num_blocks=cfg["num_blocks"], token_budget=cfg["token_budget"],
                           check_every=199)
    assert len(steps) > 100


def test_serving_trace_with_preemption(native_lib):
    """A pool too small for every admitted request to finish: with admission
    reserving only the prefill, requests are preempted and recomputed.  The
    recomputed keys and values are the same (they are a function of request
    and position), so sampled rows still match the oracle's own history."""
    reqs = W.serving_trace(num_requests=120, prompt_median=200, prompt_cap=2048, out_median=30,
                           out_min=5, out_max=60)
    stats = {}
    _run_and_check(reqs, num_layers=2, num_blocks=300, token_budget=1024, check_every=5,
                   admission="prompt_preempt", stats_out=stats)
    assert stats["num_preempted"] > 0 and stats["recomputed_tokens"] > 0


def test_serving_trace_graph_full_size(native_lib):
    """The full trace served by one CUDA-graph replay per step (the planned,
    captured path the bench's trace_graph workload times), with one output
    buffer per layer: every 199th step, every layer's replayed rows of one
    random sequence (plus the step's last sequence on the first and last
    layers) against the oracle."""
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import assert_tolerance, oracle_rows
    cfg = W.SERVING_TRACE
    rng = np.random.default_rng(1)
    samples = []

    def on_step(step, bt, outs):
        if step % 199:
            return
        for layer, out in enumerate(outs):
            seqs = {int(rng.integers(bt.num_seqs))}
            if layer in (0, len(outs) - 1):
                seqs.add(bt.num_seqs - 1)
            for s in seqs:
                q, c = int(bt.q_lens[s]), int(bt.context_lens[s])
                rows = sorted(set(rng.choice(q, min(q, 3), replace=False).tolist()) | {q - 1})
                h = int(rng.integers(32))
                idx = torch.tensor([int(bt.cu_seqlens_q[s]) + r for r in rows], device="cuda")
                got = out.index_select(0, idx)[:, h].float().cpu().numpy()
                samples.append((step, layer, int(bt.request_ids[s]), c, q, rows, h, got))

    steps = bench.run_trace_graph(torch, api, W, W.serving_trace(), num_layers=cfg["num_layers"], num_heads=32,
                                  head_dim=128, block_size=16, token_budget=cfg["token_budget"],
                                  num_blocks=cfg["num_blocks"], seed=4, on_step=on_step, per_layer_outs=True)
    assert len(steps) > 100
    got, exp = [], []
    for _, layer, rid, c, q, rows, h, g in samples:
        b = W.RaggedBatch(num_heads=32, head_dim=128, block_size=16, dtype="bf16", seed=4,
                          layer=layer, seq_ids=np.array([rid]), p=np.array([c - q]),
                          q_len=np.array([q]), block_tables=np.zeros((1, 1), np.int32), num_blocks=1)
        exp.append(oracle_rows(b, 0, [h], rows)[:, 0])
        got.append(g)
    assert len({st for st, *_ in samples}) >= 10
    assert {layer for _, layer, *_ in samples} == set(range(cfg["num_layers"]))
    assert_tolerance(np.concatenate(got).astype(np.float64), np.concatenate(exp))
