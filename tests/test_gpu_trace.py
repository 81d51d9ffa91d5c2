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

    def on_layer(step, layer, bt, out):
        if step % check_every or layer not in (0, num_layers - 1):
            return
        q_lens = bt.q_lens
        for s in {int(rng.integers(bt.num_seqs)), bt.num_seqs - 1}:
            q, c = int(q_lens[s]), int(bt.context_lens[s])
            rows = sorted(set(rng.choice(q, min(q, 3), replace=False).tolist()) | {q - 1})
            h = int(rng.integers(32))
            idx = torch.tensor([int(bt.cu_seqlens_q[s]) + r for r in rows], device="cuda")
            got = out.index_select(0, idx)[:, h].float().cpu().numpy()
            samples.append((layer, int(bt.request_ids[s]), c, q, rows, h, got))

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
