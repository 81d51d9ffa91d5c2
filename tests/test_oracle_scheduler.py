"""Pins for the scheduler oracle: hand-derived fixtures from the pages' examples
and the invariants the pages' rules imply, checked on every step of traces."""
import json
import math
import os

import numpy as np
import pytest

from continuous_batching_ragged_gb300 import workloads
from oracle import attention as oa
from oracle.scheduler import Scheduler

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    return json.load(open(os.path.join(GOLDEN, name)))


def _run_fixture(g):
    s = Scheduler(g["token_budget"], g["block_size"], g["num_blocks"], g.get("max_num_seqs", 0))
    reqs = g.get("requests") or [g["request"]]
    for r in reqs:
        s.add_request(r["id"], r["arrival_step"], r["prompt_len"], r["output_len"])
    got = []
    for _ in g["steps"]:
        got.append(s.build_batch())
        s.complete_step()
    return got


@pytest.mark.parametrize("name", ["scheduler_p2_replay.json", "scheduler_eviction.json",
                                  "scheduler_decode_over_budget.json", "p1_chunked_prefill.json"])
def test_scheduler_fixture(name):
    g = _load(name)
    got = _run_fixture(g)
    for b, exp in zip(got, g["steps"]):
        for key in ("request_ids", "q_lens", "cu_seqlens_q", "context_lens", "slot_mapping", "evicted_ids"):
            if key in exp:
                assert getattr(b, key).tolist() == exp[key], (name, key)
        if "block_tables" in exp:
            assert b.block_tables.tolist() == exp["block_tables"]
        if "row_key_limits" in exp:
            assert oa.row_key_limits(b.cu_seqlens_q, b.context_lens).tolist() == exp["row_key_limits"]


def test_p1_chunk_count_is_ceil_n_over_m():
    for n in range(1, 30):
        for m in range(1, 9):
            s = Scheduler(m, 4, 64)
            s.add_request(0, 0, n, 1)
            chunks = []
            while True:
                b = s.build_batch()
                s.complete_step()
                if b.num_seqs == 0:
                    break
                chunks.append(int(b.q_lens[0]))
            assert len(chunks) == math.ceil(n / m)
            assert sum(chunks) == n and all(c == m for c in chunks[:-1])


def test_rejects_requests_that_can_never_fit():
    s = Scheduler(8, 4, 2)
    with pytest.raises(ValueError):
        s.add_request(0, 0, 6, 3)          # ceil(9/4) = 3 blocks > 2
    with pytest.raises(ValueError):
        s.add_request(1, 0, 0, 3)


def check_trace_invariants(sched_factory, requests, m, B, NB, max_steps=10 ** 6):
    """Run a trace to completion, asserting on every step:
    * sum of q_lens <= m and every decode sequence has q_len 1 and comes first;
    * decode sequences are exactly the running requests past their prompt (up to m);
    * physical blocks of live requests are disjoint, in range, and free + held = NB;
    * slots follow block tables; context_lens = cached + q_len;
    * admission is FIFO by (arrival, id) and never before arrival;
    * every request ends with prompt_len + output_len - 1 processed tokens.
    """
    s = sched_factory()
    for r in requests:
        s.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
    by_id = {r.id: r for r in requests}
    cached = {}                # id -> tokens in cache
    produced = {}              # id -> output tokens
    blocks = {}                # id -> physical blocks
    admitted = []
    finished = set()
    step = 0
    while True:
        b = s.build_batch()
        for e in b.evicted_ids.tolist():
            assert produced[e] == by_id[e].output_len
            finished.add(e)
            blocks.pop(e)
        S = b.num_seqs
        assert b.T <= m
        assert np.all(b.q_lens >= 1)
        assert np.all(b.q_lens[:b.num_decode] == 1)
        live_decoders = [i for i in cached if i not in finished and cached[i] >= by_id[i].prompt_len]
        for pos, rid in enumerate(b.request_ids.tolist()):
            if rid not in cached:
                admitted.append(rid)
                cached[rid] = 0
                produced[rid] = 0
                blocks[rid] = []
                assert by_id[rid].arrival_step <= step
            is_decode = pos < b.num_decode
            assert is_decode == (cached[rid] >= by_id[rid].prompt_len)
            n = int(b.q_lens[pos])
            assert int(b.context_lens[pos]) == cached[rid] + n
            ctx = int(b.context_lens[pos])
            nblk = math.ceil(ctx / B)
            row = b.block_tables[pos].tolist()
            assert all(x >= 0 for x in row[:nblk]) and all(x == -1 for x in row[nblk:])
            assert row[:len(blocks[rid])] == blocks[rid]       # blocks never move
            blocks[rid] = row[:nblk]
            for k in range(n):
                p = cached[rid] + k
                assert b.slot_mapping[b.cu_seqlens_q[pos] + k] == row[p // B] * B + p % B
        # decode-first: if the batch has room left, every live decoder is in it
        if b.num_decode < len(live_decoders):
            assert b.T == m
        held = [x for v in blocks.values() for x in v]
        assert len(held) == len(set(held)) and all(0 <= x < NB for x in held)
        s.complete_step()
        for pos, rid in enumerate(b.request_ids.tolist()):
            n = int(b.q_lens[pos])
            was_decode = pos < b.num_decode
            cached[rid] += n
            if was_decode or cached[rid] == by_id[rid].prompt_len:
                produced[rid] += 1
        step += 1
        if S == 0 and s.idle:
            break
        assert step < max_steps
    order = sorted(requests, key=lambda r: (r.arrival_step, r.id))
    assert admitted == [r.id for r in order]
    assert finished == set(by_id)
    for r in requests:
        assert cached[r.id] == r.prompt_len + r.output_len - 1
        assert produced[r.id] == r.output_len
    return step


def test_random_small_traces_keep_invariants():
    for seed in range(6):
        rng = np.random.default_rng(seed)
        n = 40
        reqs = [workloads.Request(i, int(rng.integers(0, 30)), int(rng.integers(1, 40)),
                                  int(rng.integers(1, 12))) for i in range(n)]
        m, B, NB = int(rng.integers(4, 64)), int(rng.choice([1, 2, 4, 16])), 64
        reqs = [r for r in reqs if math.ceil((r.prompt_len + r.output_len) / B) <= NB]
        mx = int(rng.integers(0, 5))
        check_trace_invariants(lambda: Scheduler(m, B, NB, mx), reqs, m, B, NB)


def test_max_num_seqs_caps_running_set():
    s = Scheduler(100, 4, 100, max_num_seqs=2)
    for i in range(5):
        s.add_request(i, 0, 3, 4)
    b = s.build_batch()
    assert b.request_ids.tolist() == [0, 1]
    s.complete_step()


@pytest.mark.slow
def test_serving_trace_invariants():
    cfg = workloads.SERVING_TRACE
    reqs = workloads.serving_trace()
    steps = check_trace_invariants(
        lambda: Scheduler(cfg["token_budget"], cfg["block_size"], cfg["num_blocks"]),
        reqs, cfg["token_budget"], cfg["block_size"], cfg["num_blocks"])
    assert steps > 100
