"""The C++ scheduler (cb_build_batch) against the oracle's Python scheduler,
bit-exact on every array of every step, plus its error handling."""
import json
import math
import os

import numpy as np
import pytest

from continuous_batching_ragged_gb300 import native, workloads
from oracle.scheduler import Scheduler as OracleScheduler

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _native(*args, **kw):
    from continuous_batching_ragged_gb300.api import Scheduler
    return Scheduler(*args, **kw)


def run_both(m, B, NB, requests, max_num_seqs=0, max_steps=10 ** 6):
    a = _native(m, B, NB, max_num_seqs)
    o = OracleScheduler(m, B, NB, max_num_seqs)
    for r in requests:
        a.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
        o.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
    steps = 0
    while True:
        x = a.build_batch()
        y = o.build_batch()
        for key in ("cu_seqlens_q", "context_lens", "block_tables", "slot_mapping", "request_ids",
                    "evicted_ids"):
            gx, gy = getattr(x, key), getattr(y, key)
            assert gx.dtype == gy.dtype, key
            assert gx.shape == gy.shape and np.array_equal(gx, gy), (steps, key)
        assert x.num_decode == y.num_decode
        assert x.max_q_len == (int(y.q_lens.max()) if y.num_seqs else 0)
        assert x.max_context_len == (int(y.context_lens.max()) if y.num_seqs else 0)
        a.complete_step()
        o.complete_step()
        steps += 1
        st = a.stats()
        assert st.step == steps
        assert st.num_waiting == len(o.waiting) and st.num_running == len(o.running)
        assert st.free_blocks == len(o.free) and st.reserved_blocks == o.reserved_total
        if y.num_seqs == 0 and o.idle:
            assert a.idle
            break
        assert steps < max_steps
    return steps


@pytest.mark.parametrize("name", ["scheduler_p2_replay.json", "scheduler_eviction.json",
                                  "scheduler_decode_over_budget.json", "p1_chunked_prefill.json"])
def test_native_matches_golden(native_lib, name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    reqs = [workloads.Request(r["id"], r["arrival_step"], r["prompt_len"], r["output_len"])
            for r in (g.get("requests") or [g["request"]])]
    s = _native(g["token_budget"], g["block_size"], g["num_blocks"])
    for r in reqs:
        s.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
    for exp in g["steps"]:
        b = s.build_batch()
        for key in ("request_ids", "cu_seqlens_q", "context_lens", "slot_mapping", "evicted_ids"):
            if key in exp:
                assert getattr(b, key).tolist() == exp[key], key
        if "block_tables" in exp:
            assert b.block_tables.tolist() == exp["block_tables"]
        s.complete_step()
    run_both(g["token_budget"], g["block_size"], g["num_blocks"], reqs)


def test_native_matches_oracle_on_random_traces(native_lib):
    for seed in range(20):
        rng = np.random.default_rng(100 + seed)
        B = int(rng.choice([1, 2, 4, 8, 16]))
        NB = int(rng.integers(8, 200))
        m = int(rng.integers(1, 80))
        reqs = []
        for i in range(int(rng.integers(1, 60))):
            r = workloads.Request(int(rng.integers(0, 10 ** 6)) * 100 + i, int(rng.integers(0, 40)),
                                  int(rng.integers(1, 60)), int(rng.integers(1, 20)))
            if math.ceil((r.prompt_len + r.output_len) / B) <= NB:
                reqs.append(r)
        run_both(m, B, NB, reqs, max_num_seqs=int(rng.integers(0, 6)))


@pytest.mark.slow
def test_native_matches_oracle_on_serving_trace(native_lib):
    cfg = workloads.SERVING_TRACE
    steps = run_both(cfg["token_budget"], cfg["block_size"], cfg["num_blocks"], workloads.serving_trace())
    assert steps > 100


def test_native_scheduler_errors(native_lib):
    s = _native(8, 4, 2)
    with pytest.raises(native.CBError) as e:
        s.add_request(0, 0, 6, 3)
    assert e.value.status == native.CB_ERR_NO_BLOCKS
    with pytest.raises(native.CBError) as e:
        s.add_request(1, 0, 0, 3)
    assert e.value.status == native.CB_ERR_INVALID
    s.add_request(2, 0, 2, 2)
    with pytest.raises(native.CBError):
        s.add_request(2, 0, 2, 2)                      # duplicate id
    with pytest.raises(native.CBError):
        s.complete_step()                              # nothing built
    s.build_batch()
    with pytest.raises(native.CBError):
        s.build_batch()                                # previous batch not completed
    with pytest.raises(native.CBError):
        _native(0, 4, 2)
