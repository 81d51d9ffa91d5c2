"""Admission that reserves only the prefill, with preemption by recompute
(hassanahmed.net, the paragraph on the memory manager under continuous
batching: when the card fills, a request is evicted for a while and brought
back later).  Pins: a hand-derived fixture, and invariants checked on every
step of traces whose pools are small enough to force preemptions; then the
C++ scheduler against the oracle, bit-exact."""
import json
import math
import os

import numpy as np
import pytest

from continuous_batching_ragged_gb300 import workloads
from oracle.scheduler import Scheduler

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KEYS = ("request_ids", "q_lens", "cu_seqlens_q", "context_lens", "slot_mapping", "evicted_ids",
        "preempted_ids")


def test_preemption_fixture():
    g = json.load(open(os.path.join(GOLDEN, "scheduler_preempt_recompute.json")))
    s = Scheduler(g["token_budget"], g["block_size"], g["num_blocks"], admission=g["admission"])
    for r in g["requests"]:
        s.add_request(r["id"], r["arrival_step"], r["prompt_len"], r["output_len"])
    for exp in g["steps"]:
        b = s.build_batch()
        for key in KEYS:
            assert getattr(b, key).tolist() == exp[key], key
        assert b.num_decode == exp["num_decode"]
        if "block_tables" in exp:
            assert b.block_tables.tolist() == exp["block_tables"]
        s.complete_step()
    assert s.idle
    assert s.num_preempted == g["final"]["num_preempted"]
    assert s.recomputed_tokens == g["final"]["recomputed_tokens"]


def check_preemption_invariants(sched, requests, m, B, NB, max_steps=10 ** 6):
    """Every step of a trace run to completion:
    * T <= m, decode rows first with q_len 1, a decode row is a request whose
      cache holds its whole current prefill;
    * slots follow the block tables, context = cached + q_len, the blocks of
      live requests are disjoint and in range, a request's blocks never move;
    * a preemption takes the latest admitted running requests, newest first,
      and is not followed by an admission in the same step; the preempted
      request restarts with an empty cache and a prefill of prompt + produced
      tokens;
    * at the end every request produced output_len tokens and the tokens run
      equal sum(prompt + output - 1) + the tokens recomputed.
    """
    for r in requests:
        sched.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
    by_id = {r.id: r for r in requests}
    cached, produced, prefill, blocks = {}, {}, {}, {}
    running = []                         # admission order, as the checker sees it
    first_admission, finished = [], set()
    processed = 0
    step = 0
    preemptions = 0
    while True:
        b = sched.build_batch()
        for e in b.evicted_ids.tolist():
            assert produced[e] == by_id[e].output_len
            finished.add(e)
            blocks.pop(e)
            running.remove(e)
        pre = b.preempted_ids.tolist()
        if pre:
            # victims are the latest admitted, newest first.  A request admitted
            # in a step without room for its prefill has not appeared in a batch
            # yet; such requests are the newest, so they come first.
            seen = [rid for rid in pre if rid in running]
            k = len(pre) - len(seen)
            assert pre[k:] == seen and seen == running[::-1][:len(seen)]
            for rid in pre[:k]:
                assert rid not in finished and by_id[rid].arrival_step <= step
                produced.setdefault(rid, 0)
                if rid not in cached:
                    first_admission.append(rid)
            for rid in pre:
                if rid in running:
                    running.remove(rid)
                blocks.pop(rid, None)
                cached[rid] = 0
                prefill[rid] = by_id[rid].prompt_len + produced[rid]
                preemptions += 1
        assert b.T <= m
        assert np.all(b.q_lens[:b.num_decode] == 1)
        for pos, rid in enumerate(b.request_ids.tolist()):
            if rid not in running:
                assert not pre, "no admission in a step that preempted"
                if rid not in cached:
                    first_admission.append(rid)
                    produced[rid] = 0
                    prefill[rid] = by_id[rid].prompt_len
                cached[rid] = 0
                blocks[rid] = []
                running.append(rid)
                assert by_id[rid].arrival_step <= step
            is_decode = pos < b.num_decode
            assert is_decode == (cached[rid] >= prefill[rid])
            n = int(b.q_lens[pos])
            ctx = int(b.context_lens[pos])
            assert ctx == cached[rid] + n
            if not is_decode:
                assert ctx <= prefill[rid]
            row = [x for x in b.block_tables[pos].tolist() if x >= 0]
            assert row[:len(blocks[rid])] == blocks[rid]        # blocks never move
            assert len(row) >= math.ceil(ctx / B)
            blocks[rid] = row
            for k in range(n):
                p = cached[rid] + k
                assert b.slot_mapping[b.cu_seqlens_q[pos] + k] == row[p // B] * B + p % B
        held = [x for v in blocks.values() for x in v]
        assert len(held) == len(set(held)) and all(0 <= x < NB for x in held)
        sched.complete_step()
        for pos, rid in enumerate(b.request_ids.tolist()):
            n = int(b.q_lens[pos])
            processed += n
            was_decode = pos < b.num_decode
            cached[rid] += n
            if was_decode or cached[rid] == prefill[rid]:
                produced[rid] += 1
        step += 1
        if b.num_seqs == 0 and sched.idle:
            break
        assert step < max_steps
    order = sorted(requests, key=lambda r: (r.arrival_step, r.id))
    assert first_admission == [r.id for r in order]
    assert finished == set(by_id)
    assert all(produced[r.id] == r.output_len for r in requests)
    assert processed == sum(r.prompt_len + r.output_len - 1 for r in requests) + sched.recomputed_tokens
    assert sched.num_preempted == preemptions
    return step, preemptions


def _tight_trace(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([1, 2, 4, 16]))
    NB = int(rng.integers(6, 40))
    m = int(rng.integers(2, 48))
    reqs = []
    for i in range(int(rng.integers(5, 50))):
        r = workloads.Request(i, int(rng.integers(0, 20)), int(rng.integers(1, 30)), int(rng.integers(1, 25)))
        if math.ceil((r.prompt_len + r.output_len) / B) <= NB:
            reqs.append(r)
    return m, B, NB, reqs, int(rng.integers(0, 6))


def test_random_tight_pools_keep_invariants_and_preempt():
    total = 0
    for seed in range(25):
        m, B, NB, reqs, mx = _tight_trace(seed)
        _, n = check_preemption_invariants(Scheduler(m, B, NB, mx, admission="prompt_preempt"), reqs, m, B, NB)
        total += n
    assert total > 50            # the pools are tight enough that preemption is exercised


def test_roomy_pool_never_preempts():
    reqs = [workloads.Request(i, i // 3, 5 + i % 7, 3 + i % 5) for i in range(30)]
    s = Scheduler(16, 4, 1000, admission="prompt_preempt")
    _, n = check_preemption_invariants(s, reqs, 16, 4, 1000)
    assert n == 0 and s.recomputed_tokens == 0


def _native(*args, **kw):
    from continuous_batching_ragged_gb300.api import Scheduler as NativeScheduler
    return NativeScheduler(*args, **kw)


def test_native_preemption_matches_oracle(native_lib):
    for seed in range(25):
        m, B, NB, reqs, mx = _tight_trace(seed)
        a = _native(m, B, NB, mx, admission="prompt_preempt")
        o = Scheduler(m, B, NB, mx, admission="prompt_preempt")
        for r in reqs:
            a.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
            o.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
        steps = 0
        while True:
            x, y = a.build_batch(), o.build_batch()
            for key in ("cu_seqlens_q", "context_lens", "block_tables", "slot_mapping", "request_ids",
                        "evicted_ids", "preempted_ids"):
                gx, gy = getattr(x, key), getattr(y, key)
                assert gx.dtype == gy.dtype and gx.shape == gy.shape and np.array_equal(gx, gy), (seed, steps, key)
            assert x.num_decode == y.num_decode
            a.complete_step()
            o.complete_step()
            steps += 1
            st = a.stats()
            assert st.num_preempted == o.num_preempted and st.recomputed_tokens == o.recomputed_tokens
            assert st.free_blocks == len(o.free) and st.num_running == len(o.running)
            if y.num_seqs == 0 and o.idle:
                assert a.idle
                break


def test_native_preemption_fixture(native_lib):
    g = json.load(open(os.path.join(GOLDEN, "scheduler_preempt_recompute.json")))
    s = _native(g["token_budget"], g["block_size"], g["num_blocks"], admission=g["admission"])
    for r in g["requests"]:
        s.add_request(r["id"], r["arrival_step"], r["prompt_len"], r["output_len"])
    for exp in g["steps"]:
        b = s.build_batch()
        for key in KEYS:
            if key != "q_lens":
                assert getattr(b, key).tolist() == exp[key], key
        s.complete_step()
    st = s.stats()
    assert st.num_preempted == 1 and st.recomputed_tokens == 3


def test_unknown_admission_policy_is_refused(native_lib):
    from continuous_batching_ragged_gb300 import native
    import ctypes
    cfg = native.cb_sched_config(8, 4, 16, 0, 7)
    h = ctypes.c_void_p()
    assert native.lib().cb_scheduler_create(ctypes.byref(cfg), ctypes.byref(h)) == native.CB_ERR_INVALID
    with pytest.raises(ValueError):
        Scheduler(8, 4, 16, admission="bogus")
