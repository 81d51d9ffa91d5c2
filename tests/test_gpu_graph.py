"""Planned steps and CUDA-graph capture.

One plan per step reused by every layer (cb_plan_step +
cb_ragged_attention_planned) must give the same bits as cb_ragged_attention,
and a step captured once as a CUDA graph over capacity buffers, replayed with
the metadata of each new step of a scheduler-driven trace, must give the same
bits (outputs and cache contents) as the eager calls on exact-size tensors."""
import math

import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

H, A, B = 4, 128, 16


def _regular(st):
    from continuous_batching_ragged_gb300 import api
    b = st.b
    api.cb_ragged_attention(st.q, st.cache, st.cu, st.ctx, st.bt, max_q_len=b.max_q_len,
                            max_context_len=b.max_context_len, scale=st.scale, out=st.out, workspace=st.ws)


@pytest.mark.parametrize("p,q", [([513, 0, 2000, 77, 1023], [1, 1, 1, 1, 1]),
                                 ([300], [450]),
                                 ([0, 300, 5, 40, 1000, 2], [600, 1, 77, 1, 129, 257]),
                                 ([6000, 40, 2500], [512, 1, 300])])
def test_planned_equals_unplanned_bitwise(native_lib, p, q):
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep
    layers = [DeviceStep(W.make_batch(p, q, num_heads=H, head_dim=A, block_size=B, dtype="bf16", seed=120,
                                      layer=layer)) for layer in range(3)]
    ref = []
    for st in layers:
        st.append()
        _regular(st)
        ref.append(st.out.clone())
    api.cb_check_device_errors()
    st0 = layers[0]
    b = st0.b
    api.cb_plan_step(st0.cache, st0.cu, st0.ctx, num_tokens=b.T, max_blocks_per_seq=b.block_tables.shape[1],
                     max_q_len=b.max_q_len, max_context_len=b.max_context_len, workspace=st0.ws)
    for st, r in zip(layers, ref):
        st.out.zero_()
        api.cb_ragged_attention_planned(st.q, st.cache, st0.cu, st0.ctx, st0.bt, max_q_len=b.max_q_len,
                                        max_context_len=b.max_context_len, scale=st.scale, out=st.out,
                                        workspace=st0.ws)
    api.cb_check_device_errors()
    for st, r in zip(layers, ref):
        assert torch.equal(st.out.view(torch.int16), r.view(torch.int16))


def test_planned_call_refuses_a_foreign_workspace(native_lib):
    from continuous_batching_ragged_gb300 import api, native
    from gpu_harness import DeviceStep
    st = DeviceStep(W.make_batch([5, 9], [1, 1], num_heads=H, head_dim=A, block_size=B, dtype="bf16", seed=3))
    other = torch.empty_like(st.ws)
    with pytest.raises(native.CBError, match="no cb_plan_step"):
        api.cb_ragged_attention_planned(st.q, st.cache, st.cu, st.ctx, st.bt, max_q_len=1,
                                        max_context_len=st.b.max_context_len, scale=st.scale, out=st.out,
                                        workspace=other)


def _synth_layer(api, seed, layer, rows, pos, tensors):
    for kind, t in zip((W.KIND_Q, W.KIND_K, W.KIND_V), tensors):
        api.cb_synth_tokens(t, seed, kind, layer, rows, pos)


def test_captured_step_replays_a_trace_bitwise(native_lib):
    """A small scheduler-driven trace (2 layers, budget 256): every step is run
    eagerly on exact-size tensors and by replaying one captured graph; the
    two agree bit for bit, and sampled replayed rows of every step and layer
    match the oracle."""
    from continuous_batching_ragged_gb300 import api
    from continuous_batching_ragged_gb300.step_graph import StepGraph
    from gpu_harness import assert_tolerance, oracle_rows
    rng = np.random.default_rng(2)
    samples = []
    seed, layers, budget, num_blocks = 11, 2, 256, 600
    reqs = W.serving_trace(seed=7, num_requests=24, prompt_median=120, prompt_cap=500, out_median=12,
                           out_min=3, out_max=30)
    max_blocks = math.ceil((500 + 30) / B) + 1
    scale = 1 / math.sqrt(A)
    eager = [api.KVCache.empty(num_blocks, H, B, A) for _ in range(layers)]
    graphed = [api.KVCache.empty(num_blocks, H, B, A) for _ in range(layers)]
    for c in eager + graphed:
        c.k.zero_()
        c.v.zero_()
    cap = lambda: torch.zeros((budget, H, A), dtype=torch.bfloat16, device="cuda")   # noqa: E731
    gq, gk, gv, go = ([cap() for _ in range(layers)] for _ in range(4))
    sg = StepGraph(graphed, gq, gk, gv, go, max_seqs=budget, max_blocks_per_seq=max_blocks, scale=scale)
    sched = api.Scheduler(budget, B, num_blocks)
    for r in reqs:
        sched.add_request(r.id, r.arrival_step, r.prompt_len, r.output_len)
    steps = 0
    while not sched.idle and steps < 400:
        bt = sched.build_batch()
        S, T = len(bt.context_lens), len(bt.slot_mapping)
        if S == 0:
            sched.complete_step()
            continue
        rows = torch.from_numpy(np.repeat(bt.request_ids, bt.q_lens).astype(np.int64)).cuda()
        pos = torch.from_numpy(np.concatenate([np.arange(c - q, c) for c, q in
                                               zip(bt.context_lens, bt.q_lens)]).astype(np.int32)).cuda()
        cu = torch.from_numpy(bt.cu_seqlens_q).cuda()
        ctx = torch.from_numpy(bt.context_lens).cuda()
        btab = torch.from_numpy(bt.block_tables).cuda()
        slots = torch.from_numpy(bt.slot_mapping).cuda()
        ws = torch.empty(api.cb_attention_workspace_size(eager[0], S, T, bt.max_context_len),
                         dtype=torch.uint8, device="cuda")
        ref = []
        for layer in range(layers):
            q, k, v = (torch.empty((T, H, A), dtype=torch.bfloat16, device="cuda") for _ in range(3))
            _synth_layer(api, seed, layer, rows, pos, (q, k, v))
            out = torch.empty_like(q)
            api.cb_append_kv(k, v, slots, eager[layer])
            api.cb_ragged_attention(q, eager[layer], cu, ctx, btab, max_q_len=bt.max_q_len,
                                    max_context_len=bt.max_context_len, scale=scale, out=out, workspace=ws)
            ref.append(out)
            _synth_layer(api, seed, layer, rows, pos, (gq[layer][:T], gk[layer][:T], gv[layer][:T]))
        sg.load(bt.cu_seqlens_q, bt.context_lens, bt.block_tables, bt.slot_mapping, bt.max_q_len,
                bt.max_context_len)
        if sg.graph is None:
            sg.run_eager()            # per-device state, then the graph; this step runs twice on graphed
            torch.cuda.synchronize()  # caches, which is harmless: the append rewrites the same slots
            sg.capture()
        sg.replay()
        api.cb_check_device_errors()
        for layer in range(layers):
            assert torch.equal(go[layer][:T].view(torch.int16), ref[layer].view(torch.int16)), (steps, layer)
            # the replayed rows themselves against the oracle: one random
            # sequence per layer and step, up to 4 of its rows, every head
            s = int(rng.integers(S))
            q_len, c = int(bt.q_lens[s]), int(bt.context_lens[s])
            rows = sorted(set(rng.choice(q_len, min(q_len, 3), replace=False).tolist()) | {q_len - 1})
            got = go[layer][int(bt.cu_seqlens_q[s]) + np.array(rows)].float().cpu().numpy()
            samples.append((layer, int(bt.request_ids[s]), c, q_len, rows, got))
        sched.complete_step()
        steps += 1
    assert sched.idle and steps > 20
    got, exp = [], []
    for layer, rid, c, q_len, rows, g in samples:
        b1 = W.RaggedBatch(num_heads=H, head_dim=A, block_size=B, dtype="bf16", seed=seed, layer=layer,
                           seq_ids=np.array([rid]), p=np.array([c - q_len]), q_len=np.array([q_len]),
                           block_tables=np.zeros((1, 1), np.int32), num_blocks=1)
        exp.append(oracle_rows(b1, 0, None, rows))
        got.append(g)
    assert_tolerance(np.concatenate(got).astype(np.float64), np.concatenate(exp))
    for e, g in zip(eager, graphed):
        assert torch.equal(e.k.view(torch.int16), g.k.view(torch.int16))
        assert torch.equal(e.v.view(torch.int16), g.v.view(torch.int16))


def test_captured_grouped_query_step_equals_eager_bitwise(native_lib):
    """A 2-layer step of 8 query / 2 key-value heads captured once and replayed
    with the metadata of three different steps (decode rows, prefill chunks, a
    chunk long enough to be cut into KV segments) gives the eager grouped
    calls' bits, and every replayed row matches the oracle."""
    from continuous_batching_ragged_gb300 import api
    from continuous_batching_ragged_gb300.step_graph import StepGraph
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    Hq, Hkv, layers, cap_tokens, cap_seqs = 8, 2, 2, 1024, 8
    steps = [([513, 0, 2000, 77], [1, 129, 1, 1]), ([6000, 40, 300], [300, 1, 200]), ([10, 20, 30], [1, 1, 1])]
    batches = [[W.make_batch(p, q, num_heads=Hq, head_dim=128, block_size=16, dtype="bf16", seed=240 + i,
                             layer=layer, num_kv_heads=Hkv) for layer in range(layers)]
               for i, (p, q) in enumerate(steps)]
    max_blocks = max(b.block_tables.shape[1] for bs in batches for b in bs)
    num_blocks = max(b.num_blocks for bs in batches for b in bs)
    scale = 1 / math.sqrt(A)
    caches = [api.KVCache.empty(num_blocks, Hkv, B, A) for _ in range(layers)]
    gq = [torch.zeros((cap_tokens, Hq, A), dtype=torch.bfloat16, device="cuda") for _ in range(layers)]
    gk = [torch.zeros((cap_tokens, Hkv, A), dtype=torch.bfloat16, device="cuda") for _ in range(layers)]
    gv = [torch.zeros((cap_tokens, Hkv, A), dtype=torch.bfloat16, device="cuda") for _ in range(layers)]
    go = [torch.zeros((cap_tokens, Hq, A), dtype=torch.bfloat16, device="cuda") for _ in range(layers)]
    sg = StepGraph(caches, gq, gk, gv, go, max_seqs=cap_seqs, max_blocks_per_seq=max_blocks, scale=scale)
    for i, bs in enumerate(batches):
        eager = [DeviceStep(b) for b in bs]          # its own cache, filled with the batch's history
        ref = []
        for st in eager:
            st.append()
            st.attend()
            ref.append(st.out.clone())
        api.cb_check_device_errors()
        b = bs[0]
        T = b.T
        for layer, st in enumerate(eager):          # the graph's caches start from the same history
            caches[layer].k.zero_()
            caches[layer].v.zero_()
            caches[layer].k[:st.cache.k.shape[0]].copy_(st.cache.k)
            caches[layer].v[:st.cache.v.shape[0]].copy_(st.cache.v)
            gq[layer][:T].copy_(st.q)
            gk[layer][:T].copy_(st.k_new)
            gv[layer][:T].copy_(st.v_new)
        bt = np.full((b.num_seqs, max_blocks), -1, dtype=np.int32)
        bt[:, :b.block_tables.shape[1]] = b.block_tables
        sg.load(b.cu_seqlens_q, b.context_lens, bt, b.slot_mapping, b.max_q_len, b.max_context_len)
        if sg.graph is None:
            sg.run_eager()
            torch.cuda.synchronize()
            sg.capture()
        sg.replay()
        api.cb_check_device_errors()
        for layer in range(layers):
            assert torch.equal(go[layer][:T].view(torch.int16), ref[layer].view(torch.int16)), (i, layer)
            assert_tolerance(to_np(go[layer][:T]), oracle_packed(bs[layer]))   # every replayed row
