"""Prefill chunks on tcgen05 (and mixed steps) against the oracle, plus the
invariants the pages state: chunked == single pass, packed == alone,
incremental decode == recompute, no leakage."""
import math

import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [16, 8, 64, 128])
def test_prefill_chunks_small(native_lib, B):
    """Chunk lengths around the 128-row tile, cached prefixes around the
    128-key tile and block edges; the pool's unused slots hold NaN."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    p = [0, 0, 5, 16, 127, 128, 1000, 3]
    q = [2, 128, 127, 129, 300, 64, 33, 1]
    b = W.make_batch(p, q, num_heads=2, head_dim=128, block_size=B, dtype="bf16", seed=50 + B)
    got = to_np(DeviceStep(b).run())
    assert_tolerance(got, oracle_packed(b))


def test_mixed_step_scaled_down(native_lib):
    """Decode rows and prefill chunks in one step (both kernels concurrently)."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    b = W.mixed_step(num_decode=12, ctx_lo=100, ctx_hi=700, chunks=(61, 130, 200),
                     chunk_p=(0, 129, 300), num_heads=4, seed=7)
    got = to_np(DeviceStep(b).run())
    assert_tolerance(got, oracle_packed(b))


def test_mixed_step_full_size_every_row(native_lib):
    """The full mixed step, in the launch configuration the bench times: 64
    decode rows (contexts 256-4096) plus chunks of 661/661/662 rows at cached
    lengths 0/1024/2048, 32 heads.  Every row of each prefill chunk on 2 heads
    and every decode row on 4 heads against the oracle (each tolerance applied
    per chunk and to the decode rows)."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_rows, to_np
    b = W.mixed_step()
    out = to_np(DeviceStep(b, source="device").run())
    assert np.all(np.isfinite(out))
    rng = np.random.default_rng(3)
    cu = b.cu_seqlens_q
    for s in range(b.num_seqs - 3, b.num_seqs):
        heads = sorted(rng.choice(32, 2, replace=False).tolist())
        assert_tolerance(out[cu[s]:cu[s + 1]][:, heads], oracle_rows(b, s, heads))
    got, exp = [], []
    for s in range(b.num_seqs - 3):
        heads = sorted(rng.choice(32, 4, replace=False).tolist())
        exp.append(oracle_rows(b, s, heads))
        got.append(out[cu[s]:cu[s] + 1][:, heads])
    assert_tolerance(np.concatenate(got), np.concatenate(exp))


def _header(ws):
    """The step plan's header at the start of the workspace (white-box: [9] is
    the KV tiles per prefill segment, 0 when units were not segmented)."""
    return ws[:64].view(torch.int32).tolist()


@pytest.mark.parametrize("B,kv_heads", [(16, 4), (8, 4), (128, 4), (16, 2)])
def test_prefill_kv_segments(native_lib, B, kv_heads):
    """Few prefill units over long contexts: the plan cuts each query pair's
    keys into segments (16 KV tiles here) that run on different SMs and are
    merged by log-sum-exp.  Covers rows that see no key of a later segment
    (the first query tile of a pair), a one-tile last segment, a pair of one
    query tile, decode rows beside it, block sizes and grouped KV heads."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    p = [6000, 40, 2500, 3000, 0]
    q = [512, 1, 300, 1, 129]
    b = W.make_batch(p, q, num_heads=4, head_dim=128, block_size=B, dtype="bf16", seed=140 + B,
                     num_kv_heads=kv_heads)
    st = DeviceStep(b)
    got = to_np(st.run())
    assert _header(st.ws)[9] == 16
    assert_tolerance(got, oracle_packed(b))
    # the tickets are back at zero: the same call again gives the same bits
    again = st.out.clone()
    st.attend()
    torch.cuda.synchronize()
    assert torch.equal(st.out.view(torch.int16), again.view(torch.int16))


def _run_chunked_prompt(prompt, chunk, H=32, seed=3):
    """Process one prompt chunk by chunk through append + attention on one
    cache; returns (cache, output of the last chunk)."""
    from gpu_harness import DeviceStep
    cache = None
    st = None
    for k in range(prompt // chunk):
        b = W.long_prompt_chunk(k, seed=seed, prompt=prompt, chunk=chunk, num_heads=H)
        st = DeviceStep(b, source="device", cache=cache) if cache is not None else DeviceStep(b, source="device")
        cache = st.cache
        st.run()
    return st


def test_long_prompt_chunked_equals_single_pass(native_lib):
    """A 32768-token prompt in 16 chunks of 2048, each appended and attended
    over the paged cache; the last chunk equals rows 30720.. of one pass over
    all 32768 tokens, and every row of it matches the oracle on 4 heads."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_rows, to_np
    prompt, chunk = 32768, 2048
    last = _run_chunked_prompt(prompt, chunk)
    got_last = last.out.clone()
    single_b = W.long_prompt_chunk(0, prompt=prompt, chunk=chunk, single_pass=True)
    single = DeviceStep(single_b, source="device")
    single.run()
    ref_rows = single.out[prompt - chunk:]
    # The single pass streams each query pair's keys in one piece; the last
    # chunk alone (256 units for the whole GPU) is cut into KV segments merged
    # by log-sum-exp.  Each segment rounds its probabilities to bf16 against
    # its own running max (2^-9 relative per term) and the merged row is
    # rounded to bf16 once more (1.2e-4 at |o| ~ 0.02): the two agree far
    # inside the oracle tolerance, not bit for bit.
    assert _header(last.ws)[9] > 0 and _header(single.ws)[9] == 0
    assert_tolerance(to_np(got_last), to_np(ref_rows), max_abs=1e-3, mean_abs=1e-4)
    # every row of the last chunk on 4 heads against the oracle (32768 keys)
    heads = [0, 9, 17, 30]
    exp = oracle_rows(last.b, 0, heads)
    got = to_np(got_last)[:, heads]
    assert_tolerance(got, exp)


def test_prefill_packed_equals_alone_bitwise(native_lib):
    from gpu_harness import DeviceStep
    b = W.make_batch([0, 300, 5, 40], [200, 1, 77, 1], num_heads=2, head_dim=128, block_size=16,
                     dtype="bf16", seed=61)
    full = DeviceStep(b)
    out = full.run().clone()
    cu = b.cu_seqlens_q
    for s in range(b.num_seqs):
        sub = W.RaggedBatch(num_heads=2, head_dim=128, block_size=16, dtype="bf16", seed=61, layer=0,
                            seq_ids=b.seq_ids[s:s + 1], p=b.p[s:s + 1], q_len=b.q_len[s:s + 1],
                            block_tables=b.block_tables[s:s + 1], num_blocks=b.num_blocks)
        st = DeviceStep(sub, cache=full.cache)
        st.attend()
        torch.cuda.synchronize()
        assert torch.equal(st.out.view(torch.int16), out[cu[s]:cu[s + 1]].view(torch.int16))


def test_prefill_no_cross_sequence_leakage(native_lib):
    from gpu_harness import DeviceStep
    b = W.make_batch([10, 0, 200], [150, 90, 40], num_heads=2, head_dim=128, block_size=16,
                     dtype="bf16", seed=71)
    st = DeviceStep(b)
    base = st.run().clone()
    cu = b.cu_seqlens_q
    for s in (0, 2):
        blk = torch.from_numpy(b.block_tables[s][b.block_tables[s] >= 0]).long().cuda()
        st.cache.k[blk] = st.cache.k[blk] * -2
        st.cache.v[blk] = st.cache.v[blk] + 3
        st.q[cu[s]:cu[s + 1]] *= 3
    st.attend()
    torch.cuda.synchronize()
    assert torch.equal(st.out[cu[1]:cu[2]].view(torch.int16), base[cu[1]:cu[2]].view(torch.int16))
    assert not torch.equal(st.out[cu[0]:cu[1]], base[cu[0]:cu[1]])


def test_incremental_decode_matches_single_pass(native_lib):
    """KV cache: prefill 300 tokens, then decode 5 tokens one step at a time;
    each decode row matches the corresponding row of a single causal pass."""
    from gpu_harness import DeviceStep, assert_tolerance, to_np
    P, D, H = 300, 5, 4
    total = P + D
    ids = np.random.default_rng(0).permutation(64).astype(np.int32)
    bt = ids[:math.ceil(total / 16)].reshape(1, -1)

    def batch(p, q):
        return W.RaggedBatch(num_heads=H, head_dim=128, block_size=16, dtype="bf16", seed=81, layer=0,
                             seq_ids=np.zeros(1, np.int64), p=np.array([p]), q_len=np.array([q]),
                             block_tables=bt.copy(), num_blocks=64)

    st = DeviceStep(batch(0, P))
    st.run()
    dec = []
    for t in range(P, total):
        s2 = DeviceStep(batch(t, 1), cache=st.cache)
        dec.append(to_np(s2.run())[0])
    full = DeviceStep(batch(0, total))
    ref = to_np(full.run())[P:]
    assert_tolerance(np.stack(dec), ref)
