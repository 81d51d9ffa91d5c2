"""Split-KV attention (decode rows, and every row of fp32 caches) against the oracle."""
import math

import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import native
from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_tiny_fp32_step_matches_oracle(native_lib):
    """3 sequences, T=6: a 4-token prefill and decodes over 7 and 12 cached tokens."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    b = W.tiny_fp32()
    got = to_np(DeviceStep(b).run())
    exp = oracle_packed(b)
    stats = assert_tolerance(got, exp)
    assert stats["max_abs"] < 1e-5           # fp32 end to end


@pytest.mark.parametrize("dtype,A,B", [("bf16", 128, 16), ("bf16", 128, 8), ("bf16", 128, 64),
                                       ("f32", 64, 4), ("f32", 128, 16)])
def test_decode_edge_contexts(native_lib, dtype, A, B):
    """Context lengths at 1, around block, tile (16) and split (512) edges."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    ctx = [1, 2, 15, 16, 17, 31, 33, 511, 512, 513, 1024, 1025, 1537, 2049]
    b = W.make_batch([c - 1 for c in ctx], [1] * len(ctx), num_heads=4, head_dim=A, block_size=B,
                     dtype=dtype, seed=11)
    got = to_np(DeviceStep(b).run())
    assert_tolerance(got, oracle_packed(b))


def test_decode_step_scaled_down(native_lib):
    """The decode workload's shape (32 x 128, block 16, permuted pool) with 24 sequences;
    every row checked on 4 of the 32 heads."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_rows, to_np
    b = W.decode_step(num_seqs=24, seed=21)
    got = to_np(DeviceStep(b, source="device").run())
    heads = [0, 7, 19, 31]
    exp = np.concatenate([oracle_rows(b, s, heads) for s in range(b.num_seqs)])
    assert_tolerance(got[:, heads], exp)


def test_decode_step_full_size_every_row(native_lib):
    """The full decode step, in the launch configuration the bench times: 256
    sequences, contexts U[512, 4096]; every output row checked for finiteness,
    and every sequence against the oracle on 4 heads (a different 4 per
    sequence, so all 32 heads are covered)."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_rows, to_np
    b = W.decode_step()
    st = DeviceStep(b, source="device")
    out = to_np(st.run())
    assert np.all(np.isfinite(out))
    rng = np.random.default_rng(5)
    got, exp = [], []
    for s in range(b.num_seqs):
        heads = sorted(rng.choice(32, 4, replace=False).tolist())
        exp.append(oracle_rows(b, s, heads))
        got.append(out[b.cu_seqlens_q[s]:b.cu_seqlens_q[s] + 1][:, heads])
    assert_tolerance(np.concatenate(got), np.concatenate(exp))


def test_packed_equals_alone_bitwise(native_lib):
    """Ragged batching changes nothing per sequence: each sequence run alone
    (same cache, same blocks) gives bit-identical rows."""
    from gpu_harness import DeviceStep
    b = W.make_batch([700, 0, 3000, 40, 1999], [1] * 5, num_heads=4, head_dim=128, block_size=16,
                     dtype="bf16", seed=31)
    full = DeviceStep(b)
    out = full.run().clone()
    for s in range(b.num_seqs):
        sub = W.RaggedBatch(num_heads=4, head_dim=128, block_size=16, dtype="bf16", seed=31, layer=0,
                            seq_ids=b.seq_ids[s:s + 1], p=b.p[s:s + 1], q_len=b.q_len[s:s + 1],
                            block_tables=b.block_tables[s:s + 1], num_blocks=b.num_blocks)
        st = DeviceStep(sub, cache=full.cache)
        st.attend()
        torch.cuda.synchronize()
        assert torch.equal(st.out.view(torch.int16), out[s:s + 1].view(torch.int16))


def test_no_cross_sequence_leakage_bitwise(native_lib):
    from gpu_harness import DeviceStep
    b = W.make_batch([100, 600, 50], [1, 1, 1], num_heads=2, head_dim=128, block_size=16,
                     dtype="bf16", seed=41)
    st = DeviceStep(b)
    base = st.run().clone()
    # scramble every other sequence's cache blocks and queries
    for s in (0, 2):
        blk = torch.from_numpy(b.block_tables[s][b.block_tables[s] >= 0]).long().cuda()
        st.cache.k[blk] = -st.cache.k[blk] * 3
        st.cache.v[blk] = st.cache.v[blk] + 1
        st.q[s] = st.q[s] * 2
    st.attend()
    torch.cuda.synchronize()
    assert torch.equal(st.out[1].view(torch.int16), base[1].view(torch.int16))
    assert not torch.equal(st.out[0], base[0])


def test_bad_block_id_and_metadata_are_reported(native_lib):
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep
    b = W.make_batch([40, 7], [1, 1], num_heads=2, head_dim=128, block_size=16, dtype="bf16", seed=3)
    st = DeviceStep(b)
    st.run()
    st.bt[0, 1] = b.num_blocks + 3                # physical block outside the pool
    st.attend()
    with pytest.raises(native.CBError) as e:
        api.cb_check_device_errors()
    assert e.value.status == native.CB_ERR_BOUNDS
    st.bt.copy_(torch.from_numpy(b.block_tables).cuda())
    st.ctx[1] = b.max_context_len + 5              # contradicts the host bound
    st.attend()
    with pytest.raises(native.CBError) as e:
        api.cb_check_device_errors()
    assert e.value.status == native.CB_ERR_INVALID
    st.ctx.copy_(torch.from_numpy(b.context_lens).cuda())
    st.attend()
    api.cb_check_device_errors()
