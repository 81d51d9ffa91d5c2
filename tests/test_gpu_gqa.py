"""Grouped-query attention (fewer key/value heads than query heads; not on the
pages): query head h attends with key/value head h // (H / H_kv).  Decode rows
(all query heads of a key/value head as the rows of one tensor-core unit),
prefill chunks and mixed steps against the oracle, for groups of 2 to 32
heads and for one key/value head (MQA)."""
import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = [(8, 2), (8, 1), (12, 4), (16, 2), (6, 6)]


@pytest.mark.parametrize("H,Hkv", SHAPES)
def test_gqa_decode_prefill_and_mixed(native_lib, H, Hkv):
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    # decode rows around split and block edges, prefill chunks around tile edges, one mixed step
    p = [0, 1, 511, 512, 2047, 4100, 300, 0, 129]
    q = [1, 1, 1, 1, 1, 1, 200, 129, 300]
    b = W.make_batch(p, q, num_heads=H, head_dim=128, block_size=16, dtype="bf16", seed=200 + H + Hkv,
                     num_kv_heads=Hkv)
    got = to_np(DeviceStep(b).run())
    assert_tolerance(got, oracle_packed(b))


@pytest.mark.parametrize("Hkv", [8, 4, 1])
def test_gqa_decode_full_size_every_row(native_lib, Hkv):
    """The decode workload with 32 query heads over 8, 4 and 1 key/value heads
    (groups of 4 on the CUDA-core path; 8 and 32 on the tensor-core path): 256
    sequences, contexts 512-4096; every sequence on 4 query heads against the
    oracle."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_rows, to_np
    b = W.decode_step(num_kv_heads=Hkv)
    st = DeviceStep(b, source="device")
    out = to_np(st.run())
    assert np.all(np.isfinite(out))
    rng = np.random.default_rng(3)
    got, exp = [], []
    for s in range(b.num_seqs):
        heads = sorted(rng.choice(32, 4, replace=False).tolist())
        exp.append(oracle_rows(b, s, heads)[0])
        got.append(out[int(b.cu_seqlens_q[s])][heads])
    assert_tolerance(np.stack(got), np.stack(exp))


@pytest.mark.parametrize("H,Hkv,B", [(64, 2, 16), (16, 2, 32), (40, 8, 64), (16, 1, 128), (96, 4, 16),
                                     (4, 2, 32), (16, 4, 64)])
def test_gqa_decode_groups_and_block_sizes(native_lib, H, Hkv, B):
    """Grouped decode rows: groups of 5 to 32 query heads (the tensor-core
    path; 32 fills its softmax warp) and of 2 and 4 (the CUDA-core path), every
    block size, contexts around the 128-key tile, the 512-key split and block
    edges, up to 9 splits per row; twice in a row, so the split tickets are
    back at zero between calls."""
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    ctx = [1, 2, 127, 128, 129, 511, 512, 513, 1025, 2300, 4097]
    b = W.make_batch([c - 1 for c in ctx], [1] * len(ctx), num_heads=H, head_dim=128, block_size=B,
                     dtype="bf16", seed=300 + H + B, num_kv_heads=Hkv)
    st = DeviceStep(b)
    exp = oracle_packed(b)
    first = st.run().clone()
    assert_tolerance(to_np(first), exp)
    st.attend()
    torch.cuda.synchronize()
    assert torch.equal(st.out.view(torch.int16), first.view(torch.int16))


def test_gqa_head_groups_do_not_leak(native_lib):
    """Changing key/value head 0 changes exactly the outputs of query heads in
    group 0, bit for bit everywhere else."""
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep
    H, Hkv = 8, 2
    b = W.make_batch([700, 0, 40], [1, 150, 1], num_heads=H, head_dim=128, block_size=16, dtype="bf16",
                     seed=77, num_kv_heads=Hkv)
    st = DeviceStep(b)
    base = st.run().clone()
    st.cache.k[:, 0] = st.cache.k[:, 0] * -1.5
    st.attend()
    api.cb_check_device_errors()
    changed = [not torch.equal(st.out[:, h].view(torch.int16), base[:, h].view(torch.int16)) for h in range(H)]
    assert changed == [h // (H // Hkv) == 0 for h in range(H)]


@pytest.mark.parametrize("H,Hkv", [(8, 2), (32, 8)])
def test_gqa_planned_equals_unplanned_bitwise(native_lib, H, Hkv):
    """One grouped-query plan (cb_plan_step_gqa) serves every layer of a step
    and gives the bits of cb_ragged_attention_gqa, decode rows, prefill
    chunks and a chunk cut into KV segments included."""
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep
    p, q = [513, 0, 2000, 77, 6000, 300], [1, 129, 1, 1, 300, 40]
    layers = [DeviceStep(W.make_batch(p, q, num_heads=H, head_dim=128, block_size=16, dtype="bf16",
                                      seed=230, layer=layer, num_kv_heads=Hkv)) for layer in range(2)]
    ref = []
    for st in layers:
        st.append()
        st.attend()
        ref.append(st.out.clone())
    api.cb_check_device_errors()
    st0 = layers[0]
    b = st0.b
    api.cb_plan_step(st0.cache, st0.cu, st0.ctx, num_tokens=b.T, max_blocks_per_seq=b.block_tables.shape[1],
                     max_q_len=b.max_q_len, max_context_len=b.max_context_len, workspace=st0.ws, num_q_heads=H)
    for st in layers:
        st.out.zero_()
        api.cb_ragged_attention_planned(st.q, st.cache, st0.cu, st0.ctx, st0.bt, max_q_len=b.max_q_len,
                                        max_context_len=b.max_context_len, scale=st.scale, out=st.out,
                                        workspace=st0.ws)
    api.cb_check_device_errors()
    for st, r in zip(layers, ref):
        assert torch.equal(st.out.view(torch.int16), r.view(torch.int16))


def test_gqa_plan_refuses_other_head_counts(native_lib):
    """A plan made for one number of query heads serves no call with another."""
    from continuous_batching_ragged_gb300 import api, native
    from gpu_harness import DeviceStep
    st = DeviceStep(W.make_batch([40, 0], [1, 50], num_heads=8, head_dim=128, block_size=16, dtype="bf16",
                                 seed=231, num_kv_heads=2))
    b = st.b
    api.cb_plan_step(st.cache, st.cu, st.ctx, num_tokens=b.T, max_blocks_per_seq=b.block_tables.shape[1],
                     max_q_len=b.max_q_len, max_context_len=b.max_context_len, workspace=st.ws, num_q_heads=4)
    with pytest.raises(native.CBError, match="other metadata"):
        api.cb_ragged_attention_planned(st.q, st.cache, st.cu, st.ctx, st.bt, max_q_len=b.max_q_len,
                                        max_context_len=b.max_context_len, scale=st.scale, out=st.out,
                                        workspace=st.ws)
