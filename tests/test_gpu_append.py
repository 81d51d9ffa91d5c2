"""K1: the cache after cb_append_kv equals the oracle's cache, bit for bit;
every slot not addressed keeps its sentinel."""
import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import native
from continuous_batching_ragged_gb300 import workloads as W
from oracle import kv_cache as okv

pytestmark = pytest.mark.gpu


def _check_append(b, slots=None):
    from gpu_harness import DeviceStep, device_pool_bits, value_bits
    st = DeviceStep(b, source="host")
    if slots is not None:
        st.slots = torch.from_numpy(np.asarray(slots, np.int64)).cuda()
    st.append()
    from continuous_batching_ragged_gb300 import api
    api.cb_check_device_errors()
    sm = b.slot_mapping if slots is None else np.asarray(slots, np.int64)
    for kind, pool in ((W.KIND_K, st.cache.k), (W.KIND_V, st.cache.v)):
        new_bits = value_bits(b.packed(kind), b.dtype)
        exp = okv.append_kv(st.initial_bits[kind], new_bits, sm, b.block_size)
        assert np.array_equal(device_pool_bits(pool), exp)


@pytest.mark.parametrize("dtype,H,A,B", [("bf16", 32, 128, 16), ("f32", 4, 64, 4), ("bf16", 2, 64, 8),
                                         ("f32", 3, 128, 32)])
def test_append_matches_oracle(native_lib, dtype, H, A, B):
    rng = np.random.default_rng(H * A + B)
    S = 9
    p = rng.integers(0, 70, S)
    q = rng.integers(1, 40, S)
    b = W.make_batch(p, q, num_heads=H, head_dim=A, block_size=B, dtype=dtype, seed=int(B),
                     num_blocks=int(sum(np.ceil((p + q) / B))) + 5)
    _check_append(b)


def test_append_mixed_step_full_size(native_lib):
    """The mixed step's 2048 appended tokens (64 decode + 661/661/662 prefill),
    in the launch configuration the bench times: the K and V bits of every
    appended (token, head) row, read back at its slot, equal the host
    generator's values, and every other slot of both pools is unchanged."""
    b = W.mixed_step()
    from gpu_harness import DeviceStep, value_bits
    from continuous_batching_ragged_gb300 import api
    st = DeviceStep(b, source="device")
    slots = torch.from_numpy(b.slot_mapping).cuda()
    blk, off = slots // b.block_size, slots % b.block_size
    pools = ((W.KIND_K, st.cache.k), (W.KIND_V, st.cache.v))
    befores = [pool.view(torch.int16).clone() for _, pool in pools]
    st.append()
    api.cb_check_device_errors()
    for (kind, pool), before in zip(pools, befores):
        after = pool.view(torch.int16)
        rows = after[blk, :, off, :].cpu().numpy().view(np.uint16)
        assert np.array_equal(rows, value_bits(b.packed(kind), "bf16"))
        after_rest = after.clone()
        after_rest[blk, :, off, :] = 0
        before[blk, :, off, :] = 0
        assert torch.equal(after_rest, before)
        del after_rest


def test_append_skips_negative_slots(native_lib):
    b = W.make_batch([0, 3], [2, 1], num_heads=2, head_dim=64, block_size=4, dtype="f32", seed=5,
                     num_blocks=4)
    sm = b.slot_mapping.copy()
    sm[1] = -1
    _check_append(b, sm)


def test_append_out_of_pool_slot_is_reported_not_written(native_lib):
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep, device_pool_bits
    b = W.make_batch([0], [3], num_heads=2, head_dim=64, block_size=4, dtype="f32", seed=6, num_blocks=2)
    st = DeviceStep(b, source="host")
    before = [device_pool_bits(st.cache.k), device_pool_bits(st.cache.v)]
    st.slots = torch.tensor([8, 100, 2 ** 40], dtype=torch.int64, device="cuda")   # pool has 8 slots
    st.append()
    with pytest.raises(native.CBError) as e:
        api.cb_check_device_errors()
    assert e.value.status == native.CB_ERR_BOUNDS
    assert np.array_equal(device_pool_bits(st.cache.k), before[0])
    assert np.array_equal(device_pool_bits(st.cache.v), before[1])
    api.cb_check_device_errors()          # the word was cleared by the previous check
