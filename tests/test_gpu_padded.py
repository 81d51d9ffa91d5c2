"""The padded baseline: a left-padded rectangular batch through the kernels.

Hugging Face blog "Continuous batching from first principles", section
"Continuous batching": before ragged batching, a batch is a rectangle whose
shorter sequences are padded on the left and masked; inserting an n-token
prompt into B decoding sequences costs (n - 1)(B - 1) pad tokens.
cb_padded_attention runs such a batch through the same kernels at its full
padded cost; its real rows must equal the ragged batch's (the oracle), and
its pad rows are never written.
"""
import math

import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import native
from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check_padded(b, heads=None, source="host", literal=False):
    from gpu_harness import DeviceStep, assert_tolerance, oracle_rows, to_np
    pb = W.left_padded(b)
    st = DeviceStep(pb, source=source)
    out = to_np(st.run())
    rr = W.real_rows(pb)
    pad_rows = np.setdiff1d(np.arange(pb.T), rr)
    assert np.all(np.isnan(out[pad_rows])), "pad rows must not be written"
    sel = slice(None) if heads is None else heads
    got = out[rr][:, sel]
    exp = np.concatenate([oracle_rows(b, s, heads) for s in range(b.num_seqs)])
    assert_tolerance(got, exp)
    if literal:
        # the oracle's literal masked definition of each padded chunk agrees
        from oracle import attention as oa
        for s in range(pb.num_seqs):
            hs = list(range(pb.num_heads)) if heads is None else heads
            kvh = [h // (pb.num_heads // pb.kv_heads) for h in hs]
            p, n = int(pb.p[s]), int(pb.q_len[s])
            ref = oa.attend_left_padded(pb.values(W.KIND_Q, s, np.arange(p, p + n), hs),
                                        pb.history(s, W.KIND_K, heads=kvh), pb.history(s, W.KIND_V, heads=kvh),
                                        p, int(pb.pad_lens[s]), 1 / math.sqrt(pb.head_dim))
            cu = pb.cu_seqlens_q
            pad = int(pb.pad_lens[s])
            assert_tolerance(out[cu[s] + pad:cu[s + 1]][:, sel], ref[pad:])
    return st, out


@pytest.mark.parametrize("B", [16, 64])
def test_padded_small_batch_matches_oracle(native_lib, B):
    """Decode rows and chunks of 37, 130 and 300 rows padded to 300: pads in
    the middle of long histories, pad keys spanning several KV tiles and a
    tile boundary, a sequence with no padding."""
    b = W.make_batch([0, 300, 5, 1000, 40], [37, 1, 130, 300, 1], num_heads=4, head_dim=128, block_size=B,
                     dtype="bf16", seed=160 + B)
    _check_padded(b, literal=True)


def test_padded_insertion_example_full_size(native_lib):
    """The blog's insertion example at the Llama-2-7B attention shape: 7
    sequences decoding over 512 cached tokens plus a new 100-token prompt,
    padded to 8 x 100 (693 pad tokens); every real row on all 32 heads."""
    b = W.page_insertion_example()
    pb = W.left_padded(b)
    assert int(pb.pad_lens.sum()) == 693
    _check_padded(b)


def test_padded_mixed_step_full_size(native_lib):
    """The mixed step (64 decode rows and chunks of 661/661/662) padded to
    67 x 662 rows, inputs generated on the device: every real row on 2 heads."""
    _check_padded(W.mixed_step(), heads=[3, 28], source="device")


def test_padded_without_pads_equals_ragged_bitwise(native_lib):
    """pad_lens all zero: the same plan and kernels as cb_ragged_attention."""
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep
    b = W.make_batch([0, 300, 5], [37, 1, 130], num_heads=4, head_dim=128, block_size=16, dtype="bf16", seed=170)
    st = DeviceStep(b)
    ref = st.run().clone()
    zeros = torch.zeros(b.num_seqs, dtype=torch.int32, device="cuda")
    out = torch.empty_like(ref)
    api.cb_padded_attention(st.q, st.cache, st.cu, st.ctx, st.bt, zeros, max_q_len=b.max_q_len,
                            max_context_len=b.max_context_len, scale=st.scale, out=out, workspace=st.ws)
    api.cb_check_device_errors()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_padded_bad_pad_counts_are_reported(native_lib):
    """A pad count >= q_len (no real row) or < 0 is refused on the device:
    the sequence is left out and CB_ERR_INVALID reported; the next call runs."""
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep
    b = W.make_batch([10, 0], [4, 6], num_heads=2, head_dim=128, block_size=16, dtype="bf16", seed=171)
    pb = W.left_padded(b)
    st = DeviceStep(pb)
    st.run()
    for bad in ([6, 0], [-1, 0], [2, 6]):
        st.pads.copy_(torch.tensor(bad, dtype=torch.int32))
        st.attend()
        with pytest.raises(native.CBError) as e:
            api.cb_check_device_errors()
        assert e.value.status == native.CB_ERR_INVALID
    st.pads.copy_(torch.from_numpy(pb.pad_lens))
    st.attend()
    api.cb_check_device_errors()
