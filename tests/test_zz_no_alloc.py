"""cb_decode_attention_noalloc, called through the C ABI, against cb_ragged_attention
and the oracle.

Some callers cannot allocate device memory: an op inside a host framework
whose caching allocator (or a KV pool sized to fill the GPU) already owns all
device memory, behind a plugin interface that hands over only the op's inputs
and outputs, has neither cudaMalloc nor a workspace to lend.  For them the
library offers a decode entry point whose split-KV scratch is a fixed array
reserved in device memory.  It must return the same rows as the workspace-based
entry point and the oracle, call after call (the array keeps the previous
call's contents, so the second call checks that whatever must start at zero is
cleared), and a call must leave the device's free memory unchanged.

This file is collected last; it must pass both alone in a fresh process and
after every other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import native
from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(lib, st, out):
    b = st.b
    c = st.cache.c_struct()
    return lib.cb_decode_attention_noalloc(
        st.q.data_ptr(), ctypes.byref(c), st.cu.data_ptr(), st.ctx.data_ptr(), st.bt.data_ptr(),
        b.num_seqs, b.T, b.max_blocks_per_seq, b.max_context_len, st.scale, out.data_ptr(),
        int(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", ["bf16_decode", "f32_decode"])
def test_noalloc_matches_workspace_entry_point_twice(native_lib, case):
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep, assert_tolerance, fill_sentinel, oracle_rows, to_np
    heads = None
    if case == "bf16_decode":
        # contexts 512..4096: up to 9 splits per row, so the ticketed merge runs
        b = W.decode_step(num_seqs=64, seed=5)
        st = DeviceStep(b, source="device")
        heads = [0, 9, 22, 31]                    # every row on 4 of the 32 heads against the oracle
    else:
        b = W.make_batch([0, 6, 700, 1500, 63], [1] * 5, num_heads=4, head_dim=64, block_size=4,
                         dtype="f32", seed=9)
        st = DeviceStep(b)
    ref = to_np(st.run())
    exp = np.concatenate([oracle_rows(b, s, heads) for s in range(b.num_seqs)])
    sel = slice(None) if heads is None else heads
    assert api.cb_attention_workspace_size(st.cache, b.num_seqs, b.T, b.max_context_len) \
        <= native.NOALLOC_SCRATCH_BYTES
    outs = [torch.empty_like(st.out) for _ in range(2)]
    for i, out in enumerate(outs):
        fill_sentinel(out)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        status = _noalloc(native_lib, st, out)
        assert status == native.CB_OK, native_lib.cb_last_error()
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if i == 1:
            # the first call may load the library's device image (which holds
            # the static array); the second must leave free memory unchanged
            assert free_after == free_before, (free_before, free_after)
        api.cb_check_device_errors()
        got = to_np(out)
        assert_tolerance(got, ref, max_abs=2e-2, mean_abs=2e-3)
        assert_tolerance(got[:, sel], exp)


def test_noalloc_rejects_steps_beyond_its_scratch(native_lib):
    """A step whose split-KV scratch exceeds the static array is refused on the
    host before any launch.  Every argument is consistent (a [64, 2048] block
    table for contexts up to 32768), so nothing could read out of bounds even
    if the check were missing."""
    from continuous_batching_ragged_gb300 import api
    S, H, A, B, max_ctx = 64, 32, 128, 16, 32768
    cache = api.KVCache.empty(4, H, B, A, torch.bfloat16)
    q = torch.zeros((S, H, A), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    cu = torch.arange(S + 1, dtype=torch.int32, device="cuda")
    ctx = torch.ones(S, dtype=torch.int32, device="cuda")
    bt = torch.zeros((S, max_ctx // B), dtype=torch.int32, device="cuda")
    need = api.cb_attention_workspace_size(cache, S, S, max_ctx)
    assert need > native.NOALLOC_SCRATCH_BYTES
    c = cache.c_struct()
    status = native_lib.cb_decode_attention_noalloc(
        q.data_ptr(), ctypes.byref(c), cu.data_ptr(), ctx.data_ptr(), bt.data_ptr(), S, S,
        max_ctx // B, max_ctx, 1 / math.sqrt(A), out.data_ptr(), None)
    assert status == native.CB_ERR_INVALID
    assert b"static scratch" in native_lib.cb_last_error()
    # more query tokens than sequences: not a decode step, refused before launch
    status = native_lib.cb_decode_attention_noalloc(
        q.data_ptr(), ctypes.byref(c), cu.data_ptr(), ctx.data_ptr(), bt.data_ptr(), S - 1, S,
        max_ctx // B, 64, 1 / math.sqrt(A), out.data_ptr(), None)
    assert status == native.CB_ERR_INVALID
    assert b"decode only" in native_lib.cb_last_error()
