"""The step plan: the work lists that the GPU builds from a step's metadata and
that the persistent decode and prefill kernels claim.  A step's output must
depend only on the step's inputs: never on what the workspace held before the
call, and never on which CTA claimed which unit.  The batches cover each route
through cb_ragged_attention (decode only, one prefill chunk alone, mixed) and
the plan's special cases (exactly one prefill item; several sorted by cost;
query pairs cut into KV segments, whose arrival tickets live in the workspace)."""
import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    "decode_only": ([513, 0, 2000, 77, 1023], [1, 1, 1, 1, 1]),
    "prefill_only": ([300], [450]),
    "mixed_one_prefill_item": ([100, 700, 0, 40], [1, 1, 200, 1]),
    "mixed_sorted_items": ([0, 300, 5, 40, 1000, 2], [600, 1, 77, 1, 129, 257]),
    "prefill_kv_segments": ([6000, 40, 2500], [512, 1, 300]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_output_independent_of_workspace_contents(native_lib, case):
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep, assert_tolerance, fill_sentinel, oracle_packed, to_np
    p, q = CASES[case]
    b = W.make_batch(p, q, num_heads=4, head_dim=128, block_size=16, dtype="bf16", seed=83)
    st = DeviceStep(b)
    st.append()
    st.ws.zero_()
    st.attend()
    api.cb_check_device_errors()
    ref = st.out.clone()
    assert_tolerance(to_np(ref), oracle_packed(b))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    for _ in range(25):
        st.ws.random_(0, 256, generator=gen)
        fill_sentinel(st.out)
        st.attend()
        api.cb_check_device_errors()
        assert torch.equal(st.out.view(torch.int16), ref.view(torch.int16))


def test_repeated_steps_reuse_one_workspace(native_lib):
    """Steps of different shapes back to back on one workspace, no host sync in
    between: each step's list is built and consumed before the next overwrites it."""
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import DeviceStep, to_np
    steps = [DeviceStep(W.make_batch(p, q, num_heads=4, head_dim=128, block_size=16, dtype="bf16",
                                     seed=90 + i))
             for i, (p, q) in enumerate(CASES[c] for c in sorted(CASES))]
    refs = []
    for st in steps:
        refs.append(to_np(st.run()).copy())
    need = max(st.ws.numel() for st in steps)
    shared = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for _ in range(10):
        for st in steps:
            st.ws = shared
            st.attend()
    api.cb_check_device_errors()
    for st, r in zip(steps, refs):
        np.testing.assert_array_equal(to_np(st.out), r)
