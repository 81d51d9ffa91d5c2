"""The device generator reproduces the host generator bit for bit."""
import numpy as np
import pytest
import torch

from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_synth_tokens_bit_exact(native_lib, dtype):
    from continuous_batching_ragged_gb300 import api
    from gpu_harness import TORCH_DT, value_bits
    rng = np.random.default_rng(1)
    n, H, A = 97, 4, 64
    seq = rng.integers(0, 2 ** 31, n).astype(np.int64)
    pos = rng.integers(0, 2 ** 20, n).astype(np.int32)
    out = torch.empty((n, H, A), dtype=TORCH_DT[dtype], device="cuda")
    api.cb_synth_tokens(out, 0x1234_5678_9ABC, W.KIND_V, 7, torch.from_numpy(seq).cuda(),
                        torch.from_numpy(pos).cuda())
    got = out.view(torch.int16 if dtype == "bf16" else torch.int32).cpu().numpy()
    for i in range(n):
        exp = W.token_values(0x1234_5678_9ABC, W.KIND_V, 7, int(seq[i]), [pos[i]], range(H), A, dtype)[0]
        assert np.array_equal(got[i].view(np.uint16 if dtype == "bf16" else np.uint32),
                              value_bits(exp, dtype))


def test_synth_fill_cache_matches_host_pool(native_lib):
    from gpu_harness import DeviceStep, device_pool_bits, host_pool_bits
    b = W.make_batch([5, 0, 33, 16], [1, 3, 1, 2], num_heads=2, head_dim=128, block_size=16,
                     dtype="bf16", seed=3, num_blocks=12)
    st = DeviceStep(b, source="device")
    torch.cuda.synchronize()
    for kind, pool in ((W.KIND_K, st.cache.k), (W.KIND_V, st.cache.v)):
        got = device_pool_bits(pool)
        exp = host_pool_bits(b, kind)
        assert np.array_equal(got, exp)
