"""The seeded generator: Philox known-answer vectors, exactness and statistics."""
import json
import os

import numpy as np

from continuous_batching_ragged_gb300 import workloads as w

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    g = json.load(open(os.path.join(GOLDEN, "philox4x32_10_kat.json")))
    for vec in g["vectors"]:
        c = [int(x, 16) for x in vec["counter"]]
        k = [int(x, 16) for x in vec["key"]]
        out = w.philox4x32_10(*c, *k)
        assert [int(x) for x in out] == [int(x, 16) for x in vec["output"]]


def test_irwin_hall_moments_and_range():
    x = w.token_values(123, w.KIND_K, 0, 5, np.arange(2048), range(8), 128, "f32")
    assert abs(float(x.mean())) < 5e-3
    assert abs(float(x.std()) - 1.0) < 5e-3
    assert float(np.abs(x).max()) <= 4.0 * np.sqrt(1.5) + 1e-6


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is halfway between bf16 1.0 and 1.0078125 -> even (1.0)
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], dtype=np.float32)
    r = w.round_to_bf16(x)
    assert r.tolist() == [1.0, 1.015625, -2.5, 0.0]
    import torch
    t = torch.from_numpy(np.random.default_rng(0).standard_normal(4096).astype(np.float32))
    assert np.array_equal(w.round_to_bf16(t.numpy()), t.to(torch.bfloat16).float().numpy())


def test_values_independent_of_packing():
    b = w.make_batch([3, 0], [2, 4], num_heads=2, head_dim=8, block_size=4, dtype="bf16", seed=9)
    q = b.packed(w.KIND_K)
    h0 = b.history(0, w.KIND_K)
    h1 = b.history(1, w.KIND_K)
    assert np.array_equal(q[0:2], h0[3:5])
    assert np.array_equal(q[2:6], h1[0:4])


def test_batch_metadata_shapes():
    b = w.tiny_fp32()
    assert b.cu_seqlens_q.tolist() == [0, 4, 5, 6]
    assert b.context_lens.tolist() == [4, 8, 13]
    assert b.T == 6
    sm = b.slot_mapping
    assert len(set(sm.tolist())) == 6
    m = w.mixed_step()
    assert m.T == 2048 and m.num_seqs == 67
    assert m.q_len[-3:].tolist() == [661, 661, 662] and m.p[-3:].tolist() == [0, 1024, 2048]
    d = w.decode_step(num_seqs=16)
    assert np.all((d.p >= 512) & (d.p <= 4096))


def test_padding_count_matches_the_blog_example():
    """Blog 'Continuous batching from first principles', section 'Continuous
    batching': B=8, n=100 -> (n-1)(B-1) = 693 padding tokens."""
    b = w.page_insertion_example()
    assert b.T == 7 + 100
    assert w.padding_tokens(b) == 693 == (100 - 1) * (8 - 1)
    pb = w.left_padded(b)
    assert pb.T == 8 * 100 and pb.T - b.T == 693 == int(pb.pad_lens.sum())
    # pads come first in each chunk, after the cached prefix; the real rows follow
    assert np.array_equal(pb.context_lens - pb.q_len, b.p)
    assert np.array_equal(pb.context_lens[:-1], b.p[:-1] + 100)
    assert pb.pad_lens.tolist() == [99] * 7 + [0]


def test_compiled_generator_equals_numpy_bitwise():
    """The compiled host generator (used for the oracle's large inputs) gives
    the numpy definition's bits, over seeds above 2^32, every kind, layers,
    large sequence ids and positions, scattered heads, both dtypes."""
    assert w._values_lib() is not None, "gcc should build hostgen/token_values.c"
    rng = np.random.default_rng(17)
    for seed, kind, layer, seq, dtype in [(0, 0, 0, 0, "bf16"), (2 ** 40 + 12345, 1, 31, 1999, "bf16"),
                                          (0xFFFF_FFFF_FFFF, 2, 65535, 2 ** 31 + 7, "f32"),
                                          (7, 1, 3, 123456, "f32")]:
        pos = np.concatenate([np.arange(40), rng.integers(0, 2 ** 32 - 1, 24)])
        heads = [0, 5, 31, 1000]
        a = w.token_values_numpy(seed, kind, layer, seq, pos, heads, 128, dtype)
        b = w.token_values(seed, kind, layer, seq, pos, heads, 128, dtype)
        assert a.shape == b.shape == (64, 4, 128)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # head_dim 64 and an empty request
    a = w.token_values_numpy(3, 2, 1, 9, np.arange(5), range(4), 64, "f32")
    assert np.array_equal(a.view(np.uint32), w.token_values(3, 2, 1, 9, np.arange(5), range(4), 64, "f32").view(np.uint32))
    assert w.token_values(3, 2, 1, 9, np.arange(0), range(4), 64, "f32").shape == (0, 4, 64)


def test_drift_shapes_scores_only_through_q_and_k():
    """A drifted batch adds q_shift * u to every query and k_slope * j * u to
    the key at position j (u = ones / sqrt(A)), rounded to the dtype; values
    are untouched and the undrifted batch is the plain generator."""
    plain = w.make_batch([10], [3], num_heads=2, head_dim=128, block_size=16, dtype="f32", seed=4)
    drift = w.make_batch([10], [3], num_heads=2, head_dim=128, block_size=16, dtype="f32", seed=4,
                         drift=(4.0, 0.5))
    u = 1 / np.sqrt(128)
    np.testing.assert_allclose(drift.history(0, w.KIND_K) - plain.history(0, w.KIND_K),
                               (0.5 * np.arange(13) * u)[:, None, None] * np.ones((1, 2, 128)), atol=1e-5)
    np.testing.assert_allclose(drift.packed(w.KIND_Q) - plain.packed(w.KIND_Q), 4.0 * u, atol=1e-6)
    assert np.array_equal(drift.history(0, w.KIND_V), plain.history(0, w.KIND_V))
    bf = w.make_batch([10], [3], num_heads=2, head_dim=128, block_size=16, dtype="bf16", seed=4, drift=(4.0, 0.5))
    k = bf.history(0, w.KIND_K)
    assert np.array_equal(k, w.round_to_bf16(k))
