"""Pins for the attention oracle, each independent of the oracle's own code.

Closed forms, library routines (torch SDPA, scipy softmax), 50-digit brute
force, the worked example of the page "continuous-batching"
(zhangchitc.github.io) and the invariants the pages state.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_row_key_limits_p2_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "p2_worked_example.json")))
    lim = oa.row_key_limits(np.array(g["cu_seqlens_q"]), np.array(g["context_lens"]))
    assert lim.tolist() == g["row_key_limits"]
    # score block of each request: q_len rows x context_len columns
    cu = g["cu_seqlens_q"]
    for s, (rows, cols) in enumerate(g["score_block_shapes"]):
        assert cu[s + 1] - cu[s] == rows
        assert g["context_lens"][s] == cols
        assert lim[cu[s + 1] - 1] == cols          # the last row sees every key


def test_row_key_limits_rejects_bad_metadata():
    with pytest.raises(ValueError):
        oa.row_key_limits(np.array([0, 2]), np.array([1]))      # context < q_len
    with pytest.raises(ValueError):
        oa.row_key_limits(np.array([0, 0]), np.array([3]))      # empty sequence


def test_p2_worked_example_values_against_library_softmax():
    """D (4 new, causal), B (1 over 5 keys), C (1 over 3 keys): each row equals
    scipy's softmax over its visible scores times V."""
    g = json.load(open(os.path.join(GOLDEN, "p2_worked_example.json")))
    rng = np.random.default_rng(11)
    H, A = 2, 8
    ctx = g["context_lens"]
    k = [_rand(rng, c, H, A) for c in ctx]
    v = [_rand(rng, c, H, A) for c in ctx]
    q = _rand(rng, 6, H, A)
    scale = 1 / math.sqrt(A)
    out = oa.ragged_attention(q, np.array(g["cu_seqlens_q"]), np.array(ctx), k, v, scale)
    for t, (s, lim) in enumerate(zip([0, 0, 0, 0, 1, 2], g["row_key_limits"])):
        for h in range(H):
            w = scipy.special.softmax(scale * (k[s][:lim, h] @ q[t, h]))
            np.testing.assert_allclose(out[t, h], w @ v[s][:lim, h], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("n", [1, 5, 37])
def test_single_pass_prefill_matches_torch_sdpa(n):
    rng = np.random.default_rng(n)
    H, A = 3, 16
    q, k, v = (_rand(rng, n, H, A) for _ in range(3))
    ours = oa.attend_sequence(q, k, v, 0, 1 / math.sqrt(A))
    tq, tk, tv = (torch.from_numpy(x).permute(1, 0, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    np.testing.assert_allclose(ours, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("p,n", [(1, 1), (5, 3), (64, 17), (100, 1), (7, 40)])
def test_chunk_with_cached_prefix_matches_rows_of_single_pass_sdpa(p, n):
    """Chunked prefill reaches the single-pass result (blog, section Chunked
    prefill): rows p..p+n-1 of a causal pass over all p+n tokens."""
    rng = np.random.default_rng(1000 + p * 7 + n)
    H, A = 2, 32
    L = p + n
    q, k, v = (_rand(rng, L, H, A) for _ in range(3))
    ours = oa.attend_sequence(q[p:], k, v, p, 1 / math.sqrt(A))
    tq, tk, tv = (torch.from_numpy(x).permute(1, 0, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    np.testing.assert_allclose(ours, ref.permute(1, 0, 2).numpy()[p:], rtol=1e-11, atol=1e-12)


def test_non_default_scale_matches_sdpa_scale_argument():
    rng = np.random.default_rng(5)
    q, k, v = (_rand(rng, 9, 2, 8) for _ in range(3))
    ours = oa.attend_sequence(q[4:], k, v, 4, 0.77)
    tq, tk, tv = (torch.from_numpy(x).permute(1, 0, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=0.77)
    np.testing.assert_allclose(ours, ref.permute(1, 0, 2).numpy()[4:], rtol=1e-11, atol=1e-12)


def test_single_key_returns_its_value_exactly():
    rng = np.random.default_rng(3)
    q, k, v = (_rand(rng, 1, 4, 8) for _ in range(3))
    out = oa.attend_sequence(q, k, v, 0, 0.3)
    assert np.array_equal(out, v)


def test_equal_values_give_that_value():
    rng = np.random.default_rng(4)
    p, n, H, A = 6, 5, 2, 8
    q = _rand(rng, n, H, A)
    k = _rand(rng, p + n, H, A)
    v = np.broadcast_to(_rand(rng, 1, H, A), (p + n, H, A)).copy()
    out = oa.attend_sequence(q, k, v, p, 0.5)
    np.testing.assert_allclose(out, np.broadcast_to(v[:1], out.shape), rtol=1e-14, atol=1e-14)


def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(6)
    p, n, H, A = 3, 4, 2, 8
    q = np.zeros((n, H, A))
    k = _rand(rng, p + n, H, A)
    v = _rand(rng, p + n, H, A)
    out = oa.attend_sequence(q, k, v, p, 1.0)
    for i in range(n):
        np.testing.assert_allclose(out[i], v[:p + i + 1].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_value():
    """k_j = 40 q for one visible j: its score exceeds the rest by hundreds, so
    its weight is 1 to far below 1e-12."""
    rng = np.random.default_rng(8)
    p, n, H, A = 10, 3, 1, 16
    q = _rand(rng, n, H, A)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = 0.01 * _rand(rng, p + n, H, A)
    v = _rand(rng, p + n, H, A)
    j = 4
    for i in range(n):
        kk = k.copy()
        kk[j] = 40.0 * q[i]
        out = oa.attend_sequence(q, kk, v, p, 1.0)
        np.testing.assert_allclose(out[i], v[j], rtol=0, atol=1e-12)


def test_future_keys_have_no_effect():
    """Causal mask: changing keys/values after position p+i leaves row i as is."""
    rng = np.random.default_rng(9)
    p, n, H, A = 4, 6, 2, 8
    q, k, v = _rand(rng, n, H, A), _rand(rng, p + n, H, A), _rand(rng, p + n, H, A)
    base = oa.attend_sequence(q, k, v, p, 0.4)
    for i in range(n):
        k2, v2 = k.copy(), v.copy()
        k2[p + i + 1:] += 5.0
        v2[p + i + 1:] -= 3.0
        out = oa.attend_sequence(q, k2, v2, p, 0.4)
        assert np.array_equal(out[i], base[i])
        if i + 1 < n:
            assert not np.allclose(out[i + 1], base[i + 1])


def test_brute_force_50_digits():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(10)
    p, n, H, A = 2, 3, 2, 4
    q, k, v = _rand(rng, n, H, A), _rand(rng, p + n, H, A), _rand(rng, p + n, H, A)
    scale = 0.6
    out = oa.attend_sequence(q, k, v, p, scale)
    for i in range(n):
        for h in range(H):
            e = [mp.exp(mp.mpf(scale) * mp.fsum(mp.mpf(q[i, h, a]) * mp.mpf(k[j, h, a]) for a in range(A)))
                 for j in range(p + i + 1)]
            tot = mp.fsum(e)
            for a in range(A):
                ref = mp.fsum(e[j] * mp.mpf(v[j, h, a]) for j in range(p + i + 1)) / tot
                assert abs(float(ref) - out[i, h, a]) < 1e-13


def _packed_case(rng, p_list, n_list, H=2, A=8):
    k = [_rand(rng, p + n, H, A) for p, n in zip(p_list, n_list)]
    v = [_rand(rng, p + n, H, A) for p, n in zip(p_list, n_list)]
    q = [_rand(rng, n, H, A) for n in n_list]
    return q, k, v


def test_packed_equals_each_sequence_alone_in_any_order():
    """Ragged batching: packing sequences together changes nothing per sequence
    (blog, section Continuous batching; zhangchitc, Ragged batching)."""
    rng = np.random.default_rng(12)
    p_list, n_list = [0, 9, 3, 20, 1], [5, 1, 4, 1, 7]
    q, k, v = _packed_case(rng, p_list, n_list)
    alone = [oa.attend_sequence(q[s], k[s], v[s], p_list[s], 0.35) for s in range(5)]
    for order in ([0, 1, 2, 3, 4], [4, 2, 0, 3, 1], [3, 1, 4, 0, 2]):
        qs = np.concatenate([q[s] for s in order])
        cu = np.concatenate([[0], np.cumsum([n_list[s] for s in order])])
        ctx = np.array([p_list[s] + n_list[s] for s in order])
        out = oa.ragged_attention(qs, cu, ctx, [k[s] for s in order], [v[s] for s in order], 0.35)
        for pos, s in enumerate(order):
            assert np.array_equal(out[cu[pos]:cu[pos + 1]], alone[s])


def test_no_cross_sequence_leakage():
    rng = np.random.default_rng(13)
    p_list, n_list = [4, 0, 11], [3, 6, 1]
    q, k, v = _packed_case(rng, p_list, n_list)
    cu = np.array([0, 3, 9, 10])
    ctx = np.array([7, 6, 12])
    base = oa.ragged_attention(np.concatenate(q), cu, ctx, k, v, 0.5)
    q2 = [x.copy() for x in q]
    k2 = [x.copy() for x in k]
    v2 = [x.copy() for x in v]
    for s in (0, 2):
        q2[s] += 1.0
        k2[s] *= -2.0
        v2[s] += 7.0
    out = oa.ragged_attention(np.concatenate(q2), cu, ctx, k2, v2, 0.5)
    assert np.array_equal(out[3:9], base[3:9])
    assert not np.allclose(out[:3], base[:3])


def test_incremental_decode_equals_full_recompute():
    """KV cache (blog, section KV-cache): prefill P tokens, then decode one token
    at a time against the cached keys; each decode row equals the matching row of
    one causal pass over all tokens."""
    rng = np.random.default_rng(14)
    P, steps, H, A = 6, 5, 2, 8
    L = P + steps
    q, k, v = (_rand(rng, L, H, A) for _ in range(3))
    full = oa.attend_sequence(q, k, v, 0, 0.3)
    pre = oa.attend_sequence(q[:P], k[:P], v[:P], 0, 0.3)
    np.testing.assert_allclose(pre, full[:P], rtol=1e-13, atol=1e-14)
    for t in range(P, L):
        row = oa.attend_sequence(q[t:t + 1], k[:t + 1], v[:t + 1], t, 0.3)
        np.testing.assert_allclose(row[0], full[t], rtol=1e-13, atol=1e-14)


def test_chunked_prefill_equals_single_pass_every_split():
    rng = np.random.default_rng(15)
    n, H, A = 7, 2, 8
    q, k, v = (_rand(rng, n, H, A) for _ in range(3))
    full = oa.attend_sequence(q, k, v, 0, 0.25)
    for m in (1, 2, 3, 4, 6):       # blog example: n=7, m=4 -> chunks of 4 and 3
        got = []
        for start in range(0, n, m):
            end = min(n, start + m)
            got.append(oa.attend_sequence(q[start:end], k[:end], v[:end], start, 0.25))
        np.testing.assert_allclose(np.concatenate(got), full, rtol=1e-13, atol=1e-14)


def test_rows_per_pass_only_bounds_memory():
    rng = np.random.default_rng(16)
    q, k, v = _rand(rng, 50, 1, 8), _rand(rng, 80, 1, 8), _rand(rng, 80, 1, 8)
    a = oa.attend_sequence(q, k, v, 30, 0.5, rows_per_pass=7)
    b = oa.attend_sequence(q, k, v, 30, 0.5, rows_per_pass=256)
    np.testing.assert_allclose(a, b, rtol=1e-14, atol=1e-15)


def test_grouped_query_attention_equals_heads_with_repeated_keys_values():
    """Grouped-query attention (not on the pages; query head h reads key/value
    head h // G) is multi-head attention whose keys and values are each
    repeated for the G query heads of their group."""
    rng = np.random.default_rng(31)
    for H, H_kv in ((8, 2), (6, 3), (4, 1), (5, 5)):
        n, p, A = 5, 9, 16
        q = rng.standard_normal((n, H, A))
        k = rng.standard_normal((p + n, H_kv, A))
        v = rng.standard_normal((p + n, H_kv, A))
        got = oa.attend_sequence(q, k, v, p, 0.25)
        G = H // H_kv
        exp = oa.attend_sequence(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), p, 0.25)
        np.testing.assert_array_equal(got, exp)
        # and head h's output depends only on its own group's keys and values
        k2 = k.copy()
        k2[:, 0] += 1.0
        changed = np.any(oa.attend_sequence(q, k2, v, p, 0.25) != got, axis=(0, 2))
        assert changed.tolist() == [h // G == 0 for h in range(H)]


def test_grouped_query_attention_rejects_uneven_groups():
    q = np.zeros((1, 6, 4))
    k = np.zeros((1, 4, 4))
    with pytest.raises(ValueError):
        oa.attend_sequence(q, k, k, 0, 1.0)


def test_left_padded_real_rows_equal_unpadded_attention():
    """A left-padded chunk's real rows see exactly the unpadded chunk's keys:
    inserting pad tokens (masked) between the cache and the real tokens
    changes no real row.  Pad rows have no output."""
    from oracle import attention as oa
    rng = np.random.default_rng(8)
    p, n, pad, H, Hkv, A = 5, 7, 3, 4, 2, 16
    q = rng.standard_normal((n - pad, H, A))
    k = rng.standard_normal((p + n - pad, Hkv, A))
    v = rng.standard_normal((p + n - pad, Hkv, A))
    ref = oa.attend_sequence(q, k, v, p, 0.3)
    # the padded layout: pad rows (arbitrary values) first, pad keys at p .. p+pad-1
    qp = np.concatenate([rng.standard_normal((pad, H, A)) * 50, q])
    kp = np.concatenate([k[:p], rng.standard_normal((pad, Hkv, A)) * 50, k[p:]])
    vp = np.concatenate([v[:p], rng.standard_normal((pad, Hkv, A)) * 50, v[p:]])
    got = oa.attend_left_padded(qp, kp, vp, p, pad, 0.3)
    assert np.all(np.isnan(got[:pad]))
    np.testing.assert_allclose(got[pad:], ref, rtol=0, atol=1e-12)
    # no padding: the plain definition
    np.testing.assert_allclose(oa.attend_left_padded(q, k, v, p, 0, 0.3), ref, rtol=0, atol=1e-12)


def test_left_padded_hand_example():
    """p = 2 cached keys, a 3-row chunk with 2 pad rows: its one real row
    (chunk row 2, position 4) attends keys 0, 1 and 4 only."""
    from oracle import attention as oa
    q = np.zeros((3, 1, 2))
    q[2, 0] = [1.0, 0.0]
    k = np.array([[1.0, 0.0], [2.0, 0.0], [9.0, 0.0], [9.0, 0.0], [0.0, 0.0]])[:, None, :]
    v = np.array([[1.0, 0.0], [0.0, 1.0], [100.0, 100.0], [100.0, 100.0], [3.0, 3.0]])[:, None, :]
    got = oa.attend_left_padded(q, k, v, 2, 2, 1.0)[2, 0]
    w = np.exp(np.array([1.0, 2.0, 0.0]))
    w /= w.sum()
    exp = w[0] * v[0, 0] + w[1] * v[1, 0] + w[2] * v[4, 0]
    np.testing.assert_allclose(got, exp, rtol=0, atol=1e-14)


def test_left_padded_batch_layout():
    """workloads.left_padded: every sequence gets max(q_len) rows with the pads
    first; real rows carry the unpadded batch's q/k/v values and the history
    of a real row is the unpadded history with the pad tokens inserted at
    p .. p + pad - 1; the blog's insertion example costs (n-1)(B-1) pads."""
    from continuous_batching_ragged_gb300 import workloads as W
    b = W.make_batch([4, 0, 9], [1, 6, 2], num_heads=2, head_dim=8, block_size=4, dtype="bf16", seed=12)
    pb = W.left_padded(b)
    assert pb.q_len.tolist() == [6, 6, 6] and pb.pad_lens.tolist() == [5, 0, 4] and pb.useful_tokens == 9
    rr = W.real_rows(pb)
    for kind in (W.KIND_Q, W.KIND_K, W.KIND_V):
        assert np.array_equal(pb.packed(kind)[rr], b.packed(kind))
    for s in range(3):
        p, pad = int(b.p[s]), int(pb.pad_lens[s])
        h = pb.history(s, W.KIND_K)
        ref = b.history(s, W.KIND_K)
        assert np.array_equal(np.concatenate([h[:p], h[p + pad:]]), ref)
    ins = W.page_insertion_example(num_heads=2, head_dim=8)
    assert W.padding_tokens(ins) == 99 * 7 == int(W.left_padded(ins).pad_lens.sum())
