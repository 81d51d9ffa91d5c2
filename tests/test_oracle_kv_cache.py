"""Pins for the cache oracle: a hand-derived fixture and write/read round trips."""
import json
import os

import numpy as np

from oracle import kv_cache as ok

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_append_matches_hand_fixture():
    g = json.load(open(os.path.join(GOLDEN, "kv_append_small.json")))
    NB, H, B, A = g["num_blocks"], g["num_heads"], g["block_size"], g["head_dim"]
    new = np.array([[[100 * t + 10 * h + a + 1 for a in range(A)] for h in range(H)] for t in range(3)],
                   dtype=np.float64)
    pool = np.zeros((NB, H, B, A))
    out = ok.append_kv(pool, new, np.array(g["slot_mapping"]), B)
    assert np.array_equal(out, np.array(g["expected_pool"], dtype=np.float64))
    assert np.array_equal(pool, np.zeros_like(pool))          # input untouched


def test_append_then_gather_returns_history_and_leaves_other_slots():
    rng = np.random.default_rng(0)
    NB, H, B, A = 12, 3, 4, 5
    sentinel = -123.0
    pool = np.full((NB, H, B, A), sentinel)
    tables = [np.array([7, 2, 9]), np.array([0, 11])]
    lens = [10, 6]
    # write all positions of both sequences in an interleaved order
    rows, slots = [], []
    hist = [rng.standard_normal((n, H, A)) for n in lens]
    order = [(s, j) for j in range(10) for s in range(2) if j < lens[s]]
    for s, j in order:
        rows.append(hist[s][j])
        slots.append(ok.slot_of(tables[s], j, B))
    pool = ok.append_kv(pool, np.stack(rows), np.array(slots), B)
    for s in range(2):
        assert np.array_equal(ok.gather_sequence(pool, tables[s], lens[s], B), hist[s])
    used = {(int(tables[s][j // B]), j % B) for s in range(2) for j in range(lens[s])}
    for b in range(NB):
        for o in range(B):
            if (b, o) not in used:
                assert np.all(pool[b, :, o, :] == sentinel)


def test_slot_formula_examples():
    # block table [5, 1]: position 0 -> block 5 offset 0; position 5 with B=4 -> block 1 offset 1
    assert ok.slot_of(np.array([5, 1]), 0, 4) == 20
    assert ok.slot_of(np.array([5, 1]), 5, 4) == 5
    assert ok.slot_of(np.array([5, 1]), 3, 4) == 23
