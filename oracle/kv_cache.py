"""Block-paged KV cache writes and reads (oracle; test infrastructure only).

Page "continuous-batching" (zhangchitc.github.io), section "Inside the
kernel": a step first stores every new key and value row under the request
it belongs to; attention then gathers all of that request's keys and values
from the cache, one block after another.  hassanahmed.net, "How Continuous Batching Speeds Up LLM Serving",
paragraph on PagedAttention: the cache is stored in fixed-size blocks.

Pool layout: one array per K and V, [num_blocks, H, B, A].  A token with
cache slot s = block_id * B + offset occupies pool[block_id, :, offset, :].
Logical token position j of a sequence lives in block block_table[j // B] at
offset j % B.
"""
from __future__ import annotations

import numpy as np


def slot_of(block_table: np.ndarray, position: int, block_size: int) -> int:
    """Cache slot of a sequence's token at ``position``."""
    return int(block_table[position // block_size]) * block_size + position % block_size


def append_kv(pool: np.ndarray, new: np.ndarray, slot_mapping: np.ndarray,
              block_size: int) -> np.ndarray:
    """Return a copy of ``pool`` [NB, H, B, A] with row t of ``new`` [T, H, A]
    written at slot_mapping[t]; a negative slot means the row is skipped."""
    out = np.array(pool, copy=True)
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        out[blk, :, off, :] = new[t]
    return out


def gather_sequence(pool: np.ndarray, block_table: np.ndarray, length: int,
                    block_size: int) -> np.ndarray:
    """Read positions 0..length-1 of one sequence back out of ``pool``: [length, H, A]."""
    rows = []
    for j in range(length):
        blk = int(block_table[j // block_size])
        rows.append(pool[blk, :, j % block_size, :])
    return np.stack(rows) if rows else np.zeros((0,) + pool.shape[1:2] + pool.shape[3:], pool.dtype)
