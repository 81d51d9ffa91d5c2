"""Test-side staging of a RaggedBatch on the GPU and its oracle counterpart.

Inputs reach the device either from the host generator (small cases) or from
the device generator of cb_synth.h (full-size cases); the oracle always
recomputes its inputs on the host from the same seeded definition.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from continuous_batching_ragged_gb300 import api
from continuous_batching_ragged_gb300 import workloads as W
from oracle import attention as oa

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}
BF16_NAN = 0x7FC1            # sentinel for never-written bf16 pool slots
F32_NAN = 0x7FC00001

# Tolerance stated for bf16 outputs with fp32 accumulation.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


_INT_VIEW = {torch.bfloat16: torch.int16, torch.float32: torch.int32}
_NP_INT = {"bf16": np.int16, "f32": np.int32}


def value_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Bit patterns of dtype-representable fp32 values (uint16 for bf16, uint32 for f32)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16) if dtype == "bf16" else u.copy()


def host_pool_bits(b: W.RaggedBatch, kind: int) -> np.ndarray:
    """Initial pool bits: each sequence's cached prefix at its slots, sentinel NaN elsewhere."""
    sent = BF16_NAN if b.dtype == "bf16" else F32_NAN
    dt = np.uint16 if b.dtype == "bf16" else np.uint32
    bits = np.full((b.num_blocks, b.kv_heads, b.block_size, b.head_dim), sent, dtype=dt)
    for s in range(b.num_seqs):
        ps = int(b.p[s])
        if ps:
            pos = np.arange(ps)
            vals = value_bits(b.history(s, kind, upto=ps), b.dtype)
            bits[b.block_tables[s, pos // b.block_size], :, pos % b.block_size, :] = vals
    return bits


def device_pool_bits(t: torch.Tensor) -> np.ndarray:
    v = t.view(_INT_VIEW[t.dtype]).cpu().numpy()
    return v.view(np.uint16) if t.dtype == torch.bfloat16 else v.view(np.uint32)


def dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(TORCH_DT[dtype]).cuda()


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def fill_sentinel(t: torch.Tensor) -> None:
    if t.dtype == torch.bfloat16:
        t.view(torch.int16).fill_(BF16_NAN)
    else:
        t.view(torch.int32).fill_(F32_NAN)


class DeviceStep:
    """One packed step staged on the GPU: cache, this step's Q/K/V, metadata."""

    def __init__(self, b: W.RaggedBatch, source: str = "host", cache: api.KVCache = None):
        self.b = b
        dt = TORCH_DT[b.dtype]
        if cache is None:
            cache = api.KVCache.empty(b.num_blocks, b.kv_heads, b.block_size, b.head_dim, dt)
            fill_sentinel(cache.k)
            fill_sentinel(cache.v)
            self._prefill_cache(cache, source)
        self.cache = cache
        T = b.T
        if source == "host":
            self.q = dev(b.packed(W.KIND_Q), b.dtype)
            self.k_new = dev(b.packed(W.KIND_K), b.dtype)
            self.v_new = dev(b.packed(W.KIND_V), b.dtype)
        else:
            seq_rows = np.repeat(b.seq_ids, b.q_len)
            pos = np.concatenate([b.gen_positions(s, np.arange(b.p[s], b.p[s] + b.q_len[s]))
                                  for s in range(b.num_seqs)])
            sid = torch.from_numpy(seq_rows.astype(np.int64)).cuda()
            ps = torch.from_numpy(pos.astype(np.int32)).cuda()
            self.q, self.k_new, self.v_new = (torch.empty((T, b.heads_of(kind), b.head_dim), dtype=dt, device="cuda")
                                              for kind in (W.KIND_Q, W.KIND_K, W.KIND_V))
            for kind, t in ((W.KIND_Q, self.q), (W.KIND_K, self.k_new), (W.KIND_V, self.v_new)):
                api.cb_synth_tokens(t, b.seed, kind, b.layer, sid, ps)
        self.cu = torch.from_numpy(b.cu_seqlens_q).cuda()
        self.ctx = torch.from_numpy(b.context_lens).cuda()
        self.bt = torch.from_numpy(b.block_tables).cuda()
        self.slots = torch.from_numpy(b.slot_mapping).cuda()
        self.out = torch.empty_like(self.q)
        fill_sentinel(self.out)
        self.grouped = b.num_heads != b.kv_heads
        self.pads = None if b.pad_lens is None else torch.from_numpy(b.pad_lens.astype(np.int32)).cuda()
        ws = (api.cb_attention_workspace_size_gqa(self.cache, b.num_heads, b.num_seqs, T, b.max_context_len)
              if self.grouped else api.cb_attention_workspace_size(self.cache, b.num_seqs, T, b.max_context_len))
        self.ws = torch.empty(ws, dtype=torch.uint8, device="cuda")
        self.scale = 1.0 / math.sqrt(b.head_dim)

    def _prefill_cache(self, cache, source):
        b = self.b
        if source == "host":
            self.initial_bits = {}
            for kind, pool in ((W.KIND_K, cache.k), (W.KIND_V, cache.v)):
                bits = host_pool_bits(b, kind)
                self.initial_bits[kind] = bits
                pool.view(_INT_VIEW[pool.dtype]).copy_(torch.from_numpy(bits.view(_NP_INT[b.dtype])))
        elif int(b.p.max()) > 0:
            sid = torch.from_numpy(b.seq_ids).cuda()
            pl = torch.from_numpy(b.p.astype(np.int32)).cuda()
            bt = torch.from_numpy(b.block_tables).cuda()
            for kind, pool in ((W.KIND_K, cache.k), (W.KIND_V, cache.v)):
                api.cb_synth_fill_cache(pool, b.seed, kind, b.layer, sid, pl, bt, int(b.p.max()))

    def append(self):
        api.cb_append_kv(self.k_new, self.v_new, self.slots, self.cache)

    def attend(self):
        b = self.b
        kw = dict(max_q_len=b.max_q_len, max_context_len=b.max_context_len, scale=self.scale, out=self.out,
                  workspace=self.ws)
        if self.pads is not None:
            api.cb_padded_attention(self.q, self.cache, self.cu, self.ctx, self.bt, self.pads, **kw)
        else:
            fn = api.cb_ragged_attention_gqa if self.grouped else api.cb_ragged_attention
            fn(self.q, self.cache, self.cu, self.ctx, self.bt, **kw)

    def run(self):
        self.append()
        self.attend()
        api.cb_check_device_errors()
        return self.out


def oracle_rows(b: W.RaggedBatch, s: int, heads=None, rows=None) -> np.ndarray:
    """Oracle output of sequence s, [q_len (or len(rows)), len(heads), A] fp64."""
    if heads is None:
        heads = list(range(b.num_heads))
    p, n = int(b.p[s]), int(b.q_len[s])
    pos = np.arange(p, p + n) if rows is None else p + np.asarray(rows)
    c = int(b.context_lens[s]) if rows is None else int(p + np.max(rows) + 1)
    q = b.values(W.KIND_Q, s, pos, heads)
    # the key/value head of each query head (one per query head: the oracle then needs no grouping)
    kvh = [h // (b.num_heads // b.kv_heads) for h in heads]
    k = b.values(W.KIND_K, s, np.arange(c), kvh)
    v = b.values(W.KIND_V, s, np.arange(c), kvh)
    if rows is None:
        return oa.attend_sequence(q, k, v, p, 1.0 / math.sqrt(b.head_dim))
    # selected rows: row r sees keys 0..p+r; run each as a one-row chunk at its own offset
    out = np.empty((len(pos), len(heads), b.head_dim))
    for i, r in enumerate(rows):
        out[i] = oa.attend_sequence(q[i:i + 1], k[:p + r + 1], v[:p + r + 1], p + r,
                                    1.0 / math.sqrt(b.head_dim))[0]
    return out


def oracle_packed(b: W.RaggedBatch) -> np.ndarray:
    return np.concatenate([oracle_rows(b, s) for s in range(b.num_seqs)])


def assert_tolerance(got: np.ndarray, exp: np.ndarray, max_abs=MAX_ABS, mean_abs=MEAN_ABS) -> dict:
    assert got.shape == exp.shape
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - exp)
    stats = {"max_abs": float(err.max()), "mean_abs": float(err.mean())}
    assert stats["max_abs"] <= max_abs, stats
    assert stats["mean_abs"] <= mean_abs, stats
    return stats
