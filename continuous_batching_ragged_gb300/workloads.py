"""Seeded synthetic inputs for the ragged attention step.

This module is the only code shared by the CUDA path's tests/bench and the
CPU oracle's tests.  It draws numbers and lays out batches; it contains none
of the method's arithmetic (no attention, no softmax, no scheduling rule).

Values
------
Every Q/K/V element is a pure function of

    (seed, kind, layer, seq_id, position, head, dim)        kind: 0=Q 1=K 2=V

so a token's key/value is the same whether it is produced by this step's
projection or read back from the cache, and whether its sequence is packed
with others or run alone.  The function is

  1. Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
     easy as 1, 2, 3", SC'11) on counter
         (head*A + dim, position, seq_id, (kind << 16) | layer)
     with key (seed mod 2^32, seed >> 32 mod 2^32);
  2. the four 32-bit outputs split into eight 16-bit uniforms u_k;
  3. an Irwin-Hall(8) standard normal approximation, computed exactly:
         S2 = 2*sum(u_k) - 8*65535           (|S2| < 2^24, exact in fp32)
         x  = fp32(S2) * fp32(sqrt(1.5) / 131072)   (one RNE multiply)
     which has mean 0 and variance 1 (to 1 part in 2^32);
  4. for bf16 workloads, x rounded to bf16 with round-to-nearest-even.

Each step is exact IEEE arithmetic, so the CUDA generator in
``csrc/synth.cu`` (an independent implementation of the same definition)
produces bit-identical values; that is what lets the oracle recompute any
sampled row of a workload that only ever existed in GPU memory.

Batches
-------
``RaggedBatch`` describes one packed step: per sequence its cached length p
(tokens already in the cache), its query length q_len and its block table.
Derived arrays (cu_seqlens_q, context_lens, slot_mapping) follow the page
"continuous-batching" (zhangchitc.github.io), section "Inside the kernel:
cu_seqlens splits six rows back into three": an exclusive prefix sum of the
per-request token counts, and a per-token cache slot block_id*B + offset.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

KIND_Q, KIND_K, KIND_V = 0, 1, 2

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

# fp32(sqrt(1.5) / 131072); the CUDA side spells the same float as a hex literal.
IH8_SCALE = np.float32(math.sqrt(1.5) / 131072.0)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32 with 10 rounds (Salmon et al., SC'11, section 4).

    Counters are uint32 arrays (broadcast together); the key is two 32-bit ints.
    Returns four uint32 arrays.
    """
    c0 = np.asarray(c0, dtype=np.uint32)
    c1 = np.asarray(c1, dtype=np.uint32)
    c2 = np.asarray(c2, dtype=np.uint32)
    c3 = np.asarray(c3, dtype=np.uint32)
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 &= 0xFFFFFFFF
    k1 &= 0xFFFFFFFF
    for _ in range(10):
        p0 = _M0 * c0.astype(np.uint64)
        p1 = _M1 * c2.astype(np.uint64)
        hi0 = (p0 >> np.uint64(32)).astype(np.uint32)
        lo0 = (p0 & _MASK32).astype(np.uint32)
        hi1 = (p1 >> np.uint64(32)).astype(np.uint32)
        lo1 = (p1 & _MASK32).astype(np.uint32)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint32(k0), lo1,
                          hi0 ^ c3 ^ np.uint32(k1), lo0)
        k0 = (k0 + _W0) & 0xFFFFFFFF
        k1 = (k1 + _W1) & 0xFFFFFFFF
    return c0, c1, c2, c3


def irwin_hall8(w0, w1, w2, w3) -> np.ndarray:
    """Map four uint32 words to one approximately N(0,1) fp32 value (exact)."""
    s = np.zeros(np.shape(w0), dtype=np.int64)
    for w in (w0, w1, w2, w3):
        w = w.astype(np.int64)
        s += (w & 0xFFFF) + (w >> 16)
    s2 = 2 * s - 8 * 65535
    return s2.astype(np.float32) * IH8_SCALE


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest bf16 (ties to even); returned as fp32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = (r << np.uint64(16)).astype(np.uint32)
    return out.view(np.float32).reshape(np.shape(x))


_VALUES_LIB = None        # ctypes handle of libcb_values.so, False once it failed to build or load


def _values_lib():
    """The compiled host generator (hostgen/token_values.c), built on first use;
    None where no C compiler is available (token_values then runs in numpy)."""
    global _VALUES_LIB
    if _VALUES_LIB is None:
        try:
            import ctypes
            from . import build as _build
            lib = ctypes.CDLL(_build.build_values_lib())
            f = lib.cbv_token_values
            f.restype = None
            f.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                          ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32,
                          ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
            _VALUES_LIB = lib
        except Exception:          # no compiler or loader: fall back to numpy
            _VALUES_LIB = False
    return _VALUES_LIB or None


def _token_values_c(lib, seed, kind, layer, seq_id, positions, heads, head_dim, dtype):
    """token_values through libcb_values.so, positions split over host threads
    (ctypes releases the GIL for the call)."""
    import concurrent.futures
    import os
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64).reshape(-1).astype(np.uint32))
    hd = np.ascontiguousarray(np.asarray(list(heads), dtype=np.uint32))
    out = np.empty((len(pos), len(hd), head_dim), dtype=np.float32)
    if len(pos) == 0 or len(hd) == 0:
        return out
    per_pos = len(hd) * head_dim
    nthreads = max(1, min(len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 1,
                          (len(pos) * per_pos) // (1 << 16) + 1))
    bounds = np.linspace(0, len(pos), nthreads + 1).astype(np.int64)
    bf16 = 1 if dtype == "bf16" else 0

    def run(i):
        a, b = int(bounds[i]), int(bounds[i + 1])
        if b > a:
            lib.cbv_token_values(seed & 0xFFFFFFFFFFFFFFFF, kind & 0xFFFFFFFF, layer & 0xFFFFFFFF,
                                 seq_id & 0xFFFFFFFF, pos[a:].ctypes.data, b - a, hd.ctypes.data, len(hd),
                                 head_dim, bf16, out[a:].ctypes.data)

    if nthreads == 1:
        run(0)
    else:
        with concurrent.futures.ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(run, range(nthreads)))
    return out


def token_values(seed: int, kind: int, layer: int, seq_id: int,
                 positions: np.ndarray, heads: Sequence[int], head_dim: int,
                 dtype: str) -> np.ndarray:
    """Values of ``kind`` for one sequence: array [len(positions), len(heads), A].
    Runs the compiled host generator when it is available, else numpy; the two
    are pinned bit for bit to each other."""
    if dtype not in ("bf16", "f32"):
        raise ValueError(dtype)
    lib = _values_lib()
    if lib is not None:
        return _token_values_c(lib, seed, kind, layer, seq_id, positions, heads, head_dim, dtype)
    return token_values_numpy(seed, kind, layer, seq_id, positions, heads, head_dim, dtype)


def token_values_numpy(seed: int, kind: int, layer: int, seq_id: int,
                       positions: np.ndarray, heads: Sequence[int], head_dim: int,
                       dtype: str) -> np.ndarray:
    """token_values written out in numpy (the definition above, step by step)."""
    positions = np.asarray(positions, dtype=np.uint32).reshape(-1, 1, 1)
    heads = np.asarray(heads, dtype=np.uint32).reshape(1, -1, 1)
    dims = np.arange(head_dim, dtype=np.uint32).reshape(1, 1, -1)
    c0 = heads * np.uint32(head_dim) + dims
    c2 = np.uint32(seq_id)
    c3 = np.uint32(((kind & 0xFFFF) << 16) | (layer & 0xFFFF))
    w = philox4x32_10(c0, positions, c2, c3, seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    x = irwin_hall8(*w)
    if dtype == "bf16":
        x = round_to_bf16(x)
    elif dtype != "f32":
        raise ValueError(dtype)
    return x


# ---------------------------------------------------------------------------
# Batch descriptions
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class RaggedBatch:
    """One packed step.  Sequence s has p[s] cached tokens and q_len[s] new ones."""
    num_heads: int
    head_dim: int
    block_size: int
    dtype: str                      # "bf16" or "f32"
    seed: int
    layer: int
    seq_ids: np.ndarray             # [S] int64, identity for the value generator
    p: np.ndarray                   # [S] int64, cached length before the step
    q_len: np.ndarray               # [S] int64, >= 1
    block_tables: np.ndarray        # [S, max_blocks] int32, -1 padded
    num_blocks: int                 # pool size in blocks
    name: str = ""
    useful_tokens: Optional[int] = None   # of a padded batch: the real query tokens
    num_kv_heads: Optional[int] = None    # key/value heads (grouped-query attention); None = num_heads
    # (q_shift, k_slope): shaped inputs whose scores rise along the sequence.
    # Every query gets q_shift * u added and the key at position j gets
    # k_slope * j * u, u = (1, ..., 1) / sqrt(A), then the sum is rounded to the
    # dtype; so scale * q . k grows by about scale * q_shift * k_slope per key
    # and a row's running maximum keeps climbing as keys stream in.  Values of
    # such a batch exist only on the host (the device generator does not
    # shape them).
    drift: Optional[Tuple[float, float]] = None
    # Left padding (a padded batch, see left_padded): the first pad_lens[s]
    # new tokens of sequence s are pad tokens.  They occupy cache positions
    # p .. p + pad - 1 and take their values from generator positions
    # PAD_POSITION_BASE + i; the real tokens after them keep the values of
    # their unpadded positions, so real rows see exactly the unpadded data.
    pad_lens: Optional[np.ndarray] = None

    @property
    def kv_heads(self) -> int:
        return self.num_kv_heads if self.num_kv_heads else self.num_heads

    def heads_of(self, kind: int) -> int:
        return self.num_heads if kind == KIND_Q else self.kv_heads

    @property
    def num_seqs(self) -> int:
        return int(len(self.p))

    @property
    def context_lens(self) -> np.ndarray:
        return (self.p + self.q_len).astype(np.int32)

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        cu = np.zeros(self.num_seqs + 1, dtype=np.int32)
        cu[1:] = np.cumsum(self.q_len)
        return cu

    @property
    def T(self) -> int:
        return int(np.sum(self.q_len))

    @property
    def max_q_len(self) -> int:
        return int(self.q_len.max()) if self.num_seqs else 0

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def slot_mapping(self) -> np.ndarray:
        out = np.empty(self.T, dtype=np.int64)
        cu = self.cu_seqlens_q
        B = self.block_size
        for s in range(self.num_seqs):
            pos = np.arange(self.p[s], self.p[s] + self.q_len[s])
            out[cu[s]:cu[s + 1]] = self.block_tables[s, pos // B].astype(np.int64) * B + pos % B
        return out

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    # -- values ------------------------------------------------------------
    def gen_positions(self, s: int, positions) -> np.ndarray:
        """Generator positions of sequence s's cache positions (the identity
        unless the batch is left-padded)."""
        x = np.asarray(positions, dtype=np.int64)
        if self.pad_lens is None or int(self.pad_lens[s]) == 0:
            return x
        p, pad = int(self.p[s]), int(self.pad_lens[s])
        return np.where(x < p, x, np.where(x < p + pad, PAD_POSITION_BASE + (x - p), x - pad))

    def values(self, kind: int, s: int, positions, heads) -> np.ndarray:
        """Values of ``kind`` for sequence s at cache ``positions`` and ``heads``:
        [len(positions), len(heads), A], fp32 holding dtype values."""
        positions = self.gen_positions(s, positions)
        x = token_values(self.seed, kind, self.layer, int(self.seq_ids[s]), positions, heads,
                         self.head_dim, self.dtype)
        if self.drift is None or kind == KIND_V:
            return x
        q_shift, k_slope = self.drift
        u = np.full(self.head_dim, 1.0 / math.sqrt(self.head_dim), dtype=np.float32)
        if kind == KIND_Q:
            add = np.float32(q_shift) * u
        else:
            pos = np.asarray(positions, dtype=np.float32).reshape(-1, 1, 1)
            add = (np.float32(k_slope) * pos) * u
        y = (x + add).astype(np.float32)
        return round_to_bf16(y) if self.dtype == "bf16" else y

    def packed(self, kind: int) -> np.ndarray:
        """This step's tokens of ``kind`` packed as [T, heads, A] (fp32 holding dtype
        values); queries have num_heads heads, keys and values kv_heads."""
        nh = self.heads_of(kind)
        out = np.empty((self.T, nh, self.head_dim), dtype=np.float32)
        cu = self.cu_seqlens_q
        heads = range(nh)
        for s in range(self.num_seqs):
            pos = np.arange(self.p[s], self.p[s] + self.q_len[s])
            out[cu[s]:cu[s + 1]] = self.values(kind, s, pos, heads)
        return out

    def history(self, s: int, kind: int, heads: Optional[Sequence[int]] = None,
                upto: Optional[int] = None) -> np.ndarray:
        """Sequence s's keys or values for positions [0, upto) (default: context_len)."""
        if heads is None:
            heads = range(self.heads_of(kind))
        n = int(self.context_lens[s]) if upto is None else int(upto)
        return self.values(kind, s, np.arange(n), heads)

    def prefilled_pool(self, kind: int, sentinel: float = float("nan")) -> np.ndarray:
        """Host pool [num_blocks, H, B, A] holding every sequence's cached prefix
        (positions < p) at its block-table slots; every other slot holds ``sentinel``."""
        B = self.block_size
        pool = np.full((self.num_blocks, self.kv_heads, B, self.head_dim), sentinel, dtype=np.float32)
        for s in range(self.num_seqs):
            ps = int(self.p[s])
            if ps == 0:
                continue
            vals = self.history(s, kind, upto=ps)                  # [p, H, A]
            pos = np.arange(ps)
            blk = self.block_tables[s, pos // B]
            pool[blk, :, pos % B, :] = vals
        return pool


def _assign_blocks(rng: np.random.Generator, ctx: np.ndarray, block_size: int,
                   num_blocks: Optional[int] = None, permute: bool = True
                   ) -> Tuple[np.ndarray, int]:
    """Give each sequence ceil(ctx/B) distinct physical blocks from a pool."""
    need = [int(math.ceil(int(c) / block_size)) for c in ctx]
    total = sum(need)
    if num_blocks is None:
        num_blocks = total
    if num_blocks < total:
        raise ValueError("pool too small")
    ids = rng.permutation(num_blocks) if permute else np.arange(num_blocks)
    maxb = max(need) if need else 1
    bt = np.full((len(ctx), max(maxb, 1)), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(need):
        bt[s, :n] = ids[off:off + n]
        off += n
    return bt, num_blocks


def make_batch(p: Sequence[int], q_len: Sequence[int], *, num_heads: int, head_dim: int,
               block_size: int, dtype: str, seed: int, layer: int = 0,
               num_blocks: Optional[int] = None, permute: bool = True,
               seq_ids: Optional[Sequence[int]] = None, name: str = "",
               num_kv_heads: Optional[int] = None,
               drift: Optional[Tuple[float, float]] = None) -> RaggedBatch:
    p = np.asarray(p, dtype=np.int64)
    q_len = np.asarray(q_len, dtype=np.int64)
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    bt, nb = _assign_blocks(rng, p + q_len, block_size, num_blocks, permute)
    if seq_ids is None:
        seq_ids = np.arange(len(p), dtype=np.int64)
    return RaggedBatch(num_heads=num_heads, head_dim=head_dim, block_size=block_size,
                       dtype=dtype, seed=seed, layer=layer,
                       seq_ids=np.asarray(seq_ids, dtype=np.int64), p=p, q_len=q_len,
                       block_tables=bt, num_blocks=nb, name=name, num_kv_heads=num_kv_heads,
                       drift=drift)


PAD_POSITION_BASE = 1 << 30      # generator positions of pad tokens (no real token sits there)


def left_padded(b: RaggedBatch) -> RaggedBatch:
    """The same sequences as one rectangular, left-padded batch (Hugging Face
    blog "Continuous batching from first principles", section "Continuous
    batching": without ragged batching, sequences are padded on the left to a
    common length and masked; inserting an n-token prompt into B decoding
    prompts costs (n-1)(B-1) padding tokens).  Every sequence carries
    n = max(q_len) new tokens, pad_lens = n - q_len of them pads first; the
    pads are appended to the cache like real tokens and masked out of
    attention by cb_padded_attention, so a step computes B * n query rows
    over the pads' keys too, while each real row's result is that of the
    ragged batch."""
    n = int(b.q_len.max())
    pb = make_batch(b.p, np.full(b.num_seqs, n, np.int64), num_heads=b.num_heads, head_dim=b.head_dim,
                    block_size=b.block_size, dtype=b.dtype, seed=b.seed, layer=b.layer,
                    seq_ids=b.seq_ids, name=b.name + "_padded", num_kv_heads=b.num_kv_heads)
    pb.pad_lens = (n - b.q_len).astype(np.int32)
    pb.useful_tokens = b.T
    return pb


def real_rows(pb: RaggedBatch) -> np.ndarray:
    """Packed row indices of a left-padded batch's real (non-pad) rows, in
    packed order of the unpadded batch."""
    cu = pb.cu_seqlens_q
    return np.concatenate([np.arange(cu[s] + int(pb.pad_lens[s]), cu[s + 1]) for s in range(pb.num_seqs)])


def padding_tokens(b: RaggedBatch) -> int:
    """Query rows the padded equivalent adds over the ragged batch."""
    return int(b.num_seqs * b.q_len.max() - b.q_len.sum())


def page_insertion_example(seed: int = 5, batch: int = 8, n: int = 100, cached: int = 512,
                           num_heads: int = 32, head_dim: int = 128, block_size: int = 16) -> RaggedBatch:
    """B-1 prompts decoding one token each (``cached`` tokens in the cache) plus
    one newly inserted prompt of n tokens, the blog's B=8, n=100 example."""
    p = [cached] * (batch - 1) + [0]
    q = [1] * (batch - 1) + [n]
    return make_batch(p, q, num_heads=num_heads, head_dim=head_dim, block_size=block_size,
                      dtype="bf16", seed=seed, name="insertion")


# ---------------------------------------------------------------------------
# The five workloads (Llama-2-7B attention shape: 32 heads x 128, MHA)
# ---------------------------------------------------------------------------

def tiny_fp32(seed: int = 0) -> RaggedBatch:
    """3 sequences, T=6: a fresh 4-token prefill and two decodes with 7 and 12
    cached tokens; fp32, H=4, A=64, block size 4, pool of 8 permuted blocks."""
    return make_batch([0, 7, 12], [4, 1, 1], num_heads=4, head_dim=64, block_size=4,
                      dtype="f32", seed=seed, num_blocks=8, name="tiny_fp32")


def decode_step(seed: int = 1, num_seqs: int = 256, ctx_lo: int = 512, ctx_hi: int = 4096,
                num_heads: int = 32, head_dim: int = 128, block_size: int = 16,
                num_kv_heads: Optional[int] = None) -> RaggedBatch:
    """Decode-only step: every sequence has p ~ U{ctx_lo..ctx_hi} cached tokens and
    one query; blocks drawn from a randomly permuted pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    p = rng.integers(ctx_lo, ctx_hi, size=num_seqs, endpoint=True)
    return make_batch(p, np.ones(num_seqs, np.int64), num_heads=num_heads, head_dim=head_dim,
                      block_size=block_size, dtype="bf16", seed=seed, name="decode",
                      num_kv_heads=num_kv_heads)


def mixed_step(seed: int = 2, num_decode: int = 64, ctx_lo: int = 256, ctx_hi: int = 4096,
               chunks: Sequence[int] = (661, 661, 662), chunk_p: Sequence[int] = (0, 1024, 2048),
               num_heads: int = 32, head_dim: int = 128, block_size: int = 16,
               num_kv_heads: Optional[int] = None) -> RaggedBatch:
    """Mixed step, token budget 2048: decode tokens first, then prefill chunks."""
    rng = np.random.Generator(np.random.PCG64(seed))
    pd = rng.integers(ctx_lo, ctx_hi, size=num_decode, endpoint=True)
    p = np.concatenate([pd, np.asarray(chunk_p, np.int64)])
    q = np.concatenate([np.ones(num_decode, np.int64), np.asarray(chunks, np.int64)])
    return make_batch(p, q, num_heads=num_heads, head_dim=head_dim, block_size=block_size,
                      dtype="bf16", seed=seed, name="mixed", num_kv_heads=num_kv_heads)


def long_prompt_chunk(k: int, seed: int = 3, prompt: int = 32768, chunk: int = 2048,
                      num_heads: int = 32, head_dim: int = 128, block_size: int = 16,
                      single_pass: bool = False) -> RaggedBatch:
    """Chunk k (0-based) of a ``prompt``-token prompt processed ``chunk`` tokens at a
    time; with single_pass the whole prompt is one chunk.  All chunks of one prompt
    share one block table (sequence id 0, blocks 0..prompt/B-1 permuted by seed)."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    nb = int(math.ceil(prompt / block_size))
    ids = rng.permutation(nb).astype(np.int32)
    if single_pass:
        p, q = 0, prompt
    else:
        p, q = k * chunk, chunk
    nblk = int(math.ceil((p + q) / block_size))
    bt = ids[:nblk].reshape(1, -1).copy()
    return RaggedBatch(num_heads=num_heads, head_dim=head_dim, block_size=block_size,
                       dtype="bf16", seed=seed, layer=0, seq_ids=np.zeros(1, np.int64),
                       p=np.asarray([p], np.int64), q_len=np.asarray([q], np.int64),
                       block_tables=bt, num_blocks=nb, name="long_prompt")


@dataclasses.dataclass
class Request:
    id: int
    arrival_step: int
    prompt_len: int
    output_len: int


def serving_trace(seed: int = 4, num_requests: int = 2000, rate: float = 4.0,
                  prompt_median: float = 512.0, prompt_sigma: float = 1.0, prompt_cap: int = 8192,
                  out_median: float = 120.0, out_sigma: float = 0.8,
                  out_min: int = 20, out_max: int = 800) -> List[Request]:
    """Poisson arrivals (rate per scheduler step) with lognormal prompt and output
    lengths; output length is fixed at admission and stands in for <eos>."""
    rng = np.random.Generator(np.random.PCG64(seed))
    gaps = rng.exponential(1.0 / rate, size=num_requests)
    arrival = np.floor(np.cumsum(gaps)).astype(np.int64)
    prompt = np.rint(rng.lognormal(math.log(prompt_median), prompt_sigma, size=num_requests))
    prompt = np.clip(prompt, 1, prompt_cap).astype(np.int64)
    out = np.rint(rng.lognormal(math.log(out_median), out_sigma, size=num_requests))
    out = np.clip(out, out_min, out_max).astype(np.int64)
    return [Request(i, int(arrival[i]), int(prompt[i]), int(out[i])) for i in range(num_requests)]


SERVING_TRACE = dict(num_layers=32, num_heads=32, head_dim=128, block_size=16,
                     token_budget=4096, num_blocks=10240)
