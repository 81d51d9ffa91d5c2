"""Plain fp64 attention, one sequence at a time (oracle; test infrastructure only).

Definition restated from the Hugging Face blog "Continuous batching from first
principles":

* section *Attention*: scores Q K^T, a boolean mask applied to them, a row-wise
  softmax, then a product with V; Q may have n_Q rows and K, V n_K rows;
* section *Chunked prefill*: a chunk's queries see the stored keys/values of
  the earlier tokens of the same prompt plus the chunk's own keys, causally;
* section *Continuous batching* ("ragged batching"): sequences are concatenated
  and tokens of different sequences never interact;

and from the page "continuous-batching" (zhangchitc.github.io), section
"Ragged batching: attention in per-request blocks": a prefilling request's
scores form a lower-triangular block, a decoding request with c keys (cache
plus its new token) forms a 1 x c row.

Combined: query row i (0-based) of a sequence whose cache held p tokens before
the step sees keys j = 0 .. p+i, and

    o_i = sum_j exp(z_j - max z) v_j / sum_j exp(z_j - max z),  z_j = scale * q_i . k_j

The pages print scores without a scale; the 1/sqrt(A) scale is an input here.

Grouped-query attention (fewer key/value heads than query heads) is not on the
pages; it is taken as the usual grouping: with H query and H_kv key/value
heads, query head h uses key/value head h // (H / H_kv).
"""
from __future__ import annotations

import numpy as np


def row_key_limits(cu_seqlens_q: np.ndarray, context_lens: np.ndarray) -> np.ndarray:
    """Number of keys each packed query row may see.

    Sequence s owns packed rows cu[s] .. cu[s+1]-1 and has context_lens[s] keys
    after this step's append; its cached length before the step is
    p = context_lens[s] - q_len, and its row i sees p + i + 1 keys.
    """
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    ctx = np.asarray(context_lens, dtype=np.int64)
    out = np.empty(int(cu[-1]), dtype=np.int64)
    for s in range(len(ctx)):
        n = int(cu[s + 1] - cu[s])
        p = int(ctx[s]) - n
        if n < 1 or p < 0:
            raise ValueError(f"sequence {s}: q_len={n}, context_len={int(ctx[s])}")
        out[cu[s]:cu[s + 1]] = p + 1 + np.arange(n)
    return out


def attend_sequence(q: np.ndarray, k: np.ndarray, v: np.ndarray, p: int, scale: float,
                    rows_per_pass: int = 256) -> np.ndarray:
    """Attention of one sequence's new queries over its keys/values.

    q: [n, H, A] this step's queries; k, v: [p + n, H_kv, A] the whole history
    in token order (cache then new tokens), H a multiple of H_kv (query head h
    reads key/value head h // (H / H_kv)).  Returns [n, H, A] fp64.  Each row's
    softmax is taken over its full set of visible keys at once; ``rows_per_pass``
    only bounds memory.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, H, A = q.shape
    c, H_kv = k.shape[0], k.shape[1]
    if c != p + n or v.shape[0] != c:
        raise ValueError("history length must equal p + q_len")
    if H_kv < 1 or H % H_kv != 0 or v.shape[1] != H_kv:
        raise ValueError("query heads must be a multiple of key/value heads")
    group = H // H_kv
    out = np.empty((n, H, A), dtype=np.float64)
    key_idx = np.arange(c)
    for h in range(H):
        kh = k[:, h // group, :]
        vh = v[:, h // group, :]
        for r0 in range(0, n, rows_per_pass):
            r1 = min(n, r0 + rows_per_pass)
            z = scale * (q[r0:r1, h, :] @ kh.T)                       # [rows, c]
            visible = key_idx[None, :] <= (p + np.arange(r0, r1))[:, None]
            z = np.where(visible, z, -np.inf)
            m = z.max(axis=1, keepdims=True)
            w = np.exp(z - m)                                         # exp(-inf) = 0
            out[r0:r1, h, :] = (w @ vh) / w.sum(axis=1, keepdims=True)
    return out


def attend_left_padded(q: np.ndarray, k: np.ndarray, v: np.ndarray, p: int, pad: int,
                       scale: float) -> np.ndarray:
    """Attention of one left-padded chunk, the padded batching that ragged
    batching replaces (Hugging Face blog "Continuous batching from first
    principles", section "Continuous batching": sequences padded on the left
    to a common length, an attention mask keeping the pads out).

    q: [n, H, A] the chunk's rows, its `pad` pad rows first; k, v: [p + n,
    H_kv, A] the history, with the pad tokens' keys and values at positions
    p .. p + pad - 1.  Real row i (pad <= i < n) attends the keys j <= p + i
    that are not pads: j < p or j >= p + pad.  Pad rows have no output and
    come back as NaN.  Returns [n, H, A] fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, H, A = q.shape
    c, H_kv = k.shape[0], k.shape[1]
    if c != p + n or v.shape[0] != c:
        raise ValueError("history length must equal p + q_len")
    if not 0 <= pad < n:
        raise ValueError("need 0 <= pad < q_len")
    group = H // H_kv
    out = np.full((n, H, A), np.nan)
    j = np.arange(c)
    rows = np.arange(pad, n)
    visible = (j[None, :] <= (p + rows)[:, None]) & ((j[None, :] < p) | (j[None, :] >= p + pad))
    for h in range(H):
        z = scale * (q[pad:, h, :] @ k[:, h // group, :].T)
        z = np.where(visible, z, -np.inf)
        m = z.max(axis=1, keepdims=True)
        w = np.exp(z - m)
        out[pad:, h, :] = (w @ v[:, h // group, :]) / w.sum(axis=1, keepdims=True)
    return out


def ragged_attention(q_packed: np.ndarray, cu_seqlens_q: np.ndarray, context_lens: np.ndarray,
                     k_hist, v_hist, scale: float) -> np.ndarray:
    """Attention over a packed batch, each sequence computed alone and unpacked.

    q_packed: [T, H, A]; k_hist[s], v_hist[s]: [context_lens[s], H_kv, A], the
    sequence's full history (the oracle's own record, never a device cache).
    Returns [T, H, A] fp64 in packed order.
    """
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    ctx = np.asarray(context_lens, dtype=np.int64)
    row_key_limits(cu, ctx)          # validates the metadata
    out = np.empty(q_packed.shape, dtype=np.float64)
    for s in range(len(ctx)):
        a, b = int(cu[s]), int(cu[s + 1])
        p = int(ctx[s]) - (b - a)
        out[a:b] = attend_sequence(q_packed[a:b], k_hist[s], v_hist[s], p, scale)
    return out
